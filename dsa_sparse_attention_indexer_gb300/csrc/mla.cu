// Sparse MLA entry points ("vLLM 推理链路概览", Sparse MLA Attention;
// "GLM-5.3 推理全链路(一)", decode: MQA 形态与吸收): argument checks, the
// workspace contract and the launch of the tensor-core kernel in mla_tc.cu.
// Decode and prefill share one kernel: a query row is a row whatever its
// request's q_len, and causality is the per-row limit j <= p.
#include "dsa_internal.cuh"
#include "indexer_common.cuh"

namespace dsa {

int device_sm_count() {
    int dev = 0, sms = 148;
    if (cudaGetDevice(&dev) == cudaSuccess) cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    return sms > 1024 ? 1024 : sms;
}

int mla_tc_ctas(int64_t total_q, int sms);
size_t mla_tc_ws_bytes(int64_t total_q, int G);
dsa_status launch_sparse_mla_tc(const void* q, const int32_t* topk, const uint8_t* kv, const dsa_batch* b,
                                float softmax_scale, void* out, int32_t out_dtype, float* lse, void* ws,
                                int G, int32_t* st, cudaStream_t s);

dsa_status sparse_mla_launch(const void* q, const int32_t* topk, const dsa_topk_share* share,
                             const uint8_t* kv, const dsa_batch* b, float softmax_scale, void* out,
                             int32_t out_dtype, float* lse, void* ws, size_t ws_bytes, int32_t* st,
                             void* stream, bool decode);

}  // namespace dsa

using namespace dsa;

extern "C" dsa_status dsa_topk_share_get(const dsa_topk_share* s, const int32_t** topk, int64_t* rows,
                                         int32_t* layer_id);

dsa_status dsa::sparse_mla_launch(const void* q, const int32_t* topk, const dsa_topk_share* share,
                                  const uint8_t* kv, const dsa_batch* b, float softmax_scale, void* out,
                                  int32_t out_dtype, float* lse, void* ws, size_t ws_bytes, int32_t* st,
                                  void* stream, bool decode) {
    dsa_status vs = validate_batch(b);
    if (vs != DSA_OK) return vs;
    if (out_dtype != DSA_DTYPE_BF16 && out_dtype != DSA_DTYPE_F32) return DSA_ERR_INVALID_ARGUMENT;
    if (!(softmax_scale > 0.f)) return DSA_ERR_INVALID_ARGUMENT;
    if (!topk) {
        if (!share) return DSA_ERR_INVALID_ARGUMENT;
        int64_t rows = 0;
        dsa_status gs = dsa_topk_share_get(share, &topk, &rows, nullptr);
        if (gs != DSA_OK) return gs;
        if (rows != b->total_q) return DSA_ERR_INVALID_ARGUMENT;
    }
    if (b->total_q == 0) return DSA_OK;                                  // no rows
    if (!q || !kv || !out || !topk) return DSA_ERR_INVALID_ARGUMENT;
    if (!aligned16(q) || !aligned16(kv) || !aligned16(out) || !aligned16(topk)) return DSA_ERR_ALIGNMENT;
    (void)decode;
    const int G = mla_tc_ctas(b->total_q, device_sm_count());
    if (!ws) return DSA_ERR_INVALID_ARGUMENT;
    if (ws_bytes < mla_tc_ws_bytes(b->total_q, G)) return DSA_ERR_WORKSPACE_TOO_SMALL;
    if (!aligned16(ws)) return DSA_ERR_ALIGNMENT;
    if (b->total_q > 0x3fffffffLL / 2048) return DSA_ERR_UNSUPPORTED;
    if (b->num_pages * DSA_PAGE_TOKENS > 0x7fffffffLL) return DSA_ERR_UNSUPPORTED;   // int32 cache slots
    return launch_sparse_mla_tc(q, topk, kv, b, softmax_scale, out, out_dtype, lse, ws, G, st, as_stream(stream));
}

extern "C" dsa_status dsa_sparse_mla_workspace_size(const dsa_batch* b, size_t* bytes) {
    dsa_status vs = validate_batch(b);
    if (vs != DSA_OK) return vs;
    if (!bytes) return DSA_ERR_INVALID_ARGUMENT;
    // Enough for any GPU of up to 1024 SMs.
    *bytes = mla_tc_ws_bytes(b->total_q, mla_tc_ctas(b->total_q, 1024));
    return DSA_OK;
}

extern "C" dsa_status dsa_sparse_mla_decode(const void* q, const int32_t* topk, const dsa_topk_share* share,
                                            const uint8_t* kv_cache, const dsa_batch* b, float softmax_scale,
                                            void* out, int32_t out_dtype, float* lse, void* ws,
                                            size_t ws_bytes, int32_t* dev_status, void* stream) {
    return sparse_mla_launch(q, topk, share, kv_cache, b, softmax_scale, out, out_dtype, lse, ws, ws_bytes,
                             dev_status, stream, true);
}

extern "C" dsa_status dsa_sparse_mla_prefill(const void* q, const int32_t* topk, const dsa_topk_share* share,
                                             const uint8_t* kv_cache, const dsa_batch* b, float softmax_scale,
                                             void* out, int32_t out_dtype, float* lse, void* ws,
                                             size_t ws_bytes, int32_t* dev_status, void* stream) {
    return sparse_mla_launch(q, topk, share, kv_cache, b, softmax_scale, out, out_dtype, lse, ws, ws_bytes,
                             dev_status, stream, false);
}
