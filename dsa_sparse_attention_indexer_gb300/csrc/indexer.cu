// dsa_indexer_topk: index-Q quantisation -> indexer scores -> top-2048 per
// query row ("vLLM 推理链路概览", DSA Indexer; "GLM-5.3 推理全链路(十一)",
// 优化二 for the short-context rule).
#include "dsa_internal.cuh"
#include "indexer_common.cuh"
#include "topk_common.cuh"
#include "indexer_tc.cuh"

namespace dsa {

// One CTA per query row: select over the row's p + 1 visible scores.
__global__ void __launch_bounds__(kSelThreads)
indexer_select_kernel(const float* __restrict__ scores, int64_t ld, BatchDev b,
                      int32_t* __restrict__ topk, float* __restrict__ topk_scores) {
    extern __shared__ __align__(16) uint8_t sel_smem[];
    const int64_t row = blockIdx.x;
    const int r = row_request(b.q_start, b.batch, row);
    const int qn = b.q_start[r + 1] - b.q_start[r];
    const int64_t t = row - b.q_start[r];
    int64_t n = (int64_t)b.seq_len[r] - qn + t + 1;            // positions 0..p
    if (n > ld) n = ld;                                          // seq_len beyond the declared bound
    select_topk_row(scores + row * ld, n, topk + row * kTopK, topk_scores ? topk_scores + row * kTopK : nullptr,
                    sel_smem);
}

inline int64_t score_ld(const dsa_batch* b) { return ((int64_t)b->max_seq_len + 3) / 4 * 4; }

// Decode batches (one query row per request) take the fused tensor-core path;
// other batches score into full rows and select from them.
inline bool use_tc_path(const dsa_batch* b) { return b->max_q_len == 1 && b->total_q == b->batch; }

inline size_t indexer_ws_bytes(const dsa_batch* b) {
    const size_t qbytes = (q8_workspace_bytes(b->total_q) + 255) / 256 * 256;
    if (use_tc_path(b))   // row histograms + plan, for any GPU of up to 1024 SMs
        return qbytes + (size_t)b->total_q * 4096 * 4 + tc_plan_bytes(b->batch, 1024);
    const size_t sbytes = ((size_t)b->total_q * (size_t)score_ld(b) * 4 + 255) / 256 * 256;
    return qbytes + sbytes + mt_plan_bytes(b->batch, b->total_q);
}

}  // namespace dsa

using namespace dsa;

extern "C" dsa_status dsa_topk_share_publish(dsa_topk_share* s, int32_t layer_id, const int32_t* topk,
                                             int64_t rows);

extern "C" dsa_status dsa_indexer_topk_workspace_size(const dsa_batch* b, size_t* bytes) {
    dsa_status vs = validate_batch(b);
    if (vs != DSA_OK) return vs;
    if (!bytes) return DSA_ERR_INVALID_ARGUMENT;
    *bytes = indexer_ws_bytes(b);
    return DSA_OK;
}

// MXFP4 index-K cache, decode batches: the same quantised queries, plan,
// fused score kernel (E2M1 keys, block scales in the epilogue) and merge.
extern "C" dsa_status dsa_indexer_topk_mxfp4(const void* q, const float* w, const uint8_t* idxk_cache,
                                             const dsa_batch* b, int32_t* topk, float* topk_scores,
                                             dsa_topk_share* share, int32_t layer_id, void* ws,
                                             size_t ws_bytes, int32_t* dev_status, void* stream) {
    dsa_status vs = validate_batch(b);
    if (vs != DSA_OK) return vs;
    if (!q || !w || !idxk_cache || !topk) return DSA_ERR_INVALID_ARGUMENT;
    if (!aligned16(q) || !aligned16(topk) || (reinterpret_cast<uintptr_t>(idxk_cache) & 31)) return DSA_ERR_ALIGNMENT;
    if (b->total_q > 0) {
        if (!use_tc_path(b)) return DSA_ERR_UNSUPPORTED;            // decode batches only
        if (b->num_pages * 68 > 0x7fffffffLL) return DSA_ERR_UNSUPPORTED;
        if (!ws) return DSA_ERR_INVALID_ARGUMENT;
        if (!aligned16(ws)) return DSA_ERR_ALIGNMENT;
        if (ws_bytes < indexer_ws_bytes(b)) return DSA_ERR_WORKSPACE_TOO_SMALL;
        cudaStream_t s = as_stream(stream);
        uint8_t* q8 = static_cast<uint8_t*>(ws);
        float* wq = reinterpret_cast<float*>(q8 + (size_t)b->total_q * 4096);
        uint32_t* hist = reinterpret_cast<uint32_t*>(q8 + (q8_workspace_bytes(b->total_q) + 255) / 256 * 256);
        void* plan = reinterpret_cast<uint8_t*>(hist) + (size_t)b->total_q * 4096 * 4;
        dsa_status rs = launch_indexer_tc(q, w, q8, wq, hist, idxk_cache, b, topk, topk_scores, plan,
                                          device_sm_count(), dev_status, s, true);
        if (rs != DSA_OK) return rs;
    }
    if (share) return dsa_topk_share_publish(share, layer_id, topk, b->total_q);
    return DSA_OK;
}

extern "C" dsa_status dsa_indexer_topk(const void* q, const float* w, const uint8_t* idxk_cache,
                                       const dsa_batch* b, int32_t* topk, float* topk_scores,
                                       dsa_topk_share* share, int32_t layer_id, void* ws,
                                       size_t ws_bytes, int32_t* dev_status, void* stream) {
    dsa_status vs = validate_batch(b);
    if (vs != DSA_OK) return vs;
    if (!q || !w || !idxk_cache || !topk) return DSA_ERR_INVALID_ARGUMENT;
    if (!aligned16(q) || !aligned16(idxk_cache) || !aligned16(topk)) return DSA_ERR_ALIGNMENT;
    if (b->total_q > 0) {
        if (!ws) return DSA_ERR_INVALID_ARGUMENT;
        if (!aligned16(ws)) return DSA_ERR_ALIGNMENT;
        if (ws_bytes < indexer_ws_bytes(b)) return DSA_ERR_WORKSPACE_TOO_SMALL;
        cudaStream_t s = as_stream(stream);
        uint8_t* q8 = static_cast<uint8_t*>(ws);
        float* wq = reinterpret_cast<float*>(q8 + (size_t)b->total_q * 4096);
        float* sc = reinterpret_cast<float*>(q8 + (q8_workspace_bytes(b->total_q) + 255) / 256 * 256);
        const int64_t ld = score_ld(b);
        if (b->num_pages * 66 > 0x7fffffffLL) return DSA_ERR_UNSUPPORTED;
        const bool tc = use_tc_path(b);
        if (tc) {
            uint32_t* hist = reinterpret_cast<uint32_t*>(sc);
            const int G = device_sm_count();
            void* plan = reinterpret_cast<uint8_t*>(sc) + (size_t)b->total_q * 4096 * 4;
            dsa_status rs = launch_indexer_tc(q, w, q8, wq, hist, idxk_cache, b, topk, topk_scores, plan, G,
                                              dev_status, s);
            if (rs != DSA_OK) return rs;
            if (share) return dsa_topk_share_publish(share, layer_id, topk, b->total_q);
            return DSA_OK;
        }
        dsa_status rs = launch_index_q_quant(q, w, b->total_q, q8, wq, nullptr, s);
        if (rs != DSA_OK) return rs;
        void* plan = reinterpret_cast<uint8_t*>(sc) + ((size_t)b->total_q * (size_t)ld * 4 + 255) / 256 * 256;
        rs = launch_indexer_rows(q8, wq, idxk_cache, b, sc, ld, true, false, plan, device_sm_count(), dev_status, s);
        if (rs != DSA_OK) return rs;
        BatchDev bd = to_dev(b);
        if (ensure_smem_limit(reinterpret_cast<const void*>(&indexer_select_kernel), kSelSmem) != DSA_OK)
            return DSA_ERR_CUDA;
        indexer_select_kernel<<<(unsigned)b->total_q, kSelThreads, kSelSmem, s>>>(sc, ld, bd, topk, topk_scores);
        DSA_CHECK_LAUNCH();
    }
    if (share) return dsa_topk_share_publish(share, layer_id, topk, b->total_q);
    return DSA_OK;
}
