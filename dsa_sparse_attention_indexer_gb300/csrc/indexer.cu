// dsa_indexer_topk: index-Q quantisation -> indexer scores -> top-2048 per
// query row ("vLLM 推理链路概览", DSA Indexer; "GLM-5.3 推理全链路(十一)",
// 优化二 for the short-context rule).
#include "dsa_internal.cuh"
#include "indexer_common.cuh"
#include "indexer_tc.cuh"

namespace dsa {

// Decode batches (one query row per request) take the fused tensor-core path;
// other batches the multi-row tensor-core path, which streams each row's
// candidates into workspace slots (no score row is written).
inline bool use_tc_path(const dsa_batch* b) { return b->max_q_len == 1 && b->total_q == b->batch; }

inline size_t round256(size_t x) { return (x + 255) / 256 * 256; }

// The fused decode path for T query rows: quantised queries, row histograms and
// its plan, for any GPU of up to 1024 SMs.
inline size_t decode_ws_bytes(int64_t T, int64_t batch) {
    return round256(q8_workspace_bytes(T)) + (size_t)T * 4096 * 4 + tc_plan_bytes(batch, 1024);
}
// MXFP4 cache, several rows per request: every query row becomes a request of
// its own (context = its position + 1, its request's page-table row), built in
// the workspace after the decode path's part.
inline size_t mx_rows_virtual_bytes(const dsa_batch* b) {
    return round256((size_t)(2 * b->total_q + 1) * 4) + round256((size_t)b->total_q * b->max_pages * 4);
}

// Decode batches: the fused path.  Other batches: row histograms + the
// multi-row plan with its candidate slots for the current device's SM count
// (O(T x 6144) candidates, no score rows), or the MXFP4 call's virtual decode
// batch, whichever is larger.
inline size_t indexer_ws_bytes(const dsa_batch* b) {
    if (use_tc_path(b)) return decode_ws_bytes(b->total_q, b->batch);
    const size_t fp8 = round256(q8_workspace_bytes(b->total_q)) + (size_t)b->total_q * 4096 * 4 +
                       mt_topk_bytes(b->batch, b->total_q, device_sm_count());
    const size_t mx = decode_ws_bytes(b->total_q, b->total_q) + mx_rows_virtual_bytes(b);
    return fp8 > mx ? fp8 : mx;
}

// Row i of a multi-row batch as request i of a decode batch.
__global__ void __launch_bounds__(256)
virtual_rows_kernel(BatchDev b, int32_t* __restrict__ seq_v, int32_t* __restrict__ qs_v,
                    int32_t* __restrict__ pt_v) {
    const int64_t row = blockIdx.x;
    const int r = row_request(b.q_start, b.batch, row);
    const int qn = b.q_start[r + 1] - b.q_start[r];
    const int p = b.seq_len[r] - qn + (int)(row - b.q_start[r]);
    if (threadIdx.x == 0) {
        seq_v[row] = p + 1;
        qs_v[row] = (int32_t)row;
        if (row == b.total_q - 1) qs_v[row + 1] = (int32_t)(row + 1);
    }
    const int32_t* src = b.page_table + (int64_t)r * b.max_pages;
    int32_t* dst = pt_v + row * b.max_pages;
    for (int k = threadIdx.x; k < b.max_pages; k += 256) dst[k] = src[k];
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

// MXFP4 index-K cache: the same quantised queries, plan, fused score kernel
// (E2M1 keys, block scales in the epilogue) and merge as the decode path.  A
// batch with several rows per request runs as a virtual decode batch of one
// request per row (each row reads its request's keys up to its position).
extern "C" dsa_status dsa_indexer_topk_mxfp4(const void* q, const float* w, const uint8_t* idxk_cache,
                                             const dsa_batch* b, int32_t* topk, float* topk_scores,
                                             dsa_topk_share* share, int32_t layer_id, void* ws,
                                             size_t ws_bytes, int32_t* dev_status, void* stream) {
    dsa_status vs = validate_batch(b);
    if (vs != DSA_OK) return vs;
    if (b->total_q == 0) return share ? dsa_topk_share_publish(share, layer_id, topk, 0) : DSA_OK;   // no rows
    if (!q || !w || !idxk_cache || !topk) return DSA_ERR_INVALID_ARGUMENT;
    if (!aligned16(q) || !aligned16(topk) || (reinterpret_cast<uintptr_t>(idxk_cache) & 31)) return DSA_ERR_ALIGNMENT;
    if (b->total_q > 0) {
        if (b->num_pages * 68 > 0x7fffffffLL) return DSA_ERR_UNSUPPORTED;
        if (!use_tc_path(b) && b->total_q > 65535) return DSA_ERR_UNSUPPORTED;   // rows as requests
        if (!ws) return DSA_ERR_INVALID_ARGUMENT;
        if (!aligned16(ws)) return DSA_ERR_ALIGNMENT;
        if (ws_bytes < indexer_ws_bytes(b)) return DSA_ERR_WORKSPACE_TOO_SMALL;
        cudaStream_t s = as_stream(stream);
        uint8_t* q8 = static_cast<uint8_t*>(ws);
        float* wq = reinterpret_cast<float*>(q8 + (size_t)b->total_q * 4096);
        uint32_t* hist = reinterpret_cast<uint32_t*>(q8 + round256(q8_workspace_bytes(b->total_q)));
        void* plan = reinterpret_cast<uint8_t*>(hist) + (size_t)b->total_q * 4096 * 4;
        dsa_batch vb = *b;
        if (!use_tc_path(b)) {
            uint8_t* vbase = static_cast<uint8_t*>(ws) + decode_ws_bytes(b->total_q, b->total_q);
            int32_t* seq_v = reinterpret_cast<int32_t*>(vbase);
            int32_t* qs_v = seq_v + b->total_q;
            int32_t* pt_v = reinterpret_cast<int32_t*>(vbase + round256((size_t)(2 * b->total_q + 1) * 4));
            virtual_rows_kernel<<<(unsigned)b->total_q, 256, 0, s>>>(to_dev(b), seq_v, qs_v, pt_v);
            DSA_CHECK_LAUNCH();
            vb.batch = (int32_t)b->total_q;
            vb.max_q_len = 1;
            vb.seq_len = seq_v;
            vb.q_start = qs_v;
            vb.page_table = pt_v;
        }
        dsa_status rs = launch_indexer_tc(q, w, q8, wq, hist, idxk_cache, &vb, topk, topk_scores, plan,
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
    if (b->total_q == 0) return share ? dsa_topk_share_publish(share, layer_id, topk, 0) : DSA_OK;   // no rows
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
        uint32_t* hist = reinterpret_cast<uint32_t*>(sc);
        dsa_status rs = launch_index_q_quant(q, w, b->total_q, q8, wq, hist, s);   // also clears hist
        if (rs != DSA_OK) return rs;
        void* plan = reinterpret_cast<uint8_t*>(sc) + (size_t)b->total_q * 4096 * 4;
        rs = launch_indexer_rows_topk(q8, wq, hist, idxk_cache, b, topk, topk_scores, plan, device_sm_count(),
                                      dev_status, s);
        if (rs != DSA_OK) return rs;
    }
    if (share) return dsa_topk_share_publish(share, layer_id, topk, b->total_q);
    return DSA_OK;
}
