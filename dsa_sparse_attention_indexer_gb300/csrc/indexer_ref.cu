// Index-Q quantisation for the multi-token indexer and the dsa_indexer_scores
// hook: FP8 E4M3 with one ue8m0 scale per head, folded into the head weight
// (w'_m = w_m * 2^e_m, exact) - "GLM-5.3 推理全链路(十一)", 读取路径里的两条
// "非缓存"字节: Q is [tokens, 32, 128] FP8 plus a scale per 128 dims.  The
// scores themselves come from the tensor-core kernels (indexer_tc.cu for
// decode batches, indexer_mt.cu for the others and for dsa_indexer_scores).
#include "dsa_internal.cuh"
#include "indexer_common.cuh"
#include "indexer_tc.cuh"

namespace dsa {

// One warp per (row, head): 128 bf16 -> 128 E4M3 codes + w * 2^e (row histogram reset).
__global__ void __launch_bounds__(256)
index_q_quant_kernel(const uint16_t* __restrict__ q, const float* __restrict__ w, int64_t rows,
                     uint8_t* __restrict__ q8, float* __restrict__ wq, uint32_t* __restrict__ hist) {
    const int lane = threadIdx.x & 31;
    const int64_t g = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);   // row*32 + head
    if (g >= rows * 32) return;
    index_q_quant_warp(q, w, g, lane, q8, wq, hist);
}

}  // namespace dsa

using namespace dsa;

namespace dsa {
dsa_status launch_index_q_quant(const void* q, const float* w, int64_t rows, uint8_t* q8, float* wq,
                                uint32_t* hist, cudaStream_t s) {
    const int64_t warps = rows * 32;
    const int64_t blocks = (warps + 7) / 8;
    if (blocks == 0) return DSA_OK;
    index_q_quant_kernel<<<(unsigned)blocks, 256, 0, s>>>(static_cast<const uint16_t*>(q), w, rows, q8, wq, hist);
    DSA_CHECK_LAUNCH();
    return DSA_OK;
}
}  // namespace dsa

extern "C" dsa_status dsa_indexer_scores_workspace_size(const dsa_batch* b, size_t* bytes) {
    dsa_status vs = validate_batch(b);
    if (vs != DSA_OK) return vs;
    if (!bytes) return DSA_ERR_INVALID_ARGUMENT;
    *bytes = (q8_workspace_bytes(b->total_q) + 255) / 256 * 256 + mt_plan_bytes(b->batch, b->total_q);
    return DSA_OK;
}

extern "C" dsa_status dsa_indexer_scores(const void* q, const float* w, const uint8_t* idxk_cache,
                                         const dsa_batch* b, float* scores, int64_t ld, void* ws,
                                         size_t ws_bytes, int32_t* dev_status, void* stream) {
    dsa_status vs = validate_batch(b);
    if (vs != DSA_OK) return vs;
    if (!q || !w || !idxk_cache || !scores) return DSA_ERR_INVALID_ARGUMENT;
    if (ld < b->max_seq_len) return DSA_ERR_INVALID_ARGUMENT;
    if (!aligned16(q) || !aligned16(idxk_cache)) return DSA_ERR_ALIGNMENT;
    if (b->total_q == 0) return DSA_OK;
    if (!ws || !aligned16(ws)) return ws ? DSA_ERR_ALIGNMENT : DSA_ERR_INVALID_ARGUMENT;
    const size_t qbytes = (q8_workspace_bytes(b->total_q) + 255) / 256 * 256;
    if (ws_bytes < qbytes + mt_plan_bytes(b->batch, b->total_q)) return DSA_ERR_WORKSPACE_TOO_SMALL;
    if (b->num_pages * 66 > 0x7fffffffLL) return DSA_ERR_UNSUPPORTED;
    uint8_t* q8 = static_cast<uint8_t*>(ws);
    float* wq = reinterpret_cast<float*>(q8 + (size_t)b->total_q * 4096);
    cudaStream_t s = as_stream(stream);
    dsa_status rs = launch_index_q_quant(q, w, b->total_q, q8, wq, nullptr, s);
    if (rs != DSA_OK) return rs;
    return launch_indexer_rows(q8, wq, idxk_cache, b, scores, ld, false, true, q8 + qbytes, device_sm_count(),
                               dev_status, s);
}
