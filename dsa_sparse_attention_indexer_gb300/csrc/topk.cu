// Top-2048 selection over fp32 score rows ("vLLM 推理链路概览", DSA Indexer:
// I_i = TopK_{j,2048}(s_ij); "GLM-5.3 推理全链路(十一)", 优化二: a context of
// at most 2048 tokens selects [0, 1, ..., L-1, -1, ...]).
//
// One CTA per row.  Scores become order-preserving uint32 keys (-0 folded onto
// +0); select_topk_row reads the row twice (a histogram of the top 12 key
// bits, then the keys at or above the bin of the 2048th) and selects the rest
// exactly inside that bin (ties -> lower position), writing the kept positions
// in ascending order.
#include "dsa_internal.cuh"
#include "topk_common.cuh"

namespace dsa {

__global__ void __launch_bounds__(kSelThreads)
topk_from_scores_kernel(const float* __restrict__ scores, int64_t ld, const int32_t* __restrict__ valid_len,
                        int64_t max_len, int32_t* __restrict__ topk) {
    extern __shared__ __align__(16) uint8_t sel_smem[];
    const int64_t r = blockIdx.x;
    const int64_t n = max((int64_t)0, min((int64_t)valid_len[r], max_len));   // never past the row
    select_topk_row(scores + r * ld, n, topk + r * kTopK, nullptr, sel_smem);
}

}  // namespace dsa

using namespace dsa;

extern "C" dsa_status dsa_topk_from_scores_workspace_size(int32_t rows, int64_t max_len, size_t* bytes) {
    if (!bytes || rows < 0 || max_len < 0) return DSA_ERR_INVALID_ARGUMENT;
    *bytes = 0;
    return DSA_OK;
}

extern "C" dsa_status dsa_topk_from_scores(const float* scores, int64_t ld, const int32_t* valid_len,
                                           int32_t rows, int64_t max_len, int32_t* topk, void* ws,
                                           size_t ws_bytes, void* stream) {
    (void)ws;
    (void)ws_bytes;
    if (rows < 0 || max_len < 0 || ld < max_len) return DSA_ERR_INVALID_ARGUMENT;
    if (rows == 0) return DSA_OK;
    if (!scores || !valid_len || !topk) return DSA_ERR_INVALID_ARGUMENT;
    if (max_len > 0x7fffffffLL) return DSA_ERR_UNSUPPORTED;
    if (ensure_smem_limit(reinterpret_cast<const void*>(&topk_from_scores_kernel), kSelSmem) != DSA_OK)
        return DSA_ERR_CUDA;
    topk_from_scores_kernel<<<rows, kSelThreads, kSelSmem, as_stream(stream)>>>(scores, ld, valid_len, max_len, topk);
    DSA_CHECK_LAUNCH();
    return DSA_OK;
}
