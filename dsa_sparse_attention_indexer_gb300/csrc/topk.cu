// Top-2048 selection over fp32 score rows ("vLLM 推理链路概览", DSA Indexer:
// I_i = TopK_{j,2048}(s_ij); "GLM-5.3 推理全链路(十一)", 优化二: a context of
// at most 2048 tokens selects [0, 1, ..., L-1, -1, ...]).
//
// One CTA per row.  Scores become order-preserving uint32 keys (-0 folded onto
// +0).  A three-pass radix select (11 + 11 + 10 bits) finds the 2048th largest
// key K* and how many keys equal to K* are needed; a final ordered pass keeps
// key > K*, plus the first `need` keys == K* in position order (ties -> lower
// position), and writes the kept positions in ascending order.
#include "dsa_internal.cuh"
#include "topk_common.cuh"

namespace dsa {

struct ScoreRowSource {
    const float* row;
    __device__ __forceinline__ uint32_t key(int64_t j) const { return score_key(__ldg(row + j)); }
    __device__ __forceinline__ float score(int64_t j) const { return __ldg(row + j); }
};

__global__ void __launch_bounds__(kSelThreads)
topk_from_scores_kernel(const float* __restrict__ scores, int64_t ld,
                        const int32_t* __restrict__ valid_len, int32_t* __restrict__ topk) {
    __shared__ SelectSmem sm;
    const int64_t r = blockIdx.x;
    const int64_t n = valid_len[r];
    ScoreRowSource src{scores + r * ld};
    select_topk_row(src, n, topk + r * kTopK, (float*)nullptr, sm);
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
    topk_from_scores_kernel<<<rows, kSelThreads, 0, as_stream(stream)>>>(scores, ld, valid_len, topk);
    DSA_CHECK_LAUNCH();
    return DSA_OK;
}
