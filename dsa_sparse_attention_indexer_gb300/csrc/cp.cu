// Context-parallel split of long requests over G ranks ("GLM-5.3 推理全链路(十一)",
// 两个框架的对照: with prefill context parallelism the indexer's reads are spread
// over the ranks; "Accelerating GLM-5.3-Flash on H200", prefill 的重点是少搬一次、
// 少等一次: CP4 on the prefill side).
//
// Each rank holds a disjoint slice of a request's positions in its own caches
// and runs the single-GPU calls on it: the indexer gives the slice's top-2048
// with scores, sparse MLA gives attention over the selected positions the rank
// holds together with their log-sum-exp.  Two exchanges between the ranks
// (the caller's collective) carry at most 2048 (score, position) pairs and one
// [64 x 512] partial per query row and rank; the kernels here merge them:
//   topk_merge_kernel       the global top-2048 of the union of the ranks'
//                           lists (every globally selected position is also
//                           selected within its own slice), same order and
//                           tie rule as the indexer;
//   topk_localize_kernel    a rank's share of the global list, in its own
//                           local positions, compacted to the front;
//   attention_merge_kernel  softmax attention over the union from the ranks'
//                           parts: out = sum_g w_g out_g / sum_g w_g with
//                           w_g = exp(lse_g - max lse).
#include "dsa_internal.cuh"
#include "select_common.cuh"

namespace dsa {
namespace cp {

constexpr int kMaxRanks = 8;
constexpr int kMergeThreads = 1024;
constexpr int kCand = kMaxRanks * kTopK;                    // candidates of one row, at most
// shared memory of the merge: keys and positions of the candidates, a 4096-bin
// histogram, scan scratch and the radix-select result
constexpr int kMergeSmem = kCand * 8 + 4096 * 4 + 64 * 4 + 16;

// One block per query row.
__global__ void __launch_bounds__(kMergeThreads)
topk_merge_kernel(const int32_t* __restrict__ cand_pos, const float* __restrict__ cand_scores,
                  const int64_t* __restrict__ pos_offset, int G, int64_t rows, int32_t* __restrict__ topk,
                  float* __restrict__ topk_scores, int32_t* __restrict__ st) {
    extern __shared__ __align__(16) uint8_t msm[];
    uint32_t* key = reinterpret_cast<uint32_t*>(msm);
    int32_t* pos = reinterpret_cast<int32_t*>(msm + kCand * 4);
    uint32_t* hist = reinterpret_cast<uint32_t*>(msm + kCand * 8);
    int* scratch = reinterpret_cast<int*>(msm + kCand * 8 + 4096 * 4);
    sel::Found* found = reinterpret_cast<sel::Found*>(msm + kCand * 8 + 4096 * 4 + 64 * 4);
    __shared__ int s_n;
    const int64_t row = blockIdx.x;
    const int gt = threadIdx.x;
    // gather the ranks' candidates with their global positions
    int n = 0;
    const int total_in = G * kTopK;
    for (int base = 0; base < total_in; base += kMergeThreads) {
        const int i = base + gt;
        bool have = false;
        uint32_t kk = 0;
        int32_t pp = 0;
        if (i < total_in) {
            const int g = i / kTopK;
            const int64_t at = ((int64_t)g * rows + row) * kTopK + (i % kTopK);
            const int32_t lp = cand_pos[at];
            if (lp >= 0) {
                const int64_t gp = (int64_t)lp + pos_offset[(int64_t)g * rows + row];
                if (gp < 0 || gp > 0x7ffffffeLL) {
                    record_error(st, DSA_DEVERR_INDEX_RANGE, gp);
                } else {
                    have = true;
                    kk = score_key(cand_scores[at]);
                    pp = (int32_t)gp;
                }
            }
        }
        int tot;
        const int rank = sel::excl_scan<kMergeThreads, 0>(have ? 1 : 0, gt, scratch, &tot);
        if (have) {
            key[n + rank] = kk;
            pos[n + rank] = pp;
        }
        n += tot;
    }
    if (gt == 0) s_n = n;
    __syncthreads();
    if (n > kTopK) sel::compact_topk<kMergeThreads, 0>(key, pos, &s_n, kTopK, gt, hist, scratch, found);
    __syncthreads();
    n = s_n;
    // ascending positions: pad to 2048 with the largest position, sort, write
    for (int i = n + gt; i < kTopK; i += kMergeThreads) {
        pos[i] = 0x7fffffff;
        key[i] = 0u;
    }
    __syncthreads();
    sel::bitonic_sort_by_pos<kMergeThreads, 0>(pos, key, kTopK, gt);
    for (int i = gt; i < kTopK; i += kMergeThreads) {
        const bool v = i < n;
        topk[row * kTopK + i] = v ? pos[i] : -1;
        if (topk_scores) topk_scores[row * kTopK + i] = v ? key_score(key[i]) : 0.f;
    }
}

// One block per query row: entries of the global list inside [lo, lo + len),
// as local positions j - lo, in their order, then -1.
constexpr int kLocThreads = 1024;
__global__ void __launch_bounds__(kLocThreads)
topk_localize_kernel(const int32_t* __restrict__ topk, int64_t rows, const int64_t* __restrict__ lo,
                     const int64_t* __restrict__ len, int32_t* __restrict__ out) {
    __shared__ int scratch[32];
    const int64_t row = blockIdx.x;
    const int gt = threadIdx.x;
    const int64_t a = lo[row], n = len[row];
    int done = 0;
    for (int base = 0; base < kTopK; base += kLocThreads) {
        const int e = base + gt;
        const int32_t j = topk[row * kTopK + e];
        const bool mine = j >= 0 && (int64_t)j >= a && (int64_t)j < a + n;
        int tot;
        const int rank = sel::excl_scan<kLocThreads, 0>(mine ? 1 : 0, gt, scratch, &tot);
        if (mine) out[row * kTopK + done + rank] = (int32_t)((int64_t)j - a);
        done += tot;
    }
    for (int e = done + gt; e < kTopK; e += kLocThreads) out[row * kTopK + e] = -1;
}

// One block per (row, head): 128 threads, four of the 512 dims each.
constexpr int kAttThreads = 128;
__global__ void __launch_bounds__(kAttThreads)
attention_merge_kernel(const float* __restrict__ o_parts, const float* __restrict__ lse_parts, int G,
                       int64_t rows, void* __restrict__ out, int out_f32, float* __restrict__ lse_out) {
    const int64_t row = blockIdx.x;
    const int h = blockIdx.y;
    const int tid = threadIdx.x;
    float M = -INFINITY;
    for (int g = 0; g < G; ++g) M = fmaxf(M, lse_parts[((int64_t)g * rows + row) * 64 + h]);
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    float den = 0.f;
    if (M != -INFINITY) {
        for (int g = 0; g < G; ++g) {
            const float lg = lse_parts[((int64_t)g * rows + row) * 64 + h];
            if (lg == -INFINITY) continue;
            const float wg = expf(lg - M);
            den += wg;
            const float4 v = reinterpret_cast<const float4*>(o_parts + (((int64_t)g * rows + row) * 64 + h) * 512)[tid];
            acc.x = fmaf(wg, v.x, acc.x);
            acc.y = fmaf(wg, v.y, acc.y);
            acc.z = fmaf(wg, v.z, acc.z);
            acc.w = fmaf(wg, v.w, acc.w);
        }
    }
    const float inv = den > 0.f ? 1.f / den : 0.f;
    const int64_t o = (row * 64 + h) * 512 + tid * 4;
    if (out_f32) {
        *reinterpret_cast<float4*>(static_cast<float*>(out) + o) =
            make_float4(acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv);
    } else {
        __nv_bfloat162 lo2 = __floats2bfloat162_rn(acc.x * inv, acc.y * inv);
        __nv_bfloat162 hi2 = __floats2bfloat162_rn(acc.z * inv, acc.w * inv);
        *reinterpret_cast<uint2*>(static_cast<__nv_bfloat16*>(out) + o) =
            make_uint2(*reinterpret_cast<uint32_t*>(&lo2), *reinterpret_cast<uint32_t*>(&hi2));
    }
    if (lse_out && tid == 0) lse_out[row * 64 + h] = den > 0.f ? M + logf(den) : -INFINITY;
}

}  // namespace cp
}  // namespace dsa

using namespace dsa;

extern "C" dsa_status dsa_cp_topk_merge(const int32_t* cand_pos, const float* cand_scores, const int64_t* pos_offset,
                                        int32_t ranks, int64_t rows, int32_t* topk, float* topk_scores,
                                        int32_t* dev_status, void* stream) {
    if (ranks < 1 || ranks > cp::kMaxRanks || rows < 0) return DSA_ERR_INVALID_ARGUMENT;
    if (rows == 0) return DSA_OK;
    if (!cand_pos || !cand_scores || !pos_offset || !topk) return DSA_ERR_INVALID_ARGUMENT;
    if (rows > 0x7fffffffLL) return DSA_ERR_UNSUPPORTED;
    if (!aligned16(cand_pos) || !aligned16(cand_scores) || !aligned16(topk)) return DSA_ERR_ALIGNMENT;
    if (ensure_smem_limit(reinterpret_cast<const void*>(&cp::topk_merge_kernel), cp::kMergeSmem) != DSA_OK)
        return DSA_ERR_CUDA;
    cp::topk_merge_kernel<<<(unsigned)rows, cp::kMergeThreads, cp::kMergeSmem, as_stream(stream)>>>(
        cand_pos, cand_scores, pos_offset, ranks, rows, topk, topk_scores, dev_status);
    DSA_CHECK_LAUNCH();
    return DSA_OK;
}

extern "C" dsa_status dsa_cp_topk_localize(const int32_t* topk, int64_t rows, const int64_t* slice_start,
                                           const int64_t* slice_len, int32_t* local_topk, void* stream) {
    if (rows < 0) return DSA_ERR_INVALID_ARGUMENT;
    if (rows == 0) return DSA_OK;
    if (!topk || !slice_start || !slice_len || !local_topk) return DSA_ERR_INVALID_ARGUMENT;
    if (rows > 0x7fffffffLL) return DSA_ERR_UNSUPPORTED;
    if (topk == local_topk) return DSA_ERR_INVALID_ARGUMENT;          // rows are read while others are written
    cp::topk_localize_kernel<<<(unsigned)rows, cp::kLocThreads, 0, as_stream(stream)>>>(topk, rows, slice_start,
                                                                                        slice_len, local_topk);
    DSA_CHECK_LAUNCH();
    return DSA_OK;
}

extern "C" dsa_status dsa_cp_attention_merge(const float* o_parts, const float* lse_parts, int32_t ranks,
                                             int64_t rows, void* out, int32_t out_dtype, float* lse,
                                             void* stream) {
    if (ranks < 1 || ranks > cp::kMaxRanks || rows < 0) return DSA_ERR_INVALID_ARGUMENT;
    if (out_dtype != DSA_DTYPE_BF16 && out_dtype != DSA_DTYPE_F32) return DSA_ERR_INVALID_ARGUMENT;
    if (rows == 0) return DSA_OK;
    if (!o_parts || !lse_parts || !out) return DSA_ERR_INVALID_ARGUMENT;
    if (rows > 0x7fffffffLL) return DSA_ERR_UNSUPPORTED;
    if (!aligned16(o_parts) || !aligned16(out)) return DSA_ERR_ALIGNMENT;
    cp::attention_merge_kernel<<<dim3((unsigned)rows, 64), cp::kAttThreads, 0, as_stream(stream)>>>(
        o_parts, lse_parts, ranks, rows, out, out_dtype == DSA_DTYPE_F32, lse);
    DSA_CHECK_LAUNCH();
    return DSA_OK;
}
