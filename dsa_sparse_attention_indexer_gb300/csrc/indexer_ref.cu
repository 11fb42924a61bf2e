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

// CUDA-core scorer for decode batches (one query row per request), kept to
// measure the tensor-core kernels against: a CTA per (request, 128-token
// tile), a thread per token.  The row's 32 x 128 query values sit in shared
// memory as fp32; a thread widens its key row 16 values at a time (exact:
// E4M3 -> fp32) and adds each chunk's products to its 32 head sums with
// packed f32x2 FMAs, so its arithmetic is the tensor-core path's (E4M3
// products, fp32 sums) in another order.  Then ReLU, the head weights and the
// key scale; tokens past the context and pages out of range get -inf.
namespace dsa {
constexpr int kSimtTok = 128;
__global__ void __launch_bounds__(kSimtTok)
simt_score_kernel(const uint8_t* __restrict__ q8, const float* __restrict__ wq, const uint8_t* __restrict__ cache,
                  BatchDev b, float* __restrict__ scores, int64_t ld, int32_t* __restrict__ st) {
    __shared__ __align__(16) float2 qf[32 * 64];       // [head][dim pair]
    __shared__ float wsh[32];
    const int r = blockIdx.y;
    const int L = b.seq_len[r];
    const int t0 = blockIdx.x * kSimtTok;
    if (t0 >= L) return;                               // the whole block
    const int64_t row = b.q_start[r];
    const uint16_t* qrow = reinterpret_cast<const uint16_t*>(q8 + row * 4096);
    for (int i = threadIdx.x; i < 2048; i += kSimtTok) qf[i] = e4m3x2_to_f32x2(qrow[i]);
    if (threadIdx.x < 32) wsh[threadIdx.x] = wq[row * 32 + threadIdx.x];
    __syncthreads();
    const int t = t0 + threadIdx.x;
    if (t >= L) return;
    const int pi = t >> 6;
    const int64_t pg = pi < b.max_pages ? (int64_t)b.page_table[(int64_t)r * b.max_pages + pi] : -2;
    float out = -INFINITY;
    if (pg >= 0 && pg < b.num_pages) {
        const uint8_t* page = cache + pg * (int64_t)kIdxPageBytes;
        const uint4* krow = reinterpret_cast<const uint4*>(page + (t & 63) * 128);
        const float ks = *reinterpret_cast<const float*>(page + kIdxPayloadBytes + (t & 63) * 4);
        float2 acc[32];
#pragma unroll
        for (int m = 0; m < 32; ++m) acc[m] = make_float2(0.f, 0.f);
#pragma unroll 1
        for (int c = 0; c < 8; ++c) {                  // 16 key values per chunk
            const uint4 raw = __ldg(krow + c);
            const uint32_t wds[4] = {raw.x, raw.y, raw.z, raw.w};
            float2 kf[8];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                kf[2 * u] = e4m3x2_to_f32x2((uint16_t)(wds[u] & 0xffffu));
                kf[2 * u + 1] = e4m3x2_to_f32x2((uint16_t)(wds[u] >> 16));
            }
#pragma unroll
            for (int m = 0; m < 32; ++m) {
                const float4* qq = reinterpret_cast<const float4*>(qf + m * 64 + c * 8);
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    const float4 q4 = qq[u];
                    acc[m] = __ffma2_rn(make_float2(q4.x, q4.y), kf[2 * u], acc[m]);
                    acc[m] = __ffma2_rn(make_float2(q4.z, q4.w), kf[2 * u + 1], acc[m]);
                }
            }
        }
        float sum = 0.f;
#pragma unroll
        for (int m = 0; m < 32; ++m) sum = fmaf(wsh[m], fmaxf(acc[m].x + acc[m].y, 0.f), sum);
        out = sum * ks;
    } else {
        record_error(st, pg == -2 ? DSA_DEVERR_INDEX_RANGE : DSA_DEVERR_PAGE_RANGE, pg == -2 ? t : pg);
    }
    scores[row * ld + t] = out;
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
    if (b->total_q == 0) return DSA_OK;                                  // no rows
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

extern "C" dsa_status dsa_indexer_scores_cuda_core(const void* q, const float* w, const uint8_t* idxk_cache,
                                                   const dsa_batch* b, float* scores, int64_t ld, void* ws,
                                                   size_t ws_bytes, int32_t* dev_status, void* stream) {
    dsa_status vs = validate_batch(b);
    if (vs != DSA_OK) return vs;
    if (b->total_q == 0) return DSA_OK;                                  // no rows
    if (!q || !w || !idxk_cache || !scores) return DSA_ERR_INVALID_ARGUMENT;
    if (ld < b->max_seq_len) return DSA_ERR_INVALID_ARGUMENT;
    if (!aligned16(q) || !aligned16(idxk_cache)) return DSA_ERR_ALIGNMENT;
    if (b->max_q_len > 1 || b->total_q != b->batch) return DSA_ERR_UNSUPPORTED;   // decode batches
    if (b->total_q == 0) return DSA_OK;
    if (!ws || !aligned16(ws)) return ws ? DSA_ERR_ALIGNMENT : DSA_ERR_INVALID_ARGUMENT;
    if (ws_bytes < q8_workspace_bytes(b->total_q)) return DSA_ERR_WORKSPACE_TOO_SMALL;
    if (b->batch > 65535) return DSA_ERR_UNSUPPORTED;
    uint8_t* q8 = static_cast<uint8_t*>(ws);
    float* wq = reinterpret_cast<float*>(q8 + (size_t)b->total_q * 4096);
    cudaStream_t s = as_stream(stream);
    dsa_status rs = launch_index_q_quant(q, w, b->total_q, q8, wq, nullptr, s);
    if (rs != DSA_OK) return rs;
    const unsigned tiles = (unsigned)((b->max_seq_len + kSimtTok - 1) / kSimtTok);
    if (tiles == 0) return DSA_OK;
    simt_score_kernel<<<dim3(tiles, (unsigned)b->batch), kSimtTok, 0, s>>>(q8, wq, idxk_cache, to_dev(b), scores, ld,
                                                                           dev_status);
    DSA_CHECK_LAUNCH();
    return DSA_OK;
}
