// Seed rows for top-k reuse across MTP draft steps ("GLM-5.3 推理全链路(十一)",
// 优化四: PD 分离下的 seed 传输 - the seed buffer receives a plain copy of the
// selected top-k rows, 2048 int32 per request, and the kpool tail slots).
//
// One CTA per seed row: 8 KB copied as 16-byte vectors when the row stride
// keeps every row 16-byte aligned, else as int32.  Pure copy, HBM-bound.
#include "dsa_internal.cuh"

namespace dsa {
namespace {

constexpr int kSeedThreads = 256;

__global__ void __launch_bounds__(kSeedThreads)
mtp_seed_write_kernel(const int32_t* __restrict__ topk, int64_t topk_rows, const int32_t* __restrict__ src_row,
                      int32_t* __restrict__ seed, int32_t width, int32_t* st) {
    const int64_t r = blockIdx.x;
    const int64_t s = src_row ? (int64_t)src_row[r] : r;
    const bool ok = s >= 0 && s < topk_rows;
    if (!ok && threadIdx.x == 0) record_error(st, DSA_DEVERR_INDEX_RANGE, s);
    int32_t* dst = seed + r * (int64_t)width;
    if ((width & 3) == 0) {
        const int4* src4 = reinterpret_cast<const int4*>(topk + (ok ? s : 0) * (int64_t)kTopK);
        int4* dst4 = reinterpret_cast<int4*>(dst);
        const int4 pad = make_int4(-1, -1, -1, -1);
        for (int i = threadIdx.x; i < kTopK / 4; i += kSeedThreads) dst4[i] = ok ? __ldg(src4 + i) : pad;
        for (int i = kTopK / 4 + threadIdx.x; i < width / 4; i += kSeedThreads) dst4[i] = pad;
    } else {
        const int32_t* src = topk + (ok ? s : 0) * (int64_t)kTopK;
        for (int i = threadIdx.x; i < width; i += kSeedThreads)
            dst[i] = (ok && i < kTopK) ? __ldg(src + i) : -1;
    }
}

}  // namespace
}  // namespace dsa

extern "C" dsa_status dsa_mtp_seed_write(const int32_t* topk, int64_t topk_rows, const int32_t* src_row, int64_t n,
                                         int32_t* seed, int32_t width, int32_t* dev_status, void* stream) {
    if (n < 0 || topk_rows < 0 || width < DSA_TOPK) return DSA_ERR_INVALID_ARGUMENT;
    if (n == 0) return DSA_OK;
    if (!seed || !topk) return DSA_ERR_INVALID_ARGUMENT;
    if (n > INT32_MAX) return DSA_ERR_UNSUPPORTED;
    if ((reinterpret_cast<uintptr_t>(topk) & 15) || (reinterpret_cast<uintptr_t>(seed) & 15))
        return DSA_ERR_ALIGNMENT;
    dsa::mtp_seed_write_kernel<<<(unsigned)n, dsa::kSeedThreads, 0, dsa::as_stream(stream)>>>(
        topk, topk_rows, src_row, seed, width, dev_status);
    return cudaGetLastError() == cudaSuccess ? DSA_OK : DSA_ERR_CUDA;
}
