// Internal helpers shared by the libdsa kernels (device side) and the C-ABI
// layer (host side).  Not part of the public ABI.
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <stdint.h>

#include "dsa.h"

namespace dsa {

constexpr int kPage = DSA_PAGE_TOKENS;
constexpr int kIdxPageBytes = DSA_IDXK_PAGE_BYTES;
constexpr int kIdxPayloadBytes = DSA_PAGE_TOKENS * DSA_INDEX_HEAD_DIM;   // 8192
constexpr int kKvTokenBytes = DSA_KV_TOKEN_BYTES;
constexpr int kKvPageBytes = DSA_KV_PAGE_BYTES;
constexpr int kTopK = DSA_TOPK;
constexpr float kE4M3Max = 448.0f;

// --------------------------------------------------------------------------
// Device status block: [0] OR of DSA_DEVERR_* bits, [1] count, [2] a value.
// --------------------------------------------------------------------------
__device__ __forceinline__ void record_error(int32_t* st, int bit, int64_t value) {
    if (st != nullptr) {
        atomicOr(st, bit);
        atomicAdd(st + 1, 1);
        atomicExch(st + 2, (int32_t)value);
    }
}

// --------------------------------------------------------------------------
// Order-preserving uint32 key of an fp32 score: a > b  <=>  key(a) > key(b).
// -0.0 is folded onto +0.0 so the two compare equal (ties go by position).
// Key 0 is never produced by a finite float and marks "no score".
// --------------------------------------------------------------------------
__device__ __forceinline__ uint32_t score_key(float f) {
    uint32_t b = __float_as_uint(f);
    if (b == 0x80000000u) b = 0u;
    return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}
__device__ __forceinline__ float key_score(uint32_t k) {
    uint32_t b = (k & 0x80000000u) ? (k & 0x7fffffffu) : ~k;
    return __uint_as_float(b);
}

// --------------------------------------------------------------------------
// ue8m0 block scale: the smallest e with amax <= 448 * 2^e (amax == 0 -> 0).
// frexpf gives a first guess; exact comparisons against 448 * 2^e settle it.
// --------------------------------------------------------------------------
__device__ __forceinline__ int ue8m0_exponent(float amax) {
    if (!(amax > 0.0f)) return 0;
    int e;
    frexpf(amax / kE4M3Max, &e);
    while (amax > ldexpf(kE4M3Max, e)) ++e;
    while (amax <= ldexpf(kE4M3Max, e - 1)) --e;
    return e;
}

// Two floats -> two E4M3 codes (round to nearest even), low byte = a.
__device__ __forceinline__ uint16_t f32x2_to_e4m3x2(float a, float b) {
    return (uint16_t)__nv_cvt_float2_to_fp8x2(make_float2(a, b), __NV_SATFINITE, __NV_E4M3);
}

// Two E4M3 codes (low byte first) -> two floats (exact).
__device__ __forceinline__ float2 e4m3x2_to_f32x2(uint16_t v) {
    __half2_raw h = __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)v, __NV_E4M3);
    __half2 hh = *reinterpret_cast<__half2*>(&h);
    return __half22float2(hh);
}

__device__ __forceinline__ float bf16_bits_to_f32(uint16_t b) {
    return __uint_as_float(((uint32_t)b) << 16);
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}
__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}

// Request index of query row `row`: the r with q_start[r] <= row < q_start[r+1].
__device__ __forceinline__ int row_request(const int32_t* q_start, int B, int64_t row) {
    // In a decode batch (one query row per request) row r is request r: two
    // independent loads confirm that in one round trip.  The test accepts only
    // the one request whose rows contain `row` (an empty request never passes
    // it), so the search below gives the same answer whenever it is skipped.
    const int g = (int)(row < (int64_t)(B - 1) ? row : (int64_t)(B - 1));
    if (g >= 0 && (int64_t)__ldg(q_start + g) <= row && row < (int64_t)__ldg(q_start + g + 1)) return g;
    int lo = 0, hi = B - 1;
    while (lo < hi) {
        int mid = (lo + hi + 1) >> 1;
        if ((int64_t)__ldg(q_start + mid) <= row) lo = mid; else hi = mid - 1;
    }
    return lo;
}

}  // namespace dsa

// --------------------------------------------------------------------------
// Host-side launch helpers (used by the .cu files that implement the ABI).
// --------------------------------------------------------------------------
#define DSA_CHECK_LAUNCH()                                                   \
    do {                                                                     \
        cudaError_t e_ = cudaGetLastError();                                 \
        if (e_ != cudaSuccess) return DSA_ERR_CUDA;                          \
    } while (0)
#define DSA_CHECK(call)                                                      \
    do {                                                                     \
        if ((call) != cudaSuccess) return DSA_ERR_CUDA;                      \
    } while (0)

namespace dsa {
inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
inline cudaStream_t as_stream(void* s) { return reinterpret_cast<cudaStream_t>(s); }

// Limit of the pipeline waits of later launches that take it (the decode
// score kernel); 2 s unless dsa_debug_set_wait_limit_ns changed it.
uint64_t wait_limit_ns();

// Programmatic dependent launch.  A kernel launched by launch_pdl may begin
// while the stream's previous kernel is still running; before its first
// access to global memory it calls pdl_wait(), which returns once that kernel
// has finished and its writes are visible (at once when there is none).  A
// kernel calls pdl_trigger() after its own pdl_wait() to let the next one
// start early, so everything before its predecessor has finished by the time
// the next kernel runs any code.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*k)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                              unsigned cluster, Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    unsigned n = 0;
    attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[n].val.programmaticStreamSerializationAllowed = 1;
    ++n;
    if (cluster > 1) {
        attr[n].id = cudaLaunchAttributeClusterDimension;
        attr[n].val.clusterDim.x = cluster;
        attr[n].val.clusterDim.y = 1;
        attr[n].val.clusterDim.z = 1;
        ++n;
    }
    cfg.attrs = attr;
    cfg.numAttrs = n;
    return cudaLaunchKernelEx(&cfg, k, args...);
}

// Raises kernel `func`'s dynamic shared-memory limit to `bytes` on the current
// device.  The limit is a per-device setting, so it is applied once per
// (kernel, device); the record of what was applied is guarded by a lock, so
// host threads may call concurrently.
dsa_status ensure_smem_limit(const void* func, int bytes);

// The driver's cuTensorMapEncodeTiled (CUDA 12.0 ABI), looked up once per
// process (thread-safe); NULL if the driver does not provide it.
void* tensor_map_encode_fn();
}  // namespace dsa
