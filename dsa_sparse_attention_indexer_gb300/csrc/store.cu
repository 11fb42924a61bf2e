// Cache writers: the index-K store (k_norm LayerNorm -> interleaved RoPE on
// dims 0..63 -> FP8 E4M3 with a ue8m0 scale; "GLM-5.3 推理全链路(十一)",
// section 索引器缓存里存的是什么) and the latent-row store (512 FP8 + four
// scales + 64 bf16 RoPE dims = 656 B; same page, section 主 KV 缓存里存的是什么).
//
// Both are tiny (n new tokens per step) and write-only; one warp per token,
// every lane writes one contiguous 4- or 16-byte piece so the row leaves the
// SM as full 128-byte segments.
#include <cmath>

#include "dsa_internal.cuh"

namespace dsa {

// Rotation frequencies base^(-2i/64), i < 32, computed once on the host in fp64.
struct RopeFreqs {
    double theta[32];
};

// E2M1 code of y (OCP Microscaling FP4: values 0, 0.5, 1, 1.5, 2, 3, 4, 6 with
// a sign bit): nearest value, ties to the even code, |y| > 6 saturates to 6;
// the sign bit follows y.  The thresholds are the midpoints between
// neighbouring values; a midpoint goes to the neighbour whose code is even.
__device__ __forceinline__ uint32_t e2m1_code(float y) {
    const uint32_t sign = (__float_as_uint(y) >> 31) << 3;
    const float a = fabsf(y);
    uint32_t m;
    if (a <= 0.25f) m = 0;
    else if (a < 0.75f) m = 1;
    else if (a <= 1.25f) m = 2;
    else if (a < 1.75f) m = 3;
    else if (a <= 2.5f) m = 4;
    else if (a < 3.5f) m = 5;
    else if (a <= 5.0f) m = 6;
    else m = 7;
    return sign | m;
}

// One warp per token; lane l owns dims [4l, 4l+4).  RoPE pairs (2i, 2i+1)
// never straddle lanes.  kMx: the MXFP4 page layout ("GLM-5.3 推理全链路(十一)",
// 两个框架的对照): lanes 8b .. 8b+7 hold block b of 32 dims, whose shared
// exponent is floor(log2(amax)) - 2 (OCP MX, E2M1's largest value is 1.5 * 2^2),
// clamped to [-127, 127]; each lane writes its 4 codes as 2 packed bytes.
template <bool kMx>
__device__ __forceinline__ void store_index_key(const uint16_t* __restrict__ krow, int32_t tpos, int64_t s,
                                                const float* __restrict__ gamma, const float* __restrict__ beta,
                                                float eps, const RopeFreqs& fr, uint8_t* __restrict__ cache,
                                                int lane) {
    const uint2 raw = *reinterpret_cast<const uint2*>(krow + lane * 4);
    float x[4] = {bf16_bits_to_f32(raw.x & 0xffffu), bf16_bits_to_f32(raw.x >> 16),
                  bf16_bits_to_f32(raw.y & 0xffffu), bf16_bits_to_f32(raw.y >> 16)};
    // LayerNorm over 128 dims, biased variance, fp32.
    const float mean = warp_sum(x[0] + x[1] + x[2] + x[3]) * (1.0f / 128.0f);
    float d2 = 0.f;
#pragma unroll
    for (int i = 0; i < 4; ++i) { x[i] -= mean; d2 += x[i] * x[i]; }
    const float var = warp_sum(d2) * (1.0f / 128.0f);
    const float inv = 1.0f / sqrtf(var + eps);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        float y = x[i] * inv;
        if (gamma) y *= gamma[lane * 4 + i];
        if (beta) y += beta[lane * 4 + i];
        x[i] = y;
    }
    // Interleaved RoPE on dims 0..63: lanes 0..15 hold pairs i = 2l, 2l+1.
    // The angle pos * theta_i and its reduction modulo 2*pi are formed in
    // fp64 (at positions near 2^20 an fp32 angle would be off by ~0.1 rad);
    // the reduced angle, |r| <= pi, goes through fp32 sincos.
    if (lane < 16) {
        const double p = (double)tpos;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int i = 2 * lane + h;
            const double ang = p * fr.theta[i];
            const double red = fma(-6.283185307179586, rint(ang * 0.15915494309189535), ang);
            float si, c;
            sincosf((float)red, &si, &c);
            const float a = x[2 * h], b = x[2 * h + 1];
            x[2 * h] = a * c - b * si;
            x[2 * h + 1] = a * si + b * c;
        }
    }
    float amax = fmaxf(fmaxf(fabsf(x[0]), fabsf(x[1])), fmaxf(fabsf(x[2]), fabsf(x[3])));
    if constexpr (kMx) {
#pragma unroll
        for (int o = 4; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
        int k2 = 0;
        frexpf(amax, &k2);                               // amax = m * 2^k2, m in [0.5, 1)
        const int e = amax > 0.f ? max(-127, min(127, k2 - 1 - 2)) : 0;
        const uint32_t c0 = e2m1_code(ldexpf(x[0], -e)), c1 = e2m1_code(ldexpf(x[1], -e));
        const uint32_t c2 = e2m1_code(ldexpf(x[2], -e)), c3 = e2m1_code(ldexpf(x[3], -e));
        const int64_t page = s / kPage;
        const int row = (int)(s % kPage);
        uint8_t* pg = cache + page * (int64_t)DSA_IDXK_MXFP4_PAGE_BYTES;
        *reinterpret_cast<uint16_t*>(pg + row * 64 + lane * 2) = (uint16_t)(c0 | (c1 << 4) | (c2 << 8) | (c3 << 12));
        if ((lane & 7) == 0) pg[kPage * 64 + row * 4 + (lane >> 3)] = (uint8_t)(e + 127);
        return;
    }
    amax = warp_max(amax);
    const int e = ue8m0_exponent(amax);
    const uint32_t lo = f32x2_to_e4m3x2(ldexpf(x[0], -e), ldexpf(x[1], -e));
    const uint32_t hi = f32x2_to_e4m3x2(ldexpf(x[2], -e), ldexpf(x[3], -e));
    const int64_t page = s / kPage;
    const int row = (int)(s % kPage);
    uint8_t* pg = cache + page * (int64_t)kIdxPageBytes;
    *reinterpret_cast<uint32_t*>(pg + row * 128 + lane * 4) = lo | (hi << 16);
    if (lane == 0) *reinterpret_cast<float*>(pg + kIdxPayloadBytes + row * 4) = ldexpf(1.0f, e);
}

template <bool kMx>
__global__ void __launch_bounds__(256)
index_k_store_kernel(const uint16_t* __restrict__ k, const int32_t* __restrict__ pos,
                     const int64_t* __restrict__ slot, int64_t n,
                     const float* __restrict__ gamma, const float* __restrict__ beta,
                     float eps, RopeFreqs fr, uint8_t* __restrict__ cache,
                     int64_t num_pages, int32_t* __restrict__ st) {
    pdl_wait();
    pdl_trigger();
    const int lane = threadIdx.x & 31;
    const int64_t t = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    if (t >= n) return;
    const int64_t s = slot[t];
    if (s < 0) return;                                   // padded row: K write skipped
    if (s >= num_pages * kPage) {
        if (lane == 0) record_error(st, DSA_DEVERR_SLOT_RANGE, s);
        return;
    }
    store_index_key<kMx>(k + t * 128, pos[t], s, gamma, beta, eps, fr, cache, lane);
}

// The latent row from the A-projection outputs, in one pass ("GLM-5.3 推理全链路
// (一)", 4.3 两个 RMSNorm 与 RoPE: kv_a_layernorm over kv_c, RoPE on k_pe, the
// result written into the KV pool, and on a layer with an indexer the index key
// into the index cache as well).  One warp per token: lane l owns latent dims
// [16l, 16l+16) (block l/8) and the RoPE pair (2l, 2l+1).
__global__ void __launch_bounds__(256)
latent_store_fused_kernel(const uint16_t* __restrict__ kv_c, const uint16_t* __restrict__ k_pe,
                          const int32_t* __restrict__ pos, const int64_t* __restrict__ slot, int64_t n,
                          const float* __restrict__ kv_gamma, float rms_eps, RopeFreqs fr,
                          uint8_t* __restrict__ kv_cache, int64_t num_pages,
                          const uint16_t* __restrict__ idx_k, const float* __restrict__ idx_gamma,
                          const float* __restrict__ idx_beta, float ln_eps, uint8_t* __restrict__ idxk_cache,
                          int64_t idx_num_pages, int32_t* __restrict__ st) {
    const int lane = threadIdx.x & 31;
    const int64_t t = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    if (t >= n) return;
    const int64_t s = slot[t];
    if (s < 0) return;
    if (s < num_pages * kPage) {
        const uint4* src = reinterpret_cast<const uint4*>(kv_c + t * 512 + lane * 16);
        const uint4 r0 = src[0], r1 = src[1];
        const uint32_t w[8] = {r0.x, r0.y, r0.z, r0.w, r1.x, r1.y, r1.z, r1.w};
        float x[16];
        float ss = 0.f;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            x[2 * i] = bf16_bits_to_f32(w[i] & 0xffffu);
            x[2 * i + 1] = bf16_bits_to_f32(w[i] >> 16);
            ss = fmaf(x[2 * i], x[2 * i], ss);
            ss = fmaf(x[2 * i + 1], x[2 * i + 1], ss);
        }
        const float inv = 1.0f / sqrtf(warp_sum(ss) * (1.0f / 512.0f) + rms_eps);   // RMSNorm, fp32
        float amax = 0.f;
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            x[i] *= inv;
            if (kv_gamma) x[i] *= kv_gamma[lane * 16 + i];
            amax = fmaxf(amax, fabsf(x[i]));
        }
#pragma unroll
        for (int o = 4; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
        const int e = ue8m0_exponent(amax);
        uint32_t q[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const uint32_t a = f32x2_to_e4m3x2(ldexpf(x[4 * i], -e), ldexpf(x[4 * i + 1], -e));
            const uint32_t b = f32x2_to_e4m3x2(ldexpf(x[4 * i + 2], -e), ldexpf(x[4 * i + 3], -e));
            q[i] = a | (b << 16);
        }
        // RoPE pair (2l, 2l+1) of k_pe: angle reduced in fp64 as for the index key
        const uint32_t pr = reinterpret_cast<const uint32_t*>(k_pe + t * 64)[lane];
        const float a = bf16_bits_to_f32(pr & 0xffffu), b = bf16_bits_to_f32(pr >> 16);
        const double ang = (double)pos[t] * fr.theta[lane];
        const double red = fma(-6.283185307179586, rint(ang * 0.15915494309189535), ang);
        float si, co;
        sincosf((float)red, &si, &co);
        const __nv_bfloat16 ra = __float2bfloat16_rn(a * co - b * si), rb = __float2bfloat16_rn(a * si + b * co);
        const uint32_t rp = (uint32_t)__bfloat16_as_ushort(ra) | ((uint32_t)__bfloat16_as_ushort(rb) << 16);
        uint8_t* row = kv_cache + (s / kPage) * (int64_t)kKvPageBytes + (s % kPage) * kKvTokenBytes;
        *reinterpret_cast<uint4*>(row + lane * 16) = make_uint4(q[0], q[1], q[2], q[3]);
        if ((lane & 7) == 0) *reinterpret_cast<float*>(row + 512 + (lane >> 3) * 4) = ldexpf(1.0f, e);
        *reinterpret_cast<uint32_t*>(row + 528 + lane * 4) = rp;
    } else if (lane == 0) {
        record_error(st, DSA_DEVERR_SLOT_RANGE, s);
    }
    if (idx_k) {
        if (s < idx_num_pages * kPage)
            store_index_key<false>(idx_k + t * 128, pos[t], s, idx_gamma, idx_beta, ln_eps, fr, idxk_cache, lane);
        else if (lane == 0)
            record_error(st, DSA_DEVERR_SLOT_RANGE, s);
    }
}

// One warp per token; lane l owns latent dims [16l, 16l+16) (block l/8) and,
// for l < 8, RoPE dims [8l, 8l+8).
__global__ void __launch_bounds__(256)
latent_store_kernel(const uint16_t* __restrict__ c, const uint16_t* __restrict__ rope,
                    const int64_t* __restrict__ slot, int64_t n, uint8_t* __restrict__ cache,
                    int64_t num_pages, int32_t* __restrict__ st) {
    pdl_wait();
    pdl_trigger();
    const int lane = threadIdx.x & 31;
    const int64_t t = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    if (t >= n) return;
    const int64_t s = slot[t];
    if (s < 0) return;
    if (s >= num_pages * kPage) {
        if (lane == 0) record_error(st, DSA_DEVERR_SLOT_RANGE, s);
        return;
    }
    const uint4* src = reinterpret_cast<const uint4*>(c + t * 512 + lane * 16);
    const uint4 r0 = src[0], r1 = src[1];
    const uint32_t w[8] = {r0.x, r0.y, r0.z, r0.w, r1.x, r1.y, r1.z, r1.w};
    float x[16];
    float amax = 0.f;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        x[2 * i] = bf16_bits_to_f32(w[i] & 0xffffu);
        x[2 * i + 1] = bf16_bits_to_f32(w[i] >> 16);
        amax = fmaxf(amax, fmaxf(fabsf(x[2 * i]), fabsf(x[2 * i + 1])));
    }
#pragma unroll
    for (int o = 4; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    const int e = ue8m0_exponent(amax);
    uint32_t q[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const uint32_t a = f32x2_to_e4m3x2(ldexpf(x[4 * i], -e), ldexpf(x[4 * i + 1], -e));
        const uint32_t b = f32x2_to_e4m3x2(ldexpf(x[4 * i + 2], -e), ldexpf(x[4 * i + 3], -e));
        q[i] = a | (b << 16);
    }
    uint8_t* row = cache + (s / kPage) * (int64_t)kKvPageBytes + (s % kPage) * kKvTokenBytes;
    *reinterpret_cast<uint4*>(row + lane * 16) = make_uint4(q[0], q[1], q[2], q[3]);
    if ((lane & 7) == 0) *reinterpret_cast<float*>(row + 512 + (lane >> 3) * 4) = ldexpf(1.0f, e);
    if (lane < 8)
        *reinterpret_cast<uint4*>(row + 528 + lane * 16) =
            reinterpret_cast<const uint4*>(rope + t * 64)[lane];
}

}  // namespace dsa

using namespace dsa;

extern "C" dsa_status dsa_index_k_store(const void* k, const int32_t* pos, const int64_t* slot,
                                        int64_t n, const float* gamma, const float* beta,
                                        float ln_eps, float rope_base, uint8_t* idxk_cache,
                                        int64_t num_pages, int32_t* dev_status, void* stream) {
    if (n < 0 || num_pages < 0) return DSA_ERR_INVALID_ARGUMENT;
    if (n == 0) return DSA_OK;
    if (!k || !pos || !slot || !idxk_cache) return DSA_ERR_INVALID_ARGUMENT;
    if (!(ln_eps >= 0.f) || !(rope_base > 0.f)) return DSA_ERR_INVALID_ARGUMENT;
    if (!aligned16(k) || !aligned16(idxk_cache)) return DSA_ERR_ALIGNMENT;
    const int warps = 8;
    const int64_t blocks = (n + warps - 1) / warps;
    if (blocks > 0x7fffffff) return DSA_ERR_UNSUPPORTED;
    RopeFreqs fr;
    for (int i = 0; i < 32; ++i) fr.theta[i] = std::pow((double)rope_base, -2.0 * (double)i / 64.0);
    DSA_CHECK(launch_pdl(index_k_store_kernel<false>, dim3((unsigned)blocks), dim3(warps * 32), 0, as_stream(stream), 1,
                         static_cast<const uint16_t*>(k), pos, slot, n, gamma, beta, ln_eps, fr, idxk_cache, num_pages,
                         dev_status));
    return DSA_OK;
}

extern "C" dsa_status dsa_index_k_store_mxfp4(const void* k, const int32_t* pos, const int64_t* slot,
                                              int64_t n, const float* gamma, const float* beta,
                                              float ln_eps, float rope_base, uint8_t* idxk_cache,
                                              int64_t num_pages, int32_t* dev_status, void* stream) {
    if (n < 0 || num_pages < 0) return DSA_ERR_INVALID_ARGUMENT;
    if (n == 0) return DSA_OK;
    if (!k || !pos || !slot || !idxk_cache) return DSA_ERR_INVALID_ARGUMENT;
    if (!(ln_eps >= 0.f) || !(rope_base > 0.f)) return DSA_ERR_INVALID_ARGUMENT;
    if (!aligned16(k) || (reinterpret_cast<uintptr_t>(idxk_cache) & 31)) return DSA_ERR_ALIGNMENT;
    const int warps = 8;
    const int64_t blocks = (n + warps - 1) / warps;
    if (blocks > 0x7fffffff) return DSA_ERR_UNSUPPORTED;
    RopeFreqs fr;
    for (int i = 0; i < 32; ++i) fr.theta[i] = std::pow((double)rope_base, -2.0 * (double)i / 64.0);
    DSA_CHECK(launch_pdl(index_k_store_kernel<true>, dim3((unsigned)blocks), dim3(warps * 32), 0, as_stream(stream), 1,
                         static_cast<const uint16_t*>(k), pos, slot, n, gamma, beta, ln_eps, fr, idxk_cache, num_pages,
                         dev_status));
    return DSA_OK;
}

extern "C" dsa_status dsa_latent_kv_store_fused(const void* kv_c, const void* k_pe, const int32_t* pos,
                                                const int64_t* slot, int64_t n, const float* kv_gamma,
                                                float rms_eps, float rope_base, uint8_t* kv_cache, int64_t num_pages,
                                                const void* idx_k, const float* idx_gamma, const float* idx_beta,
                                                float ln_eps, uint8_t* idxk_cache, int64_t idx_num_pages,
                                                int32_t* dev_status, void* stream) {
    if (n < 0 || num_pages < 0 || idx_num_pages < 0) return DSA_ERR_INVALID_ARGUMENT;
    if (n == 0) return DSA_OK;
    if (!kv_c || !k_pe || !pos || !slot || !kv_cache) return DSA_ERR_INVALID_ARGUMENT;
    if (idx_k && !idxk_cache) return DSA_ERR_INVALID_ARGUMENT;
    if (!(rms_eps >= 0.f) || !(ln_eps >= 0.f) || !(rope_base > 0.f)) return DSA_ERR_INVALID_ARGUMENT;
    if (!aligned16(kv_c) || (reinterpret_cast<uintptr_t>(k_pe) & 3) || !aligned16(kv_cache)) return DSA_ERR_ALIGNMENT;
    if (idx_k && (!aligned16(idx_k) || !aligned16(idxk_cache))) return DSA_ERR_ALIGNMENT;
    const int warps = 8;
    const int64_t blocks = (n + warps - 1) / warps;
    if (blocks > 0x7fffffff) return DSA_ERR_UNSUPPORTED;
    RopeFreqs fr;
    for (int i = 0; i < 32; ++i) fr.theta[i] = std::pow((double)rope_base, -2.0 * (double)i / 64.0);
    latent_store_fused_kernel<<<(unsigned)blocks, warps * 32, 0, as_stream(stream)>>>(
        static_cast<const uint16_t*>(kv_c), static_cast<const uint16_t*>(k_pe), pos, slot, n, kv_gamma, rms_eps,
        fr, kv_cache, num_pages, static_cast<const uint16_t*>(idx_k), idx_gamma, idx_beta, ln_eps, idxk_cache,
        idx_num_pages, dev_status);
    DSA_CHECK_LAUNCH();
    return DSA_OK;
}

extern "C" dsa_status dsa_latent_kv_store(const void* c, const void* rope, const int64_t* slot,
                                          int64_t n, uint8_t* kv_cache, int64_t num_pages,
                                          int32_t* dev_status, void* stream) {
    if (n < 0 || num_pages < 0) return DSA_ERR_INVALID_ARGUMENT;
    if (n == 0) return DSA_OK;
    if (!c || !rope || !slot || !kv_cache) return DSA_ERR_INVALID_ARGUMENT;
    if (!aligned16(c) || !aligned16(rope) || !aligned16(kv_cache)) return DSA_ERR_ALIGNMENT;
    const int warps = 8;
    const int64_t blocks = (n + warps - 1) / warps;
    if (blocks > 0x7fffffff) return DSA_ERR_UNSUPPORTED;
    DSA_CHECK(launch_pdl(latent_store_kernel, dim3((unsigned)blocks), dim3(warps * 32), 0, as_stream(stream), 1,
                         static_cast<const uint16_t*>(c), static_cast<const uint16_t*>(rope), slot, n, kv_cache,
                         num_pages, dev_status));
    return DSA_OK;
}
