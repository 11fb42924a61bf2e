// Batch descriptor handling shared by the indexer and sparse-MLA entry points.
#pragma once
#include "dsa_internal.cuh"

namespace dsa {

// By-value copy of dsa_batch passed to kernels.
struct BatchDev {
    int32_t batch;
    int32_t max_pages;
    int32_t max_seq_len;
    int32_t max_q_len;
    int64_t total_q;
    int64_t num_pages;
    const int32_t* seq_len;
    const int32_t* q_start;
    const int32_t* page_table;
    uint64_t wait_ns;      // limit of the decode score kernel's pipeline waits (normally 2 s)
};

inline BatchDev to_dev(const dsa_batch* b) {
    BatchDev d;
    d.batch = b->batch;
    d.max_pages = b->max_pages;
    d.max_seq_len = b->max_seq_len;
    d.max_q_len = b->max_q_len;
    d.total_q = b->total_q;
    d.num_pages = b->num_pages;
    d.seq_len = b->seq_len;
    d.q_start = b->q_start;
    d.page_table = b->page_table;
    d.wait_ns = wait_limit_ns();
    return d;
}

// Host-side checks of a batch descriptor (before any launch).
inline dsa_status validate_batch(const dsa_batch* b) {
    if (!b) return DSA_ERR_INVALID_ARGUMENT;
    if (b->batch < 1 || b->max_pages < 1 || b->max_seq_len < 1 || b->max_q_len < 0 ||
        b->total_q < 0 || b->num_pages < 1)
        return DSA_ERR_INVALID_ARGUMENT;
    if (!b->seq_len || !b->q_start || !b->page_table) return DSA_ERR_INVALID_ARGUMENT;
    if ((int64_t)b->max_pages * DSA_PAGE_TOKENS < b->max_seq_len) return DSA_ERR_INVALID_ARGUMENT;
    if (b->total_q > (int64_t)b->batch * b->max_q_len) return DSA_ERR_INVALID_ARGUMENT;
    if (b->total_q > 0x7fffffffLL || b->batch > 65535) return DSA_ERR_UNSUPPORTED;
    return DSA_OK;
}

// Quantised index query + folded head weights: T * (4096 B codes + 128 B weights).
inline size_t q8_workspace_bytes(int64_t total_q) { return (size_t)total_q * (4096 + 128); }

dsa_status launch_index_q_quant(const void* q, const float* w, int64_t rows, uint8_t* q8, float* wq,
                                uint32_t* hist, cudaStream_t s);

// Index-Q quantisation of one (row, head) g = row * 32 + head by one warp:
// 128 bf16 -> 128 E4M3 codes with one ue8m0 scale 2^e, folded into the head
// weight (w' = w * 2^e, exact); also clears the row's 128-word slice of the
// top-12-bit histogram when hist is given.
__device__ __forceinline__ void index_q_quant_warp(const uint16_t* __restrict__ q, const float* __restrict__ w,
                                                   int64_t g, int lane, uint8_t* __restrict__ q8,
                                                   float* __restrict__ wq, uint32_t* __restrict__ hist) {
    if (hist) reinterpret_cast<uint4*>(hist + g * 128)[lane] = make_uint4(0, 0, 0, 0);
    const uint2 raw = *reinterpret_cast<const uint2*>(q + g * 128 + lane * 4);
    const float x0 = bf16_bits_to_f32(raw.x & 0xffffu), x1 = bf16_bits_to_f32(raw.x >> 16);
    const float x2 = bf16_bits_to_f32(raw.y & 0xffffu), x3 = bf16_bits_to_f32(raw.y >> 16);
    float amax = fmaxf(fmaxf(fabsf(x0), fabsf(x1)), fmaxf(fabsf(x2), fabsf(x3)));
    amax = warp_max(amax);
    const int e = ue8m0_exponent(amax);
    const uint32_t lo = f32x2_to_e4m3x2(ldexpf(x0, -e), ldexpf(x1, -e));
    const uint32_t hi = f32x2_to_e4m3x2(ldexpf(x2, -e), ldexpf(x3, -e));
    *reinterpret_cast<uint32_t*>(q8 + g * 128 + lane * 4) = lo | (hi << 16);
    if (lane == 0) wq[g] = w[g] * ldexpf(1.0f, e);
}

}  // namespace dsa
