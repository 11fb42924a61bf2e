// Sparse MLA in absorbed (MQA) form ("vLLM 推理链路概览", Sparse MLA Attention;
// "GLM-5.3 推理全链路(一)", decode: MQA 形态与吸收):
//   S_hj = scale * <q_h, [c_j * s_j | r_j]>,  out_h = sum_j softmax_j(S_hj) c_j
// over the selected positions j of each query row (j <= p).
//
// Work split: the T x 2048 (row, entry) slots are cut into one contiguous,
// equal share per CTA (at least 256 slots each).  For each row piece in its
// share a CTA gathers the valid entries, streams them in tiles of 64 tokens (656-B rows
// copied with cp.async into a staging buffer while the previous tile computes),
// dequantises each tile into fp16 (c * scale is exact in fp16 for scales in
// [2^-15, 2^7]; the RoPE part converts from bf16), and runs
//   S^T = K Q^T      (M = 64 tokens, N = 64 heads, K = 576)
//   O^T += V^T P^T   (M = 512 latent dims, N = 64 heads, K = 64 tokens)
// on warp-level fp16 tensor-core MMAs with fp32 accumulation and an online
// softmax in fp32 (P is rounded to fp16 for the second product).
// A row covered by several CTAs is merged by log-sum-exp: each piece writes a
// partial (unnormalised O, max, sum) and the last CTA to finish the row (an
// atomic counter per row) combines them.
#include "dsa_internal.cuh"
#include "indexer_common.cuh"

namespace dsa {

constexpr int kMlaThreads = 256;
constexpr int kTile = 64;                 // tokens per tile
constexpr int kQS = 584;                  // fp16 row stride of Q and K tiles (576 + 8)
constexpr int kPS = 72;                   // fp16 row stride of P^T (64 + 8)
constexpr int kSmemQ = 64 * kQS * 2;      // 74,752
constexpr int kSmemK = kTile * kQS * 2;   // 74,752
constexpr int kSmemRaw = kTile * kKvTokenBytes;   // 41,984
constexpr int kSmemP = 64 * kPS * 2;      // 9,216
constexpr int kSmemSlots = kTopK * 8;     // 16,384
constexpr int kOffQ = 0;
constexpr int kOffK = kOffQ + kSmemQ;
constexpr int kOffRaw = kOffK + kSmemK;
constexpr int kOffP = kOffRaw + kSmemRaw;
constexpr int kOffSlots = kOffP + kSmemP;
constexpr int kOffRed = kOffSlots + kSmemSlots;        // red_max[4][64], red_sum[4][64]
constexpr int kOffStat = kOffRed + 2 * 4 * 64 * 4;     // m_run, l_run, alpha [64] each
constexpr int kOffMisc = kOffStat + 3 * 64 * 4;        // scan scratch
constexpr int kMlaSmem = kOffMisc + 64;

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return (uint32_t)__cvta_generic_to_shared(p);
}
__device__ __forceinline__ void ldsm_x4(uint32_t a, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];\n"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3) : "r"(a));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t a, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];\n"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3) : "r"(a));
}
__device__ __forceinline__ void mma16816(float* d, uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1) {
    asm volatile("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
                 "{%8,%9}, {%0,%1,%2,%3};\n"
                 : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
                 : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}
__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(dst), "l"(src));
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::); }
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_group 0;\n" ::); }

__device__ __forceinline__ uint32_t pack_half2(float a, float b) {
    __half2 h = __floats2half2_rn(a, b);
    return *reinterpret_cast<uint32_t*>(&h);
}

// Block-wide exclusive scan for kMlaThreads threads.
__device__ __forceinline__ int mla_block_scan(int v, int* warp_tot, int* total) {
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
    int x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) warp_tot[wid] = x;
    __syncthreads();
    if (wid == 0) {
        int w = (lane < 8) ? warp_tot[lane] : 0;
#pragma unroll
        for (int o = 1; o < 8; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, w, o);
            if (lane >= o) w += y;
        }
        if (lane < 8) warp_tot[lane] = w;
    }
    __syncthreads();
    const int base = wid > 0 ? warp_tot[wid - 1] : 0;
    *total = warp_tot[7];
    __syncthreads();
    return base + x - v;
}

struct MlaArgs {
    const uint16_t* q;          // [T,64,576] bf16
    const int32_t* topk;        // [T,2048]
    const uint8_t* kv;          // latent cache
    BatchDev b;
    float scale_log2;           // softmax_scale * log2(e)
    int64_t n_slots;            // T * 2048
    int G;                      // CTAs sharing the slots
    void* out;
    int out_f32;
    float* lse;
    float* part_o;              // [2G, 64, 512]: a CTA's first / last row piece
    float* part_ml;             // [2G, 64, 2]
    int32_t* row_done;          // [T] pieces finished per row (zero on entry, reset to zero)
    int32_t* st;
};

__device__ __forceinline__ int64_t mla_cta_start(int64_t g, int64_t N, int64_t G) { return g * N / G; }
__device__ __forceinline__ int64_t mla_cta_of(int64_t x, int64_t N, int64_t G) { return ((x + 1) * G + N - 1) / N - 1; }

// Partial slot of CTA g's piece of row r: 2g for the CTA's first row, 2g+1 otherwise.
__device__ __forceinline__ int64_t mla_slot(int64_t g, int64_t r, int64_t N, int64_t G) {
    return 2 * g + ((mla_cta_start(g, N, G) / kTopK == r) ? 0 : 1);
}

__global__ void __launch_bounds__(kMlaThreads, 1)
sparse_mla_kernel(MlaArgs a) {
    extern __shared__ __align__(128) uint8_t smem[];
    __half* Qs = reinterpret_cast<__half*>(smem + kOffQ);
    __half* Ks = reinterpret_cast<__half*>(smem + kOffK);
    uint8_t* Raw = smem + kOffRaw;
    __half* Ps = reinterpret_cast<__half*>(smem + kOffP);
    int64_t* slots = reinterpret_cast<int64_t*>(smem + kOffSlots);
    float* red_max = reinterpret_cast<float*>(smem + kOffRed);
    float* red_sum = red_max + 4 * 64;
    float* m_run = reinterpret_cast<float*>(smem + kOffStat);
    float* l_run = m_run + 64;
    float* alpha = l_run + 64;
    int* misc = reinterpret_cast<int*>(smem + kOffMisc);

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const BatchDev& b = a.b;
    const int64_t N = a.n_slots, G = a.G, g = blockIdx.x;
    const int64_t e_begin = mla_cta_start(g, N, G), e_end = mla_cta_start(g + 1, N, G);
    for (int64_t row = e_begin / kTopK; row * kTopK < e_end; ++row) {
    const int64_t lo_e = max(e_begin, row * kTopK) - row * kTopK;
    const int64_t hi_e = min(e_end, (row + 1) * kTopK) - row * kTopK;
    const int64_t g0 = mla_cta_of(row * kTopK, N, G), g1 = mla_cta_of(row * kTopK + kTopK - 1, N, G);
    const int r = row_request(b.q_start, b.batch, row);
    const int qn = b.q_start[r + 1] - b.q_start[r];
    const int L = b.seq_len[r];
    const int p = L - qn + (int)(row - b.q_start[r]);
    __syncthreads();                                   // shared state of the previous piece is free

    // ---- 1. collect the piece's valid entries (ordered) ------------------
    const int chunk = (int)(hi_e - lo_e);
    const int e0 = (int)lo_e;
    int ntok = 0;
    for (int base = 0; base < chunk; base += kMlaThreads * 8) {
        int64_t sl[8];
        int cnt = 0;
#pragma unroll
        for (int q = 0; q < 8; ++q) {
            const int e = base + tid * 8 + q;
            sl[q] = -1;
            if (e < chunk) {
                const int j = a.topk[row * kTopK + e0 + e];
                if (j >= 0 && j <= p) {
                    if (j >= L || j / kPage >= b.max_pages) {
                        record_error(a.st, DSA_DEVERR_INDEX_RANGE, j);
                    } else {
                        const int64_t pg = b.page_table[(int64_t)r * b.max_pages + j / kPage];
                        if (pg < 0 || pg >= b.num_pages) record_error(a.st, DSA_DEVERR_PAGE_RANGE, pg);
                        else sl[q] = pg * kPage + (j % kPage);
                    }
                }
            }
            cnt += sl[q] >= 0;
        }
        int total;
        int off = ntok + mla_block_scan(cnt, misc, &total);
#pragma unroll
        for (int q = 0; q < 8; ++q)
            if (sl[q] >= 0) slots[off++] = sl[q];
        ntok += total;
    }

    // ---- 2. Q (bf16 -> fp16) and softmax state ----------------------------
    const uint16_t* qrow = a.q + row * (64 * 576);
    for (int c = tid; c < 64 * 72; c += kMlaThreads) {          // 8 values per item
        const int h = c / 72, d = (c % 72) * 8;
        const uint4 v = *reinterpret_cast<const uint4*>(qrow + h * 576 + d);
        const uint32_t w4[4] = {v.x, v.y, v.z, v.w};
        uint32_t o[4];
#pragma unroll
        for (int i = 0; i < 4; ++i)
            o[i] = pack_half2(bf16_bits_to_f32(w4[i] & 0xffffu), bf16_bits_to_f32(w4[i] >> 16));
        *reinterpret_cast<uint4*>(Qs + h * kQS + d) = make_uint4(o[0], o[1], o[2], o[3]);
    }
    if (tid < 64) {
        m_run[tid] = -INFINITY;
        l_run[tid] = 0.f;
        alpha[tid] = 1.f;
    }
    __syncthreads();

    const int ntiles = (ntok + kTile - 1) / kTile;
    auto issue_tile = [&](int tile) {
        const int n_in = min(kTile, ntok - tile * kTile);
        for (int c = tid; c < kTile * 41; c += kMlaThreads) {
            const int tk = c / 41, part = c % 41;
            if (tk < n_in) {
                const int64_t s = slots[tile * kTile + tk];
                const uint8_t* src = a.kv + (s / kPage) * (int64_t)kKvPageBytes + (s % kPage) * kKvTokenBytes + part * 16;
                cp_async16(smem_u32(Raw + tk * kKvTokenBytes + part * 16), src);
            }
        }
        cp_async_commit();
    };
    if (ntiles > 0) issue_tile(0);

    float oacc[4][8][4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int n = 0; n < 8; ++n)
#pragma unroll
            for (int k = 0; k < 4; ++k) oacc[i][n][k] = 0.f;

    const int g8 = lane >> 2, cq = lane & 3;
    for (int tile = 0; tile < ntiles; ++tile) {
        const int n_in = min(kTile, ntok - tile * kTile);
        cp_async_wait_all();
        __syncthreads();
        // ---- dequantise the staged rows into fp16 Ks ----------------------
        for (int c = tid; c < kTile * 40; c += kMlaThreads) {
            const int tk = c / 40, part = c % 40;
            uint4 outv[2];
            if (tk >= n_in) {
                outv[0] = outv[1] = make_uint4(0, 0, 0, 0);
                if (part < 32) {
                    *reinterpret_cast<uint4*>(Ks + tk * kQS + part * 16) = outv[0];
                    *reinterpret_cast<uint4*>(Ks + tk * kQS + part * 16 + 8) = outv[1];
                } else {
                    *reinterpret_cast<uint4*>(Ks + tk * kQS + 512 + (part - 32) * 8) = outv[0];
                }
                continue;
            }
            const uint8_t* rw = Raw + tk * kKvTokenBytes;
            if (part < 32) {
                const float sc = reinterpret_cast<const float*>(rw + 512)[part >> 3];
                if (sc < 0x1p-15f || sc > 0x1p7f) record_error(a.st, DSA_DEVERR_FP16_RANGE, part);
                const uint4 v = *reinterpret_cast<const uint4*>(rw + part * 16);
                const uint32_t w4[4] = {v.x, v.y, v.z, v.w};
                uint32_t o[8];
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const float2 f0 = e4m3x2_to_f32x2((uint16_t)(w4[i] & 0xffffu));
                    const float2 f1 = e4m3x2_to_f32x2((uint16_t)(w4[i] >> 16));
                    o[2 * i] = pack_half2(f0.x * sc, f0.y * sc);
                    o[2 * i + 1] = pack_half2(f1.x * sc, f1.y * sc);
                }
                *reinterpret_cast<uint4*>(Ks + tk * kQS + part * 16) = make_uint4(o[0], o[1], o[2], o[3]);
                *reinterpret_cast<uint4*>(Ks + tk * kQS + part * 16 + 8) = make_uint4(o[4], o[5], o[6], o[7]);
            } else {
                const uint4 v = *reinterpret_cast<const uint4*>(rw + 528 + (part - 32) * 16);
                const uint32_t w4[4] = {v.x, v.y, v.z, v.w};
                uint32_t o[4];
#pragma unroll
                for (int i = 0; i < 4; ++i)
                    o[i] = pack_half2(bf16_bits_to_f32(w4[i] & 0xffffu), bf16_bits_to_f32(w4[i] >> 16));
                *reinterpret_cast<uint4*>(Ks + tk * kQS + 512 + (part - 32) * 8) = make_uint4(o[0], o[1], o[2], o[3]);
            }
        }
        __syncthreads();
        if (tile + 1 < ntiles) issue_tile(tile + 1);     // staging buffer is free again

        // ---- S^T = K Q^T: warp -> tokens 16*(warp&3).., heads 32*(warp>>2).. ----
        const int mt = warp & 3, nh = warp >> 2;
        float sacc[4][4];
#pragma unroll
        for (int n = 0; n < 4; ++n)
#pragma unroll
            for (int k = 0; k < 4; ++k) sacc[n][k] = 0.f;
        {
            const uint32_t a_base = smem_u32(Ks + (mt * 16 + (lane & 7) + ((lane >> 3) & 1) * 8) * kQS + (lane >> 4) * 8);
            const uint32_t b_base0 = smem_u32(Qs + (nh * 32 + (lane & 7) + (lane >> 4) * 8) * kQS + ((lane >> 3) & 1) * 8);
            const uint32_t b_base1 = b_base0 + 16 * kQS * 2;
#pragma unroll 4
            for (int ks = 0; ks < 36; ++ks) {
                uint32_t a0, a1, a2, a3, b0, b1, b2, b3, c0, c1, c2, c3;
                ldsm_x4(a_base + ks * 32, a0, a1, a2, a3);
                ldsm_x4(b_base0 + ks * 32, b0, b1, b2, b3);
                ldsm_x4(b_base1 + ks * 32, c0, c1, c2, c3);
                mma16816(sacc[0], a0, a1, a2, a3, b0, b1);
                mma16816(sacc[1], a0, a1, a2, a3, b2, b3);
                mma16816(sacc[2], a0, a1, a2, a3, c0, c1);
                mma16816(sacc[3], a0, a1, a2, a3, c2, c3);
            }
        }
        // ---- online softmax over the tile (columns = heads) -----------------
        const int tok0 = mt * 16 + g8, tok1 = tok0 + 8;
        const bool v0 = tok0 < n_in, v1 = tok1 < n_in;
#pragma unroll
        for (int n = 0; n < 4; ++n) {
            sacc[n][0] = v0 ? sacc[n][0] * a.scale_log2 : -INFINITY;
            sacc[n][1] = v0 ? sacc[n][1] * a.scale_log2 : -INFINITY;
            sacc[n][2] = v1 ? sacc[n][2] * a.scale_log2 : -INFINITY;
            sacc[n][3] = v1 ? sacc[n][3] * a.scale_log2 : -INFINITY;
            float m0 = fmaxf(sacc[n][0], sacc[n][2]), m1 = fmaxf(sacc[n][1], sacc[n][3]);
#pragma unroll
            for (int o = 4; o < 32; o <<= 1) {
                m0 = fmaxf(m0, __shfl_xor_sync(0xffffffffu, m0, o));
                m1 = fmaxf(m1, __shfl_xor_sync(0xffffffffu, m1, o));
            }
            if (g8 == 0) {
                red_max[mt * 64 + nh * 32 + n * 8 + 2 * cq] = m0;
                red_max[mt * 64 + nh * 32 + n * 8 + 2 * cq + 1] = m1;
            }
        }
        __syncthreads();
        if (tid < 64) {
            const float tm = fmaxf(fmaxf(red_max[tid], red_max[64 + tid]), fmaxf(red_max[128 + tid], red_max[192 + tid]));
            const float mo = m_run[tid];
            const float mn = fmaxf(mo, tm);
            alpha[tid] = (mn == -INFINITY) ? 1.f : exp2f(mo - mn);
            m_run[tid] = mn;
        }
        __syncthreads();
#pragma unroll
        for (int n = 0; n < 4; ++n) {
            const int h0 = nh * 32 + n * 8 + 2 * cq;
            const float mh0 = m_run[h0], mh1 = m_run[h0 + 1];
            const float p0 = (mh0 == -INFINITY) ? 0.f : exp2f(sacc[n][0] - mh0);
            const float p1 = (mh1 == -INFINITY) ? 0.f : exp2f(sacc[n][1] - mh1);
            const float p2 = (mh0 == -INFINITY) ? 0.f : exp2f(sacc[n][2] - mh0);
            const float p3 = (mh1 == -INFINITY) ? 0.f : exp2f(sacc[n][3] - mh1);
            Ps[h0 * kPS + tok0] = __float2half_rn(p0);
            Ps[(h0 + 1) * kPS + tok0] = __float2half_rn(p1);
            Ps[h0 * kPS + tok1] = __float2half_rn(p2);
            Ps[(h0 + 1) * kPS + tok1] = __float2half_rn(p3);
            float s0 = p0 + p2, s1 = p1 + p3;
#pragma unroll
            for (int o = 4; o < 32; o <<= 1) {
                s0 += __shfl_xor_sync(0xffffffffu, s0, o);
                s1 += __shfl_xor_sync(0xffffffffu, s1, o);
            }
            if (g8 == 0) {
                red_sum[mt * 64 + h0] = s0;
                red_sum[mt * 64 + h0 + 1] = s1;
            }
        }
        __syncthreads();
        if (tid < 64)
            l_run[tid] = l_run[tid] * alpha[tid] + red_sum[tid] + red_sum[64 + tid] + red_sum[128 + tid] + red_sum[192 + tid];

        // ---- O^T = alpha * O^T + V^T P^T: warp -> latent dims 64*warp.. -------
#pragma unroll
        for (int n = 0; n < 8; ++n) {
            const float al0 = alpha[n * 8 + 2 * cq], al1 = alpha[n * 8 + 2 * cq + 1];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                oacc[i][n][0] *= al0;
                oacc[i][n][1] *= al1;
                oacc[i][n][2] *= al0;
                oacc[i][n][3] *= al1;
            }
        }
        {
            const uint32_t a_base = smem_u32(Ks + ((lane & 7) + (lane >> 4) * 8) * kQS + warp * 64 + ((lane >> 3) & 1) * 8);
            const uint32_t b_base = smem_u32(Ps + ((lane & 7) + (lane >> 4) * 8) * kPS + ((lane >> 3) & 1) * 8);
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
                uint32_t af[4][4];
#pragma unroll
                for (int i = 0; i < 4; ++i)
                    ldsm_x4_t(a_base + (kk * 16 * kQS + i * 16) * 2, af[i][0], af[i][1], af[i][2], af[i][3]);
#pragma unroll
                for (int np = 0; np < 4; ++np) {
                    uint32_t b0, b1, b2, b3;
                    ldsm_x4(b_base + (np * 16 * kPS + kk * 16) * 2, b0, b1, b2, b3);
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        mma16816(oacc[i][2 * np], af[i][0], af[i][1], af[i][2], af[i][3], b0, b1);
                        mma16816(oacc[i][2 * np + 1], af[i][0], af[i][1], af[i][2], af[i][3], b2, b3);
                    }
                }
            }
        }
        __syncthreads();    // Ks / Ps are rewritten by the next tile
    }

    // ---- 3. write the result ---------------------------------------------
    __syncthreads();
    if (g0 == g1) {
#pragma unroll
        for (int n = 0; n < 8; ++n) {
            const int h0 = n * 8 + 2 * cq;
            const float l0 = l_run[h0], l1 = l_run[h0 + 1];
            const float i0 = l0 > 0.f ? 1.f / l0 : 0.f, i1 = l1 > 0.f ? 1.f / l1 : 0.f;
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int d0 = warp * 64 + i * 16 + g8, d1 = d0 + 8;
                const int64_t o00 = (row * 64 + h0) * 512, o01 = (row * 64 + h0 + 1) * 512;
                const float v00 = oacc[i][n][0] * i0, v01 = oacc[i][n][1] * i1;
                const float v10 = oacc[i][n][2] * i0, v11 = oacc[i][n][3] * i1;
                if (a.out_f32) {
                    float* o = static_cast<float*>(a.out);
                    o[o00 + d0] = v00; o[o01 + d0] = v01; o[o00 + d1] = v10; o[o01 + d1] = v11;
                } else {
                    __nv_bfloat16* o = static_cast<__nv_bfloat16*>(a.out);
                    o[o00 + d0] = __float2bfloat16_rn(v00); o[o01 + d0] = __float2bfloat16_rn(v01);
                    o[o00 + d1] = __float2bfloat16_rn(v10); o[o01 + d1] = __float2bfloat16_rn(v11);
                }
            }
        }
        if (a.lse && tid < 64) {
            const float l = l_run[tid];
            a.lse[row * 64 + tid] = l > 0.f ? (m_run[tid] + log2f(l)) * 0.69314718055994531f : -INFINITY;
        }
        continue;
    }
    // several CTAs share the row: write this piece's partial
    {
        const int64_t unit = mla_slot(g, row, N, G);
        float* po = a.part_o + unit * 64 * 512;
#pragma unroll
        for (int n = 0; n < 8; ++n) {
            const int h0 = n * 8 + 2 * cq;
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int d0 = warp * 64 + i * 16 + g8, d1 = d0 + 8;
                po[h0 * 512 + d0] = oacc[i][n][0];
                po[(h0 + 1) * 512 + d0] = oacc[i][n][1];
                po[h0 * 512 + d1] = oacc[i][n][2];
                po[(h0 + 1) * 512 + d1] = oacc[i][n][3];
            }
        }
        if (tid < 64) {
            a.part_ml[(unit * 64 + tid) * 2] = m_run[tid];
            a.part_ml[(unit * 64 + tid) * 2 + 1] = l_run[tid];
        }
    }
    __threadfence();
    __syncthreads();
    if (tid == 0) misc[8] = (atomicAdd(&a.row_done[row], 1) == (int)(g1 - g0)) ? 1 : 0;
    __syncthreads();
    if (misc[8]) {
        // last piece of the row: combine all partials by log-sum-exp
        __threadfence();
        for (int h = warp; h < 64; h += 8) {
            float M = -INFINITY;
            for (int64_t gg = g0; gg <= g1; ++gg) {
                const int64_t u = mla_slot(gg, row, N, G);
                const float m = __ldcg(&a.part_ml[(u * 64 + h) * 2]), l = __ldcg(&a.part_ml[(u * 64 + h) * 2 + 1]);
                if (l > 0.f) M = fmaxf(M, m);
            }
            float acc[16];
#pragma unroll
            for (int j = 0; j < 16; ++j) acc[j] = 0.f;
            float Ltot = 0.f;
            for (int64_t gg = g0; gg <= g1; ++gg) {
                const int64_t u = mla_slot(gg, row, N, G);
                const float m = __ldcg(&a.part_ml[(u * 64 + h) * 2]), l = __ldcg(&a.part_ml[(u * 64 + h) * 2 + 1]);
                if (!(l > 0.f)) continue;
                const float wgt = exp2f(m - M);
                Ltot += wgt * l;
                const float4* src = reinterpret_cast<const float4*>(a.part_o + (u * 64 + h) * 512) + lane;
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const float4 v = __ldcg(src + j * 32);
                    acc[4 * j] += wgt * v.x; acc[4 * j + 1] += wgt * v.y;
                    acc[4 * j + 2] += wgt * v.z; acc[4 * j + 3] += wgt * v.w;
                }
            }
            const float inv = Ltot > 0.f ? 1.f / Ltot : 0.f;
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int64_t o = (row * 64 + h) * 512 + (lane + j * 32) * 4;
                if (a.out_f32) {
                    reinterpret_cast<float4*>(static_cast<float*>(a.out) + o)[0] =
                        make_float4(acc[4 * j] * inv, acc[4 * j + 1] * inv, acc[4 * j + 2] * inv, acc[4 * j + 3] * inv);
                } else {
                    __nv_bfloat16* ob = static_cast<__nv_bfloat16*>(a.out) + o;
                    ob[0] = __float2bfloat16_rn(acc[4 * j] * inv); ob[1] = __float2bfloat16_rn(acc[4 * j + 1] * inv);
                    ob[2] = __float2bfloat16_rn(acc[4 * j + 2] * inv); ob[3] = __float2bfloat16_rn(acc[4 * j + 3] * inv);
                }
            }
            if (a.lse && lane == 0)
                a.lse[row * 64 + h] = Ltot > 0.f ? (M + log2f(Ltot)) * 0.69314718055994531f : -INFINITY;
        }
        if (tid == 0) a.row_done[row] = 0;             // ready for the next call
    }
    }   // row pieces
}

// CTAs sharing the T x 2048 slots: at most one per SM, and at least 256 slots
// (four 64-token tiles) per CTA.
inline int mla_ctas(int64_t total_q, int sms) {
    const int64_t n = total_q * kTopK;
    int64_t gcount = n / 256;
    if (gcount < 1) gcount = 1;
    if (gcount > sms) gcount = sms;
    return (int)gcount;
}

// Workspace: partials for two row pieces per CTA, their (max, sum), and the
// per-row counters.
inline size_t mla_ws_bytes(int64_t total_q, int G) {
    size_t b = (size_t)2 * G * 64 * 512 * 4 + (size_t)2 * G * 64 * 2 * 4;
    b = (b + 255) / 256 * 256;
    return b + (size_t)total_q * 4;
}

int device_sm_count() {
    int dev = 0, sms = 148;
    if (cudaGetDevice(&dev) == cudaSuccess) cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    return sms > 1024 ? 1024 : sms;
}

dsa_status sparse_mla_launch(const void* q, const int32_t* topk, const dsa_topk_share* share,
                             const uint8_t* kv, const dsa_batch* b, float softmax_scale, void* out,
                             int32_t out_dtype, float* lse, void* ws, size_t ws_bytes, int32_t* st,
                             void* stream, bool decode);

}  // namespace dsa

using namespace dsa;

extern "C" dsa_status dsa_topk_share_get(const dsa_topk_share* s, const int32_t** topk, int64_t* rows,
                                         int32_t* layer_id);

dsa_status dsa::sparse_mla_launch(const void* q, const int32_t* topk, const dsa_topk_share* share,
                                  const uint8_t* kv, const dsa_batch* b, float softmax_scale, void* out,
                                  int32_t out_dtype, float* lse, void* ws, size_t ws_bytes, int32_t* st,
                                  void* stream, bool decode) {
    dsa_status vs = validate_batch(b);
    if (vs != DSA_OK) return vs;
    if (!q || !kv || !out) return DSA_ERR_INVALID_ARGUMENT;
    if (out_dtype != DSA_DTYPE_BF16 && out_dtype != DSA_DTYPE_F32) return DSA_ERR_INVALID_ARGUMENT;
    if (!(softmax_scale > 0.f)) return DSA_ERR_INVALID_ARGUMENT;
    if (!topk) {
        if (!share) return DSA_ERR_INVALID_ARGUMENT;
        int64_t rows = 0;
        dsa_status gs = dsa_topk_share_get(share, &topk, &rows, nullptr);
        if (gs != DSA_OK) return gs;
        if (rows != b->total_q) return DSA_ERR_INVALID_ARGUMENT;
    }
    if (!aligned16(q) || !aligned16(kv) || !aligned16(out) || !aligned16(topk)) return DSA_ERR_ALIGNMENT;
    if (b->total_q == 0) return DSA_OK;
    (void)decode;
    const int G = mla_ctas(b->total_q, device_sm_count());
    if (!ws) return DSA_ERR_INVALID_ARGUMENT;
    if (ws_bytes < mla_ws_bytes(b->total_q, G)) return DSA_ERR_WORKSPACE_TOO_SMALL;
    if (!aligned16(ws)) return DSA_ERR_ALIGNMENT;
    if (b->total_q > 0x3fffffffLL / 2048) return DSA_ERR_UNSUPPORTED;
    static bool attr_set = false;
    if (!attr_set) {
        if (cudaFuncSetAttribute(sparse_mla_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kMlaSmem) !=
            cudaSuccess)
            return DSA_ERR_CUDA;
        attr_set = true;
    }
    MlaArgs a;
    a.q = static_cast<const uint16_t*>(q);
    a.topk = topk;
    a.kv = kv;
    a.b = to_dev(b);
    a.scale_log2 = softmax_scale * 1.4426950408889634f;
    a.n_slots = b->total_q * kTopK;
    a.G = G;
    a.out = out;
    a.out_f32 = out_dtype == DSA_DTYPE_F32;
    a.lse = lse;
    a.part_o = static_cast<float*>(ws);
    a.part_ml = a.part_o + (size_t)2 * G * 64 * 512;
    const size_t cnt_off = ((size_t)2 * G * 64 * 512 * 4 + (size_t)2 * G * 64 * 2 * 4 + 255) / 256 * 256;
    a.row_done = reinterpret_cast<int32_t*>(static_cast<uint8_t*>(ws) + cnt_off);
    a.st = st;
    cudaStream_t s = as_stream(stream);
    if (cudaMemsetAsync(a.row_done, 0, (size_t)b->total_q * 4, s) != cudaSuccess) return DSA_ERR_CUDA;
    sparse_mla_kernel<<<(unsigned)G, kMlaThreads, kMlaSmem, s>>>(a);
    DSA_CHECK_LAUNCH();
    return DSA_OK;
}

extern "C" dsa_status dsa_sparse_mla_workspace_size(const dsa_batch* b, size_t* bytes) {
    dsa_status vs = validate_batch(b);
    if (vs != DSA_OK) return vs;
    if (!bytes) return DSA_ERR_INVALID_ARGUMENT;
    // Enough for any GPU of up to 1024 SMs.
    *bytes = mla_ws_bytes(b->total_q, mla_ctas(b->total_q, 1024));
    return DSA_OK;
}

extern "C" dsa_status dsa_sparse_mla_decode(const void* q, const int32_t* topk, const dsa_topk_share* share,
                                            const uint8_t* kv_cache, const dsa_batch* b, float softmax_scale,
                                            void* out, int32_t out_dtype, float* lse, void* ws,
                                            size_t ws_bytes, int32_t* dev_status, void* stream) {
    return sparse_mla_launch(q, topk, share, kv_cache, b, softmax_scale, out, out_dtype, lse, ws, ws_bytes,
                             dev_status, stream, true);
}

extern "C" dsa_status dsa_sparse_mla_prefill(const void* q, const int32_t* topk, const dsa_topk_share* share,
                                             const uint8_t* kv_cache, const dsa_batch* b, float softmax_scale,
                                             void* out, int32_t out_dtype, float* lse, void* ws,
                                             size_t ws_bytes, int32_t* dev_status, void* stream) {
    return sparse_mla_launch(q, topk, share, kv_cache, b, softmax_scale, out, out_dtype, lse, ws, ws_bytes,
                             dev_status, stream, false);
}
