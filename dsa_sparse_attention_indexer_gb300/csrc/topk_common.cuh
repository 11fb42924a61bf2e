// Block-wide top-2048 of one fp32 score row (device code shared by the
// standalone top-k kernel and the multi-token indexer), "vLLM 推理链路概览",
// DSA Indexer: I_i = TopK_{j,2048}(s_ij), ties to the lower position.
//
// Two reads of the row, with float4 loads several in flight per thread:
//   1. a 4096-bin histogram of the top 12 key bits; the bin b* that holds the
//      2048th largest key and the count A of keys above it;
//   2. keys above b* go straight to the selection (exactly A of them), keys in
//      b* to a shared-memory boundary buffer.
// The remaining 2048 - A are selected exactly inside b* (radix passes on the
// low 20 bits, ties -> lower position).  The selected positions are written in
// ascending order from a bitmap of the row and its popcount prefix.  Rows
// whose boundary bin overflows the buffer select inside b* straight from the
// row; rows longer than the bitmap sort the 2048 by position instead.
#pragma once
#include "dsa_internal.cuh"
#include "select_common.cuh"

namespace dsa {

constexpr int kSelThreads = 1024;
constexpr int kSelBndCap = 16384;                                 // boundary entries in shared memory
constexpr int kSelOffHist = 0;                                    // 4096 bins
constexpr int kSelOffPos = kSelOffHist + 4096 * 4;                // selected positions [2048]
constexpr int kSelOffKey = kSelOffPos + 2048 * 4;                 // selected keys [2048]
constexpr int kSelOffChunk = kSelOffKey + 2048 * 4;               // [1024] chunk prefix
constexpr int kSelOffBndKey = kSelOffChunk + 1024 * 4;            // boundary keys, later the bitmap
constexpr int kSelOffBndPos = kSelOffBndKey + kSelBndCap * 4;
constexpr int kSelOffMisc = kSelOffBndPos + kSelBndCap * 4;
constexpr int kSelSmem = kSelOffMisc + 256;                       // dynamic shared memory per CTA
constexpr int64_t kSelBitmapRows = (int64_t)kSelBndCap * 64;      // positions the bitmap covers (2^20)

struct SelMisc {
    int32_t n_sure, n_bnd, n_sel;
    sel::Found found;
    int32_t scratch[32];
};
static_assert(sizeof(SelMisc) <= 256, "select misc block");

// Positions 0..n-1 of a score row, in uniform rounds (every thread makes the
// same number of calls, so f may use warp votes): f(active, key, position).
// float4 loads, four in flight per thread, when the row is 16-byte aligned.
struct SelRow {
    const float* row;
    int64_t n;
    template <class F>
    __device__ __forceinline__ void visit(int gt, F&& f) const {
        constexpr int U = 4;
        const bool vec = (reinterpret_cast<uintptr_t>(row) & 15) == 0;
        const int64_t nv = vec ? n / 4 : 0;
        const float4* r4 = reinterpret_cast<const float4*>(row);
        for (int64_t base = 0; base < nv; base += (int64_t)kSelThreads * U) {
            float4 x[U];
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int64_t v = base + u * kSelThreads + gt;
                x[u] = v < nv ? __ldg(r4 + v) : make_float4(0.f, 0.f, 0.f, 0.f);
            }
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int64_t v = base + u * kSelThreads + gt;
                const bool a = v < nv;
                f(a, score_key(x[u].x), (int32_t)(4 * v));
                f(a, score_key(x[u].y), (int32_t)(4 * v + 1));
                f(a, score_key(x[u].z), (int32_t)(4 * v + 2));
                f(a, score_key(x[u].w), (int32_t)(4 * v + 3));
            }
        }
        for (int64_t base = 4 * nv; base < n; base += kSelThreads) {
            const int64_t j = base + gt;
            const bool a = j < n;
            f(a, a ? score_key(__ldg(row + j)) : 0u, (int32_t)j);
        }
    }
};

// The keys of one bin of a row, as a selection source.
struct SelRowBin {
    SelRow r;
    uint32_t bin;
    template <class F>
    __device__ __forceinline__ void visit(int gt, F&& f) const {
        r.visit(gt, [&](bool a, uint32_t k, int32_t j) { f(a && (k >> 20) == bin, k, j); });
    }
};

// Appends (key, pos) of the lanes with `take` at warp-aggregated slots of a
// shared-memory list with counter *ctr; slots from cap on are dropped.  Every
// lane of the warp calls it.
__device__ __forceinline__ void warp_append(bool take, uint32_t key, int32_t pos, int32_t* ctr, uint32_t* keys,
                                            int32_t* poss, int cap) {
    const uint32_t m = __ballot_sync(0xffffffffu, take);
    if (m == 0u) return;
    const int lane = threadIdx.x & 31, leader = __ffs(m) - 1;
    int base = 0;
    if (lane == leader) base = atomicAdd(ctr, __popc(m));
    base = __shfl_sync(0xffffffffu, base, leader);
    if (take) {
        const int i = base + __popc(m & ((1u << lane) - 1u));
        if (i < cap) {
            keys[i] = key;
            poss[i] = pos;
        }
    }
}

// The top-2048 positions of the n visible scores of `row` into out[2048] in
// ascending position order, -1 padded; out_scores (optional) gets their scores.
// A row of at most 2048 takes every position.  The whole CTA (kSelThreads
// threads) calls it; smem: kSelSmem bytes, 16-byte aligned.
inline __device__ void select_topk_row(const float* __restrict__ row, int64_t n, int32_t* __restrict__ out,
                                float* __restrict__ out_scores, uint8_t* smem) {
    constexpr int NT = kSelThreads;
    const int t = threadIdx.x;
    if (n <= kTopK) {
        for (int i = t; i < kTopK; i += NT) {
            out[i] = i < n ? i : -1;
            if (out_scores) out_scores[i] = 0.f;
        }
        return;
    }
    uint32_t* hist = reinterpret_cast<uint32_t*>(smem + kSelOffHist);
    int32_t* sel_pos = reinterpret_cast<int32_t*>(smem + kSelOffPos);
    uint32_t* sel_key = reinterpret_cast<uint32_t*>(smem + kSelOffKey);
    int32_t* chunk = reinterpret_cast<int32_t*>(smem + kSelOffChunk);
    uint32_t* bnd_key = reinterpret_cast<uint32_t*>(smem + kSelOffBndKey);
    int32_t* bnd_pos = reinterpret_cast<int32_t*>(smem + kSelOffBndPos);
    SelMisc* mm = reinterpret_cast<SelMisc*>(smem + kSelOffMisc);
    const SelRow src{row, n};
    // ---- 1. histogram of the top 12 key bits, and the bin of the 2048th key
    for (int i = t; i < 4096; i += NT) hist[i] = 0u;
    if (t == 0) {
        mm->n_sure = 0;
        mm->n_bnd = 0;
    }
    __syncthreads();
    src.visit(t, [&](bool a, uint32_t k, int32_t) {
        if (a) atomicAdd(&hist[k >> 20], 1u);
    });
    __syncthreads();
    {
        uint32_t c[4];
        int mine = 0;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            c[q] = hist[4095 - (t * 4 + q)];
            mine += (int)c[q];
        }
        int tot;
        int above = sel::excl_scan<NT, 0>(mine, t, mm->scratch, &tot);
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            if (above < kTopK && above + (int)c[q] >= kTopK) {
                mm->found.bin = (uint32_t)(4095 - (t * 4 + q));
                mm->found.above = above;
            }
            above += (int)c[q];
        }
        __syncthreads();
    }
    const uint32_t b1 = mm->found.bin;
    // ---- 2. keys above b1 join the selection; keys in b1 go to the boundary buffer
    src.visit(t, [&](bool a, uint32_t k, int32_t j) {
        const uint32_t bin = k >> 20;
        warp_append(a && bin > b1, k, j, &mm->n_sure, sel_key, sel_pos, kTopK);
        warp_append(a && bin == b1, k, j, &mm->n_bnd, bnd_key, bnd_pos, kSelBndCap);
    });
    __syncthreads();
    const int n_sure = min(mm->n_sure, kTopK), n_bnd = mm->n_bnd;
    const int need = kTopK - n_sure;
    int ns = n_sure;
    if (need > 0 && n_bnd <= need) {                             // the whole bin is in
        for (int i = t; i < n_bnd; i += NT) {
            sel_pos[n_sure + i] = bnd_pos[i];
            sel_key[n_sure + i] = bnd_key[i];
        }
        ns = n_sure + n_bnd;
        __syncthreads();
    } else if (need > 0) {                                       // the rest exactly, inside b1
        if (t == 0) mm->n_sel = n_sure;
        __syncthreads();
        if (n_bnd <= kSelBndCap) {
            const sel::SmemSrc<NT> bs{bnd_key, bnd_pos, n_bnd};
            const sel::Threshold th = sel::topk_threshold<NT, 0>(bs, need, t, hist, mm->scratch, &mm->found, 1, b1);
            for (int i = t; i < n_bnd; i += NT) {
                if (th.keep(bnd_key[i], bnd_pos[i])) {
                    const int jj = atomicAdd(&mm->n_sel, 1);
                    if (jj < kTopK) {
                        sel_pos[jj] = bnd_pos[i];
                        sel_key[jj] = bnd_key[i];
                    }
                }
            }
        } else {                                                 // bin too large for shared memory
            const SelRowBin bs{src, b1};
            const sel::Threshold th = sel::topk_threshold<NT, 0>(bs, need, t, hist, mm->scratch, &mm->found, 1, b1);
            bs.visit(t, [&](bool a, uint32_t k, int32_t j) {
                warp_append(a && th.keep(k, j), k, j, &mm->n_sel, sel_key, sel_pos, kTopK);
            });
        }
        __syncthreads();
        ns = min(mm->n_sel, kTopK);
    }
    // ---- 3. ascending positions
    if (n <= kSelBitmapRows) {                                   // the boundary buffers, free now, hold its bitmap
        sel::write_ranked<NT>(sel_pos, sel_key, ns, n, bnd_key, chunk, reinterpret_cast<uint16_t*>(hist), mm->scratch,
                              out, out_scores, t);
        return;
    }
    for (int i = ns + t; i < kTopK; i += NT) {
        sel_pos[i] = 0x7fffffff;
        sel_key[i] = 0u;
    }
    __syncthreads();
    sel::bitonic_sort_by_pos<NT, 0>(sel_pos, sel_key, kTopK, t);
    for (int i = t; i < kTopK; i += NT) {
        const bool h = i < ns;
        out[i] = h ? sel_pos[i] : -1;
        if (out_scores) out_scores[i] = h ? key_score(sel_key[i]) : 0.f;
    }
}

}  // namespace dsa
