// Block-wide radix top-2048 of one row of keys (device code shared by the
// standalone top-k kernel and the indexer kernels).
#pragma once
#include "dsa_internal.cuh"

namespace dsa {

constexpr int kSelThreads = 1024;
constexpr int kSelWarps = kSelThreads / 32;

struct SelectSmem {
    uint32_t hist[2048];
    int32_t warp_tot[kSelWarps];
    int32_t warp_tot2[kSelWarps];
    uint32_t found_bin;
    int32_t found_above;
};

// Exclusive scan of one int per thread over the CTA; *total gets the sum.
__device__ __forceinline__ int block_exclusive_scan(int v, int32_t* warp_tot, int* total) {
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
        int w = (lane < kSelWarps) ? warp_tot[lane] : 0;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, w, o);
            if (lane >= o) w += y;
        }
        if (lane < kSelWarps) warp_tot[lane] = w;
    }
    __syncthreads();
    const int base = (wid > 0) ? warp_tot[wid - 1] : 0;
    *total = warp_tot[kSelWarps - 1];
    __syncthreads();
    return base + x - v;
}

// Histogram atomics with same-bin lanes of a warp folded into one add.
__device__ __forceinline__ void hist_add(uint32_t* hist, uint32_t bin, bool active) {
    const unsigned m = __ballot_sync(0xffffffffu, active);
    if (!active) return;
    const unsigned peers = __match_any_sync(m, bin);
    const int leader = __ffs(peers) - 1;
    if ((threadIdx.x & 31) == leader) atomicAdd(&hist[bin], (uint32_t)__popc(peers));
}

// Find bin b (counting from the top) where the running count crosses k_rem:
// count(bins > b) < k_rem <= count(bins >= b).  nbins is 1024 or 2048.
__device__ __forceinline__ void find_crossing_bin(SelectSmem& sm, int nbins, int k_rem) {
    const int per = nbins / kSelThreads;              // 1 or 2 bins per thread
    const int t = threadIdx.x;
    uint32_t c[2] = {0, 0};
    for (int q = 0; q < per; ++q) c[q] = sm.hist[nbins - 1 - (t * per + q)];
    int total;
    int above = block_exclusive_scan((int)(c[0] + c[1]), sm.warp_tot, &total);
    for (int q = 0; q < per; ++q) {
        const int b = nbins - 1 - (t * per + q);
        if (above < k_rem && above + (int)c[q] >= k_rem) {
            sm.found_bin = (uint32_t)b;
            sm.found_above = above;
        }
        above += (int)c[q];
    }
    __syncthreads();
}

// Select the top-2048 positions of keys src.key(0..n-1) into out[2048] in
// ascending position order, -1 padded.  Optionally writes the selected
// scores (src.score) into out_scores.  All threads of the CTA must call it.
template <typename Src>
__device__ void select_topk_row(const Src& src, int64_t n, int32_t* __restrict__ out,
                                float* __restrict__ out_scores, SelectSmem& sm) {
    const int t = threadIdx.x;
    if (n <= kTopK) {
        for (int i = t; i < kTopK; i += kSelThreads) {        // context fits: take all
            out[i] = (i < n) ? i : -1;
            if (out_scores) out_scores[i] = 0.0f;
        }
        return;
    }
    uint32_t prefix = 0, pmask = 0;
    int k_rem = kTopK;
    const int shifts[3] = {21, 10, 0};
    const int bits[3] = {11, 11, 10};
#pragma unroll 1
    for (int pass = 0; pass < 3; ++pass) {
        const int nb = 1 << bits[pass];
        for (int i = t; i < 2048; i += kSelThreads) sm.hist[i] = 0;
        __syncthreads();
        const int64_t n_round = (n + kSelThreads - 1) / kSelThreads * kSelThreads;
        for (int64_t j = t; j < n_round; j += kSelThreads) {
            uint32_t k = 0;
            bool act = false;
            if (j < n) {
                k = src.key(j);
                act = (k & pmask) == prefix;
            }
            hist_add(sm.hist, (k >> shifts[pass]) & (uint32_t)(nb - 1), act);
        }
        __syncthreads();
        find_crossing_bin(sm, nb, k_rem);
        prefix |= sm.found_bin << shifts[pass];
        pmask |= (uint32_t)(nb - 1) << shifts[pass];
        k_rem -= sm.found_above;
        __syncthreads();
    }
    const uint32_t kth = prefix;      // the 2048th largest key
    const int need_eq = k_rem;        // keys == kth to keep, lowest positions first
    // Ordered compaction: 4 consecutive positions per thread per round.
    constexpr int kItems = 4;
    int eq_seen = 0, out_pos = 0;
    for (int64_t base = 0; base < n; base += (int64_t)kSelThreads * kItems) {
        uint32_t keys[kItems];
        int n_eq = 0;
#pragma unroll
        for (int q = 0; q < kItems; ++q) {
            const int64_t j = base + (int64_t)t * kItems + q;
            keys[q] = (j < n) ? src.key(j) : 0u;
            n_eq += (j < n && keys[q] == kth) ? 1 : 0;
        }
        int tot_eq;
        int eq_rank = eq_seen + block_exclusive_scan(n_eq, sm.warp_tot, &tot_eq);
        bool sel[kItems];
        int n_sel = 0;
#pragma unroll
        for (int q = 0; q < kItems; ++q) {
            const int64_t j = base + (int64_t)t * kItems + q;
            bool s = false;
            if (j < n) {
                if (keys[q] > kth) s = true;
                else if (keys[q] == kth) { s = eq_rank < need_eq; ++eq_rank; }
            }
            sel[q] = s;
            n_sel += s ? 1 : 0;
        }
        int tot_sel;
        int pos = out_pos + block_exclusive_scan(n_sel, sm.warp_tot2, &tot_sel);
#pragma unroll
        for (int q = 0; q < kItems; ++q) {
            if (sel[q] && pos < kTopK) {
                const int64_t j = base + (int64_t)t * kItems + q;
                out[pos] = (int32_t)j;
                if (out_scores) out_scores[pos] = key_score(keys[q]);
                ++pos;
            }
        }
        eq_seen += tot_eq;
        out_pos += tot_sel;
        if (out_pos >= kTopK) break;
    }
    for (int i = out_pos + t; i < kTopK; i += kSelThreads) {   // only if keys were missing
        out[i] = -1;
        if (out_scores) out_scores[i] = 0.0f;
    }
}

}  // namespace dsa
