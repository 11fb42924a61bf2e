// Radix top-k helpers for a group of NT threads synchronised by named barrier
// BAR (0 = the whole CTA).  Keys are order-preserving uint32 score keys; the
// order is (key descending, position ascending), so ties go to the lower
// position as the indexer's selection rule requires.
#pragma once
#include "dsa_internal.cuh"

namespace dsa {
namespace sel {

template <int NT, int BAR>
__device__ __forceinline__ void gsync() {
    if constexpr (BAR == 0) {
        __syncthreads();
    } else {
        asm volatile("bar.sync %0, %1;" ::"n"(BAR), "n"(NT) : "memory");
    }
}

// Exclusive scan of one int per thread of the group (gt = group thread id).
template <int NT, int BAR>
__device__ __forceinline__ int excl_scan(int v, int gt, int* scratch, int* total) {
    constexpr int NW = NT / 32;
    const int lane = gt & 31, wid = gt >> 5;
    int x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) scratch[wid] = x;
    gsync<NT, BAR>();
    if (wid == 0) {
        int w = (lane < NW) ? scratch[lane] : 0;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, w, o);
            if (lane >= o) w += y;
        }
        if (lane < NW) scratch[lane] = w;
    }
    gsync<NT, BAR>();
    const int base = wid > 0 ? scratch[wid - 1] : 0;
    *total = scratch[NW - 1];
    gsync<NT, BAR>();
    return base + x - v;
}

// Histogram add with the same-bin lanes of a warp folded into one atomic.
// Every lane of the warp must call it (active or not).
__device__ __forceinline__ void hist_add(uint32_t* hist, uint32_t bin, bool active) {
    const unsigned m = __ballot_sync(0xffffffffu, active);
    if (!active) return;
    const unsigned peers = __match_any_sync(m, bin);
    if ((int)(threadIdx.x & 31) == __ffs(peers) - 1) atomicAdd(&hist[bin], (uint32_t)__popc(peers));
}

struct Found {
    uint32_t bin;
    int32_t above;
};

// The k-th largest key (k >= 1) among the active elements a source visits, and
// how many elements equal to it belong to the top k.  Three passes of
// 12 + 12 + 8 bits over the source.  hist: 4096 words of shared memory.
// A caller that knows every active key shares the top 12 bits `top12` passes
// pass0 = 1 and skips the first pass.
//
// Src::visit(gt, f) calls f(active, key, pos) for its elements with the same
// trip count on every thread of the group.
template <int NT, int BAR, class Src>
__device__ void radix_kth(const Src& src, int k, int gt, uint32_t* hist, int* scratch, Found* found,
                          uint32_t* kth_out, int* need_eq_out, int* n_eq_out, int pass0 = 0,
                          uint32_t top12 = 0) {
    uint32_t prefix = pass0 ? top12 << 20 : 0u, pmask = pass0 ? 0xfff00000u : 0u;
    int krem = k;
#pragma unroll 1
    for (int pass = pass0; pass < 3; ++pass) {
        const int shift = pass == 0 ? 20 : (pass == 1 ? 8 : 0);
        const int nb = pass < 2 ? 4096 : 256;
        for (int i = gt; i < nb; i += NT) hist[i] = 0;
        gsync<NT, BAR>();
        src.visit(gt, [&](bool act, uint32_t key, int32_t) {
            act = act && ((key & pmask) == prefix);
            hist_add(hist, (key >> shift) & (uint32_t)(nb - 1), act);
        });
        gsync<NT, BAR>();
        const int per = nb >= NT ? nb / NT : 1;
        int mine = 0;
        for (int q = 0; q < per; ++q) {
            const int b = nb - 1 - (gt * per + q);
            if (b >= 0) mine += (int)hist[b];
        }
        int total;
        int above = excl_scan<NT, BAR>(mine, gt, scratch, &total);
        for (int q = 0; q < per; ++q) {
            const int b = nb - 1 - (gt * per + q);
            if (b < 0) break;
            const int c = (int)hist[b];
            if (above < krem && above + c >= krem) {
                found->bin = (uint32_t)b;
                found->above = above;
            }
            above += c;
        }
        gsync<NT, BAR>();
        const uint32_t fb = found->bin;
        const int fa = found->above;
        if (pass == 2 && n_eq_out) *n_eq_out = (int)hist[fb];
        gsync<NT, BAR>();
        prefix |= fb << shift;
        pmask |= (uint32_t)(nb - 1) << shift;
        krem -= fa;
    }
    *kth_out = prefix;
    *need_eq_out = krem;
}

// Source over shared-memory arrays key[0..n), pos[0..n).
template <int NT>
struct SmemSrc {
    const uint32_t* key;
    const int32_t* pos;
    int n;
    template <class F>
    __device__ __forceinline__ void visit(int gt, F&& f) const {
        const int nr = (n + NT - 1) / NT * NT;
        for (int i = gt; i < nr; i += NT) {
            const bool a = i < n;
            f(a, a ? key[i] : 0u, a ? pos[i] : 0);
        }
    }
};

// Elements of a source whose key equals `kth`, keyed by position so that the
// largest transformed key is the lowest position.
template <class Src>
struct TieSrc {
    const Src& src;
    uint32_t kth;
    template <class F>
    __device__ __forceinline__ void visit(int gt, F&& f) const {
        src.visit(gt, [&](bool a, uint32_t key, int32_t pos) {
            f(a && key == kth, 0x7fffffffu - (uint32_t)pos, pos);
        });
    }
};

// Selection threshold of the top-k of a source: keep key > kth, or key == kth
// and pos <= pmax.
struct Threshold {
    uint32_t kth;
    int32_t pmax;
    __device__ __forceinline__ bool keep(uint32_t key, int32_t pos) const {
        return key > kth || (key == kth && pos <= pmax);
    }
};

template <int NT, int BAR, class Src>
__device__ Threshold topk_threshold(const Src& src, int k, int gt, uint32_t* hist, int* scratch, Found* found,
                                    int pass0 = 0, uint32_t top12 = 0) {
    uint32_t kth;
    int need_eq, n_eq = 0;
    radix_kth<NT, BAR>(src, k, gt, hist, scratch, found, &kth, &need_eq, &n_eq, pass0, top12);
    Threshold t{kth, 0x7fffffff};
    if (n_eq > need_eq) {
        TieSrc<Src> ts{src, kth};
        uint32_t tk;
        int ne2;
        radix_kth<NT, BAR>(ts, need_eq, gt, hist, scratch, found, &tk, &ne2, nullptr);
        t.pmax = (int32_t)(0x7fffffffu - tk);
    }
    return t;
}

// Keep the top-k of key/pos[0..*n) in place (stable); returns the threshold.
// Requires *n > k.  All NT threads call it; *n is updated.
template <int NT, int BAR>
__device__ Threshold compact_topk(uint32_t* key, int32_t* pos, int* n, int k, int gt, uint32_t* hist,
                                  int* scratch, Found* found) {
    const int cnt = *n;
    SmemSrc<NT> src{key, pos, cnt};
    const Threshold th = topk_threshold<NT, BAR>(src, k, gt, hist, scratch, found);
    int out = 0;
    for (int base = 0; base < cnt; base += NT) {
        const int i = base + gt;
        const bool have = i < cnt;
        const uint32_t kk = have ? key[i] : 0u;
        const int32_t pp = have ? pos[i] : 0;
        const bool keep = have && th.keep(kk, pp);
        int total;
        const int rank = excl_scan<NT, BAR>(keep ? 1 : 0, gt, scratch, &total);   // all reads done
        if (keep) {
            key[out + rank] = kk;
            pos[out + rank] = pp;
        }
        out += total;
        gsync<NT, BAR>();
    }
    if (gt == 0) *n = out;
    gsync<NT, BAR>();
    return th;
}

// Bitonic sort of n (a power of two) (pos, key) pairs by ascending position.
template <int NT, int BAR>
__device__ void bitonic_sort_by_pos(int32_t* pos, uint32_t* key, int n, int gt) {
    for (int size = 2; size <= n; size <<= 1) {
        for (int stride = size >> 1; stride > 0; stride >>= 1) {
            for (int i = gt; i < n / 2; i += NT) {
                const int lo = 2 * i - (i & (stride - 1));
                const int hi = lo + stride;
                const bool up = (lo & size) == 0;
                const int32_t a = pos[lo], b = pos[hi];
                if ((a > b) == up) {
                    pos[lo] = b;
                    pos[hi] = a;
                    const uint32_t t = key[lo];
                    key[lo] = key[hi];
                    key[hi] = t;
                }
            }
            gsync<NT, BAR>();
        }
    }
}

// Writes the ns selected (position, key) pairs to out / outs in ascending
// position order, then -1 (score 0) up to 2048.  Positions are distinct and
// below n_valid (<= 2^20), so the output index of p is the number of selected
// positions below p: a bitmap of the row and its popcount prefix give it
// without a sort.  Shared memory: bm, 32 * ceil(n_valid / 1024) words;
// chunk_pre, 1024 ints; sub_pre, 8192 uint16 (the in-chunk prefix of every
// 2^gsh-word sub-chunk, so a rank adds at most 3 words).  The whole CTA of
// 1024 threads calls it.
template <int NT>
__device__ void write_ranked(const int32_t* pos, const uint32_t* key, int ns, int64_t n_valid, uint32_t* bm,
                             int32_t* chunk_pre, uint16_t* sub_pre, int* scratch, int32_t* out, float* outs,
                             int gt) {
    static_assert(NT == 1024, "one 32-word chunk prefix per thread");
    const int nwords = (int)((n_valid + 31) >> 5);
    const int nchunks = (nwords + 31) >> 5;                         // <= 1024
    for (int w = gt; w < nchunks * 32; w += NT) bm[w] = 0u;
    __syncthreads();
    for (int i = gt; i < ns; i += NT) atomicOr(&bm[pos[i] >> 5], 1u << (pos[i] & 31));
    __syncthreads();
    int gsh = 0;
    while ((nwords >> gsh) > 8192) ++gsh;                            // <= 2
    const int lane = gt & 31, wid = gt >> 5;
    for (int c = wid; c < nchunks; c += NT / 32) {                  // a warp counts a chunk, a lane a word
        const int pc = __popc(bm[c * 32 + lane]);
        int x = pc;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, x, o);
            if (lane >= o) x += y;
        }
        if ((lane & ((1 << gsh) - 1)) == 0) sub_pre[(c * 32 + lane) >> gsh] = (uint16_t)(x - pc);
        if (lane == 31) chunk_pre[c] = x;
    }
    __syncthreads();
    const int ccount = gt < nchunks ? chunk_pre[gt] : 0;
    int total;
    const int cpre = excl_scan<NT, 0>(ccount, gt, scratch, &total);   // every read is done
    if (gt < nchunks) chunk_pre[gt] = cpre;
    __syncthreads();
    for (int i = gt; i < ns; i += NT) {
        const int32_t pp = pos[i];
        const int w = pp >> 5, sub = w >> gsh;
        int rank = chunk_pre[w >> 5] + sub_pre[sub];
        for (int v = sub << gsh; v < w; ++v) rank += __popc(bm[v]);
        rank += __popc(bm[w] & ((1u << (pp & 31)) - 1u));
        out[rank] = pp;
        if (outs) outs[rank] = key_score(key[i]);
    }
    for (int i = ns + gt; i < 2048; i += NT) {                      // only if candidates were missing
        out[i] = -1;
        if (outs) outs[i] = 0.f;
    }
}

}  // namespace sel
}  // namespace dsa
