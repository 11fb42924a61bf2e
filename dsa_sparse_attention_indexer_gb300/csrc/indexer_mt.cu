// Lightning-indexer scores for batches with several query rows per request
// (speculative verify, prefill chunks) on the 5th-generation tensor cores
// ("vLLM 推理链路概览", DSA Indexer: s_j = sum_m w_m ReLU(<q_m, k_j>);
// "GLM-5.3 推理全链路(十一)", 优化一: the index-K cache is read page by page).
//
// For a request the score is a dense FP8 contraction: its index-K tiles
// (128 tokens = two 64-token pages) are the A operand (M = 128) and a block of
// up to 8 of its query rows x 32 heads the B operand (N = 32 R <= 256), so
// every page is read once per row block instead of once per row.  Row t of a
// request sees positions 0..p_t (p_t = L - q_len + t); a row block scores the
// tiles up to its last row's position.
//
//  1. plan kernel: row blocks of every request (optionally only requests with
//     context > 2048, whose rows need scoring), their tile counts, and the
//     prefix of (row block, tile) items; each CTA takes one contiguous, equal
//     share of the items.
//  2. score kernel (persistent, one CTA per SM, warp-specialised):
//       warp 0     producer: a row block's quantised queries by one TMA box
//                  (double-buffered), each tile's two pages by TMA (128-byte
//                  swizzle) plus their 256-B scale rows, into an 8-stage ring;
//       warp 1     tcgen05.mma issuer (kind::f8f6f4, M=128, N=32R, K=4x32)
//                  into a double-buffered TMEM accumulator of 256 columns;
//       warps 2-13 three epilogue groups of four warps, all on every tile:
//                  group g takes its third of the block's rows (three warps
//                  per SM sub-partition on the same tile, so TMEM loads and
//                  arithmetic of different warps overlap while the MMA fills
//                  the other accumulator); per token and row, ReLU,
//                  head-weighted sum (packed f32x2 FMA; the block's head
//                  weights staged in shared memory), times the key scale.
//  3. top-k (dsa_indexer_topk): no score row is written.  A CTA's share of a
//     row block is a piece; each row of a piece streams its candidates into a
//     slot of 6144 in the workspace: scores above the row's rising threshold
//     are appended (a warp reserves its rows' room with one shared atomic per
//     tile and stores the entries after its next tile's arithmetic).  A slot
//     takes at most 128 entries a tile, so the epilogue checks the slots
//     (6144 - fullest) / 128 tiles after the last check; a slot that may not
//     hold the next four tiles is compacted: loaded into registers (16-byte
//     loads), one histogram pass over its key range finds the bin of its
//     2048th key, the entries from that bin up stay (at least 2048; an exact
//     radix selection when the bin is crowded) and the threshold rises to the
//     bin's lower edge.  At the piece end the slot's keys join the row's
//     12-bit key histogram.
//     The merge of the decode indexer (per-slot filter at the bin of the row's
//     2048th key, then an exact per-row selection) gives the row's top-2048.
//     The global top-2048 is inside the union of the pieces' top-2048s.
//     Scores (dsa_indexer_scores): the rows are written coalesced (32
//     consecutive positions per warp store); positions beyond a row's own
//     position, and pages outside the pool, get -inf.
// Every wait is time-bounded; a timeout is recorded and the CTA winds down.
#include "dsa_internal.cuh"
#include "indexer_common.cuh"
#include "indexer_tc.cuh"
#include "select_common.cuh"
#include "sm100.cuh"

#include <cudaTypedefs.h>

namespace dsa {
namespace imt {

using namespace sm100;

constexpr int kRows = 8;                        // query rows per row block
constexpr int kStages = 8;
constexpr int kStageBytes = 16384;              // 2 x 8192 FP8 payload (two 64-token pages)
constexpr int kQBytes = kRows * 32 * 128;       // one row block's quantised queries (256 x 128 B)
constexpr int kPidChunk = 64;                   // tiles whose page ids the producer fetches at once
constexpr int kGroups = 3;                      // epilogue groups of 4 warps, all on every tile
constexpr int kEpiThreads = 128 * kGroups;
constexpr int kEpiWarps = kEpiThreads / 32;
constexpr int kPerGrp = (kRows + kGroups - 1) / kGroups;   // rows of a block one group scores, at most
constexpr int kThreads = 64 + kEpiThreads;
constexpr int kTmemCols = 512;                  // 2 accumulators x 256 columns

constexpr int kOffStages = 0;
constexpr int kOffQ = kOffStages + kStages * kStageBytes;          // 2 row-block buffers
constexpr int kOffScales = kOffQ + 2 * kQBytes;                     // 2 x 256 B of key scales per stage
constexpr int kOffBars = kOffScales + kStages * 512;
constexpr int kOffPid = kOffBars + (2 * kStages + 9) * 8;
constexpr int kOffHist = kOffPid + kPidChunk * 2 * 8;          // 4096-bin radix histogram (compaction)
constexpr int kOffMisc = kOffHist + 4096 * 4;
constexpr int kMiscBytes = 512;
constexpr int kOffW = (kOffMisc + kMiscBytes + 15) / 16 * 16;   // the row block's head weights (fp32)
static_assert(kOffW % 16 == 0, "16-byte loads of the head weights");
constexpr int kSmemUsed = kOffW + kRows * 32 * 4;
constexpr int kSmemAlloc = kSmemUsed + 1024;
static_assert(kSmemAlloc <= 232448, "shared memory budget");
static_assert(kOffQ % 1024 == 0 && kQBytes % 1024 == 0, "swizzle atoms need 1 KB alignment");
constexpr int kEpiBar = 1;                      // named barrier of the two epilogue groups
constexpr int kSlotCap = kRowSlotCandidates;    // candidate entries of one row of a piece
constexpr int kCheckEvery = 4;                  // tiles between epilogue-wide checks of the slots
static_assert(kSlotCap - kCheckEvery * 128 > kTopK, "room above the 2048 kept by a compaction");

struct Misc {
    int32_t stage_valid[kStages];
    uint32_t tmem_base;
    int32_t abort;
    int32_t cnt[kRows];                         // candidates in each row's slot of the current piece
    uint32_t theta[kRows];                      // each row's threshold: only keys above it are candidates
    int32_t bad;                                // an epilogue warp gave up
    sel::Found found;
    int32_t scratch[32];
};
static_assert(sizeof(Misc) <= kMiscBytes, "misc block");

// Work plan (device buffers in the caller's workspace).
struct MtPlan {
    int32_t* rb_first;     // [B+1] first row block of each request
    int32_t* rb_req;       // [NBmax] request of each row block
    int64_t* item_start;   // [NBmax+1] (row block, tile) prefix
    int32_t* nb;           // [1] row blocks in this batch
    // streaming top-k only (NULL otherwise): the pieces (CTA shares) of each
    // row block, and the candidate slots of their rows.  Row rr of row block
    // rb's j-th piece owns slot 8 piece_first[rb] + rr npieces(rb) + j, so
    // each query row's slots are contiguous.
    int32_t* piece_first;  // [NBmax+1]
    int32_t* slot_row;     // [8 (NBmax + G)] query row of each slot, -1 = unused
    int32_t* row_seg0;     // [T] first slot of each query row
    int32_t* row_segn;     // [T] its slot count
    int32_t* nslots;       // [1]
    uint32_t* cand_key;    // [8 (NBmax + G), kSlotCap]
    int32_t* cand_pos;
    int32_t* cand_cnt;     // [8 (NBmax + G)]
    uint32_t* hist;        // [T, 4096] top-12-bit key histogram of each row's candidates
    int32_t G;             // CTAs the items are cut for
};

__device__ __forceinline__ int64_t cta_start(int64_t g, int64_t N, int64_t G) { return g * N / G; }
__device__ __forceinline__ int64_t cta_of_item(int64_t x, int64_t N, int64_t G) { return ((x + 1) * G + N - 1) / N - 1; }

// Rows [t0, t0 + R) of request r: R and the tiles to score -- up to its last
// row's position, or (full_rows) the whole context.
__device__ __forceinline__ void block_shape(const BatchDev& b, int r, int t0, bool full_rows, int* R, int* tiles) {
    const int L = b.seq_len[r];
    const int qn = b.q_start[r + 1] - b.q_start[r];
    *R = min(kRows, qn - t0);
    const int last = full_rows ? L - 1 : L - qn + t0 + *R - 1;
    *tiles = last >= 0 ? (last + 128) / 128 : 0;
}

// Single CTA of 1024 threads.
__global__ void __launch_bounds__(1024)
plan_kernel(BatchDev b, int skip_short, int full_rows, MtPlan p) {
    __shared__ int32_t scratch[32];
    const int gt = threadIdx.x;
    // pass 1: row blocks per request, and their prefix
    int32_t run = 0;
    for (int base = 0; base < b.batch; base += 1024) {
        const int r = base + gt;
        int nb = 0;
        if (r < b.batch) {
            const int L = b.seq_len[r];
            const int qn = b.q_start[r + 1] - b.q_start[r];
            if (qn > 0 && (!skip_short || L > kTopK)) nb = (qn + kRows - 1) / kRows;
        }
        int total;
        const int ex = sel::excl_scan<1024, 0>(nb, gt, scratch, &total);
        if (r < b.batch) p.rb_first[r] = run + ex;
        run += total;
    }
    const int32_t NB = run;
    if (gt == 0) {
        p.rb_first[b.batch] = NB;
        *p.nb = NB;
    }
    __syncthreads();
    // pass 2: request of each row block, its tiles, and the item prefix
    int64_t irun = 0;
    for (int base = 0; base < NB; base += 1024) {
        const int rb = base + gt;
        int tiles = 0;
        if (rb < NB) {
            int lo = 0, hi = b.batch - 1;                 // last request whose first row block <= rb
            while (lo < hi) {
                const int mid = (lo + hi + 1) >> 1;
                if (p.rb_first[mid] <= rb) lo = mid; else hi = mid - 1;
            }
            p.rb_req[rb] = lo;
            int R;
            block_shape(b, lo, (rb - p.rb_first[lo]) * kRows, full_rows != 0, &R, &tiles);
        }
        int total;
        const int ex = sel::excl_scan<1024, 0>(tiles, gt, scratch, &total);
        if (rb < NB) p.item_start[rb] = irun + ex;
        irun += total;
    }
    if (gt == 0) p.item_start[NB] = irun;
    if (!p.piece_first) return;
    __syncthreads();
    // pass 3 (streaming top-k): pieces of each row block, and the slots of their rows
    const int64_t N = irun;
    const int64_t G = p.G;
    int32_t prun = 0;
    for (int base = 0; base < NB; base += 1024) {
        const int rb = base + gt;
        int np = 0;
        if (rb < NB) {
            const int64_t s0 = p.item_start[rb], s1 = p.item_start[rb + 1];
            if (s1 > s0) np = (int)(cta_of_item(s1 - 1, N, G) - cta_of_item(s0, N, G) + 1);
        }
        int total;
        const int ex = sel::excl_scan<1024, 0>(np, gt, scratch, &total);
        if (rb < NB) p.piece_first[rb] = prun + ex;
        prun += total;
    }
    if (gt == 0) {
        p.piece_first[NB] = prun;
        *p.nslots = kRows * prun;
    }
    for (int i = gt; i < kRows * prun; i += 1024) p.slot_row[i] = -1;
    for (int64_t i = gt; i < b.total_q; i += 1024) {          // rows without slots: not scored
        p.row_seg0[i] = 0;
        p.row_segn[i] = 0;
    }
    __syncthreads();
    for (int rb = gt; rb < NB; rb += 1024) {
        const int r = p.rb_req[rb];
        const int t0 = (rb - p.rb_first[r]) * kRows;
        const int qn = b.q_start[r + 1] - b.q_start[r];
        const int R = min(kRows, qn - t0);
        const int np = p.piece_first[rb + 1] - p.piece_first[rb];
        const int base = kRows * p.piece_first[rb];
        for (int rr = 0; rr < R; ++rr) {
            const int64_t row = (int64_t)b.q_start[r] + t0 + rr;
            p.row_seg0[row] = base + rr * np;
            p.row_segn[row] = np;
            for (int j = 0; j < np; ++j) p.slot_row[base + rr * np + j] = (int32_t)row;
        }
    }
}

// Row block holding item i (item_start is non-decreasing, item_start[NB] = N).
__device__ __forceinline__ int find_block(const MtPlan& p, int NB, int64_t i) {
    int lo = 0, hi = NB - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (p.item_start[mid] <= i) lo = mid; else hi = mid - 1;
    }
    return lo;
}

// Walks the CTA's items in order: row block, tile, and the running counts the
// roles use to derive stages, accumulators and row-block buffers.
struct Walk {
    int64_t i, i_end;
    int rb;           // current row block
    int64_t rb_end;   // first item of the next row block
    int j;            // row blocks entered so far (0 for the first)
};

__device__ __forceinline__ void walk_begin(Walk& w, const MtPlan& p, int NB, int64_t i0, int64_t i1) {
    w.i = i0;
    w.i_end = i1;
    w.j = 0;
    w.rb = i0 < i1 ? find_block(p, NB, i0) : 0;
    w.rb_end = i0 < i1 ? p.item_start[w.rb + 1] : 0;
}
// Advance to the next item; returns true when it starts a new row block.
__device__ __forceinline__ bool walk_next(Walk& w, const MtPlan& p) {
    ++w.i;
    if (w.i < w.i_end && w.i >= w.rb_end) {
        do {
            ++w.rb;
        } while (p.item_start[w.rb + 1] <= w.i);         // skip row blocks without tiles
        w.rb_end = p.item_start[w.rb + 1];
        ++w.j;
        return true;
    }
    return false;
}

__device__ __forceinline__ void epi_sync() { asm volatile("bar.sync %0, %1;" ::"n"(kEpiBar), "n"(kEpiThreads) : "memory"); }

constexpr int kSlotPer = kSlotCap / kEpiThreads;   // slot entries per epilogue thread
static_assert(kSlotCap % (4 * kEpiThreads) == 0, "whole groups of four slot entries per thread");

// Slot entry held in register u of epilogue thread et: groups of four
// consecutive entries (one 16-byte load), the thread's groups kEpiThreads apart.
__device__ __forceinline__ int slot_entry(int u, int et) { return ((u >> 2) * kEpiThreads + et) * 4 + (u & 3); }

// A slot's entries held in the epilogue threads' registers (entry
// slot_entry(u, et) in k[u], p[u]), as a selection source.
struct RegSrc {
    const uint32_t (&k)[kSlotPer];
    const int32_t (&p)[kSlotPer];
    int n, et;
    template <class F>
    __device__ __forceinline__ void visit(int, F&& f) const {
#pragma unroll
        for (int u = 0; u < kSlotPer; ++u) {
            const bool a = slot_entry(u, et) < n;
            f(a, a ? k[u] : 0u, a ? p[u] : 0);
        }
    }
};

// Entries a compaction may keep before it falls back to the exact selection.
constexpr int kKeepMax = kTopK + 512;
static_assert(kKeepMax <= kSlotCap - kCheckEvery * 128, "a compaction always makes room");

// Compaction of a slot of *n > 2048 entries in global memory, all epilogue
// threads: one batch of loads into registers, then one histogram pass of
// 4096 equal-width bins over the slot's key range [lo, hi] gives the bin b*
// of the 2048th largest key.  T = the lower edge of b*: the slot keeps every
// key >= T (at least 2048 entries), and a later key <= T cannot enter the
// top-2048 (2048 kept entries are at or above it, at lower positions).  When
// b* is crowded (ties, a narrow range) and more than kKeepMax would stay, the
// exact radix selection keeps exactly the top-2048 (key, then lower position)
// and T is the 2048th key.  Survivors are written back in any order; returns
// T, the slot's new threshold.
__device__ uint32_t compact_slot(uint32_t* key, int32_t* pos, int* n, int et, uint32_t* hist, int* scratch,
                                 sel::Found* found) {
    const int cnt = *n;
    const int lane = et & 31, wid = et >> 5;
    uint32_t k[kSlotPer];
    int32_t ps[kSlotPer];
    uint32_t lo = 0xffffffffu, hi = 0u;
#pragma unroll
    for (int g = 0; g < kSlotPer / 4; ++g) {          // 16-byte loads (slots are 16-byte aligned, kSlotCap long)
        const int i0 = (g * kEpiThreads + et) * 4;
        uint4 kv = make_uint4(0u, 0u, 0u, 0u), pv = make_uint4(0u, 0u, 0u, 0u);
        if (i0 < cnt) {
            kv = __ldcg(reinterpret_cast<const uint4*>(key + i0));
            pv = __ldcg(reinterpret_cast<const uint4*>(pos + i0));
        }
        k[4 * g + 0] = kv.x; k[4 * g + 1] = kv.y; k[4 * g + 2] = kv.z; k[4 * g + 3] = kv.w;
        ps[4 * g + 0] = (int32_t)pv.x; ps[4 * g + 1] = (int32_t)pv.y;
        ps[4 * g + 2] = (int32_t)pv.z; ps[4 * g + 3] = (int32_t)pv.w;
    }
#pragma unroll
    for (int u = 0; u < kSlotPer; ++u) {
        if (slot_entry(u, et) < cnt) {
            lo = min(lo, k[u]);
            hi = max(hi, k[u]);
        }
    }
    lo = __reduce_min_sync(0xffffffffu, lo);
    hi = __reduce_max_sync(0xffffffffu, hi);
    if (lane == 0) {
        scratch[wid] = (int)lo;
        scratch[kEpiWarps + wid] = (int)hi;
    }
    for (int i = et; i < 4096; i += kEpiThreads) hist[i] = 0u;
    epi_sync();
#pragma unroll
    for (int v = 0; v < kEpiWarps; ++v) {
        lo = min(lo, (uint32_t)scratch[v]);
        hi = max(hi, (uint32_t)scratch[kEpiWarps + v]);
    }
    const uint32_t span = hi - lo;
    const int shift = (span >> 12) ? 32 - __clz((int)(span >> 12)) : 0;   // (span >> shift) < 4096
#pragma unroll
    for (int u = 0; u < kSlotPer; ++u)
        if (slot_entry(u, et) < cnt) atomicAdd(&hist[(k[u] - lo) >> shift], 1u);
    epi_sync();                                        // every scratch read above is done too
    constexpr int kPer = (4096 + kEpiThreads - 1) / kEpiThreads;   // bins per thread, from the top
    int mine = 0;
#pragma unroll
    for (int q = 0; q < kPer; ++q) {
        const int bin = 4095 - (et * kPer + q);
        if (bin >= 0) mine += (int)hist[bin];
    }
    int total;
    int above = sel::excl_scan<kEpiThreads, kEpiBar>(mine, et, scratch, &total);
#pragma unroll
    for (int q = 0; q < kPer; ++q) {
        const int bin = 4095 - (et * kPer + q);
        const int c = bin >= 0 ? (int)hist[bin] : 0;
        if (above < kTopK && above + c >= kTopK) {
            found->bin = (uint32_t)bin;
            found->above = above + c;                  // entries in bins >= b*
        }
        above += c;
    }
    epi_sync();
    sel::Threshold th{lo + (found->bin << shift), 0x7fffffff};
    if (found->above > kKeepMax) {
        epi_sync();                                    // found is rewritten by the selection
        RegSrc src{k, ps, cnt, et};
        th = sel::topk_threshold<kEpiThreads, kEpiBar>(src, kTopK, et, hist, scratch, found);
    }
    // survivors in warp order, then u, then lane: one scan of the warps' counts,
    // and each store instruction of a warp writes consecutive entries
    unsigned km[kSlotPer];
    int wcount = 0;
#pragma unroll
    for (int u = 0; u < kSlotPer; ++u) {
        km[u] = __ballot_sync(0xffffffffu, slot_entry(u, et) < cnt && th.keep(k[u], ps[u]));
        wcount += __popc(km[u]);
    }
    const int wbase = sel::excl_scan<kEpiThreads, kEpiBar>(lane == 0 ? wcount : 0, et, scratch, &total);
    int at = __shfl_sync(0xffffffffu, wbase, 0);                 // every load is done
    const unsigned below = (1u << lane) - 1u;
#pragma unroll
    for (int u = 0; u < kSlotPer; ++u) {
        if ((km[u] >> lane) & 1u) {
            const int o = at + __popc(km[u] & below);
            key[o] = k[u];
            pos[o] = ps[u];
        }
        at += __popc(km[u]);
    }
    if (et == 0) *n = total;
    epi_sync();
    return th.kth;
}

// Head-weighted ReLU sum of one token's 32 head logits (TMEM words) for one
// query row: sum_m w_m max(l_m, 0), eight partial sums in four packed pairs.
// w: the row's 32 weights in shared memory (copied once per row block; global
// loads of them on every tile cost about 5 % of the kernel).
__device__ __forceinline__ float head_sum(const uint32_t (&v)[32], const float* __restrict__ w) {
    const float4* w4 = reinterpret_cast<const float4*>(w);
    float2 a[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) a[j] = make_float2(0.f, 0.f);
#pragma unroll
    for (int m4 = 0; m4 < 8; ++m4) {
        const float4 ww = w4[m4];
        const float2 x01 = make_float2(fmaxf(__uint_as_float(v[4 * m4 + 0]), 0.f),
                                       fmaxf(__uint_as_float(v[4 * m4 + 1]), 0.f));
        const float2 x23 = make_float2(fmaxf(__uint_as_float(v[4 * m4 + 2]), 0.f),
                                       fmaxf(__uint_as_float(v[4 * m4 + 3]), 0.f));
        a[(2 * m4) & 3] = __ffma2_rn(make_float2(ww.x, ww.y), x01, a[(2 * m4) & 3]);
        a[(2 * m4 + 1) & 3] = __ffma2_rn(make_float2(ww.z, ww.w), x23, a[(2 * m4 + 1) & 3]);
    }
    return ((a[0].x + a[0].y) + (a[1].x + a[1].y)) + ((a[2].x + a[2].y) + (a[3].x + a[3].y));
}

// Wait for this thread's TMEM loads, then pin the loaded registers after the
// wait (the compiler sees them defined here, so no use moves above it).
__device__ __forceinline__ void tmem_wait_regs(uint32_t (&r)[32]) {
    asm volatile("tcgen05.wait::ld.sync.aligned;");
    asm volatile(""
                 : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]), "+r"(r[7]),
                   "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]), "+r"(r[12]), "+r"(r[13]), "+r"(r[14]),
                   "+r"(r[15]), "+r"(r[16]), "+r"(r[17]), "+r"(r[18]), "+r"(r[19]), "+r"(r[20]), "+r"(r[21]),
                   "+r"(r[22]), "+r"(r[23]), "+r"(r[24]), "+r"(r[25]), "+r"(r[26]), "+r"(r[27]), "+r"(r[28]),
                   "+r"(r[29]), "+r"(r[30]), "+r"(r[31]));
}
__device__ __forceinline__ void reg_fence(uint32_t (&r)[32]) {
    asm volatile(""
                 : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]), "+r"(r[7]),
                   "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]), "+r"(r[12]), "+r"(r[13]), "+r"(r[14]),
                   "+r"(r[15]), "+r"(r[16]), "+r"(r[17]), "+r"(r[18]), "+r"(r[19]), "+r"(r[20]), "+r"(r[21]),
                   "+r"(r[22]), "+r"(r[23]), "+r"(r[24]), "+r"(r[25]), "+r"(r[26]), "+r"(r[27]), "+r"(r[28]),
                   "+r"(r[29]), "+r"(r[30]), "+r"(r[31]));
}

// Scores of this thread's token (TMEM lane) for nr <= kPerGrp consecutive rows:
// tbase + 32 j holds row j's 32 head logits, w + 32 j its head weights.  Rows
// go in pairs: both loads, one wait, both sums.
__device__ __forceinline__ void row_scores(uint32_t tbase, const float* __restrict__ w, int nr, float sk,
                                           float (&s)[kPerGrp]) {
#pragma unroll
    for (int j = 0; j < kPerGrp; j += 2) {
        if (j < nr) {
            uint32_t va[32], vb[32];
            tmem_ld_32x32b_x32(tbase + j * 32, va);
            if (j + 1 < nr) tmem_ld_32x32b_x32(tbase + (j + 1) * 32, vb);
            tmem_wait_regs(va);
            reg_fence(vb);
            s[j] = head_sum(va, w + j * 32) * sk;
            if (j + 1 < nr) s[j + 1] = head_sum(vb, w + (j + 1) * 32) * sk;
        }
    }
}

// kStream: stream each row's candidates into its slots (dsa_indexer_topk);
// otherwise write the score rows (dsa_indexer_scores).
template <bool kStream>
__global__ void __launch_bounds__(kThreads, 1)
score_rows_kernel(const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap qmap,
                  const uint8_t* __restrict__ cache, const float* __restrict__ wq, BatchDev b, MtPlan p,
                  float* __restrict__ scores, int64_t ld, int32_t* __restrict__ st) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + kOffBars);
    uint64_t* empty = full + kStages;
    uint64_t* accf = empty + kStages;
    uint64_t* acce = accf + 2;
    uint64_t* qfull = acce + 2;
    uint64_t* qempty = qfull + 2;
    uint64_t* drain = qempty + 2;
    int64_t* pid = reinterpret_cast<int64_t*>(smem + kOffPid);
    Misc* misc = reinterpret_cast<Misc*>(smem + kOffMisc);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1 + kEpiWarps);  // MMA commit + one arrive per epilogue warp
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(&accf[a], 1);
            mbar_init(&acce[a], kEpiWarps);
            mbar_init(&qfull[a], 1);
            mbar_init(&qempty[a], 1);
        }
        mbar_init(drain, 1);
        misc->abort = 0;
        misc->bad = 0;
        fence_barrier_init();
    }
    if (warp == 1) {
        tmem_alloc(&misc->tmem_base, kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = misc->tmem_base;
    volatile int32_t* abort_flag = &misc->abort;
    const int NB = *p.nb;
    const int64_t N = NB > 0 ? p.item_start[NB] : 0;
    const int64_t G = gridDim.x;
    const int64_t i0 = cta_start(blockIdx.x, N, G), i1 = cta_start(blockIdx.x + 1, N, G);

    if (warp == 0) {
        // ------------------------------------------------------------ producer
        Walk w;
        walk_begin(w, p, NB, i0, i1);
        int stage = 0;
        uint32_t phase = 0;
        int inflight = 0;
        bool stop = false;
        bool new_block = true;
        while (w.i < w.i_end && !stop) {
            const int r = p.rb_req[w.rb];
            const int t0 = (w.rb - p.rb_first[r]) * kRows;
            const int L = b.seq_len[r];
            const int32_t* pt = b.page_table + (int64_t)r * b.max_pages;
            const int tile0 = (int)(w.i - p.item_start[w.rb]);
            const int nt = (int)min((int64_t)kPidChunk, min(w.rb_end, w.i_end) - w.i);   // within the row block and the share
            // page ids of the next nt tiles of this row block
            for (int k = lane; k < 2 * nt; k += 32) {
                const int idx = tile0 * 2 + k;
                pid[k] = idx < b.max_pages ? (int64_t)pt[idx] : (int64_t)-2;
            }
            __syncwarp();
            int ok = 1;
            if (lane == 0) {
                if (new_block) {
                    // quantised queries of the row block: 256 rows x 128 B from row (q_start + t0) * 32
                    const int qb = w.j & 1;
                    if (w.j >= 2 && !mbar_wait(&qempty[qb], (uint32_t)(((w.j >> 1) - 1) & 1))) {
                        ok = 0;
                        record_error(st, DSA_DEVERR_TIMEOUT, 511);
                    }
                    if (ok) {
                        mbar_arrive_expect_tx(&qfull[qb], kQBytes);
                        tma_load_2d(smem + kOffQ + qb * kQBytes, &qmap, 0,
                                    (int32_t)((b.q_start[r] + t0) * 32), &qfull[qb]);
                    }
                }
                for (int k = 0; k < nt && ok; ++k) {
                    if (*abort_flag || !mbar_wait(&empty[stage], phase ^ 1)) {
                        if (!*abort_flag) record_error(st, DSA_DEVERR_TIMEOUT, 512);
                        ok = 0;
                        break;
                    }
                    const int t_abs = (tile0 + k) * 128;
                    const int pages = (L - t_abs > 64) ? 2 : 1;
                    uint32_t bytes = 0;
                    int vmask = 0;
                    int64_t pg[2];
                    for (int jj = 0; jj < pages; ++jj) {
                        pg[jj] = pid[k * 2 + jj];
                        if (pg[jj] >= 0 && pg[jj] < b.num_pages) {
                            vmask |= 1 << jj;
                            bytes += 8192 + 256;
                        } else if (pg[jj] == -2) {
                            record_error(st, DSA_DEVERR_INDEX_RANGE, t_abs + jj * 64);
                        } else {
                            record_error(st, DSA_DEVERR_PAGE_RANGE, pg[jj]);
                        }
                    }
                    misc->stage_valid[stage] = vmask;
                    uint8_t* sb = smem + kOffStages + stage * kStageBytes;
                    mbar_arrive_expect_tx(&full[stage], bytes);
                    for (int jj = 0; jj < pages; ++jj) {
                        if (!(vmask & (1 << jj))) continue;
                        tma_load_2d(sb + jj * 8192, &kmap, 0, (int32_t)(pg[jj] * 66), &full[stage]);
                        bulk_load(smem + kOffScales + stage * 512 + jj * 256,
                                  cache + pg[jj] * (int64_t)kIdxPageBytes + kIdxPayloadBytes, 256, &full[stage]);
                    }
                    ++inflight;
                    if (++stage == kStages) {
                        stage = 0;
                        phase ^= 1;
                    }
                }
            }
            ok = __shfl_sync(0xffffffffu, ok, 0);
            __syncwarp();
            if (!ok) {
                stop = true;
                break;
            }
            new_block = false;
            for (int k = 0; k < nt; ++k)
                if (walk_next(w, p)) new_block = true;
        }
        if (lane == 0 && stop) {
            if (!*abort_flag) record_error(st, DSA_DEVERR_TIMEOUT, 51);
            *abort_flag = 1;
            for (int k = 0; k < kStages && inflight > 0; ++k, --inflight) {   // let issued copies land
                stage = (stage + kStages - 1) % kStages;
                if (stage == kStages - 1) phase ^= 1;
                mbar_wait(&full[stage], phase, 500000000ull);
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        Walk w;
        walk_begin(w, p, NB, i0, i1);
        int stage = 0, acc = 0;
        uint32_t phase = 0, acc_phase = 0;
        bool stop = false, issued = false;
        bool new_block = true;
        while (w.i < w.i_end) {
            const int r = p.rb_req[w.rb];
            const int t0 = (w.rb - p.rb_first[r]) * kRows;
            const int qn = b.q_start[r + 1] - b.q_start[r];
            const int R = min(kRows, qn - t0);
            const uint32_t idesc = idesc_e4m3_f32(128, 32 * R);
            const int qb = w.j & 1;
            int ok = 1;
            if (lane == 0) {
                ok = (!*abort_flag && mbar_wait(&acce[acc], acc_phase ^ 1)) ? 1 : 0;
                if (!ok && !*abort_flag) record_error(st, DSA_DEVERR_TIMEOUT, 521);
                if (ok && new_block) {
                    ok = mbar_wait(&qfull[qb], (uint32_t)((w.j >> 1) & 1)) ? 1 : 0;
                    if (!ok) record_error(st, DSA_DEVERR_TIMEOUT, 522);
                }
                if (ok) {
                    ok = mbar_wait(&full[stage], phase) ? 1 : 0;
                    if (!ok) record_error(st, DSA_DEVERR_TIMEOUT, 523);
                }
                if (ok) {
                    tc_fence_after();
                    const uint32_t a0 = smem_addr(smem + kOffStages + stage * kStageBytes);
                    const uint32_t b0 = smem_addr(smem + kOffQ + qb * kQBytes);
#pragma unroll
                    for (int k = 0; k < 4; ++k)
                        mma_f8f6f4(tmem + acc * 256, desc_kmajor_sw128(a0 + 32 * k), desc_kmajor_sw128(b0 + 32 * k),
                                   idesc, k > 0 ? 1u : 0u);
                    mma_commit(&empty[stage]);
                    mma_commit(&accf[acc]);
                    issued = true;
                }
            }
            ok = __shfl_sync(0xffffffffu, ok, 0);
            if (!ok) {
                stop = true;
                break;
            }
            if (++stage == kStages) {
                stage = 0;
                phase ^= 1;
            }
            if (++acc == 2) {
                acc = 0;
                acc_phase ^= 1;
            }
            const int64_t rb_end = w.rb_end;
            new_block = walk_next(w, p);
            if (w.i >= rb_end || w.i >= w.i_end) {          // the row block's last tile: its Q buffer frees on completion
                if (lane == 0) mma_commit(&qempty[qb]);
            }
            __syncwarp();
        }
        if (lane == 0) {
            if (stop) {
                record_error(st, DSA_DEVERR_TIMEOUT, 52);
                *abort_flag = 1;
            }
            if (issued) {                                     // no MMA in flight when the TMEM is released
                mma_commit(drain);
                mbar_wait(drain, 0, 500000000ull);
            }
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------------ epilogue
        // Every group takes every tile (accumulator = running index parity),
        // group g its share of the block's rows.  Warp w reads TMEM lanes
        // 32 (w % 4) .., i.e. tokens 32 (w % 4) .. of the tile.  Streaming: the
        // groups meet at a named barrier at each piece start, every kCheckEvery
        // tiles of a piece and at its end, where full slots are compacted.
        const int grp = (warp - 2) >> 2;
        const int quarter = warp & 3;
        const int tok = quarter * 32 + lane;
        const int et = threadIdx.x - 64;                 // 0 .. kEpiThreads - 1
        uint32_t* hist = reinterpret_cast<uint32_t*>(smem + kOffHist);
        float* wsm = reinterpret_cast<float*>(smem + kOffW);
        Walk w;
        walk_begin(w, p, NB, i0, i1);
        int64_t gidx = 0;
        bool bad = false;
        bool piece_start = true;
        int ptile = 0;                                   // tiles of the current piece walked so far
        // The next check of the slots: a slot takes at most 128 entries a tile, so
        // a check after (capacity - fullest slot) / 128 tiles finds none overflowed.
        int next_check = kSlotCap / 128;
        int slot0 = 0, np = 0;                           // the piece's slot of row 0 and the row block's pieces
        uint32_t th[kPerGrp];                              // the group's rows' thresholds (copies of misc->theta)
#pragma unroll
        for (int j = 0; j < kPerGrp; ++j) th[j] = 0u;
        // Values of the current row block, read when it starts.
        int r = 0, t0 = 0, qn = 0, R = 0, rlo = 0, nr = 0, p0 = 0;
        int64_t row0 = 0, item0 = 0;
        // Streaming: the previous tile's candidates, stored once its reservation
        // (a shared atomic) has returned, i.e. after the next tile's arithmetic.
        unsigned pend_m[kPerGrp];
        uint32_t pend_key[kPerGrp];
        int pend_pos = 0, pend_base = 0;
        uint32_t* kslot = nullptr;                       // the group's first row's slot in this piece
        int32_t* pslot = nullptr;
        int64_t rstride = 0;                             // from one row's slot to the next row's
#pragma unroll
        for (int j = 0; j < kPerGrp; ++j) pend_m[j] = 0u;
        auto flush = [&]() {
            if constexpr (kStream) {
                const unsigned below = (1u << lane) - 1u;
#pragma unroll
                for (int j = 0; j < kPerGrp; ++j) {
                    const int b_j = __shfl_sync(0xffffffffu, pend_base, j);
                    if ((pend_m[j] >> lane) & 1u) {
                        const int64_t at = j * rstride + b_j + __popc(pend_m[j] & below);
                        kslot[at] = pend_key[j];
                        pslot[at] = pend_pos;
                    }
                    pend_m[j] = 0u;
                }
            }
        };
        bool new_block = true;
        while (w.i < w.i_end) {
            if (new_block) {
                r = p.rb_req[w.rb];
                t0 = (w.rb - p.rb_first[r]) * kRows;
                qn = b.q_start[r + 1] - b.q_start[r];
                R = min(kRows, qn - t0);
                rlo = (grp * R + kGroups - 1) / kGroups;           // the group's rows: rlo .. rlo + nr - 1
                nr = ((grp + 1) * R + kGroups - 1) / kGroups - rlo;
                row0 = b.q_start[r] + t0;
                p0 = b.seq_len[r] - qn + t0;                      // position of the block's first row
                item0 = p.item_start[w.rb];
            }
            if (!kStream && new_block) {                 // the block's head weights, once per block
                epi_sync();
                if (et < R * 32) wsm[et] = wq[row0 * 32 + et];
                epi_sync();
            }
            if (kStream && piece_start) {
                const int64_t N = p.item_start[NB];
                const int64_t g0 = cta_of_item(p.item_start[w.rb], N, G);
                np = p.piece_first[w.rb + 1] - p.piece_first[w.rb];
                slot0 = kRows * p.piece_first[w.rb] + (int)(blockIdx.x - g0);
                epi_sync();                              // the previous piece is finished
                if (et < R * 32) wsm[et] = wq[row0 * 32 + et];   // the block's head weights
                if (et < kRows) {
                    misc->cnt[et] = 0;
                    misc->theta[et] = 0u;                // key 0: below every score
                }
                epi_sync();
#pragma unroll
                for (int j = 0; j < kPerGrp; ++j) th[j] = 0u;
                rstride = (int64_t)np * kSlotCap;
                kslot = p.cand_key + (int64_t)(slot0 + rlo * np) * kSlotCap;
                pslot = p.cand_pos + (int64_t)(slot0 + rlo * np) * kSlotCap;
                ptile = 0;
                next_check = kSlotCap / 128;
            }
            if (!bad && __any_sync(0xffffffffu, *abort_flag != 0)) bad = true;   // another role gave up
            if (!bad) {
                const int tile = (int)(w.i - item0);
                const int stage = (int)(gidx % kStages);
                const uint32_t phase = (uint32_t)((gidx / kStages) & 1);
                const int acc = (int)(gidx & 1);
                const uint32_t acc_phase = (uint32_t)((gidx >> 1) & 1);
                int ok = __all_sync(0xffffffffu, mbar_wait(&accf[acc], acc_phase));
                if (!ok && lane == 0) record_error(st, DSA_DEVERR_TIMEOUT, 531);
                if (ok) {
                    ok = __all_sync(0xffffffffu, mbar_wait(&full[stage], phase));   // scales + page mask
                    if (!ok && lane == 0) record_error(st, DSA_DEVERR_TIMEOUT, 532);
                }
                if (ok) {
                    tc_fence_after();
                    const int vmask = misc->stage_valid[stage];
                    const float sk = reinterpret_cast<const float*>(smem + kOffScales + stage * 512)[tok];
                    const int pos = tile * 128 + tok;
                    const bool page_ok = (vmask >> (tok >> 6)) & 1;
                    float sc[kPerGrp];
                    if (nr > 0)
                        row_scores(tmem + ((uint32_t)(quarter * 32) << 16) + acc * 256 + rlo * 32,
                                   wsm + rlo * 32, nr, sk, sc);
                    if constexpr (kStream) {
                        // candidates above each row's threshold: one ballot per row, then lane j
                        // reserves row rlo + j's room (the group's atomics go out together);
                        // the previous tile's candidates are stored first
                        flush();
                        unsigned mine = 0;
#pragma unroll
                        for (int j = 0; j < kPerGrp; ++j) {
                            const uint32_t key = score_key(sc[j]);
                            const bool pass = j < nr && page_ok && pos <= p0 + rlo + j && key > th[j];
                            pend_m[j] = __ballot_sync(0xffffffffu, pass);
                            pend_key[j] = key;
                            if (lane == j) mine = pend_m[j];
                        }
                        pend_base = 0;
                        if (mine) pend_base = atomicAdd(&misc->cnt[rlo + lane], __popc(mine));
                        pend_pos = pos;
                    } else {
#pragma unroll
                        for (int j = 0; j < kPerGrp; ++j)
                            if (j < nr && pos < ld)
                                scores[(row0 + rlo + j) * ld + pos] = (page_ok && pos <= p0 + rlo + j) ? sc[j] : -INFINITY;
                    }
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) {
                        mbar_arrive(&acce[acc]);
                        mbar_arrive(&empty[stage]);
                    }
                } else {
                    bad = true;                             // this warp stops; the others time out too
                    if (lane == 0) {
                        record_error(st, DSA_DEVERR_TIMEOUT, 53);
                        *abort_flag = 1;
                    }
                }
            }
            ++gidx;
            ++ptile;
            const bool piece_end = w.i + 1 >= w.rb_end || w.i + 1 >= w.i_end;
            if (kStream && (piece_end || ptile == next_check)) {
                // every tile of the piece so far is in the slots: compact the slots that
                // may not hold the next kCheckEvery tiles, schedule the next check, and at
                // the piece end publish the slots (up to kSlotCap entries each, no compaction)
                flush();
                if (lane == 0 && bad) misc->bad = 1;
                epi_sync();
                const bool any_bad = misc->bad != 0;
                if (!any_bad) {
                    if (!piece_end) {
                        for (int rr = 0; rr < R; ++rr) {
                            if (misc->cnt[rr] <= kSlotCap - kCheckEvery * 128) continue;
                            const int64_t sl = (int64_t)(slot0 + rr * np) * kSlotCap;
                            const uint32_t t = compact_slot(p.cand_key + sl, p.cand_pos + sl, &misc->cnt[rr], et,
                                                            hist, misc->scratch, &misc->found);
                            if (et == 0) misc->theta[rr] = t;
                            epi_sync();
                        }
#pragma unroll
                        for (int j = 0; j < kPerGrp; ++j) th[j] = misc->theta[rlo + j];
                    }
                    int fullest = 0;                        // the same value in every thread
                    for (int rr = 0; rr < R; ++rr) fullest = max(fullest, misc->cnt[rr]);
                    next_check = ptile + max(1, (kSlotCap - fullest) / 128);
                } else {
                    next_check = ptile + kCheckEvery;
                }
                if (piece_end) {
                    for (int rr = 0; rr < kRows; ++rr) {
                        const int slot = slot0 + rr * np;
                        if (rr >= R) break;
                        const int cnt = any_bad ? 0 : misc->cnt[rr];
                        if (et == 0) p.cand_cnt[slot] = cnt;
                        uint32_t* gh = p.hist + (row0 + rr) * 4096;
                        for (int i = et; i < cnt; i += kEpiThreads)
                            atomicAdd(&gh[__ldcg(p.cand_key + (int64_t)slot * kSlotCap + i) >> 20], 1u);
                    }
                }
                epi_sync();                             // every read of the shared state above is done
            }
            piece_start = walk_next(w, p);
            new_block = piece_start;
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

}  // namespace imt

namespace {
struct QMapCache {
    const void* ptr = nullptr;
    int64_t rows = 0;
    CUtensorMap map;
};
}  // namespace

bool make_index_tmap(const uint8_t* cache, int64_t num_pages, bool mx, CUtensorMap* out);

static bool make_q8_tmap(const uint8_t* q8, int64_t total_q, CUtensorMap* out) {
    static thread_local QMapCache mc;                  // per host thread: no lock needed
    if (mc.ptr == q8 && mc.rows == total_q) {
        *out = mc.map;
        return true;
    }
    const auto encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(tensor_map_encode_fn());
    if (!encode) return false;
    // q8 viewed as a [T * 32, 128] byte matrix (row = one head of one query row);
    // a box is one row block: 256 rows, rows past T * 32 read as zeros.
    cuuint64_t dims[2] = {128, (cuuint64_t)total_q * 32};
    cuuint64_t strides[1] = {128};
    cuuint32_t box[2] = {128, (cuuint32_t)(imt::kRows * 32)};
    cuuint32_t estr[2] = {1, 1};
    CUresult res = encode(out, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<uint8_t*>(q8), dims, strides, box, estr,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (res != CUDA_SUCCESS) return false;
    mc.ptr = q8;
    mc.rows = total_q;
    mc.map = *out;
    return true;
}

// Workspace of the multi-row plan; with `slots` (streaming top-k) also the
// pieces, the slot index and the candidate slots for a grid of G CTAs.
static size_t mt_plan_layout(int64_t batch, int64_t total_q, int G, bool slots, imt::MtPlan* p, void* base) {
    const int64_t nb_max = (total_q + imt::kRows - 1) / imt::kRows + batch;
    const int64_t nslots = (int64_t)imt::kRows * (nb_max + G);
    uint8_t* q = static_cast<uint8_t*>(base);
    size_t off = 0;
    auto take = [&](size_t bytes, size_t align) -> uint8_t* {
        off = (off + align - 1) / align * align;
        uint8_t* at = q ? q + off : nullptr;
        off += bytes;
        return at;
    };
    imt::MtPlan m{};
    m.rb_first = reinterpret_cast<int32_t*>(take((size_t)(batch + 1) * 4, 16));
    m.rb_req = reinterpret_cast<int32_t*>(take((size_t)nb_max * 4, 16));
    m.item_start = reinterpret_cast<int64_t*>(take((size_t)(nb_max + 1) * 8, 16));
    m.nb = reinterpret_cast<int32_t*>(take(16, 16));
    m.G = G;
    if (slots) {
        m.piece_first = reinterpret_cast<int32_t*>(take((size_t)(nb_max + 1) * 4, 16));
        m.slot_row = reinterpret_cast<int32_t*>(take((size_t)nslots * 4, 16));
        m.row_seg0 = reinterpret_cast<int32_t*>(take((size_t)total_q * 4, 16));
        m.row_segn = reinterpret_cast<int32_t*>(take((size_t)total_q * 4, 16));
        m.nslots = reinterpret_cast<int32_t*>(take(16, 16));
        m.cand_cnt = reinterpret_cast<int32_t*>(take((size_t)nslots * 4, 256));
        m.cand_key = reinterpret_cast<uint32_t*>(take((size_t)nslots * imt::kSlotCap * 4, 256));
        m.cand_pos = reinterpret_cast<int32_t*>(take((size_t)nslots * imt::kSlotCap * 4, 256));
    }
    if (p) *p = m;
    return (off + 255) / 256 * 256;
}

size_t mt_plan_bytes(int64_t batch, int64_t total_q) { return mt_plan_layout(batch, total_q, 0, false, nullptr, nullptr); }
size_t mt_topk_bytes(int64_t batch, int64_t total_q, int G) {
    return mt_plan_layout(batch, total_q, G, true, nullptr, nullptr);
}

static imt::MtPlan carve_mt_plan(void* base, int64_t batch, int64_t total_q) {
    imt::MtPlan p;
    mt_plan_layout(batch, total_q, 0, false, &p, base);
    return p;
}

// Scores of every query row of the batch into rows of `scores` (leading
// dimension ld).  skip_short: requests with context <= 2048 are not scored
// (their rows select everything without scores).  full_rows: every row gets
// its whole context (positions past its own are -inf); otherwise a row block
// stops at its last row's position.
dsa_status launch_indexer_rows(const uint8_t* q8, const float* wq, const uint8_t* cache, const dsa_batch* b,
                               float* scores, int64_t ld, bool skip_short, bool full_rows, void* plan_ws, int G,
                               int32_t* st, cudaStream_t s) {
    CUtensorMap kmap, qmap;
    if (!make_index_tmap(cache, b->num_pages, false, &kmap)) return DSA_ERR_CUDA;
    if (!make_q8_tmap(q8, b->total_q, &qmap)) return DSA_ERR_CUDA;
    if (ensure_smem_limit(reinterpret_cast<const void*>(&imt::score_rows_kernel<false>), imt::kSmemAlloc) != DSA_OK)
        return DSA_ERR_CUDA;
    BatchDev bd = to_dev(b);
    imt::MtPlan p = carve_mt_plan(plan_ws, b->batch, b->total_q);
    p.G = G;
    imt::plan_kernel<<<1, 1024, 0, s>>>(bd, skip_short ? 1 : 0, full_rows ? 1 : 0, p);
    DSA_CHECK_LAUNCH();
    imt::score_rows_kernel<false><<<G, imt::kThreads, imt::kSmemAlloc, s>>>(kmap, qmap, cache, wq, bd, p, scores, ld, st);
    DSA_CHECK_LAUNCH();
    return DSA_OK;
}

// Indexer top-2048 of every query row of a multi-row batch without score rows:
// plan, streaming score kernel, then the decode indexer's merge in row mode.
// hist: [T, 4096] words, cleared by the query quantisation before this call.
dsa_status launch_indexer_rows_topk(const uint8_t* q8, const float* wq, uint32_t* hist, const uint8_t* cache,
                                    const dsa_batch* b, int32_t* topk, float* topk_scores, void* plan_ws, int G,
                                    int32_t* st, cudaStream_t s) {
    CUtensorMap kmap, qmap;
    if (!make_index_tmap(cache, b->num_pages, false, &kmap)) return DSA_ERR_CUDA;
    if (!make_q8_tmap(q8, b->total_q, &qmap)) return DSA_ERR_CUDA;
    if (ensure_smem_limit(reinterpret_cast<const void*>(&imt::score_rows_kernel<true>), imt::kSmemAlloc) != DSA_OK)
        return DSA_ERR_CUDA;
    BatchDev bd = to_dev(b);
    imt::MtPlan p;
    mt_plan_layout(b->batch, b->total_q, G, true, &p, plan_ws);
    p.hist = hist;
    imt::plan_kernel<<<1, 1024, 0, s>>>(bd, 1, 0, p);
    DSA_CHECK_LAUNCH();
    imt::score_rows_kernel<true><<<G, imt::kThreads, imt::kSmemAlloc, s>>>(kmap, qmap, cache, wq, bd, p, nullptr, 0, st);
    DSA_CHECK_LAUNCH();
    Plan mp{};
    mp.cand_key = p.cand_key;
    mp.cand_pos = p.cand_pos;
    mp.cand_cnt = p.cand_cnt;
    mp.hist = hist;
    mp.slot_row = p.slot_row;
    mp.row_seg0 = p.row_seg0;
    mp.row_segn = p.row_segn;
    mp.nslots = p.nslots;
    mp.seg_stride = imt::kSlotCap;
    const int64_t nb_max = (b->total_q + imt::kRows - 1) / imt::kRows + b->batch;
    return launch_topk_merge(b, mp, (int64_t)imt::kRows * (nb_max + G), topk, topk_scores, s);
}

}  // namespace dsa
