// Fused lightning indexer + top-2048 for decode rows (one query token per
// request) on the 5th-generation tensor cores ("vLLM 推理链路概览", DSA
// Indexer: s_j = sum_m w_m ReLU(<q_m, k_j>), I = TopK_{j,2048}(s_j);
// "GLM-5.3 推理全链路(十一)", 优化一: the index-K cache is read page by page).
//
// Per request the score is a dense contraction [L tokens x 128] x [128 x 32
// heads] in FP8: the index-K tile (128 tokens = two 64-token pages) is the A
// operand (M = 128), the request's quantised query the B operand (N = 32).
//
//  1. prep kernel: block 0 cuts the concatenated tiles of all requests that
//     need scoring (context > 2048) into one contiguous, equal share per CTA
//     (a share is split at request boundaries into segments); the other
//     blocks quantise the index queries, a warp per head, and clear the row
//     histograms.
//  2. score kernel (persistent, one CTA per SM, warp-specialised, 11 warps):
//       warps 0, 10  TMA producers, taking alternate tiles: per tile, two 8 KB
//                    payload boxes through a 128-byte-swizzled tensor map into
//                    a 9-stage ring the two warps share, and the two 256-B
//                    key-scale rows by bulk copy into a ring of their own;
//       warp 1       tcgen05.mma issuer (kind::f8f6f4, M=128, N=32, K=4x32)
//                    into one of 16 TMEM accumulators, so the tensor pipe runs
//                    up to 16 tiles ahead of the epilogue;
//       warps 2-9    epilogue, two groups of four warps taking alternate
//                    tiles: tcgen05.ld of a token's 32 head dots, ReLU, head-
//                    weighted sum, times the token's key scale; keys above the
//                    running threshold are appended to a shared-memory
//                    candidate buffer (4608 entries with a 4096-bin histogram
//                    of 16-bit counts), compacted by radix select whenever it
//                    fills; the threshold rises to the 2048th key.  At a
//                    segment end the buffer and its histogram go to the
//                    workspace.
//     No full score row is ever written to memory.
//  3. merge: one block per segment keeps the candidates at or above the bin
//     of its row's 2048th key (the row histogram of all segment candidates
//     gives that bin); one block per query row then selects the rest of the
//     2048 inside that bin exactly (ties -> lower position) and sorts by
//     position.
// The global top-2048 is inside the union of the segment top-2048s, and the
// shared (key desc, position asc) order makes ties consistent.
#include "dsa_internal.cuh"
#include "indexer_common.cuh"
#include "indexer_tc.cuh"
#include "select_common.cuh"
#include "sm100.cuh"

#include <cudaTypedefs.h>

namespace dsa {
namespace itc {

using namespace sm100;

constexpr int kStages = 9;
constexpr int kAcc = 16;                        // TMEM accumulators (32 columns each) in flight
constexpr int kSSlots = 16;                     // key-scale slots (512 B each), released by the epilogue
constexpr int kStageBytes = 16384;              // 2 x 8192 FP8 payload (two 64-token pages)
constexpr int kPidChunk = 64;                   // tiles whose page ids a producer fetches at once
constexpr int kCheckEvery = 4;                  // tiles between epilogue-wide checks
constexpr int kMinTiles = 16;                   // smallest per-CTA share of tiles
constexpr int kCap = 4608;                      // candidate buffer entries
constexpr int kSegCand = kCap;                  // candidate slots of one segment in the workspace
static_assert(kSegCand == kSegCandidates, "segment slots shared with the multi-row indexer");
constexpr int kEpiThreads = 256;                // two epilogue groups of 4 warps, alternating tiles
constexpr int kThreads = 96 + kEpiThreads;      // + two producer warps + MMA warp
constexpr int kProducer2Warp = (64 + kEpiThreads) / 32;   // the second producer, after the epilogue warps
constexpr int kEpiBar = 1;
constexpr int kTmemCols = 32 * kAcc;
constexpr uint32_t kIdesc = idesc_e4m3_f32(128, 32);
constexpr uint32_t kIdescMx = kIdesc | (5u << 7);       // A operand E2M1 (the MXFP4 keys), B E4M3

constexpr int kOffStages = 0;
// A tile's key scales (2 x 256 B) and page mask sit in a ring of their own,
// held until the epilogue has read them, so a 16 KB payload stage is free as
// soon as its MMAs are done and the MMA can run kAcc tiles ahead of the
// epilogue (a compaction of the candidate buffer then stalls no copy).
constexpr int kOffScales = kOffStages + kStages * kStageBytes;   // kSSlots x 512 B of key scales
constexpr int kOffB = (kOffScales + kSSlots * 512 + 1023) / 1024 * 1024;   // quantised query, 2 x 4 KB
constexpr int kOffCbKey = kOffB + 2 * 4096;                      // candidate keys
constexpr int kOffCbPos = kOffCbKey + kCap * 4;                  // candidate positions
constexpr int kOffHist = kOffCbPos + kCap * 4;                   // top-12-bit histogram of the candidates,
                                                                 // 16-bit counts, two bins per word
constexpr int kOffHist2 = kOffHist + 4096 * 2;                   // compaction scratch histogram
constexpr int kOffSideKey = kOffHist2;                           // survivors (reuse the scratch histogram)
constexpr int kOffSidePos = kOffSideKey + kTopK * 4;
constexpr int kOffBars = kOffHist2 + 4096 * 4;
constexpr int kOffPid = kOffBars + (2 * kStages + 2 * kAcc + 2 * kSSlots + 2) * 8;
constexpr int kOffMisc = kOffPid + 2 * kPidChunk * 2 * 8;      // one page-id buffer per producer warp
constexpr int kMiscBytes = 512;
constexpr int kSmemUsed = kOffMisc + kMiscBytes;
constexpr int kSmemAlloc = kSmemUsed + 1024;                     // slack for 1 KB alignment
static_assert(kSmemAlloc <= 232448, "shared memory budget");

struct Misc {
    int32_t slot_valid[kSSlots];                // page mask of the tile in each scale slot
    uint32_t tmem_base;
    int32_t cb_count;
    uint32_t theta;
    int32_t abort;
    sel::Found found;
    int32_t scratch[32];
    int32_t wtot[8];
    int64_t plast[2];                           // last tile each producer warp issued (-1: none)
};
static_assert(sizeof(Misc) <= kMiscBytes, "misc block");
static_assert(kAcc % 2 == 0 && kTmemCols <= 512, "accumulators alternate between two epilogue groups");
static_assert(kSSlots >= kStages, "scale ring at least as deep as the payload ring");
static_assert(kCap < 65536, "16-bit histogram counts");
static_assert(kCap % kEpiThreads == 0 && kCap / kEpiThreads <= 32, "per-thread candidate slice");

__device__ __forceinline__ int64_t cta_start(int64_t g, int64_t N, int64_t G) { return g * N / G; }
__device__ __forceinline__ int64_t cta_of_tile(int64_t x, int64_t N, int64_t G) { return ((x + 1) * G + N - 1) / N - 1; }

// The work plan, by one block of NT threads: tile prefix over the requests
// that need scoring, an equal share of tiles per CTA (at least kMinTiles), and
// the segments (request x CTA pieces) each CTA streams.
template <int NT>
__device__ void plan_block(BatchDev b, int G_launch, Plan p, int32_t* scratch) {
    int G = G_launch;                                  // CTAs that get a share (<= G_launch)
    const int gt = threadIdx.x;
    // pass 1: tile prefix over requests that need scoring
    int64_t run = 0;
    for (int base = 0; base < b.batch; base += NT) {
        const int r = base + gt;
        int tiles = 0;
        if (r < b.batch) {
            const int L = b.seq_len[r];
            const int qn = b.q_start[r + 1] - b.q_start[r];
            tiles = (qn > 0 && L > kTopK) ? (L + 127) / 128 : 0;
        }
        int total;
        const int ex = sel::excl_scan<NT, 0>(tiles, gt, scratch, &total);
        if (r < b.batch) p.tile_start[r] = run + ex;
        run += total;
    }
    const int64_t N = run;
    if (gt == 0) p.tile_start[b.batch] = N;
    // no CTA share below kMinTiles tiles: small batches use fewer CTAs
    if (N > 0 && N < (int64_t)G * kMinTiles) G = (int)max((int64_t)1, (N + kMinTiles - 1) / kMinTiles);
    __syncthreads();
    // pass 2: pieces per request (CTA boundaries inside it) and their prefix
    int32_t srun = 0;
    for (int base = 0; base < b.batch; base += NT) {
        const int r = base + gt;
        int np = 0;
        if (r < b.batch) {
            const int64_t s0 = p.tile_start[r], s1 = p.tile_start[r + 1];
            if (s1 > s0) np = (int)(cta_of_tile(s1 - 1, N, G) - cta_of_tile(s0, N, G) + 1);
        }
        int total;
        const int ex = sel::excl_scan<NT, 0>(np, gt, scratch, &total);
        if (r < b.batch) p.seg_first[r] = srun + ex;
        srun += total;
    }
    if (gt == 0) p.seg_first[b.batch] = srun;
    for (int g = gt; g < G_launch; g += NT) {          // every launched CTA, also the idle ones
        p.cta_range[2 * g] = 0;
        p.cta_range[2 * g + 1] = 0;
    }
    __syncthreads();
    // pass 3: segment records, one thread per segment
    const int32_t ns_total = srun;
    for (int s = gt; s < ns_total; s += NT) {
        int lo = 0, hi = b.batch - 1;                  // request r: seg_first[r] <= s < seg_first[r+1]
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (p.seg_first[mid] <= s) lo = mid; else hi = mid - 1;
        }
        const int r = lo;
        const int64_t s0 = p.tile_start[r], s1 = p.tile_start[r + 1];
        const int64_t g0 = cta_of_tile(s0, N, G), g1 = cta_of_tile(s1 - 1, N, G);
        const int64_t g = g0 + (s - p.seg_first[r]);
        const int64_t tlo = (g == g0) ? s0 : cta_start(g, N, G);
        const int64_t thi = (g == g1) ? s1 : cta_start(g + 1, N, G);
        p.segs[s] = Seg{r, (int32_t)(tlo - s0), (int32_t)(thi - s0), (int32_t)g};
        p.cand_cnt[s] = 0;                             // a segment the score kernel gives up on stays empty
    }
    __syncthreads();
    // pass 4: each CTA's contiguous run of segments
    const int32_t ns = srun;
    for (int s = gt; s < ns; s += NT) {
        const int32_t g = p.segs[s].cta;
        if (s == 0 || p.segs[s - 1].cta != g) p.cta_range[2 * g] = s;
        if (s == ns - 1 || p.segs[s + 1].cta != g) p.cta_range[2 * g + 1] = s + 1;
    }
}

// One launch before the score kernel: block 0 builds the plan, blocks 1.. quantise
// the index queries (one warp per (row, head)) and clear the row histograms.  The
// two jobs are independent, so they share the launch instead of running back to back.
constexpr int kPrepThreads = 256;
__global__ void __launch_bounds__(kPrepThreads)
prep_kernel(BatchDev b, int G_launch, Plan p, const uint16_t* __restrict__ q, const float* __restrict__ w,
            int64_t rows, uint8_t* __restrict__ q8, float* __restrict__ wq) {
    __shared__ int32_t scratch[32];
    pdl_wait();
    pdl_trigger();
    if (blockIdx.x == 0) {
        plan_block<kPrepThreads>(b, G_launch, p, scratch);
        return;
    }
    const int64_t g = (int64_t)(blockIdx.x - 1) * (kPrepThreads / 32) + (threadIdx.x >> 5);   // row*32 + head
    if (g < rows * 32) index_q_quant_warp(q, w, g, threadIdx.x & 31, q8, wq, p.hist);
}

__device__ __forceinline__ void epi_sync() { sel::gsync<kEpiThreads, kEpiBar>(); }

// Barrier over the epilogue threads that also returns the OR of `pred`:
// every epilogue thread gets the same answer.
__device__ __forceinline__ bool epi_any(bool pred) {
    uint32_t r;
    asm volatile("{\n .reg .pred p, q;\n setp.ne.u32 p, %1, 0;\n bar.red.or.pred q, %2, %3, p;\n"
                 " selp.u32 %0, 1, 0, q;\n}"
                 : "=r"(r) : "r"((uint32_t)pred), "n"(kEpiBar), "n"(kEpiThreads) : "memory");
    return r != 0;
}


// Crossing bin of a 4096-bin histogram read from the top: count(bins > b) <
// k <= count(bins >= b).  Thread et owns the 16 bins 4095-16et .. 4080-16et
// (four 16-byte loads of 32-bit counts, or two of 16-bit counts packed two to
// a word, bin b in half b & 1 of word b >> 1); the prefix over threads is a
// warp scan plus one exchange of warp totals.
template <bool kU16>
__device__ __forceinline__ void crossing_bin_4096(const uint32_t* h, int k, int et, Misc* misc) {
    const int lane = et & 31, wid = et >> 5;
    const uint4* h4 = reinterpret_cast<const uint4*>(h);
    uint32_t c[16];
    if constexpr (kU16) {
#pragma unroll
        for (int q = 0; q < 2; ++q) {
            const uint4 v = h4[511 - (et * 2 + q)];       // bins 4095-16et-8q-7 .. 4095-16et-8q
            const uint32_t wv[4] = {v.w, v.z, v.y, v.x};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                c[8 * q + 2 * e] = wv[e] >> 16;
                c[8 * q + 2 * e + 1] = wv[e] & 0xffffu;
            }
        }
    } else {
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const uint4 v = h4[1023 - (et * 4 + q)];      // bins 4095-16et-4q-3 .. 4095-16et-4q
            c[4 * q + 0] = v.w;
            c[4 * q + 1] = v.z;
            c[4 * q + 2] = v.y;
            c[4 * q + 3] = v.x;
        }
    }
    int mine = 0;
#pragma unroll
    for (int q = 0; q < 16; ++q) mine += (int)c[q];
    int x = mine;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) misc->wtot[wid] = x;
    epi_sync();
    int above = x - mine;
    for (int v = 0; v < wid; ++v) above += misc->wtot[v];
#pragma unroll
    for (int q = 0; q < 16; ++q) {
        if (above < k && above + (int)c[q] >= k) {
            misc->found.bin = (uint32_t)(4095 - (et * 16 + q));
            misc->found.above = above;
        }
        above += (int)c[q];
    }
    epi_sync();
}

// Same for a 256-bin histogram: one bin per thread.
__device__ __forceinline__ void crossing_bin_256(const uint32_t* h, int k, int et, Misc* misc) {
    const int lane = et & 31, wid = et >> 5;
    const int mine = (int)h[255 - et];
    int x = mine;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) misc->wtot[wid] = x;
    epi_sync();
    int above = x - mine;
    for (int v = 0; v < wid; ++v) above += misc->wtot[v];
    if (above < k && above + mine >= k) {
        misc->found.bin = (uint32_t)(255 - et);
        misc->found.above = above;
    }
    epi_sync();
}

// Keep the exact top-2048 (key desc, position asc) of the candidate buffer.
// hist holds the top-12-bit histogram of the buffer on entry and of the
// survivors on exit (16-bit counts, two bins per word).  Called by all epilogue threads with cb_count > 2048.
// The survivors' order in the buffer is not preserved (it does not matter:
// ties are resolved by position values and the merge sorts by position).
__device__ void compact_candidates(uint32_t* cb_key, int32_t* cb_pos, uint32_t* hist, uint32_t* hist2,
                                   uint32_t* side_key, int32_t* side_pos, Misc* misc, int et) {
    constexpr int NT = kEpiThreads;
    const int n = misc->cb_count;
    constexpr int kPer = kCap / NT;                // entries per thread (strided by NT)
    crossing_bin_4096<true>(hist, kTopK, et, misc);
    const uint32_t b1 = misc->found.bin;
    const int above1 = misc->found.above;            // candidates in bins above b1: all survive
    int krem = kTopK - above1;
    for (int i = et; i < 4096; i += NT) hist2[i] = 0u;
    epi_sync();
    uint32_t k[kPer];
#pragma unroll
    for (int u = 0; u < kPer; ++u) k[u] = (et + u * NT < n) ? cb_key[et + u * NT] : 0u;
#pragma unroll
    for (int u = 0; u < kPer; ++u)                   // second digit among bin b1
        if (et + u * NT < n && (k[u] >> 20) == b1) atomicAdd(&hist2[(k[u] >> 8) & 0xfffu], 1u);
    epi_sync();
    crossing_bin_4096<false>(hist2, krem, et, misc);
    const uint32_t b2 = misc->found.bin;
    krem -= misc->found.above;
    epi_sync();
    hist2[et] = 0u;                                    // 256 bins, one per thread
    epi_sync();
    const uint32_t pre = (b1 << 12) | b2;
#pragma unroll
    for (int u = 0; u < kPer; ++u)                   // third digit among prefix (b1, b2)
        if (et + u * NT < n && (k[u] >> 8) == pre) atomicAdd(&hist2[k[u] & 0xffu], 1u);
    epi_sync();
    crossing_bin_256(hist2, krem, et, misc);
    const uint32_t b3 = misc->found.bin;
    const int need_eq = krem - misc->found.above;
    const int n_eq = (int)hist2[b3];
    epi_sync();
    const uint32_t kth = (b1 << 20) | (b2 << 8) | b3;
    int32_t pmax = 0x7fffffff;
    if (n_eq > need_eq) {                          // exact ties at the cut: lowest positions win
        sel::SmemSrc<NT> src{cb_key, cb_pos, n};
        sel::TieSrc<sel::SmemSrc<NT>> ts{src, kth};
        uint32_t tk;
        int ne2;
        sel::radix_kth<NT, kEpiBar>(ts, need_eq, et, hist2, misc->scratch, &misc->found, &tk, &ne2, nullptr);
        pmax = (int32_t)(0x7fffffffu - tk);
    }
    // survivors into the side buffer (which reuses hist2): count, scan, write
    uint32_t keepm = 0;
    int cnt = 0;
#pragma unroll
    for (int u = 0; u < kPer; ++u) {
        const int i = et + u * NT;
        const bool keep = i < n && (k[u] > kth || (k[u] == kth && cb_pos[i] <= pmax));
        keepm |= (keep ? 1u : 0u) << u;
        cnt += keep ? 1 : 0;
    }
    const int lane = et & 31, wid = et >> 5;
    int x = cnt;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) misc->wtot[wid] = x;
    epi_sync();
    int off = x - cnt;
    for (int v = 0; v < wid; ++v) off += misc->wtot[v];
    int total = 0;
    for (int v = 0; v < NT / 32; ++v) total += misc->wtot[v];
#pragma unroll
    for (int u = 0; u < kPer; ++u) {
        if ((keepm >> u) & 1u) {
            if (off < kTopK) {
                side_key[off] = k[u];
                side_pos[off] = cb_pos[et + u * NT];
            }
            ++off;
        }
    }
    // survivors' histogram: bins above b1 keep their counts, b1 keeps the rest
    uint16_t* h16 = reinterpret_cast<uint16_t*>(hist);
    for (int i = et; i < 4096; i += NT) {
        if ((uint32_t)i < b1) h16[i] = 0u;
        else if ((uint32_t)i == b1) h16[i] = (uint16_t)(kTopK - above1);
    }
    epi_sync();
    total = min(total, kTopK);
    for (int i = et; i < total; i += NT) {
        cb_key[i] = side_key[i];
        cb_pos[i] = side_pos[i];
    }
    if (et == 0) {
        misc->cb_count = total;
        misc->theta = kth;
    }
    epi_sync();
}

// kMx: the MXFP4 index-K cache ("GLM-5.3 推理全链路(十一)", 两个框架的对照).  The
// TMA unpacks each page's 64 packed 64-byte rows into the same 128-byte rows as
// FP8 (16U4_ALIGN16B: eight bytes of values, eight bytes of gap, the E2M1
// operand layout of kind::f8f6f4), so the stage ring is unchanged; the MMA
// takes A as E2M1 and writes one 32-column accumulator per 32-dim block (four
// per tile), and the epilogue applies the blocks' ue8m0 scales before the ReLU.
template <bool kMx>
__global__ void __launch_bounds__(kThreads, 1)
score_topk_kernel(const __grid_constant__ CUtensorMap tmap, const uint8_t* __restrict__ cache,
                  const uint8_t* __restrict__ q8, const float* __restrict__ wq, BatchDev b, Plan p,
                  int32_t* __restrict__ st) {
    extern __shared__ uint8_t smem_raw[];
    // 1 KB alignment by offset (not through an integer cast) so that every
    // access below stays a shared-memory access.
    uint8_t* smem = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + kOffBars);
    uint64_t* empty = full + kStages;
    uint64_t* accf = empty + kStages;                      // [kAcc] accumulator written
    uint64_t* acce = accf + kAcc;                          // [kAcc] accumulator read by the epilogue
    uint64_t* sfull = acce + kAcc;                         // [kSSlots] key scales landed
    uint64_t* sempty = sfull + kSSlots;                    // [kSSlots] key scales read
    uint64_t* bdone = sempty + kSSlots;                    // [2] MMAs reading a query buffer done
    int64_t* pid = reinterpret_cast<int64_t*>(smem + kOffPid);
    Misc* misc = reinterpret_cast<Misc*>(smem + kOffMisc);
    uint32_t* cb_key = reinterpret_cast<uint32_t*>(smem + kOffCbKey);
    int32_t* cb_pos = reinterpret_cast<int32_t*>(smem + kOffCbPos);
    uint32_t* hist = reinterpret_cast<uint32_t*>(smem + kOffHist);
    uint32_t* hist2 = reinterpret_cast<uint32_t*>(smem + kOffHist2);
    uint32_t* side_key = reinterpret_cast<uint32_t*>(smem + kOffSideKey);
    int32_t* side_pos = reinterpret_cast<int32_t*>(smem + kOffSidePos);

    constexpr int kAccCols = kMx ? 128 : 32;               // TMEM columns of one tile's accumulator
    constexpr int kAccN = kTmemCols / kAccCols;            // accumulators in flight
    constexpr int kMapRows = kMx ? 68 : 66;                // 64 payload rows + the scales, per page
    constexpr int kPageBytes = kMx ? DSA_IDXK_MXFP4_PAGE_BYTES : kIdxPageBytes;
    constexpr int kPayBytes = kMx ? 64 * 64 : kIdxPayloadBytes;
    constexpr int kSt = kStages;                           // payload stages
    static_assert(kAccN % 2 == 0 && kAccN <= kAcc, "accumulator barriers");
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int s = 0; s < kSt; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);              // the MMA commit
        }
        for (int a = 0; a < kAcc; ++a) {
            mbar_init(&accf[a], 1);
            mbar_init(&acce[a], 4);
        }
        for (int j = 0; j < kSSlots; ++j) {
            mbar_init(&sfull[j], 1);
            mbar_init(&sempty[j], 4);             // one arrive per warp of the epilogue group
        }
        mbar_init(&bdone[0], 1);
        mbar_init(&bdone[1], 1);
        misc->abort = 0;
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
    pdl_wait();                                            // the plan and the quantised queries
    int s_begin = p.cta_range[2 * blockIdx.x], s_end = p.cta_range[2 * blockIdx.x + 1];
    const int nseg_max = (int)gridDim.x + b.batch;    // segment slots in the workspace
    if (s_begin < 0 || s_end > nseg_max || s_begin > s_end) {   // never for a plan from prep_kernel
        if (threadIdx.x == 0) record_error(st, DSA_DEVERR_INDEX_RANGE, s_begin);
        s_begin = s_end = 0;
    }
    volatile int32_t* abort_flag = &misc->abort;

    if (warp == 0 || warp == kProducer2Warp) {
        // ------------------------------------------------------------ producers
        // Two producer warps take alternate tiles of the CTA's running tile
        // index (one thread issuing every copy of an SM falls well short of
        // the HBM rate; two reach it).  Tile i uses stage i % kStages and
        // scale slot i % kSSlots; with an odd stage count the warps share the
        // stage ring, which is safe because tile i waits for the consumption
        // of tile i - kStages (and the warp's own previous tile already
        // waited for that of tile i - kStages - 2, so the parity cannot alias).
        // A warp fetches the page ids of up to kPidChunk tiles at once into
        // its own buffer; its lane 0 then issues the copies of its tiles
        // without waiting on global loads.
        const int me = warp == 0 ? 0 : 1;
        int64_t* mypid = pid + me * kPidChunk * 2;
        int64_t icount = 0;                                // running tile index (lane 0)
        int64_t last = -1;                                 // last tile this warp issued (lane 0)
        bool stop = false;
        for (int s = s_begin; s < s_end && !stop; ++s) {
            const Seg sg = p.segs[s];
            const int L = b.seq_len[sg.r];
            const int32_t* pt = b.page_table + (int64_t)sg.r * b.max_pages;
            for (int c0 = sg.lo; c0 < sg.hi && !stop; c0 += kPidChunk) {
                const int nt = min(kPidChunk, sg.hi - c0);
                for (int k = lane; k < 2 * nt; k += 32) {
                    const int idx = c0 * 2 + k;
                    mypid[k] = idx < b.max_pages ? (int64_t)pt[idx] : (int64_t)-2;
                }
                __syncwarp();
                int ok = 1;
                if (lane == 0) {
                    for (int tile = c0; tile < c0 + nt; ++tile, ++icount) {
                        if ((int)(icount & 1) != me) continue;
                        const int stage = (int)(icount % kSt);
                        const uint32_t phase = (uint32_t)((icount / kSt) & 1);
                        const int slot = (int)(icount % kSSlots);
                        const uint32_t sphase = (uint32_t)((icount / kSSlots) & 1);
                        if (*abort_flag || !mbar_wait(&empty[stage], phase ^ 1, b.wait_ns) ||
                            !mbar_wait(&sempty[slot], sphase ^ 1, b.wait_ns)) {
                            ok = 0;
                            break;
                        }
                        const int t0 = tile * 128;
                        const int pages = (L - t0 > 64) ? 2 : 1;
                        int nvalid = 0;                    // pages copied
                        int vmask = 0;
                        int64_t pg[2];
                        for (int j = 0; j < pages; ++j) {
                            pg[j] = mypid[(tile - c0) * 2 + j];
                            if (pg[j] >= 0 && pg[j] < b.num_pages) {
                                vmask |= 1 << j;
                                ++nvalid;
                            } else if (pg[j] == -2) {
                                record_error(st, DSA_DEVERR_INDEX_RANGE, t0 + j * 64);   // beyond the page table row
                            } else {
                                record_error(st, DSA_DEVERR_PAGE_RANGE, pg[j]);
                            }
                        }
                        misc->slot_valid[slot] = vmask;     // read after sfull[slot]
                        uint8_t* sb = smem + kOffStages + stage * kStageBytes;
                        // the copy counts the bytes read: 8192 FP8 or 4096 packed E2M1 per page
                        mbar_arrive_expect_tx(&full[stage], (uint32_t)(nvalid * kPayBytes));
                        mbar_arrive_expect_tx(&sfull[slot], (uint32_t)(nvalid * 256));
                        for (int j = 0; j < pages; ++j) {
                            if (!(vmask & (1 << j))) continue;
                            tma_load_2d(sb + j * 8192, &tmap, 0, (int32_t)(pg[j] * kMapRows), &full[stage]);
                            bulk_load(smem + kOffScales + slot * 512 + j * 256,
                                      cache + pg[j] * (int64_t)kPageBytes + kPayBytes, 256, &sfull[slot]);
                        }
                        last = icount;
                    }
                }
                ok = __shfl_sync(0xffffffffu, ok, 0);
                if (!ok) stop = true;
                __syncwarp();
            }
        }
        if (lane == 0 && stop) {
            if (!*abort_flag) record_error(st, DSA_DEVERR_TIMEOUT, 1);
            *abort_flag = 1;
        }
        if (lane == 0) misc->plast[me] = last;          // for the drain after an abort, below
        __syncwarp();
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        // Lane 0 waits and issues; every decision is broadcast so the warp
        // never diverges around its __syncwarp / shuffles.
        int stage = 0, acc = 0, bbuf = 0;
        uint32_t phase = 0, acc_phase = 0;
        bool issued_any = false, stop = false;
        int last_acc = 0;
        uint32_t last_acc_phase = 0;
        // With kAcc tiles in flight, the MMAs of two segments back may still
        // read a query buffer when it is due to be rewritten: each segment
        // commits to its buffer's bdone barrier, and the rewrite waits on it.
        uint32_t bph = 0u, bpending = 0u;                  // bit j: query buffer j
        for (int s = s_begin; s < s_end && !stop; ++s) {
            const Seg sg = p.segs[s];
            const int64_t row = b.q_start[sg.r];
            uint8_t* bq = smem + kOffB + bbuf * 4096;
            bool seg_issued = false;
            for (int tile = sg.lo; tile < sg.hi; ++tile) {
                int ok = 1;
                if (lane == 0) ok = (!*abort_flag && mbar_wait(&acce[acc], acc_phase ^ 1, b.wait_ns)) ? 1 : 0;
                ok = __shfl_sync(0xffffffffu, ok, 0);
                if (!ok) { stop = true; break; }
                if (tile == sg.lo) {
                    if ((bpending >> bbuf) & 1u) {
                        if (lane == 0) ok = mbar_wait(&bdone[bbuf], (bph >> bbuf) & 1u, b.wait_ns) ? 1 : 0;
                        ok = __shfl_sync(0xffffffffu, ok, 0);
                        if (!ok) { stop = true; break; }
                        bph ^= 1u << bbuf;
                        bpending &= ~(1u << bbuf);
                    }
                    // B operand: head `lane` row of the quantised query, 128-byte swizzled
                    const uint4* src = reinterpret_cast<const uint4*>(q8 + row * 4096 + lane * 128);
#pragma unroll
                    for (int c = 0; c < 8; ++c)
                        *reinterpret_cast<uint4*>(bq + lane * 128 + ((c ^ (lane & 7)) * 16)) = src[c];
                    fence_proxy_async_smem();
                    __syncwarp();
                }
                if (lane == 0) {
                    ok = mbar_wait(&full[stage], phase, b.wait_ns) ? 1 : 0;
                    if (ok) {
                        tc_fence_after();
                        const uint32_t a0 = smem_addr(smem + kOffStages + stage * kStageBytes);
                        const uint32_t b0 = smem_addr(bq);
#pragma unroll
                        for (int k = 0; k < 4; ++k) {
                            if constexpr (kMx)            // one accumulator per 32-dim scale block
                                mma_f8f6f4(tmem + acc * kAccCols + 32 * k, desc_kmajor_sw128(a0 + 32 * k),
                                           desc_kmajor_sw128(b0 + 32 * k), kIdescMx, 0u);
                            else
                                mma_f8f6f4(tmem + acc * 32, desc_kmajor_sw128(a0 + 32 * k),
                                           desc_kmajor_sw128(b0 + 32 * k), kIdesc, k > 0 ? 1u : 0u);
                        }
                        mma_commit(&empty[stage]);
                        mma_commit(&accf[acc]);
                        issued_any = true;
                        seg_issued = true;
                        last_acc = acc;
                        last_acc_phase = acc_phase;
                    }
                }
                ok = __shfl_sync(0xffffffffu, ok, 0);
                if (!ok) { stop = true; break; }
                if (++stage == kSt) { stage = 0; phase ^= 1; }
                if (++acc == kAccN) { acc = 0; acc_phase ^= 1; }
            }
            seg_issued = __shfl_sync(0xffffffffu, seg_issued ? 1 : 0, 0) != 0;
            if (seg_issued) {
                if (lane == 0) mma_commit(&bdone[bbuf]);
                bpending |= 1u << bbuf;
            }
            bbuf ^= 1;
        }
        issued_any = __shfl_sync(0xffffffffu, issued_any ? 1 : 0, 0) != 0;
        if (lane == 0 && stop) {
            record_error(st, DSA_DEVERR_TIMEOUT, 2);
            *abort_flag = 1;
        }
        // no MMA in flight when the TMEM is released, also when the epilogue gave up
        // after every tile was issued (MMAs complete in issue order)
        if (lane == 0 && issued_any) mbar_wait(&accf[last_acc], last_acc_phase, 500000000ull);
        __syncwarp();
    } else {
        // ------------------------------------------------------------ epilogue
        // Two groups of 4 warps; group g takes the tiles whose running index
        // has parity g (accumulator index % kAcc, so the parity of the
        // accumulator too).  Warp w may read TMEM lanes
        // 32*(w%4) .. 32*(w%4)+31, i.e. tokens 32*(w%4) .. of the tile.
        const int et = threadIdx.x - 64;
        const int grp = (warp - 2) >> 2;
        const int quarter = warp & 3;
        const int tok = quarter * 32 + lane;
        int64_t gidx = 0;                              // running tile index of this CTA
        for (int s = s_begin; s < s_end; ++s) {
            if (epi_any(*abort_flag != 0)) break;
            const Seg sg = p.segs[s];
            const int L = b.seq_len[sg.r];
            const int64_t row = b.q_start[sg.r];
            const int n_valid = L;                     // one decode row: positions 0..L-1
            float w[32];
#pragma unroll
            for (int m = 0; m < 32; ++m) w[m] = __ldg(wq + row * 32 + m);
            if (et == 0) {
                misc->cb_count = 0;
                misc->theta = 0u;
            }
            for (int i = et; i < 2048; i += kEpiThreads) hist[i] = 0u;
            epi_sync();
            bool aborted = false;
            bool warp_bad = false;                     // this warp saw a timeout
            // The next epilogue-wide check, in tiles of the segment: the buffer takes at
            // most 128 candidates a tile, so it cannot overflow before (kCap - count) / 128.
            int next_check = kCap / 128;
            for (int tile = sg.lo; tile < sg.hi; ++tile, ++gidx) {
                if ((int)(gidx & 1) == grp && !warp_bad) {
                    const int slot = (int)(gidx % kSSlots);
                    const uint32_t sphase = (uint32_t)((gidx / kSSlots) & 1);
                    const int acc = (int)(gidx % kAccN);
                    const uint32_t acc_phase = (uint32_t)((gidx / kAccN) & 1);
                    int ok = __all_sync(0xffffffffu, mbar_wait(&accf[acc], acc_phase, b.wait_ns));
                    if (ok) ok = __all_sync(0xffffffffu, mbar_wait(&sfull[slot], sphase, b.wait_ns));   // scales + page mask
                    if (ok) {
                        float score;
                        int vmask;
                        if constexpr (kMx) {
                            // x_h = sum over the 4 blocks of 2^(e_b) acc_b[h], 16 heads at a time
                            const uint32_t ew = reinterpret_cast<const uint32_t*>(smem + kOffScales + slot * 512)[tok];
                            vmask = misc->slot_valid[slot];
                            float sc[4];
#pragma unroll
                            for (int q = 0; q < 4; ++q) {
                                const uint32_t eb = (ew >> (8 * q)) & 255u;
                                sc[q] = eb ? __uint_as_float(eb << 23) : __uint_as_float(0x00400000u);   // 2^(eb - 127)
                            }
                            float a0 = 0.f, a1 = 0.f;
                            tc_fence_after();
#pragma unroll
                            for (int half = 0; half < 2; ++half) {
                                uint32_t v[4][16];
#pragma unroll
                                for (int q = 0; q < 4; ++q)
                                    tmem_ld_32x32b_x16(tmem + ((uint32_t)(quarter * 32) << 16) + acc * kAccCols + q * 32 +
                                                           half * 16, v[q]);
                                tmem_ld_wait();
                                if (half == 1) {
                                    tc_fence_before();
                                    __syncwarp();
                                    if (lane == 0) {
                                        mbar_arrive(&acce[acc]);
                                        mbar_arrive(&sempty[slot]);
                                    }
                                }
#pragma unroll
                                for (int m = 0; m < 16; m += 2) {
                                    float x0 = sc[0] * __uint_as_float(v[0][m]), x1 = sc[0] * __uint_as_float(v[0][m + 1]);
#pragma unroll
                                    for (int q = 1; q < 4; ++q) {
                                        x0 = fmaf(sc[q], __uint_as_float(v[q][m]), x0);
                                        x1 = fmaf(sc[q], __uint_as_float(v[q][m + 1]), x1);
                                    }
                                    a0 = fmaf(w[half * 16 + m], fmaxf(x0, 0.f), a0);
                                    a1 = fmaf(w[half * 16 + m + 1], fmaxf(x1, 0.f), a1);
                                }
                            }
                            score = a0 + a1;
                        } else {
                            uint32_t v[32];
                            tc_fence_after();
                            tmem_ld_32x32b_x32(tmem + ((uint32_t)(quarter * 32) << 16) + acc * 32, v);
                            tmem_ld_wait();
                            vmask = misc->slot_valid[slot];
                            const float sk = reinterpret_cast<const float*>(smem + kOffScales + slot * 512)[tok];
                            tc_fence_before();
                            __syncwarp();
                            if (lane == 0) {
                                mbar_arrive(&acce[acc]);
                                mbar_arrive(&sempty[slot]);
                            }
                            float a0 = 0.f, a1 = 0.f, a2 = 0.f, a3 = 0.f;
#pragma unroll
                            for (int m = 0; m < 32; m += 4) {
                                a0 = fmaf(w[m], fmaxf(__uint_as_float(v[m]), 0.f), a0);
                                a1 = fmaf(w[m + 1], fmaxf(__uint_as_float(v[m + 1]), 0.f), a1);
                                a2 = fmaf(w[m + 2], fmaxf(__uint_as_float(v[m + 2]), 0.f), a2);
                                a3 = fmaf(w[m + 3], fmaxf(__uint_as_float(v[m + 3]), 0.f), a3);
                            }
                            score = ((a0 + a1) + (a2 + a3)) * sk;
                        }
                        const int pos = tile * 128 + tok;
                        const bool valid = ((vmask >> (tok >> 6)) & 1) && pos < n_valid;
                        const uint32_t key = score_key(score);
                        const bool pass = valid && key > misc->theta;
                        const unsigned m = __ballot_sync(0xffffffffu, pass);
                        if (m) {
                            int base = 0;
                            if (lane == __ffs(m) - 1) base = atomicAdd(&misc->cb_count, __popc(m));
                            base = __shfl_sync(0xffffffffu, base, __ffs(m) - 1);
                            if (pass) {
                                const int idx = base + __popc(m & ((1u << lane) - 1u));
                                cb_key[idx] = key;
                                cb_pos[idx] = pos;
                                atomicAdd(&hist[key >> 21], 1u << ((key >> 16) & 16u));   // bin key >> 20, 16-bit half
                            }
                        }
                    } else {
                        warp_bad = true;
                        if (lane == 0) {
                            record_error(st, DSA_DEVERR_TIMEOUT, 4);
                            *abort_flag = 1;
                        }
                    }
                }
                // epilogue-wide decisions (abort, buffer room) when the buffer might fill, and
                // at the segment end.  The count is read between two barriers, so every
                // thread sees the same value and none appends before all have read it.
                if (tile - sg.lo + 1 == next_check || tile + 1 == sg.hi) {
                    if (epi_any(warp_bad)) { aborted = true; break; }
                    const int c = misc->cb_count;
                    if (epi_any(c > kCap - kCheckEvery * 128)) {
                        compact_candidates(cb_key, cb_pos, hist, hist2, side_key, side_pos, misc, et);
                        next_check = tile - sg.lo + 1 + (kCap - kTopK) / 128;   // at most 2048 kept
                    } else {
                        next_check = tile - sg.lo + 1 + max(1, (kCap - c) / 128);
                    }
                }
            }
            if (aborted) break;
            // segment end: the whole buffer and its histogram, written out.  It
            // holds the segment's top-2048 (the filter never rose above the
            // segment's 2048th key) and maybe more; the merge filter cuts the
            // row's candidates at the bin of the row's 2048th key, so no exact
            // selection is needed here.
            const int cnt = misc->cb_count;
            for (int i = et; i < cnt; i += kEpiThreads) {
                p.cand_key[(int64_t)s * kSegCand + i] = cb_key[i];
                p.cand_pos[(int64_t)s * kSegCand + i] = cb_pos[i];
            }
            if (et == 0) p.cand_cnt[s] = cnt;
            uint32_t* gh = p.hist + row * 4096;
            const uint16_t* h16 = reinterpret_cast<const uint16_t*>(hist);
            for (int i = et; i < 4096; i += kEpiThreads)
                if (h16[i]) atomicAdd(&gh[i], (uint32_t)h16[i]);
            epi_sync();
        }
    }
    __syncthreads();
    pdl_trigger();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
    if (threadIdx.x == 0 && *abort_flag) {
        // After an abort, let every copy in flight land before the CTA ends.  A
        // stage or scale slot is refilled only after its previous tile was
        // consumed, so the one copy into it that may still be in flight is that
        // of the latest tile issued to it by either warp: wait for exactly that
        // tile's phase (an older tile's parity can alias a newer one's when the
        // two warps share the ring).  Warp w issued every tile of parity w up
        // to plast[w].
        for (int ring = 0; ring < 2; ++ring) {
            const int n = ring == 0 ? kSt : kSSlots;
            uint64_t* bar = ring == 0 ? full : sfull;
            for (int x = 0; x < n; ++x) {
                int64_t jl = -1;
                for (int w = 0; w < 2; ++w)
                    for (int64_t j = misc->plast[w]; j >= 0 && j > misc->plast[w] - 2 * n; j -= 2)
                        if (j % n == x) {
                            jl = j > jl ? j : jl;
                            break;
                        }
                if (jl >= 0) mbar_wait(&bar[x], (uint32_t)((jl / n) & 1), 500000000ull);
            }
        }
    }
}

// ---------------------------------------------------------------- merge
// Two kernels after the score kernel.
//  merge_filter_kernel, one block per segment: the row histogram (top 12 key
//    bits of every segment candidate of the row) gives the bin b* that holds
//    the row's 2048th key.  The block compacts its segment's candidates in
//    place to [bins > b* | bin b*] and packs the two counts into cand_cnt
//    (sure | boundary << 16); lower bins cannot reach the row's top-2048.
//  merge_kernel, one block per query row: gathers the row's sure entries,
//    selects the remaining 2048 - sure among the bin-b* entries exactly (ties
//    -> lower position), sorts the 2048 by position and writes them out.
constexpr int kFiltThreads = 512;
constexpr int kFiltCap = kSegCand > kRowSlotCandidates ? kSegCand : kRowSlotCandidates;   // a segment's entries, at most
constexpr int kFiltPer = kFiltCap / kFiltThreads;  // candidates per thread
static_assert(kFiltCap % kFiltThreads == 0 && kFiltPer <= 16, "two class bits per candidate in a 32-bit word");
static_assert(4096 % (kFiltThreads * 4) == 0, "whole 16-byte histogram loads per thread");
constexpr int kFiltBins = 4096 / kFiltThreads;     // histogram bins per thread

__global__ void __launch_bounds__(kFiltThreads)
merge_filter_kernel(BatchDev b, Plan p) {
    __shared__ int32_t scratch[32];
    __shared__ uint32_t s_bstar;
    pdl_wait();
    pdl_trigger();
    const int s = blockIdx.x;
    int64_t row;
    if (p.slot_row) {                                  // row mode
        if (s >= *p.nslots || p.slot_row[s] < 0) return;
        row = p.slot_row[s];
    } else {
        if (s >= p.seg_first[b.batch]) return;         // launched for the most segments a plan can hold
        row = b.q_start[p.segs[s].r];
    }
    const int tid = threadIdx.x;
    const int cnt = min(p.cand_cnt[s], kFiltCap);
    uint32_t* key = p.cand_key + (int64_t)s * p.seg_stride;
    int32_t* pos = p.cand_pos + (int64_t)s * p.seg_stride;
    uint32_t k[kFiltPer];
#pragma unroll
    for (int u = 0; u < kFiltPer; ++u) {               // keys first: their loads overlap the scan below
        const int i = tid + u * kFiltThreads;
        k[u] = i < cnt ? key[i] : 0u;
    }
    // b*: thread tid owns the kFiltBins bins 4095 - kFiltBins tid downwards
    const uint4* h4 = reinterpret_cast<const uint4*>(p.hist + row * 4096);
    uint32_t c[kFiltBins];
#pragma unroll
    for (int q = 0; q < kFiltBins / 4; ++q) {
        const uint4 v = __ldcg(h4 + 1023 - (tid * (kFiltBins / 4) + q));
        c[4 * q + 0] = v.w;
        c[4 * q + 1] = v.z;
        c[4 * q + 2] = v.y;
        c[4 * q + 3] = v.x;
    }
    int mine = 0;
#pragma unroll
    for (int q = 0; q < kFiltBins; ++q) mine += (int)c[q];
    if (tid == 0) s_bstar = 0u;                        // fewer than 2048 candidates: keep them all
    int tot;
    int above = sel::excl_scan<kFiltThreads, 0>(mine, tid, scratch, &tot);
#pragma unroll
    for (int q = 0; q < kFiltBins; ++q) {
        if (above < kTopK && above + (int)c[q] >= kTopK) s_bstar = (uint32_t)(4095 - (tid * kFiltBins + q));
        above += (int)c[q];
    }
    __syncthreads();
    const uint32_t bstar = s_bstar;
    int32_t ps[kFiltPer];
    uint32_t cls = 0;                                  // 2 bits per entry: 1 sure, 2 boundary
    int n_s = 0, n_b = 0;
#pragma unroll
    for (int u = 0; u < kFiltPer; ++u) {
        const int i = tid + u * kFiltThreads;
        const uint32_t bin = k[u] >> 20;
        const uint32_t cu = i >= cnt ? 0u : bin > bstar ? 1u : bin == bstar ? 2u : 0u;
        ps[u] = cu ? pos[i] : 0;                       // positions of the kept entries only
        cls |= cu << (2 * u);
        n_s += cu == 1u;
        n_b += cu == 2u;
    }
    int tot_s, tot_b;
    int off_s = sel::excl_scan<kFiltThreads, 0>(n_s, tid, scratch, &tot_s);   // every read is done past here
    int off_b = tot_s + sel::excl_scan<kFiltThreads, 0>(n_b, tid, scratch, &tot_b);
#pragma unroll
    for (int u = 0; u < kFiltPer; ++u) {
        const uint32_t cu = (cls >> (2 * u)) & 3u;
        if (cu == 1u) {
            key[off_s] = k[u];
            pos[off_s] = ps[u];
            ++off_s;
        } else if (cu == 2u) {
            key[off_b] = k[u];
            pos[off_b] = ps[u];
            ++off_b;
        }
    }
    if (tid == 0) p.cand_cnt[s] = tot_s | (tot_b << 16);
}

// Largest j < n with pre[j] <= i (pre non-decreasing, pre[0] = 0 <= i).
__device__ __forceinline__ int seg_lookup(const int32_t* pre, int n, int i) {
    int lo = 0, hi = n - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (pre[mid] <= i) lo = mid; else hi = mid - 1;
    }
    return lo;
}

// The bin-b* entries of a row's filtered segment slots, as a selection source
// (slot j: sure entries [0, ns_j), then nb_j boundary entries).
struct BndSrc {
    const uint32_t* key;        // the row's first segment slot
    const int32_t* pos;
    const int32_t* ns_pre;      // [nseg + 1] prefix of sure counts (shared memory)
    const int32_t* nb_pre;      // [nseg + 1] prefix of boundary counts (shared memory)
    int nseg, n;
    int64_t stride;             // entries from one segment slot to the next
    __device__ __forceinline__ int64_t at(int i) const {
        const int j = seg_lookup(nb_pre, nseg, i);
        return (int64_t)j * stride + (ns_pre[j + 1] - ns_pre[j]) + (i - nb_pre[j]);
    }
    template <class F>
    __device__ __forceinline__ void visit(int gt, F&& f) const {
        const int nr = (n + 1023) / 1024 * 1024;
        for (int i = gt; i < nr; i += 1024) {
            const bool a = i < n;
            const int64_t x = a ? at(i) : 0;
            f(a, a ? key[x] : 0u, a ? pos[x] : 0);
        }
    }
};

// Ascending bitonic sort of 2048 packed (position << 32 | key) values by 1024
// threads.  Thread t holds elements i0 = 64 (t / 32) + 2 (t % 32) and i0 + 1
// in registers; partner distances up to 32 are exchanged by warp shuffles and
// only distances >= 64 go through shared memory (v64, 2048 words).
__device__ __forceinline__ void sort2048_regs(uint64_t& a, uint64_t& c, uint64_t* v64, int gt) {
    const int i0 = 64 * (gt >> 5) + 2 * (gt & 31);
    auto reg_stages = [&](int size, int smax) {
        const bool up = (i0 & size) == 0;
        for (int stride = smax; stride >= 1; stride >>= 1) {
            if (stride == 1) {
                if ((a > c) == up) {
                    const uint64_t t = a;
                    a = c;
                    c = t;
                }
            } else {
                const int m = stride >> 1;
                const uint64_t pa = __shfl_xor_sync(0xffffffffu, a, m);
                const uint64_t pc = __shfl_xor_sync(0xffffffffu, c, m);
                const bool take_min = ((i0 & stride) == 0) == up;
                a = take_min ? min(a, pa) : max(a, pa);
                c = take_min ? min(c, pc) : max(c, pc);
            }
        }
    };
    for (int size = 2; size <= 64; size <<= 1) reg_stages(size, size >> 1);
    for (int size = 128; size <= kTopK; size <<= 1) {
        v64[i0] = a;
        v64[i0 + 1] = c;
        __syncthreads();
        for (int stride = size >> 1; stride >= 64; stride >>= 1) {
            const int lo = 2 * gt - (gt & (stride - 1)), hi = lo + stride;
            const bool up = (lo & size) == 0;
            const uint64_t x = v64[lo], y = v64[hi];
            if ((x > y) == up) {
                v64[lo] = y;
                v64[hi] = x;
            }
            __syncthreads();
        }
        a = v64[i0];                                   // only this thread reads or writes i0, i0 + 1 until the next barrier
        c = v64[i0 + 1];
        reg_stages(size, 32);
    }
}

constexpr int kMergeThreads = 1024;
// Boundary-bin capacity of the merge (entries kept in shared memory; the same
// bytes later hold the row's position bitmap, 64 positions per entry).  The
// large one serves contexts up to 1M positions with one block per SM; the
// small one (about 72 KB of shared memory) lets two blocks share an SM, for
// batches with more rows than SMs whose contexts fit its bitmap.  A larger
// bin is selected in place from the workspace, a longer row by a sort.
constexpr int kBndCap = 16384;
constexpr int kBndSmall = 4096;
constexpr int kMaxSegs = 1024;
constexpr int kMOffHist = 0;
constexpr int kMOffSelPos = kMOffHist + 4096 * 4;                 // selected positions, then keys: 2048 x u64 for the sort
constexpr int kMOffSelKey = kMOffSelPos + kTopK * 4;
constexpr int kMOffNs = kMOffSelKey + kTopK * 4;
constexpr int kMOffNb = kMOffNs + (kMaxSegs + 1) * 4;
constexpr int kMOffBndKey = (kMOffNb + (kMaxSegs + 1) * 4 + 15) / 16 * 16;
constexpr int merge_smem(int bnd) { return kMOffBndKey + 2 * bnd * 4 + 256; }   // boundary keys, positions, misc
static_assert(kMergeThreads * 2 == kTopK, "the sort holds two elements per thread");
static_assert(kMOffSelPos % 8 == 0, "the sort reuses the selection as 64-bit words");

struct MergeMisc {
    int32_t n_sel, n_sure, n_bnd;
    sel::Found found;
    int32_t scratch[32];
};

template <int kBnd>
__global__ void __launch_bounds__(kMergeThreads, kBnd == kBndSmall ? 2 : 1)
merge_kernel(BatchDev b, Plan p, int32_t* __restrict__ topk, float* __restrict__ topk_scores) {
    extern __shared__ __align__(16) uint8_t msm[];
    uint32_t* hist = reinterpret_cast<uint32_t*>(msm + kMOffHist);
    int32_t* sel_pos = reinterpret_cast<int32_t*>(msm + kMOffSelPos);
    uint32_t* sel_key = reinterpret_cast<uint32_t*>(msm + kMOffSelKey);
    int32_t* ns_pre = reinterpret_cast<int32_t*>(msm + kMOffNs);
    int32_t* nb_pre = reinterpret_cast<int32_t*>(msm + kMOffNb);
    uint32_t* bnd_key = reinterpret_cast<uint32_t*>(msm + kMOffBndKey);
    int32_t* bnd_pos = reinterpret_cast<int32_t*>(msm + kMOffBndKey + kBnd * 4);
    MergeMisc* mm = reinterpret_cast<MergeMisc*>(msm + kMOffBndKey + 2 * kBnd * 4);
    pdl_wait();
    pdl_trigger();
    const int64_t row = blockIdx.x;
    const int gt = threadIdx.x;
    const int r = row_request(b.q_start, b.batch, row);
    const int qn = b.q_start[r + 1] - b.q_start[r];
    const int64_t n_valid = (int64_t)b.seq_len[r] - qn + (row - b.q_start[r]) + 1;
    int32_t* out = topk + row * kTopK;
    float* outs = topk_scores ? topk_scores + row * kTopK : nullptr;
    if (n_valid <= kTopK) {
        for (int i = gt; i < kTopK; i += kMergeThreads) {
            out[i] = i < n_valid ? i : -1;
            if (outs) outs[i] = 0.f;
        }
        return;
    }
    // filtered counts of the row's segments (nseg <= number of CTAs <= 1024)
    const int s0 = p.row_seg0 ? p.row_seg0[row] : p.seg_first[r];
    const int nseg = p.row_seg0 ? p.row_segn[row] : p.seg_first[r + 1] - s0;
    const int packed = gt < nseg ? p.cand_cnt[s0 + gt] : 0;
    int n_sure, n_bnd;
    const int es = sel::excl_scan<kMergeThreads, 0>(packed & 0xffff, gt, mm->scratch, &n_sure);
    const int eb = sel::excl_scan<kMergeThreads, 0>(packed >> 16, gt, mm->scratch, &n_bnd);
    if (gt <= nseg) {
        ns_pre[gt] = gt < nseg ? es : n_sure;
        nb_pre[gt] = gt < nseg ? eb : n_bnd;
    }
    if (gt == 0) mm->n_sel = 0;
    __syncthreads();
    const uint32_t* ckey = p.cand_key + (int64_t)s0 * p.seg_stride;
    const int32_t* cpos = p.cand_pos + (int64_t)s0 * p.seg_stride;
    n_sure = min(n_sure, kTopK);
    for (int i = gt; i < n_sure; i += kMergeThreads) {           // entries above the boundary bin: all in
        const int j = seg_lookup(ns_pre, nseg, i);
        const int64_t x = (int64_t)j * p.seg_stride + (i - ns_pre[j]);
        sel_pos[i] = cpos[x];
        sel_key[i] = ckey[x];
    }
    const int need = kTopK - n_sure;
    int ns = n_sure;
    if (need > 0 && n_bnd <= need) {                             // the whole boundary bin fits
        for (int i = gt; i < n_bnd; i += kMergeThreads) {
            const int j = seg_lookup(nb_pre, nseg, i);
            const int64_t x = (int64_t)j * p.seg_stride + (ns_pre[j + 1] - ns_pre[j]) + (i - nb_pre[j]);
            sel_pos[n_sure + i] = cpos[x];
            sel_key[n_sure + i] = ckey[x];
        }
        ns = n_sure + n_bnd;
    } else if (need > 0 && n_bnd <= kBnd) {                      // exact selection in shared memory
        for (int i = gt; i < n_bnd; i += kMergeThreads) {
            const int j = seg_lookup(nb_pre, nseg, i);
            const int64_t x = (int64_t)j * p.seg_stride + (ns_pre[j + 1] - ns_pre[j]) + (i - nb_pre[j]);
            bnd_pos[i] = cpos[x];
            bnd_key[i] = ckey[x];
        }
        if (gt == 0) mm->n_sel = n_sure;
        __syncthreads();
        sel::SmemSrc<kMergeThreads> bs{bnd_key, bnd_pos, n_bnd};
        const sel::Threshold th = sel::topk_threshold<kMergeThreads, 0>(bs, need, gt, hist, mm->scratch, &mm->found,
                                                                        1, bnd_key[0] >> 20);   // one bin: skip it
        for (int i = gt; i < n_bnd; i += kMergeThreads) {
            if (th.keep(bnd_key[i], bnd_pos[i])) {
                const int jj = atomicAdd(&mm->n_sel, 1);
                if (jj < kTopK) { sel_pos[jj] = bnd_pos[i]; sel_key[jj] = bnd_key[i]; }
            }
        }
        __syncthreads();
        ns = min(mm->n_sel, kTopK);
    } else if (need > 0) {                                       // boundary bin too large: select in place
        if (gt == 0) mm->n_sel = n_sure;
        __syncthreads();
        BndSrc src{ckey, cpos, ns_pre, nb_pre, nseg, n_bnd, p.seg_stride};
        const sel::Threshold th = sel::topk_threshold<kMergeThreads, 0>(src, need, gt, hist, mm->scratch, &mm->found,
                                                                        1, ckey[src.at(0)] >> 20);
        src.visit(gt, [&](bool a, uint32_t key, int32_t pos) {
            if (a && th.keep(key, pos)) {
                const int jj = atomicAdd(&mm->n_sel, 1);
                if (jj < kTopK) { sel_pos[jj] = pos; sel_key[jj] = key; }
            }
        });
        __syncthreads();
        ns = min(mm->n_sel, kTopK);
    }
    if (n_valid <= (int64_t)kBnd * 64) {                        // the boundary buffers, free now, hold its bitmap
        sel::write_ranked<kMergeThreads>(sel_pos, sel_key, ns, n_valid, reinterpret_cast<uint32_t*>(msm + kMOffBndKey),
                                         ns_pre, reinterpret_cast<uint16_t*>(hist), mm->scratch, out, outs, gt);
        return;
    }
    for (int i = ns + gt; i < kTopK; i += kMergeThreads) {    // only if candidates were missing
        sel_pos[i] = 0x7fffffff;
        sel_key[i] = 0u;
    }
    __syncthreads();
    // sort by position: registers from the two arrays, then the arrays' 16 KB as 2048 64-bit words
    const int i0 = 64 * (gt >> 5) + 2 * (gt & 31);
    uint64_t va = ((uint64_t)(uint32_t)sel_pos[i0] << 32) | sel_key[i0];
    uint64_t vc = ((uint64_t)(uint32_t)sel_pos[i0 + 1] << 32) | sel_key[i0 + 1];
    __syncthreads();
    sort2048_regs(va, vc, reinterpret_cast<uint64_t*>(msm + kMOffSelPos), gt);
    const bool ha = i0 < ns, hc = i0 + 1 < ns;
    *reinterpret_cast<int2*>(out + i0) = make_int2(ha ? (int32_t)(va >> 32) : -1, hc ? (int32_t)(vc >> 32) : -1);
    if (outs) {                                        // 4-byte aligned only
        outs[i0] = ha ? key_score((uint32_t)va) : 0.f;
        outs[i0 + 1] = hc ? key_score((uint32_t)vc) : 0.f;
    }
}

}  // namespace itc

// ---------------------------------------------------------------- host side
namespace {
struct MapCache {
    const void* ptr = nullptr;
    int64_t pages = -1;
    CUtensorMap map;
};
}  // namespace

// The last map encoded by this host thread for each cache format: a map holds
// only the address and the extents, so it is valid on whichever device owns
// the address, and a per-thread cache needs no lock.
bool make_index_tmap(const uint8_t* cache, int64_t num_pages, bool mx, CUtensorMap* out) {
    static thread_local MapCache mcs[2];
    MapCache& mc = mcs[mx ? 1 : 0];
    if (mc.ptr == cache && mc.pages == num_pages) {
        *out = mc.map;
        return true;
    }
    const auto encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(tensor_map_encode_fn());
    if (!encode) return false;
    // FP8: the cache viewed as a [num_pages * 66, 128] byte matrix: page p's 64
    // payload rows are rows 66p .. 66p+63 (its scales fill rows 66p+64, +65).
    // MXFP4: a [num_pages * 68, 128] matrix of 4-bit values (64-byte rows), page
    // p's payload rows 68p .. 68p+63; 16U4_ALIGN16B lands each row as 128 bytes,
    // eight bytes of values then eight bytes of gap per 16 values.
    cuuint64_t dims[2] = {128, (cuuint64_t)num_pages * (mx ? 68 : 66)};
    cuuint64_t strides[1] = {mx ? 64u : 128u};
    cuuint32_t box[2] = {128, 64};
    cuuint32_t estr[2] = {1, 1};
    CUresult res = encode(out, mx ? CU_TENSOR_MAP_DATA_TYPE_16U4_ALIGN16B : CU_TENSOR_MAP_DATA_TYPE_UINT8, 2,
                          const_cast<uint8_t*>(cache), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                          CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (res != CUDA_SUCCESS) return false;
    mc.ptr = cache;
    mc.pages = num_pages;
    mc.map = *out;
    return true;
}

size_t tc_plan_bytes(int64_t batch, int G) {
    const size_t nseg = (size_t)G + (size_t)batch;
    size_t b = 0;
    b += (size_t)(batch + 1) * 8;                   // tile_start
    b += (size_t)(batch + 1) * 4;                   // seg_first
    b += (size_t)G * 2 * 4;                         // cta_range
    b = (b + 15) / 16 * 16;
    b += nseg * sizeof(Seg);                        // segs
    b = (b + 255) / 256 * 256;
    b += nseg * itc::kSegCand * 4 * 2;              // cand_key, cand_pos
    b += nseg * 4;                                  // cand_cnt
    b = (b + 255) / 256 * 256;
    return b;
}

Plan carve_plan(void* base, int64_t batch, int G) {
    const size_t nseg = (size_t)G + (size_t)batch;
    uint8_t* q = static_cast<uint8_t*>(base);
    Plan p;
    p.tile_start = reinterpret_cast<int64_t*>(q);
    q += (size_t)(batch + 1) * 8;
    p.seg_first = reinterpret_cast<int32_t*>(q);
    q += (size_t)(batch + 1) * 4;
    p.cta_range = reinterpret_cast<int32_t*>(q);
    q += (size_t)G * 2 * 4;
    q = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(q) + 15) & ~uintptr_t(15));
    p.segs = reinterpret_cast<Seg*>(q);
    q += nseg * sizeof(Seg);
    q = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(q) + 255) & ~uintptr_t(255));
    p.cand_key = reinterpret_cast<uint32_t*>(q);
    q += nseg * itc::kSegCand * 4;
    p.cand_pos = reinterpret_cast<int32_t*>(q);
    q += nseg * itc::kSegCand * 4;
    p.cand_cnt = reinterpret_cast<int32_t*>(q);
    p.hist = nullptr;
    p.slot_row = p.row_seg0 = p.row_segn = p.nslots = nullptr;
    p.seg_stride = itc::kSegCand;
    return p;
}

dsa_status launch_indexer_tc(const void* q, const float* w, uint8_t* q8, float* wq, uint32_t* hist,
                             const uint8_t* cache, const dsa_batch* b, int32_t* topk, float* topk_scores, void* plan_ws,
                             int G, int32_t* st, cudaStream_t s, bool mx) {
    CUtensorMap map;
    if (!make_index_tmap(cache, b->num_pages, mx, &map)) return DSA_ERR_CUDA;
    if (ensure_smem_limit(reinterpret_cast<const void*>(&itc::score_topk_kernel<false>), itc::kSmemAlloc) != DSA_OK ||
        ensure_smem_limit(reinterpret_cast<const void*>(&itc::score_topk_kernel<true>), itc::kSmemAlloc) != DSA_OK ||
        ensure_smem_limit(reinterpret_cast<const void*>(&itc::merge_kernel<itc::kBndCap>), itc::merge_smem(itc::kBndCap)) !=
            DSA_OK)
        return DSA_ERR_CUDA;
    BatchDev bd = to_dev(b);
    Plan p = carve_plan(plan_ws, b->batch, G);
    p.hist = hist;
    const int64_t qblocks = (b->total_q * 32 + itc::kPrepThreads / 32 - 1) / (itc::kPrepThreads / 32);
    DSA_CHECK(launch_pdl(itc::prep_kernel, dim3((unsigned)(1 + qblocks)), dim3(itc::kPrepThreads), 0, s, 1, bd, G, p,
                         static_cast<const uint16_t*>(q), w, b->total_q, q8, wq));
    if (mx)
        DSA_CHECK(launch_pdl(itc::score_topk_kernel<true>, dim3(G), dim3(itc::kThreads), itc::kSmemAlloc, s, 1, map,
                             cache, q8, wq, bd, p, st));
    else
        DSA_CHECK(launch_pdl(itc::score_topk_kernel<false>, dim3(G), dim3(itc::kThreads), itc::kSmemAlloc, s, 1, map,
                             cache, q8, wq, bd, p, st));
    return launch_topk_merge(b, p, (int64_t)G + b->batch, topk, topk_scores, s);
}

dsa_status launch_topk_merge(const dsa_batch* b, Plan p, int64_t max_segs, int32_t* topk, float* topk_scores,
                             cudaStream_t s) {
    // more rows than SMs, contexts within the small bitmap: two merge blocks per SM
    const bool small = b->total_q > device_sm_count() && b->max_seq_len <= (int64_t)itc::kBndSmall * 64;
    const void* mk = small ? reinterpret_cast<const void*>(&itc::merge_kernel<itc::kBndSmall>)
                           : reinterpret_cast<const void*>(&itc::merge_kernel<itc::kBndCap>);
    const int msmem = itc::merge_smem(small ? itc::kBndSmall : itc::kBndCap);
    if (ensure_smem_limit(mk, msmem) != DSA_OK) return DSA_ERR_CUDA;
    BatchDev bd = to_dev(b);
    if (max_segs > 0) {
        DSA_CHECK(launch_pdl(itc::merge_filter_kernel, dim3((unsigned)max_segs), dim3(itc::kFiltThreads), 0, s, 1, bd, p));
    }
    if (small)
        DSA_CHECK(launch_pdl(itc::merge_kernel<itc::kBndSmall>, dim3((unsigned)b->total_q), dim3(itc::kMergeThreads), msmem,
                             s, 1, bd, p, topk, topk_scores));
    else
        DSA_CHECK(launch_pdl(itc::merge_kernel<itc::kBndCap>, dim3((unsigned)b->total_q), dim3(itc::kMergeThreads), msmem,
                             s, 1, bd, p, topk, topk_scores));
    return DSA_OK;
}

}  // namespace dsa
