// Sparse MLA on the 5th-generation tensor cores ("vLLM 推理链路概览", Sparse
// MLA Attention; "GLM-5.3 推理全链路(一)", decode: MQA 形态与吸收):
//   S_hj = scale * <q_h, [c_j * s_j | r_j]>,  out_h = sum_j softmax_j(S_hj) c_j
// over the selected positions j of each query row (j <= p), 64 heads of 576
// dims, 512-d latent output per head.
//
// Work split: each CTA takes one contiguous range of the T x 2048 (row, entry)
// slots, cut one of three ways:
//   T < SMs       each row gets c CTAs, cut on whole 96-token tiles, so no CTA
//                 crosses a row (a crossing costs a second O store, Q load and
//                 pipeline refill on that CTA's critical path).  With c = 2 or
//                 4 the row is one thread-block cluster whose CTAs merge their
//                 results through distributed shared memory: each publishes its
//                 per-head (max, sum), scales its O^T by its log-sum-exp weight,
//                 and bulk-copies every head's columns to the CTA that owns the
//                 head (64 / c heads each), which adds them up and writes the
//                 output.  Tiny batches (SMs / T >= 8) take up to one CTA per
//                 tile and merge through global partials (below);
//   T < 8 x SMs   equal slot shares (rows at share edges are split);
//   otherwise     whole rows per CTA (at most 1/8 imbalance, nothing split).
// Otherwise a row covered by several CTAs leaves one unnormalised
// partial (O, running max, sum) per CTA in global memory; a second kernel
// merges them by log-sum-exp, spread over (row, head) blocks.
//
// Per CTA, per tile of 96 selected tokens (the M = 128 MMA rows 96..127 are
// padding), in transposed form so that tokens are the MMA rows:
//   S^T = K Q^T      tcgen05.mma kind::f16, M=128 tokens, N=64 heads, K=576,
//                    A = fp16 KV tile (K-major), B = Q (K-major), D in TMEM;
//   O^T += V^T P^T   M = 4 x 128 latent dims, N = 64 heads, K = 96 tokens,
//                    A = the same KV tile read MN-major, B = P^T (MN-major),
//                    D = 256 TMEM columns that stay resident for the row piece.
// Shared memory holds one fp16 KV tile (110.6 KB) next to the fp16 Q of the
// row (73.7 KB), so tiles cannot be double-buffered.  Instead the tile is
// recycled group by group: its five 128-byte column groups (latent dims
// 128g..128g+127 for g < 4, the RoPE dims for g = 4) are released by
// separate MMA commits (the RoPE group when S^T is done, group g when the
// P.V MMAs of latent block g are done) and the next tile's group is written
// as soon as its predecessor is released, so dequantisation overlaps the
// tensor pipe and the next S^T starts right behind the last P.V.
// Warp roles (512 threads):
//   warps 0-7   softmax: each thread owns one token (TMEM lane) and 32 of the
//               64 heads; per-head max and sum by a transposing warp
//               reduction, online softmax with lazy rescaling (O^T in TMEM is
//               rescaled only when a head's max grows by more than 2^8), P
//               written as fp16 P^T rows.  At a piece start they convert the
//               row's Q to fp16 while the loaders build the slot list and
//               gather the first tile; the row is first multiplied by the
//               power of two that puts its largest |q| in [2^14, 2^15)
//               (exact), and the inverse is folded into the softmax scale, so
//               every finite q is inside fp16's range.  Thread 0 also issues the MMAs and
//               warp 0 owns the TMEM allocation.
//   warps 8-15  loaders: build the row piece's list of cache slots and gather
//               each tile's 656-B latent rows into
//               registers one tile ahead (all 18 16-byte pieces of a lane in
//               flight at once), then dequantise group by group into the
//               128-byte-swizzled fp16 tile (c * scale is exact in fp16 for
//               scales in [2^-15, 2^7]; the RoPE dims convert from bf16, exact
//               for |r| in [2^-17, 2^16)).  A scale outside that range, or a
//               RoPE value of 2^16 or more (clamped, so the scores stay
//               finite), is recorded as DSA_DEVERR_FP16_RANGE.
// Every wait is time-bounded; a timeout is recorded and the CTA winds down.
#include <type_traits>

#include "dsa_internal.cuh"
#include "indexer_common.cuh"
#include "sm100.cuh"

namespace dsa {
namespace mtc {

using namespace sm100;

constexpr int kTok = 96;                                   // tokens per tile
constexpr int kBlk = kTok * 128;                           // one 64-dim K-block of the KV tile
constexpr int kSoftWarps = 8;                              // two per TMEM lane quarter, 32 heads each
constexpr int kSoftThreads = kSoftWarps * 32;
constexpr int kLoadWarp0 = kSoftWarps;
constexpr int kLoadWarps = 8;
constexpr int kThreads = (kSoftWarps + kLoadWarps) * 32;
constexpr int kLoadThreads = kLoadWarps * 32;
constexpr int kTokPerLoadWarp = kTok / kLoadWarps;         // 12: four tokens per step, three steps
constexpr int kSoftBar = 1;
constexpr int kLoadBar = 2;
constexpr float kTau = 8.0f;                               // lazy-rescale threshold, log2 units
constexpr int kMaxPieces = 64;
constexpr int kTilesPerRow = (kTopK + kTok - 1) / kTok;    // 22
constexpr int kMaxParts = 24;                              // CTAs one row can span
static_assert(kMaxParts >= kTilesPerRow, "a row is cut into at most one piece per tile");
static_assert(kMaxParts <= 32, "one warp forms the combine weights");
constexpr uint32_t kIdescQK = idesc_f16_f32(128, 64, false, false);
constexpr uint32_t kIdescPV = idesc_f16_f32(128, 64, true, true);
constexpr uint32_t kColS = 0;                              // TMEM: S^T [128 x 64]
constexpr uint32_t kColO = 64;                             // TMEM: O^T 4 x [128 x 64]

constexpr int kOffKV = 0;                                  // 9 K-blocks of [96 tokens x 128 B]
constexpr int kOffQ = kOffKV + 9 * kBlk;                   // 9 K-blocks of [64 heads x 128 B]
constexpr int kOffP = kOffQ + 9 * 8192;                    // P^T: 96 token rows x 64 heads fp16
constexpr int kOffSlots = kOffP + kTok * 128;              // int32 cache slots of the row piece
constexpr int kOffRed = kOffSlots + 2048 * 4;              // [2][4 lane quarters][64 heads] fp32
constexpr int kOffStat = kOffRed + 2 * 4 * 64 * 4;         // m_ref, l_acc, alpha [64] (16-byte aligned)
constexpr int kOffXstat = kOffStat + 3 * 64 * 4;          // [8][64] (max, sum) of a row's cluster
constexpr int kOffBars = kOffXstat + 8 * 64 * 2 * 4;
constexpr int kOffMisc = kOffBars + 16 * 8;
constexpr int kSmemUsed = kOffMisc + 512;
constexpr int kSmemAlloc = kSmemUsed + 1024;
static_assert(kSmemAlloc <= 232448, "shared memory budget");
// in-cluster merge (c = 2 or 4): (c - 1) x 64 / c heads x 512 fp32 received plus as many staged for
// the other CTAs (2 x 48 heads at most, c = 4) fit in the tile, Q, P and slot space, all free once
// the last MMA has completed
static_assert(2 * 48 * 512 * 4 <= kOffRed, "cluster exchange area");
static_assert(kOffQ % 1024 == 0 && kOffP % 1024 == 0 && kBlk % 1024 == 0, "swizzle atoms need 1 KB alignment");
static_assert(kOffStat % 16 == 0, "reference maxima are read as float4");
// S^T rows 96..127 read 32 rows past each K-block: still inside the tile / Q.
static_assert(8 * kBlk + 128 * 128 <= kOffQ + 9 * 8192, "padding rows stay in shared memory");

enum { B_QFULL = 0, B_QEMPTY, B_FULL0, B_FULL4 = B_FULL0 + 4, B_SFULL, B_PV0, B_PV3 = B_PV0 + 3, B_DRAIN, B_XCHG,
       B_COUNT };
static_assert(B_COUNT <= 16, "barrier block");

struct Misc {
    uint32_t tmem_base;
    int32_t abort;
    int32_t scratch[8];
    uint32_t qmax[kSoftWarps];  // per softmax warp: largest bf16 magnitude of the row's q
    int32_t ntok[kMaxPieces];
};
static_assert(sizeof(Misc) <= 512, "misc block");

// How the T x 2048 slots are cut into CTA ranges (see the file comment).
enum { SPLIT_WHOLE_ROWS = 0, SPLIT_ROW_CTAS = 1, SPLIT_EQUAL = 2 };
struct Split {
    int64_t T;                  // query rows
    int64_t N;                  // T * 2048 slots
    int32_t G;                  // CTAs
    int32_t mode;
    int32_t c, extra;           // SPLIT_ROW_CTAS: rows < extra get c + 1 CTAs, the others c
    int32_t cluster;            // CTAs per thread-block cluster (one row each), 1 = no cluster
};

struct Args {
    const uint16_t* q;          // [T,64,576] bf16
    const int32_t* topk;        // [T,2048]
    const uint8_t* kv;          // latent cache
    BatchDev b;
    float scale_log2;
    Split sp;
    void* out;
    int out_f32;
    float* lse;
    float* part_o;              // [2G, 64, 512]
    float* part_ml;             // [2G, 64, 2]: running max (log2 units), sum
    int32_t* st;
};

// First slot of CTA g's range (g = G gives T x 2048).
__device__ __forceinline__ int64_t split_begin(int64_t g, const Split& sp) {
    if (g >= sp.G) return sp.N;
    if (sp.mode == SPLIT_WHOLE_ROWS) return (g * sp.T / sp.G) * kTopK;
    if (sp.mode == SPLIT_EQUAL) return g * sp.N / sp.G;
    const int64_t big = (int64_t)sp.extra * (sp.c + 1);
    int64_t r, j, n;
    if (g < big) {
        r = g / (sp.c + 1), j = g % (sp.c + 1), n = sp.c + 1;
    } else {
        r = sp.extra + (g - big) / sp.c, j = (g - big) % sp.c, n = sp.c;
    }
    return r * kTopK + min((int64_t)kTopK, (j * kTilesPerRow / n) * kTok);
}
// The CTA whose range holds slot x (the inverse of split_begin).
__device__ __forceinline__ int64_t split_owner(int64_t x, const Split& sp) {
    if (sp.mode == SPLIT_WHOLE_ROWS) return ((x / kTopK + 1) * sp.G - 1) / sp.T;
    if (sp.mode == SPLIT_EQUAL) return ((x + 1) * sp.G + sp.N - 1) / sp.N - 1;
    const int64_t r = x / kTopK, tile = (x % kTopK) / kTok;
    const int64_t big = (int64_t)sp.extra * (sp.c + 1);
    const int64_t gf = r < sp.extra ? r * (sp.c + 1) : big + (r - sp.extra) * sp.c;
    const int64_t n = r < sp.extra ? sp.c + 1 : sp.c;
    return gf + ((tile + 1) * n - 1) / kTilesPerRow;
}
// Partial slot of CTA g's piece of row r: its first row uses 2g, its last 2g + 1.
__device__ __forceinline__ int64_t slot_of(int64_t g, int64_t r, const Split& sp) {
    return 2 * g + ((split_begin(g, sp) / kTopK == r) ? 0 : 1);
}

__device__ __forceinline__ void soft_sync() { asm volatile("bar.sync %0, %1;" ::"n"(kSoftBar), "n"(kSoftThreads) : "memory"); }
__device__ __forceinline__ void load_sync() { asm volatile("bar.sync %0, %1;" ::"n"(kLoadBar), "n"(kLoadThreads) : "memory"); }
__device__ __forceinline__ bool soft_any(bool pred) {
    uint32_t r;
    asm volatile("{\n .reg .pred p, q;\n setp.ne.u32 p, %1, 0;\n bar.red.or.pred q, %2, %3, p;\n"
                 " selp.u32 %0, 1, 0, q;\n}"
                 : "=r"(r) : "r"((uint32_t)pred), "n"(kSoftBar), "n"(kSoftThreads) : "memory");
    return r != 0;
}
__device__ __forceinline__ bool load_any(bool pred) {
    uint32_t r;
    asm volatile("{\n .reg .pred p, q;\n setp.ne.u32 p, %1, 0;\n bar.red.or.pred q, %2, %3, p;\n"
                 " selp.u32 %0, 1, 0, q;\n}"
                 : "=r"(r) : "r"((uint32_t)pred), "n"(kLoadBar), "n"(kLoadThreads) : "memory");
    return r != 0;
}

// mbarrier wait that also gives up when another role has set the abort flag.
__device__ __forceinline__ bool wait_ab(uint64_t* bar, uint32_t parity, const volatile int32_t* abort_flag) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    for (uint32_t it = 1;; ++it) {
        if (mbar_try_wait_sleep(bar, parity, 20000u)) return true;
        if ((it & 63u) == 0u && (*abort_flag || globaltimer_ns() - t0 > 2000000000ull)) return false;
    }
}

// 16-byte read-only load that stays where it is written (a prefetch a tile
// ahead must not be sunk to its first use).
__device__ __forceinline__ uint4 ldg_pinned(const uint4* p) {
    uint4 r;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w) : "l"(p));
    return r;
}

// 2^x by the hardware approximation (subnormal results flush to 0): its error
// is far below the fp16 rounding that P gets next.
__device__ __forceinline__ float ex2_approx(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ uint32_t pack_h2(float a, float b) {
    __half2 h = __floats2half2_rn(a, b);
    return *reinterpret_cast<uint32_t*>(&h);
}
__device__ __forceinline__ uint32_t e4m3x2_scaled_h2(uint32_t two, __half2 sc2) {
    __half2_raw h = __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)two, __NV_E4M3);   // exact
    const __half2 p = __hmul2(*reinterpret_cast<__half2*>(&h), sc2);                     // * 2^e: exact
    return *reinterpret_cast<const uint32_t*>(&p);
}
__device__ __forceinline__ uint32_t bf16x2_to_h2(uint32_t w) {
    return pack_h2(bf16_bits_to_f32(w & 0xffffu), bf16_bits_to_f32(w >> 16));
}
// Two bf16 key RoPE values -> two fp16.  A magnitude of 2^16 or more (inf and
// NaN included) does not fit fp16: it is clamped to +-65280 (the largest bf16
// below fp16's maximum), so the scores stay finite, and bad is set.  Every
// other bf16 value converts exactly, except those below 2^-17, whose error
// (under 2^-25 absolute) is far below the attention tolerance.
__device__ __forceinline__ uint32_t rope_bf16x2_to_h2(uint32_t w, uint32_t& bad) {
    const uint32_t over = __vcmpgeu2(w & 0x7fff7fffu, 0x47804780u);   // per half: |x| >= 2^16
    bad |= over;
    return bf16x2_to_h2((w & ~over) | (over & ((w & 0x80008000u) | 0x477f477fu)));
}
// A query pair multiplied by the row's power of two `sc` (exact in fp32) ->
// two fp16.  After that scaling no |value| reaches 2^15, so nothing
// overflows; values more than 2^39 below the row's largest are rounded to
// fp16's subnormal grid (absolute error under 2^-25 after the scaling).
__device__ __forceinline__ uint32_t bf16x2_scaled_to_h2(uint32_t w, float sc) {
    return pack_h2(bf16_bits_to_f32(w & 0xffffu) * sc, bf16_bits_to_f32(w >> 16) * sc);
}

// Reduce 32 values across the 32 lanes of a warp: afterwards lane l holds the
// result for index l in v[0] (31 shuffles instead of 160).
template <bool kMax>
__device__ __forceinline__ void xreduce32(float (&v)[32], int lane) {
#pragma unroll
    for (int s = 16, n = 16; s >= 1; s >>= 1, n >>= 1) {
        const bool up = (lane & s) != 0;
#pragma unroll
        for (int i = 0; i < n; ++i) {
            const float send = up ? v[i] : v[i + n];
            const float keep = up ? v[i + n] : v[i];
            const float recv = __shfl_xor_sync(0xffffffffu, send, s);
            v[i] = kMax ? fmaxf(keep, recv) : keep + recv;
        }
    }
}

// S^T += K-blocks [B0, B0 + NB) of the KV tile x the same blocks of Q, four
// K = 16 steps per 64-dim block; the first MMA of a tile overwrites.
template <int B0, int NB>
__device__ __forceinline__ void qk_blocks(uint32_t d_tmem, uint64_t d_kv, uint64_t d_q, bool first) {
#pragma unroll
    for (int bk = B0; bk < B0 + NB; ++bk)
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
            mma_f16(d_tmem, d_kv + (uint64_t)((bk * kBlk + kk * 32) >> 4), d_q + (uint64_t)((bk * 8192 + kk * 32) >> 4),
                    kIdescQK, (first && bk == B0 && kk == 0) ? 0u : 1u);
}
// O^T rows of latent block MB (dims 128 MB ..) += V^T P^T over the tile's six
// 16-token steps, then a commit that releases the block's KV group.
template <int MB>
__device__ __forceinline__ void pv_block(uint32_t o_tmem, uint64_t d_v, uint64_t d_p, bool acc0, uint64_t* bar) {
#pragma unroll
    for (int kt = 0; kt < kTok / 16; ++kt)
        mma_f16(o_tmem + MB * 64, d_v + (uint64_t)((2 * MB * kBlk + kt * 2048) >> 4), d_p + (uint64_t)((kt * 2048) >> 4),
                kIdescPV, (acc0 || kt > 0) ? 1u : 0u);
    mma_commit(bar);
}

__global__ void __launch_bounds__(kThreads, 1)
sparse_mla_tc_kernel(Args a) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kOffBars);
    Misc* misc = reinterpret_cast<Misc*>(smem + kOffMisc);
    int32_t* slots = reinterpret_cast<int32_t*>(smem + kOffSlots);
    float* red = reinterpret_cast<float*>(smem + kOffRed);
    float* m_ref = reinterpret_cast<float*>(smem + kOffStat);
    float* l_acc = m_ref + 64;
    float* alpha = l_acc + 64;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const BatchDev& b = a.b;
    const int64_t g = blockIdx.x;
    const int64_t e_begin = split_begin(g, a.sp), e_end = split_begin(g + 1, a.sp);
    volatile int32_t* abort_flag = &misc->abort;

    if (tid < 64) {
        m_ref[tid] = -INFINITY;
        l_acc[tid] = 0.f;
    }
    if (tid == 0) {
        mbar_init(&bars[B_QFULL], kLoadWarps);
        mbar_init(&bars[B_QEMPTY], kSoftWarps);
        for (int i = 0; i < 5; ++i) mbar_init(&bars[B_FULL0 + i], kLoadWarps);
        mbar_init(&bars[B_SFULL], 1);
        for (int i = 0; i < 4; ++i) mbar_init(&bars[B_PV0 + i], 1);
        mbar_init(&bars[B_DRAIN], 1);
        mbar_init(&bars[B_XCHG], 1);
        misc->abort = 0;
        fence_barrier_init();
    }
    if (warp == 0) {
        tmem_alloc(&misc->tmem_base, 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = misc->tmem_base;

    auto timeout = [&](int where) {
        record_error(a.st, DSA_DEVERR_TIMEOUT, where);
        *abort_flag = 1;
    };

    if (warp >= kLoadWarp0) {
        // ================================================================ loaders
        // Only the loaders read what the previous kernel may write (the top-k):
        // they wait for it, while the softmax warps already convert the first Q.
        pdl_wait();
        const int lt = tid - kLoadWarp0 * 32;            // 0..255
        const int lw = lt >> 5;                            // 0..7
        const int c8 = lane & 7;                           // 16-byte piece of a 128-byte group
        int64_t gt = 0;                                    // tiles dequantised so far by this CTA
        int k = 0;
        uint4 raw[4][3], rope[3], scv[3];                  // [group][step]: the next tile, in flight
        bool ok = true;
        for (int64_t row = e_begin / kTopK; row * kTopK < e_end; ++row, ++k) {
            if (load_any(!ok || *abort_flag)) break;      // one decision for all loader warps
            const int64_t lo_e = max(e_begin, row * kTopK) - row * kTopK;
            const int64_t hi_e = min(e_end, (row + 1) * kTopK) - row * kTopK;
            const int r = row_request(b.q_start, b.batch, row);
            const int qn = b.q_start[r + 1] - b.q_start[r];
            const int L = b.seq_len[r];
            const int p = L - qn + (int)(row - b.q_start[r]);
            // ---- valid entries of the piece -> cache slots, in order
            int ntok = 0;
            for (int base = (int)lo_e; base < (int)hi_e; base += kLoadThreads * 8) {
                int32_t sl[8];
                int cnt = 0;
#pragma unroll
                for (int u = 0; u < 8; ++u) {
                    const int e = base + lt * 8 + u;
                    sl[u] = -1;
                    if (e < (int)hi_e) {
                        const int j = a.topk[row * kTopK + e];
                        if (j >= 0 && j <= p) {
                            if (j >= L || j / kPage >= b.max_pages) {
                                record_error(a.st, DSA_DEVERR_INDEX_RANGE, j);
                            } else {
                                const int64_t pg = b.page_table[(int64_t)r * b.max_pages + j / kPage];
                                if (pg < 0 || pg >= b.num_pages) record_error(a.st, DSA_DEVERR_PAGE_RANGE, pg);
                                else sl[u] = (int32_t)(pg * kPage + (j % kPage));
                            }
                        }
                    }
                    cnt += sl[u] >= 0;
                }
                int x = cnt;
#pragma unroll
                for (int o = 1; o < 32; o <<= 1) {
                    const int y = __shfl_up_sync(0xffffffffu, x, o);
                    if (lane >= o) x += y;
                }
                if (lane == 31) misc->scratch[lw] = x;
                load_sync();
                int off = ntok + x - cnt, tot = 0;
                for (int v = 0; v < kLoadWarps; ++v) {
                    if (v < lw) off += misc->scratch[v];
                    tot += misc->scratch[v];
                }
#pragma unroll
                for (int u = 0; u < 8; ++u)
                    if (sl[u] >= 0) slots[off++] = sl[u];
                ntok += tot;
                load_sync();
            }
            const int ntiles = (ntok + kTok - 1) / kTok;
            // ---- gather of tile t into registers: step i covers tokens
            //      12 lw + 4 i + lane / 8, lane % 8 picks the 16-byte piece of each group
            // Part `what` of the gather of tile t into registers: 0..3 = latent group,
            // 4 = RoPE dims, 5 = scales.  Each part of tile t + 1 is issued as soon as the
            // same part of tile t has been consumed, so every load has a whole tile
            // period to arrive.
            auto prefetch = [&](int t, int what) {
                const int n_in = min(kTok, ntok - t * kTok);
#pragma unroll
                for (int i = 0; i < 3; ++i) {
                    const int tk = lw * kTokPerLoadWarp + 4 * i + (lane >> 3);
                    if (tk < n_in) {
                        const int32_t sl = slots[t * kTok + tk];
                        const uint4* rowp = reinterpret_cast<const uint4*>(
                            a.kv + (int64_t)(sl >> 6) * kKvPageBytes + (sl & 63) * kKvTokenBytes);
                        if (what == 0) raw[0][i] = ldg_pinned(rowp + 0 * 8 + c8);
                        if (what == 1) raw[1][i] = ldg_pinned(rowp + 1 * 8 + c8);
                        if (what == 2) raw[2][i] = ldg_pinned(rowp + 2 * 8 + c8);
                        if (what == 3) raw[3][i] = ldg_pinned(rowp + 3 * 8 + c8);
                        if (what == 4) rope[i] = ldg_pinned(rowp + 33 + c8);
                        if (what == 5) scv[i] = ldg_pinned(rowp + 32);
                    } else {                               // no token: zero row (P is 0 there, V must be finite)
                        if (what == 0) raw[0][i] = make_uint4(0, 0, 0, 0);
                        if (what == 1) raw[1][i] = make_uint4(0, 0, 0, 0);
                        if (what == 2) raw[2][i] = make_uint4(0, 0, 0, 0);
                        if (what == 3) raw[3][i] = make_uint4(0, 0, 0, 0);
                        if (what == 4) rope[i] = make_uint4(0, 0, 0, 0);
                        if (what == 5) scv[i] = make_uint4(0x3f800000u, 0x3f800000u, 0x3f800000u, 0x3f800000u);
                    }
                }
            };
            if (ntiles > 0) {
                prefetch(0, 4);
                prefetch(0, 5);
                prefetch(0, 0);
                prefetch(0, 1);
                prefetch(0, 2);
                prefetch(0, 3);
            }
            // ---- the piece's token count, once the softmax group has taken the
            //      previous one (so QFULL never runs two phases ahead)
            if (k > 0 && !(ok = wait_ab(&bars[B_QEMPTY], (uint32_t)((k - 1) & 1), abort_flag))) {
                if (lane == 0) timeout(11);
                continue;                                  // the decision is taken at the loop top
            }
            if (lt == 0) misc->ntok[k % kMaxPieces] = ntok;
            __syncwarp();
            if (lane == 0) mbar_arrive(&bars[B_QFULL]);
            // ---- tiles: RoPE group first (free once S^T of the previous tile is done), then
            //      latent groups 0..3 (free once that tile's P.V of block g is done)
            for (int t = 0; t < ntiles && ok; ++t, ++gt) {
                const uint32_t ph = (uint32_t)((gt - 1) & 1);
                uint32_t bad_scale = 0;                    // a latent scale or a RoPE value fp16 cannot hold
                if (gt > 0 && !(ok = wait_ab(&bars[B_SFULL], ph, abort_flag))) break;
#pragma unroll
                for (int i = 0; i < 3; ++i) {
                    const int tk = lw * kTokPerLoadWarp + 4 * i + (lane >> 3);
                    *reinterpret_cast<uint4*>(smem + kOffKV + 8 * kBlk + tk * 128 + ((c8 ^ (tk & 7)) * 16)) =
                        make_uint4(rope_bf16x2_to_h2(rope[i].x, bad_scale), rope_bf16x2_to_h2(rope[i].y, bad_scale),
                                   rope_bf16x2_to_h2(rope[i].z, bad_scale), rope_bf16x2_to_h2(rope[i].w, bad_scale));
                }
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) mbar_arrive(&bars[B_FULL4]);
                const bool more = t + 1 < ntiles;
                if (more) prefetch(t + 1, 4);
#pragma unroll
                for (int gg = 0; gg < 4; ++gg) {
                    if (gt > 0 && !(ok = wait_ab(&bars[B_PV0 + gg], ph, abort_flag))) break;
#pragma unroll
                    for (int i = 0; i < 3; ++i) {
                        const int tk = lw * kTokPerLoadWarp + 4 * i + (lane >> 3);
                        const uint32_t scb = gg == 0 ? scv[i].x : gg == 1 ? scv[i].y : gg == 2 ? scv[i].z : scv[i].w;
                        const float sc = __uint_as_float(scb);
                        bad_scale |= (sc < 0x1p-15f || sc > 0x1p7f) ? 1u : 0u;
                        const __half2 sc2 = __float2half2_rn(sc);           // a power of two: exact
                        const uint4 w = raw[gg][i];
                        // 16 FP8 dims 128 gg + 16 c8 .. -> K-block 2 gg + c8 / 4, 16-byte chunks 2 (c8 % 4), +1
                        uint8_t* blkp = smem + kOffKV + (2 * gg + (c8 >> 2)) * kBlk + tk * 128;
                        const int ch = 2 * (c8 & 3), sw = tk & 7;
                        *reinterpret_cast<uint4*>(blkp + ((ch ^ sw) * 16)) =
                            make_uint4(e4m3x2_scaled_h2(w.x & 0xffffu, sc2), e4m3x2_scaled_h2(w.x >> 16, sc2),
                                       e4m3x2_scaled_h2(w.y & 0xffffu, sc2), e4m3x2_scaled_h2(w.y >> 16, sc2));
                        *reinterpret_cast<uint4*>(blkp + (((ch + 1) ^ sw) * 16)) =
                            make_uint4(e4m3x2_scaled_h2(w.z & 0xffffu, sc2), e4m3x2_scaled_h2(w.z >> 16, sc2),
                                       e4m3x2_scaled_h2(w.w & 0xffffu, sc2), e4m3x2_scaled_h2(w.w >> 16, sc2));
                    }
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&bars[B_FULL0 + gg]);
                    // spread over the tile: a whole tile's requests at once fill the
                    // SM's outstanding-miss capacity and stall every memory instruction
                    if (more) prefetch(t + 1, gg);
                }
                if (!ok) break;
                if (bad_scale) record_error(a.st, DSA_DEVERR_FP16_RANGE, lane);
                if (more) prefetch(t + 1, 5);
            }
            if (!ok && lane == 0) timeout(12);
        }
    } else {
        // ================================================================ softmax + MMA issue + epilogue
        // Warp w reads TMEM lane quarter w % 4 (token / latent row st) and
        // heads [32 hh, 32 hh + 32), hh = w / 4.
        const int q4 = warp & 3, hh = warp >> 2;
        const int st = q4 * 32 + lane;
        const uint32_t lane_addr = tmem + ((uint32_t)(q4 * 32) << 16);
        const uint32_t kv0 = smem_addr(smem + kOffKV), q0 = smem_addr(smem + kOffQ), p0 = smem_addr(smem + kOffP);
        bool issued = false;
        // Shared-memory descriptors of the operand bases; an MMA's descriptor is
        // base + offset / 16 with a compile-time offset, so the issuing thread
        // spends a few instructions per MMA (a dependent descriptor computation
        // per MMA would make the issuer, not the tensor pipe, the bottleneck).
        const uint64_t d_kv = desc_kmajor_sw128(kv0), d_q = desc_kmajor_sw128(q0);
        const uint64_t d_v = desc_mnmajor_sw128(kv0, kBlk), d_p = desc_mnmajor_sw128(p0, 8192);
        // S^T of tile gt_ (thread 0): groups in the order the loaders release them
        auto issue_qk = [&](int64_t gt_) -> bool {
            const uint32_t ph = (uint32_t)(gt_ & 1);
            if (!wait_ab(&bars[B_FULL4], ph, abort_flag)) return false;
            tc_fence_after();
            qk_blocks<8, 1>(tmem + kColS, d_kv, d_q, true);
            if (!wait_ab(&bars[B_FULL0], ph, abort_flag)) return false;
            tc_fence_after();
            qk_blocks<0, 2>(tmem + kColS, d_kv, d_q, false);
            if (!wait_ab(&bars[B_FULL0 + 1], ph, abort_flag)) return false;
            tc_fence_after();
            qk_blocks<2, 2>(tmem + kColS, d_kv, d_q, false);
            if (!wait_ab(&bars[B_FULL0 + 2], ph, abort_flag)) return false;
            tc_fence_after();
            qk_blocks<4, 2>(tmem + kColS, d_kv, d_q, false);
            if (!wait_ab(&bars[B_FULL0 + 3], ph, abort_flag)) return false;
            tc_fence_after();
            qk_blocks<6, 2>(tmem + kColS, d_kv, d_q, false);
            mma_commit(&bars[B_SFULL]);
            issued = true;
            return true;
        };
        // O^T += V^T P^T of a tile (thread 0); block g's commit releases KV group g
        auto issue_pv = [&](bool acc0) {
            tc_fence_after();
            pv_block<0>(tmem + kColO, d_v, d_p, acc0, &bars[B_PV0]);
            pv_block<1>(tmem + kColO, d_v, d_p, acc0, &bars[B_PV0 + 1]);
            pv_block<2>(tmem + kColO, d_v, d_p, acc0, &bars[B_PV0 + 2]);
            pv_block<3>(tmem + kColO, d_v, d_p, acc0, &bars[B_PV0 + 3]);
        };
        int64_t gt = 0;
        int k = 0;
        for (int64_t row = e_begin / kTopK; row * kTopK < e_end; ++row, ++k) {
            // ---- Q of the row -> fp16, K-major, 128-byte swizzle.  Every S^T MMA of the
            //      previous piece has completed (each was waited for), so Q is free; the
            //      loaders meanwhile build the slot list and gather the first tile.
            //      The row is first scaled by the power of two 2^kq that puts its largest |q|
            //      in [2^14, 2^15): exact, and it keeps every q value inside fp16's range
            //      whatever the row's magnitude; 2^-kq is folded into the softmax scale.
            float row_sl2 = a.scale_log2;
            {
                static_assert(64 * 72 == 18 * kSoftThreads, "18 16-byte pieces of q per thread");
                const uint4* qrow = reinterpret_cast<const uint4*>(a.q + row * (64 * 576));
                uint32_t mx = 0;                           // two bf16 magnitudes, compared as integers
#pragma unroll 1
                for (int u0 = 0; u0 < 18; u0 += 6) {       // pass 1: the row's largest |q|, 6 loads in flight
                    uint4 qv[6];
#pragma unroll
                    for (int u = 0; u < 6; ++u) qv[u] = __ldg(qrow + tid + (u0 + u) * kSoftThreads);
#pragma unroll
                    for (int u = 0; u < 6; ++u)
                        mx = __vmaxu2(mx, __vmaxu2(__vmaxu2(qv[u].x & 0x7fff7fffu, qv[u].y & 0x7fff7fffu),
                                                   __vmaxu2(qv[u].z & 0x7fff7fffu, qv[u].w & 0x7fff7fffu)));
                }
                mx = __reduce_max_sync(0xffffffffu, max(mx & 0xffffu, mx >> 16));
                if (lane == 0) misc->qmax[warp] = mx;
                soft_sync();
                uint32_t amax = 0;
#pragma unroll
                for (int v = 0; v < kSoftWarps; ++v) amax = max(amax, misc->qmax[v]);
                // exponent of the largest |q| (bf16 bits: 8 exponent bits above 7 mantissa bits)
                const int eq = amax == 0 ? 14 : (int)(amax >> 7) - 127;
                const int kq = min(126, max(-126, 14 - eq));
                const float sc = __int_as_float((127 + kq) << 23);
                row_sl2 = a.scale_log2 * __int_as_float((127 - kq) << 23);
#pragma unroll 1
                for (int u0 = 0; u0 < 18; u0 += 6) {       // pass 2 (from L2): scale, convert, store
                    uint4 qv[6];
#pragma unroll
                    for (int u = 0; u < 6; ++u) qv[u] = __ldg(qrow + tid + (u0 + u) * kSoftThreads);
#pragma unroll
                    for (int u = 0; u < 6; ++u) {
                        const int c = tid + (u0 + u) * kSoftThreads;
                        const int h = c / 72, cq = c % 72;
                        const int blk = cq >> 3, ch = cq & 7;
                        *reinterpret_cast<uint4*>(smem + kOffQ + blk * 8192 + h * 128 + ((ch ^ (h & 7)) * 16)) =
                            make_uint4(bf16x2_scaled_to_h2(qv[u].x, sc), bf16x2_scaled_to_h2(qv[u].y, sc),
                                       bf16x2_scaled_to_h2(qv[u].z, sc), bf16x2_scaled_to_h2(qv[u].w, sc));
                    }
                }
                if (tid == 0 && amax >= 0x7f80u) record_error(a.st, DSA_DEVERR_FP16_RANGE, (int64_t)row);   // inf / NaN in q
                fence_proxy_async_smem();
            }
            int ok = mbar_wait(&bars[B_QFULL], (uint32_t)(k & 1)) ? 1 : 0;
            if (soft_any(!ok || *abort_flag)) {
                if (tid == 0 && !ok) timeout(31);
                break;
            }
            const int ntok = misc->ntok[k % kMaxPieces];
            const int ntiles = (ntok + kTok - 1) / kTok;
            __syncwarp();
            if (lane == 0) mbar_arrive(&bars[B_QEMPTY]);
            if (tid < 64) {
                m_ref[tid] = -INFINITY;
                l_acc[tid] = 0.f;
            }
            soft_sync();                                    // Q and the statistics are in place
            float lsum[32];                                 // this token lane's running sums of its 32 heads
#pragma unroll
            for (int c = 0; c < 32; ++c) lsum[c] = 0.f;
            if (tid == 0 && ntiles > 0 && !issue_qk(gt)) timeout(34);
            bool failed = false;
            for (int t = 0; t < ntiles; ++t, ++gt) {
                ok = wait_ab(&bars[B_SFULL], (uint32_t)(gt & 1), abort_flag) ? 1 : 0;
                if (soft_any(!ok)) { failed = true; break; }
                const int n_in = min(kTok, ntok - t * kTok);
                const bool valid = st < n_in;
                // S^T row of this token for the warp's 32 heads, in log2 units; absent tokens -> -inf
                auto load_s = [&](float (&v)[32]) {
                    uint32_t u[32];
                    tmem_ld_32x32b_x32(lane_addr + kColS + hh * 32, u);
                    tmem_ld_wait();
#pragma unroll
                    for (int h = 0; h < 32; ++h) v[h] = valid ? __uint_as_float(u[h]) * row_sl2 : -INFINITY;
                };
                float v[32];
                tc_fence_after();
                load_s(v);
                // ---- lazy rescale: the exact tile max is needed only when a score
                //      exceeds its head's reference max by more than 2^kTau (always on
                //      the piece's first tile, where the reference is -inf)
                bool over = false;
                const float4* mr4 = reinterpret_cast<const float4*>(m_ref + hh * 32);   // 16-byte reads
#pragma unroll
                for (int c4 = 0; c4 < 8; ++c4) {
                    const float4 m = mr4[c4];
                    over |= v[4 * c4] > m.x + kTau || v[4 * c4 + 1] > m.y + kTau || v[4 * c4 + 2] > m.z + kTau ||
                            v[4 * c4 + 3] > m.w + kTau;
                }
                // S^T of tile gt is complete, and it was issued after the P.V of tile gt - 1:
                // O^T is stable and P^T is free.
                if (soft_any(over)) {
                    xreduce32<true>(v, lane);                   // per-head tile max (consumes v)
                    red[q4 * 64 + hh * 32 + lane] = v[0];
                    soft_sync();
                    if (tid < 64) {
                        const float tm = fmaxf(fmaxf(red[tid], red[64 + tid]), fmaxf(red[128 + tid], red[192 + tid]));
                        const float mo = m_ref[tid];
                        const bool need = tm > mo + kTau;
                        alpha[tid] = need ? (mo == -INFINITY ? 0.f : exp2f(mo - tm)) : 1.f;
                        if (need) m_ref[tid] = tm;
                    }
                    soft_sync();
                    if (t > 0) {                                // rescale the resident O^T columns of these heads
#pragma unroll 1
                        for (int mb = 0; mb < 4; ++mb) {
                            uint32_t o[32];
                            const uint32_t addr = lane_addr + kColO + mb * 64 + hh * 32;
                            tmem_ld_32x32b_x32(addr, o);
                            tmem_ld_wait();
#pragma unroll
                            for (int c = 0; c < 32; ++c) o[c] = __float_as_uint(__uint_as_float(o[c]) * alpha[hh * 32 + c]);
                            tmem_st_32x32b_x32(addr, o);
                        }
                        tmem_st_wait();
                    }
#pragma unroll
                    for (int c = 0; c < 32; ++c) lsum[c] *= alpha[hh * 32 + c];   // rare: first tile of a piece
                    load_s(v);
                }
                // ---- probabilities, this token's running sums, and its P^T row
                //      (heads 32 hh.. as fp16, MN-major 128-byte swizzle)
#pragma unroll
                for (int c4 = 0; c4 < 8; ++c4) {
                    const float4 m = mr4[c4];
                    const float mr[4] = {m.x, m.y, m.z, m.w};
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const int c = 4 * c4 + e;
                        v[c] = (v[c] == -INFINITY) ? 0.f : ex2_approx(v[c] - mr[e]);
                        lsum[c] += v[c];
                    }
                }
                if (st < kTok) {
                    uint8_t* prow = smem + kOffP + st * 128;
#pragma unroll
                    for (int cc = 0; cc < 4; ++cc) {
                        const int c = hh * 4 + cc;
                        *reinterpret_cast<uint4*>(prow + ((c ^ (st & 7)) * 16)) =
                            make_uint4(pack_h2(v[8 * cc], v[8 * cc + 1]), pack_h2(v[8 * cc + 2], v[8 * cc + 3]),
                                       pack_h2(v[8 * cc + 4], v[8 * cc + 5]), pack_h2(v[8 * cc + 6], v[8 * cc + 7]));
                    }
                }
                fence_proxy_async_smem();
                tc_fence_before();
                soft_sync();                                // P^T written, S^T and O^T reads / writes done
                if (tid == 0) {
                    issue_pv(t > 0);
                    if (t + 1 < ntiles && !issue_qk(gt + 1)) timeout(35);
                }
            }
            if (failed) {
                if (tid == 0) timeout(32);
                break;
            }
            // ---- piece end: O^T is final once the last P.V completes
            if (ntiles > 0) {
                ok = wait_ab(&bars[B_PV3], (uint32_t)((gt - 1) & 1), abort_flag) ? 1 : 0;
                if (soft_any(!ok)) {
                    if (tid == 0) timeout(33);
                    break;
                }
                tc_fence_after();
            }
            // ---- per-head sums over the piece: the lanes' running sums reduced
            xreduce32<false>(lsum, lane);
            red[256 + q4 * 64 + hh * 32 + lane] = lsum[0];
            soft_sync();
            if (tid < 64) l_acc[tid] = red[256 + tid] + red[320 + tid] + red[384 + tid] + red[448 + tid];
            soft_sync();
            if (a.sp.cluster > 1) break;                    // the row's only piece: merged in the cluster below
            const int64_t g0 = split_owner(row * kTopK, a.sp), g1 = split_owner(row * kTopK + kTopK - 1, a.sp);
            const bool whole = g0 == g1;
            const int64_t unit = whole ? 0 : slot_of(g, row, a.sp);
#pragma unroll 1
            for (int mb = 0; mb < 4; ++mb) {
                uint32_t o[32];
                if (ntiles > 0) {
                    tmem_ld_32x32b_x32(lane_addr + kColO + mb * 64 + hh * 32, o);
                    tmem_ld_wait();
                } else {
#pragma unroll
                    for (int c = 0; c < 32; ++c) o[c] = 0u;
                }
                const int d = mb * 128 + st;                           // latent dim of this TMEM lane
#pragma unroll
                for (int c = 0; c < 32; ++c) {                         // a warp stores 32 consecutive dims
                    const int h = hh * 32 + c;
                    const float ov = __uint_as_float(o[c]);
                    if (whole) {
                        const float l = l_acc[h];
                        const float val = l > 0.f ? ov / l : 0.f;
                        const int64_t oi = (row * 64 + h) * 512 + d;
                        if (a.out_f32) static_cast<float*>(a.out)[oi] = val;
                        else static_cast<__nv_bfloat16*>(a.out)[oi] = __float2bfloat16_rn(val);
                    } else {
                        a.part_o[(unit * 64 + h) * 512 + d] = ov;
                    }
                }
            }
            tc_fence_before();
            if (whole) {
                if (a.lse && tid < 64) {
                    const float l = l_acc[tid];
                    a.lse[row * 64 + tid] = l > 0.f ? (m_ref[tid] + log2f(l)) * 0.69314718055994531f : -INFINITY;
                }
            } else {
                if (tid < 64) {
                    a.part_ml[(unit * 64 + tid) * 2] = m_ref[tid];
                    a.part_ml[(unit * 64 + tid) * 2 + 1] = l_acc[tid];
                }
            }
            soft_sync();                                    // O^T may be reused
        }
        // no MMA may be in flight when the TMEM is released
        if (tid == 0 && issued) {
            mma_commit(&bars[B_DRAIN]);
            mbar_wait(&bars[B_DRAIN], 0, 500000000ull);
        }
    }
    tc_fence_before();
    __syncthreads();
    pdl_trigger();
    // ---- merge of the row inside its cluster (all 16 warps).  Every CTA
    //      reaches both cluster barriers and sends its full share, whatever
    //      happened above; a CTA that gave up contributes zeros (sum 0).  The
    //      cluster size is a compile-time constant so head -> owner is a shift.
    auto cluster_merge = [&](auto csize) {
        constexpr int c = decltype(csize)::value;            // 2 or 4
        tc_fence_after();
        const int j = (int)cluster_ctarank();
        const int64_t row = e_begin / kTopK;
        constexpr int hpc = 64 / c;                          // heads per CTA
        constexpr uint32_t blk = (uint32_t)hpc * 512 * 4;    // one CTA's share of one owner's heads, fp32
        float* recv = reinterpret_cast<float*>(smem + kOffKV);   // [c - 1 senders][hpc][512]
        float* stage = recv + (c - 1) * hpc * 512;               // [c - 1 owners][hpc][512]
        float* xstat = reinterpret_cast<float*>(smem + kOffXstat);   // [rank][head] (max, sum)
        if (tid == 0) mbar_arrive_expect_tx(&bars[B_XCHG], (uint32_t)(c - 1) * blk);   // armed before any send
        if (tid < 64) {                                      // this CTA's statistics to every CTA of the row
            const float ms = m_ref[tid], ls = *abort_flag ? 0.f : l_acc[tid];
            const uint32_t dst = smem_addr(xstat + (j * 64 + tid) * 2);
            for (int r = 0; r < c; ++r) {
                st_cluster_f32(mapa_shared(dst, (uint32_t)r), ms);
                st_cluster_f32(mapa_shared(dst + 4, (uint32_t)r), ls);
            }
        }
        cluster_sync();                                     // #1: statistics everywhere, MMAs drained, barriers armed
        float* scale = alpha;                               // [64]: this CTA's weight per head
        if (tid < 64) {
            float M = -INFINITY;
            for (int r = 0; r < c; ++r)
                if (xstat[(r * 64 + tid) * 2 + 1] > 0.f) M = fmaxf(M, xstat[(r * 64 + tid) * 2]);
            float L = 0.f;
            for (int r = 0; r < c; ++r) {
                const float lr = xstat[(r * 64 + tid) * 2 + 1];
                if (lr > 0.f) L += lr * exp2f(xstat[(r * 64 + tid) * 2] - M);
            }
            const float ls = xstat[(j * 64 + tid) * 2 + 1];
            scale[tid] = (ls > 0.f && L > 0.f) ? exp2f(xstat[(j * 64 + tid) * 2] - M) / L : 0.f;
            if (a.lse && tid / hpc == j)
                a.lse[row * 64 + tid] = L > 0.f ? (M + log2f(L)) * 0.69314718055994531f : -INFINITY;
        }
        __syncthreads();
        // the other owners' heads, scaled, staged as [owner slot][head - first head][dim]
        const int q4 = warp & 3, mb = warp >> 2;
        const int dim = mb * 128 + q4 * 32 + lane;
        const uint32_t taddr = tmem + ((uint32_t)(q4 * 32) << 16) + kColO + mb * 64;
#pragma unroll 1
        for (int half = 0; half < 2; ++half) {
            if (half * 32 / hpc == j && hpc >= 32) continue;    // all own heads
            uint32_t o[32];
            tmem_ld_32x32b_x32(taddr + half * 32, o);
            tmem_ld_wait();
#pragma unroll
            for (int cc = 0; cc < 32; ++cc) {
                const int h = half * 32 + cc;
                const int owner = h / hpc;
                if (owner == j) continue;
                const int slot = owner < j ? owner : owner - 1;
                const float sc = scale[h];
                stage[(slot * hpc + (h - owner * hpc)) * 512 + dim] = sc != 0.f ? __uint_as_float(o[cc]) * sc : 0.f;
            }
        }
        fence_proxy_async_smem();                           // staged by plain stores, read by the copy engine
        __syncthreads();
        if (tid < c - 1) {                                   // one bulk copy per other owner
            const int owner = tid < j ? tid : tid + 1;
            const int slot_there = j < owner ? j : j - 1;
            bulk_s2cluster(mapa_shared(smem_addr(recv + slot_there * hpc * 512), (uint32_t)owner), stage + tid * hpc * 512,
                           blk, mapa_shared(smem_addr(&bars[B_XCHG]), (uint32_t)owner));
        }
        if (!mbar_wait(&bars[B_XCHG], 0) && tid == 0) timeout(41);   // the other CTAs' shares of my heads
        cluster_sync();                                     // #2: every copy has landed: staging is free everywhere
        // own heads: this CTA's scaled columns plus the c - 1 received shares, staged
        // as the output block [head - h0][dim], then one bulk store
        {
            const int h0 = j * hpc, half = h0 >> 5;
            uint32_t o[32];
            tmem_ld_32x32b_x32(taddr + half * 32, o);
            tmem_ld_wait();
#pragma unroll
            for (int cc = 0; cc < 32; ++cc) {
                const int h = half * 32 + cc;
                if (h < h0 || h >= h0 + hpc) continue;
                const int hl = h - h0;
                const float sc = scale[h];
                float acc = sc != 0.f ? __uint_as_float(o[cc]) * sc : 0.f;
                for (int sl = 0; sl < c - 1; ++sl) acc += recv[(sl * hpc + hl) * 512 + dim];
                if (a.out_f32) stage[hl * 512 + dim] = acc;
                else reinterpret_cast<__nv_bfloat16*>(stage)[hl * 512 + dim] = __float2bfloat16_rn(acc);
            }
        }
        __syncthreads();
        // the block of rows row * 64 + h0 .. + hpc is contiguous in the output: 16-byte stores
        const int eb = a.out_f32 ? 4 : 2;
        const int n16 = hpc * 512 * eb / 16;
        const uint4* src = reinterpret_cast<const uint4*>(stage);
        uint4* dst = reinterpret_cast<uint4*>(static_cast<uint8_t*>(a.out) + (size_t)(row * 64 + j * hpc) * 512 * eb);
        for (int e = tid; e < n16; e += kThreads) dst[e] = src[e];
        tc_fence_before();
        __syncthreads();
    };
    if (a.sp.cluster == 2) cluster_merge(std::integral_constant<int, 2>{});
    else if (a.sp.cluster == 4) cluster_merge(std::integral_constant<int, 4>{});
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

// ---------------------------------------------------------------- combine
// Rows cut across CTAs.  With CTAs per row, block x merges row x when that row
// has several CTAs.  With equal shares, block x looks at CTA boundary
// bd = x + 1: the row holding slot split_begin(bd) is split when that slot is
// not the row's first, and the row's first such boundary merges it.  Per head h of the row
// over its partials u:  M = max m_u,  w_u = 2^(m_u - M),  L = sum w_u l_u,
//   out_h = sum_u w_u O_u,h / L,   lse_h = (M + log2 L) ln 2.
constexpr int kCombThreads = 128;                          // one head: 512 dims, 4 per thread

__global__ void __launch_bounds__(kCombThreads)
combine_kernel(Args a) {
    __shared__ float w_s[kMaxParts];
    __shared__ float inv_s;
    __shared__ int64_t u_s[kMaxParts];
    pdl_wait();
    pdl_trigger();
    int64_t row;
    if (a.sp.mode == SPLIT_ROW_CTAS) {
        row = blockIdx.x;
    } else {
        const int64_t bd = (int64_t)blockIdx.x + 1;
        const int64_t x = split_begin(bd, a.sp);
        row = x / kTopK;
        if (x % kTopK == 0) return;                         // a row boundary: nothing split here
        if (bd >= 2) {
            const int64_t px = split_begin(bd - 1, a.sp);
            if (px / kTopK == row && px % kTopK != 0) return;   // an earlier boundary merges this row
        }
    }
    const int64_t g0 = split_owner(row * kTopK, a.sp), g1 = split_owner(row * kTopK + kTopK - 1, a.sp);
    if (g0 == g1) return;                                   // written whole by its CTA
    const int np = (int)min(g1 - g0 + 1, (int64_t)kMaxParts);   // at most one CTA per tile of the row
    const int tid = threadIdx.x;
    const int h = blockIdx.y;
    if (tid < kMaxParts) u_s[tid] = tid < np ? slot_of(g0 + tid, row, a.sp) : 0;
    __syncthreads();
    // partial q's (max, sum) of head h, one thread each; then warp 0 forms the weights
    float2 ml = make_float2(-INFINITY, 0.f);
    if (tid < np) ml = __ldcg(reinterpret_cast<const float2*>(a.part_ml) + u_s[tid] * 64 + h);
    if (tid < 32) {
        float M = ml.y > 0.f ? ml.x : -INFINITY;
#pragma unroll
        for (int o = 16; o >= 1; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
        const float w = ml.y > 0.f ? exp2f(ml.x - M) : 0.f;
        float Lt = w * ml.y;
#pragma unroll
        for (int o = 16; o >= 1; o >>= 1) Lt += __shfl_xor_sync(0xffffffffu, Lt, o);
        if (tid < kMaxParts) w_s[tid] = w;
        if (tid == 0) {
            inv_s = Lt > 0.f ? 1.f / Lt : 0.f;
            if (a.lse) a.lse[row * 64 + h] = Lt > 0.f ? (M + log2f(Lt)) * 0.69314718055994531f : -INFINITY;
        }
    }
    __syncthreads();
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int q0 = 0; q0 < np; q0 += 8) {                    // eight partials' loads in flight
        float4 v[8];
#pragma unroll
        for (int j = 0; j < 8; ++j)
            v[j] = q0 + j < np ? __ldcg(reinterpret_cast<const float4*>(a.part_o + (u_s[q0 + j] * 64 + h) * 512) + tid)
                              : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const float w = q0 + j < np ? w_s[q0 + j] : 0.f;
            acc.x += w * v[j].x;
            acc.y += w * v[j].y;
            acc.z += w * v[j].z;
            acc.w += w * v[j].w;
        }
    }
    const float inv = inv_s;
    const int64_t o = (row * 64 + h) * 512 + tid * 4;
    if (a.out_f32) {
        *reinterpret_cast<float4*>(static_cast<float*>(a.out) + o) =
            make_float4(acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv);
    } else {
        __nv_bfloat162 lo2 = __floats2bfloat162_rn(acc.x * inv, acc.y * inv);
        __nv_bfloat162 hi2 = __floats2bfloat162_rn(acc.z * inv, acc.w * inv);
        *reinterpret_cast<uint2*>(static_cast<__nv_bfloat16*>(a.out) + o) =
            make_uint2(*reinterpret_cast<uint32_t*>(&lo2), *reinterpret_cast<uint32_t*>(&hi2));
    }
}

}  // namespace mtc

// CTAs per row when rows are fewer than SMs: a cluster of 2 or 4 when that
// fills the GPU best, else (tiny batches) up to one CTA per tile of the row,
// merged through global partials.
static int row_ctas(int64_t total_q, int sms) {
    const int64_t per = sms / total_q;
    if (per >= 8) return (int)std::min<int64_t>(per, mtc::kTilesPerRow);
    return per >= 4 ? 4 : per >= 2 ? 2 : 1;
}

// CTAs sharing the T x 2048 slots: one per SM at most.
int mla_tc_ctas(int64_t total_q, int sms) {
    if (total_q < sms) return (int)(total_q * row_ctas(total_q, sms));
    return sms;
}

static mtc::Split make_split(int64_t T, int G) {
    mtc::Split sp;
    sp.T = T;
    sp.N = T * kTopK;
    sp.G = G;
    sp.c = sp.extra = 0;
    sp.cluster = 1;
    if (T <= G) {
        sp.mode = mtc::SPLIT_ROW_CTAS;
        sp.c = (int32_t)(G / T);
        sp.extra = (int32_t)(G % T);
        if (sp.extra == 0 && (sp.c == 2 || sp.c == 4)) sp.cluster = sp.c;
    } else if (T < (int64_t)8 * G) {
        sp.mode = mtc::SPLIT_EQUAL;
    } else {
        sp.mode = mtc::SPLIT_WHOLE_ROWS;
    }
    return sp;
}

size_t mla_tc_ws_bytes(int64_t total_q, int G) {
    (void)total_q;
    const size_t b = (size_t)2 * G * 64 * 512 * 4 + (size_t)2 * G * 64 * 2 * 4;
    return (b + 255) / 256 * 256;
}

dsa_status launch_sparse_mla_tc(const void* q, const int32_t* topk, const uint8_t* kv, const dsa_batch* b,
                                float softmax_scale, void* out, int32_t out_dtype, float* lse, void* ws,
                                int G, int32_t* st, cudaStream_t s) {
    if (ensure_smem_limit(reinterpret_cast<const void*>(&mtc::sparse_mla_tc_kernel), mtc::kSmemAlloc) != DSA_OK)
        return DSA_ERR_CUDA;
    mtc::Args a;
    a.q = static_cast<const uint16_t*>(q);
    a.topk = topk;
    a.kv = kv;
    a.b = to_dev(b);
    a.scale_log2 = softmax_scale * 1.4426950408889634f;
    a.sp = make_split(b->total_q, G);
    a.out = out;
    a.out_f32 = out_dtype == DSA_DTYPE_F32;
    a.lse = lse;
    a.part_o = static_cast<float*>(ws);
    a.part_ml = a.part_o + (size_t)2 * G * 64 * 512;
    a.st = st;
    if (a.sp.cluster > 1) {                                 // one cluster per row
        DSA_CHECK(launch_pdl(mtc::sparse_mla_tc_kernel, dim3((unsigned)G), dim3(mtc::kThreads), mtc::kSmemAlloc, s,
                             (unsigned)a.sp.cluster, a));
        return DSA_OK;                                      // merged inside the clusters
    }
    DSA_CHECK(launch_pdl(mtc::sparse_mla_tc_kernel, dim3((unsigned)G), dim3(mtc::kThreads), mtc::kSmemAlloc, s, 1, a));
    unsigned nx = 0;                                        // combine blocks: candidate rows
    if (a.sp.mode == mtc::SPLIT_ROW_CTAS)                   // one CTA per row (c = 1, no extra): each row
        nx = (a.sp.c > 1 || a.sp.extra > 0) ? (unsigned)b->total_q : 0u;   // written whole, nothing to merge
    else if (a.sp.mode == mtc::SPLIT_EQUAL) nx = (unsigned)(G - 1);
    if (nx > 0) {
        DSA_CHECK(launch_pdl(mtc::combine_kernel, dim3(nx, 64), dim3(mtc::kCombThreads), 0, s, 1, a));
    }
    return DSA_OK;
}

}  // namespace dsa
