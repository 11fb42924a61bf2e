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
//       warps 2-9  two epilogue groups taking alternate tiles: per token and
//                  row, ReLU, head-weighted sum, times the key scale; the score
//                  rows are written coalesced (32 consecutive positions per warp
//                  store).  Positions beyond a row's own position, and pages
//                  outside the pool, get -inf.
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
constexpr int kEpiThreads = 256;                // two epilogue groups of 4 warps, alternating tiles
constexpr int kThreads = 64 + kEpiThreads;
constexpr int kTmemCols = 512;                  // 2 accumulators x 256 columns

constexpr int kOffStages = 0;
constexpr int kOffQ = kOffStages + kStages * kStageBytes;          // 2 row-block buffers
constexpr int kOffScales = kOffQ + 2 * kQBytes;                     // 2 x 256 B of key scales per stage
constexpr int kOffBars = kOffScales + kStages * 512;
constexpr int kOffPid = kOffBars + (2 * kStages + 9) * 8;
constexpr int kOffMisc = kOffPid + kPidChunk * 2 * 8;
constexpr int kSmemUsed = kOffMisc + 128;
constexpr int kSmemAlloc = kSmemUsed + 1024;
static_assert(kSmemAlloc <= 232448, "shared memory budget");
static_assert(kOffQ % 1024 == 0 && kQBytes % 1024 == 0, "swizzle atoms need 1 KB alignment");

struct Misc {
    int32_t stage_valid[kStages];
    uint32_t tmem_base;
    int32_t abort;
};
static_assert(sizeof(Misc) <= 128, "misc block");

// Work plan (device buffers in the caller's workspace).
struct MtPlan {
    int32_t* rb_first;     // [B+1] first row block of each request
    int32_t* rb_req;       // [NBmax] request of each row block
    int64_t* item_start;   // [NBmax+1] (row block, tile) prefix
    int32_t* nb;           // [1] row blocks in this batch
};

__device__ __forceinline__ int64_t cta_start(int64_t g, int64_t N, int64_t G) { return g * N / G; }

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
            mbar_init(&empty[s], 1 + 4);          // MMA commit + one arrive per warp of the epilogue group
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(&accf[a], 1);
            mbar_init(&acce[a], 4);
            mbar_init(&qfull[a], 1);
            mbar_init(&qempty[a], 1);
        }
        mbar_init(drain, 1);
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
        // Group g takes the tiles whose running index has parity g (= its
        // accumulator).  Warp w reads TMEM lanes 32 (w % 4) .., i.e. tokens
        // 32 (w % 4) .. of the tile.
        const int grp = (warp - 2) >> 2;
        const int quarter = warp & 3;
        const int tok = quarter * 32 + lane;
        Walk w;
        walk_begin(w, p, NB, i0, i1);
        int64_t gidx = 0;
        bool bad = false;
        while (w.i < w.i_end) {
            if (!bad && __any_sync(0xffffffffu, *abort_flag != 0)) bad = true;   // another role gave up
            if ((int)(gidx & 1) == grp && !bad) {
                const int r = p.rb_req[w.rb];
                const int t0 = (w.rb - p.rb_first[r]) * kRows;
                const int L = b.seq_len[r];
                const int qn = b.q_start[r + 1] - b.q_start[r];
                const int R = min(kRows, qn - t0);
                const int64_t row0 = b.q_start[r] + t0;
                const int tile = (int)(w.i - p.item_start[w.rb]);
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
                    const int p0 = L - qn + t0;               // position of the block's first row
                    for (int rr = 0; rr < R; ++rr) {
                        uint32_t v[32];
                        tmem_ld_32x32b_x32(tmem + ((uint32_t)(quarter * 32) << 16) + acc * 256 + rr * 32, v);
                        tmem_ld_wait();
                        const float4* w4 = reinterpret_cast<const float4*>(wq + (row0 + rr) * 32);
                        float a0 = 0.f, a1 = 0.f, a2 = 0.f, a3 = 0.f;
#pragma unroll
                        for (int m4 = 0; m4 < 8; ++m4) {
                            const float4 ww = __ldg(w4 + m4);
                            a0 = fmaf(ww.x, fmaxf(__uint_as_float(v[4 * m4 + 0]), 0.f), a0);
                            a1 = fmaf(ww.y, fmaxf(__uint_as_float(v[4 * m4 + 1]), 0.f), a1);
                            a2 = fmaf(ww.z, fmaxf(__uint_as_float(v[4 * m4 + 2]), 0.f), a2);
                            a3 = fmaf(ww.w, fmaxf(__uint_as_float(v[4 * m4 + 3]), 0.f), a3);
                        }
                        const float score = ((a0 + a1) + (a2 + a3)) * sk;
                        if (pos < ld)
                            scores[(row0 + rr) * ld + pos] = (page_ok && pos <= p0 + rr) ? score : -INFINITY;
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
            walk_next(w, p);
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

size_t mt_plan_bytes(int64_t batch, int64_t total_q) {
    const int64_t nb_max = (total_q + imt::kRows - 1) / imt::kRows + batch;
    size_t b = 0;
    b += (size_t)(batch + 1) * 4;                       // rb_first
    b = (b + 15) / 16 * 16;
    b += (size_t)nb_max * 4;                            // rb_req
    b = (b + 15) / 16 * 16;
    b += (size_t)(nb_max + 1) * 8;                      // item_start
    b += 16;                                            // nb
    return (b + 255) / 256 * 256;
}

static imt::MtPlan carve_mt_plan(void* base, int64_t batch, int64_t total_q) {
    const int64_t nb_max = (total_q + imt::kRows - 1) / imt::kRows + batch;
    uint8_t* q = static_cast<uint8_t*>(base);
    imt::MtPlan p;
    size_t off = 0;
    p.rb_first = reinterpret_cast<int32_t*>(q + off);
    off += (size_t)(batch + 1) * 4;
    off = (off + 15) / 16 * 16;
    p.rb_req = reinterpret_cast<int32_t*>(q + off);
    off += (size_t)nb_max * 4;
    off = (off + 15) / 16 * 16;
    p.item_start = reinterpret_cast<int64_t*>(q + off);
    off += (size_t)(nb_max + 1) * 8;
    p.nb = reinterpret_cast<int32_t*>(q + off);
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
    if (ensure_smem_limit(reinterpret_cast<const void*>(&imt::score_rows_kernel), imt::kSmemAlloc) != DSA_OK)
        return DSA_ERR_CUDA;
    BatchDev bd = to_dev(b);
    imt::MtPlan p = carve_mt_plan(plan_ws, b->batch, b->total_q);
    imt::plan_kernel<<<1, 1024, 0, s>>>(bd, skip_short ? 1 : 0, full_rows ? 1 : 0, p);
    DSA_CHECK_LAUNCH();
    imt::score_rows_kernel<<<G, imt::kThreads, imt::kSmemAlloc, s>>>(kmap, qmap, cache, wq, bd, p, scores, ld, st);
    DSA_CHECK_LAUNCH();
    return DSA_OK;
}

}  // namespace dsa
