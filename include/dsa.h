/*
 * dsa.h - C ABI of the GB300 (sm_103a) DSA attention step library (libdsa.so).
 *
 * The step has three parts, all run on one GPU by hand-written CUDA kernels:
 *   1. the lightning indexer: every cached token j gets the score
 *        s_j = sum_{m<32} w_m * ReLU(<q_m, k_j>)
 *      from 32 indexer query heads of 128 dims against one shared 128-d FP8
 *      index key ("vLLM 推理链路概览：以 GLM-5.2 为例", section DSA Indexer);
 *   2. top-2048 selection over those scores, I = TopK_{j,2048}(s_j) (same section);
 *   3. sparse MLA in absorbed (MQA) form over the selected tokens:
 *        alpha = softmax_{j in I, j <= i}(q k_j^T / sqrt(256)),  o = sum alpha c_j
 *      with 64 query heads of 576 dims and a 512-d latent output per head
 *      ("vLLM 推理链路概览", section Sparse MLA Attention; "GLM-5.3 推理全链路(一)",
 *      section "decode: MQA 形态与吸收").
 * Shared layers reuse the last full layer's indices ("GLM-5.3 推理全链路(一)",
 * section 4.5; "GLM-5.3 推理全链路(十一)", section "配置里的 78 个字符").
 *
 * Conventions for every call:
 *   - Every pointer documented "device" is caller-owned device memory; the
 *     library allocates nothing on the device.  Scratch comes from a caller
 *     workspace sized by the matching *_workspace_size call.
 *   - Every compute call is asynchronous on the caller's CUDA stream, passed
 *     as `void* stream` (a cudaStream_t; NULL = the legacy default stream).
 *   - Argument errors (null pointers, sizes, alignment, unsupported shapes) are
 *     detected on the host and returned before anything is launched.
 *   - A call over zero items (n = 0 tokens or rows, or a batch whose total_q
 *     is 0) checks its sizes, its batch and its share handle, launches
 *     nothing and returns DSA_OK; its buffer pointers may then be NULL.  An
 *     indexer call with no rows still publishes its (empty) top-k to a given
 *     share handle.
 *   - Errors that only the device can see (a page id outside the cache, a slot
 *     outside the cache, an index outside the context, a wait that timed out)
 *     never fault: the offending element is skipped and recorded in the
 *     optional device status block `dev_status` (DSA_DEVICE_STATUS_WORDS int32,
 *     device; NULL = do not record).  Read it with dsa_device_status_read().
 *   - No call throws, exits or traps.
 *   - A call runs on the CUDA device that is current on the calling host
 *     thread; every buffer it gets must live on that device.  The library's
 *     one-time set-up (kernel shared-memory limits, TMA descriptor encoding)
 *     is kept per device and per host thread, so several host threads and
 *     several devices may use the library at once.  Calls that share a
 *     workspace or an output buffer must still be ordered by the caller.
 *   - "bf16" buffers hold IEEE bfloat16 bit patterns (uint16).
 *
 * Token positions: request r holds seq_len[r] cached tokens, INCLUDING its
 * q_len[r] new query tokens; query token t (0-based within the request) sits at
 * position p = seq_len[r] - q_len[r] + t and sees positions 0..p.
 * Caches are paged: logical page k of request r is physical page
 * page_table[r * max_pages + k]; one page table serves the index-K cache and
 * every layer's latent cache ("GLM-5.3 推理全链路(一)", 细节二: page-interleaved
 * pools share one logical-page plan).
 */
#ifndef DSA_H_
#define DSA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ---- Layout constants ("GLM-5.3 推理全链路(十一)", sections 索引器缓存里存的是什么
 *      and 主 KV 缓存里存的是什么; page size 64 from 优化一: 按页分块打分). -------- */
#define DSA_PAGE_TOKENS      64
#define DSA_INDEX_HEADS      32
#define DSA_INDEX_HEAD_DIM   128
#define DSA_IDXK_TOKEN_BYTES 132    /* 128 B FP8 E4M3 key + 4 B scale             */
#define DSA_IDXK_PAGE_BYTES  8448   /* [64 x 128 B payload | 64 x fp32 scale]     */
/* MXFP4 index-K variant ("GLM-5.3 推理全链路(十一)", 两个框架的对照): per token 64 B of
 * packed E2M1 values (element 2i in the low nibble of byte i) and four ue8m0
 * block scales (one per 32 dims, byte e + 127).                               */
#define DSA_IDXK_MXFP4_TOKEN_BYTES 68
#define DSA_IDXK_MXFP4_PAGE_BYTES  4352 /* [64 x 64 B packed | 64 x 4 B scales]   */
#define DSA_MLA_HEADS        64
#define DSA_LATENT_DIM       512
#define DSA_ROPE_DIM         64
#define DSA_QK_DIM           576
#define DSA_KV_TOKEN_BYTES   656    /* [512 B FP8 | 4 x fp32 scale | 64 x bf16]   */
#define DSA_KV_PAGE_BYTES    41984  /* 64 token rows of 656 B                     */
#define DSA_TOPK             2048
#define DSA_DEVICE_STATUS_WORDS 4

/* ---- Status codes ------------------------------------------------------- */
typedef int32_t dsa_status;
#define DSA_OK                       0
#define DSA_ERR_INVALID_ARGUMENT     1  /* null pointer, negative size, bad enum    */
#define DSA_ERR_ALIGNMENT            2  /* a buffer is not 16-byte aligned          */
#define DSA_ERR_UNSUPPORTED          3  /* a shape the library does not support     */
#define DSA_ERR_WORKSPACE_TOO_SMALL  4
#define DSA_ERR_NO_TOPK_SOURCE       5  /* shared layer with no full layer published*/
#define DSA_ERR_CUDA                 6  /* a CUDA runtime call failed               */
#define DSA_ERR_DEVICE               7  /* dsa_device_status_read saw device errors */
#define DSA_ERR_SCRATCH_LIMIT        8  /* batch too large for the fixed scratch of
                                           dsa_indexer_topk_noalloc                 */

/* Bits of dev_status[0]; dev_status[1] counts offending elements, dev_status[2]
 * holds the low 32 bits of one offending value, dev_status[3] is reserved.      */
#define DSA_DEVERR_SLOT_RANGE    1   /* store: slot >= 64 * num_pages              */
#define DSA_DEVERR_PAGE_RANGE    2   /* page_table entry outside [0, num_pages)    */
#define DSA_DEVERR_INDEX_RANGE   4   /* top-k index >= seq_len of its request      */
#define DSA_DEVERR_TIMEOUT       8   /* a bounded wait inside a kernel gave up     */
#define DSA_DEVERR_FP16_RANGE   16   /* sparse MLA computes in fp16: a latent
                                        scale outside [2^-15, 2^7], a key RoPE
                                        value with |r| >= 2^16 (clamped) or an
                                        inf / NaN in q makes an operand inexact.
                                        q itself is scaled per row by a power of
                                        two, so any finite q is in range        */

/* Output dtypes of the sparse MLA calls. */
#define DSA_DTYPE_BF16 0
#define DSA_DTYPE_F32  1

/* Description of one batch of requests; the struct itself lives on the host. */
typedef struct dsa_batch {
    int32_t batch;              /* B >= 1 requests                                  */
    int32_t max_pages;          /* entries per page-table row                       */
    int32_t max_seq_len;        /* host upper bound on every seq_len[r]             */
    int32_t max_q_len;          /* host upper bound on every q_len[r]               */
    int64_t total_q;            /* T = q_start[B]: query rows in this batch         */
    int64_t num_pages;          /* pages in each cache buffer (device bounds check) */
    const int32_t* seq_len;     /* device [B]                                       */
    const int32_t* q_start;     /* device [B+1], q_start[0] = 0, q_len = diff       */
    const int32_t* page_table;  /* device [B * max_pages]                           */
} dsa_batch;

/* Host object that carries the last full layer's indices to the shared layers
 * ("GLM-5.3 推理全链路(十一)", section 一次前向里 topk 只算一遍: the full layer
 * updates the shared state, the following shared layers read the same tensor). */
typedef struct dsa_topk_share dsa_topk_share;

/* ---- General ------------------------------------------------------------ */
int32_t     dsa_abi_version(void);                 /* 1 for this header */
const char* dsa_status_string(dsa_status s);        /* static string, never NULL */

/* Zero the device status block (async on stream). */
dsa_status dsa_device_status_reset(int32_t* dev_status, void* stream);
/* Synchronise `stream`, copy the block into host_out[4]; returns DSA_ERR_DEVICE
 * when any error bit is set, DSA_OK otherwise. */
dsa_status dsa_device_status_read(const int32_t* dev_status, void* stream, int32_t* host_out);
/* Testing hook for failure detection, process-wide: the limit, in ns, of the
 * pipeline waits of the decode indexer's score kernel (dsa_indexer_topk and
 * dsa_indexer_topk_mxfp4 on a batch of one row per request) launched after
 * the call.  2e9 (2 s) by default; 0 makes every wait that is not already
 * satisfied give up at once.  A wait that gives up records
 * DSA_DEVERR_TIMEOUT; the kernel then lets its copies and MMAs in flight
 * finish, releases its tensor memory and returns, the merge sees only the
 * segments finished before, and the call's top-k is then meaningless.
 * Always DSA_OK. */
dsa_status dsa_debug_set_wait_limit_ns(uint64_t ns);

/* ---- Index-K store ("GLM-5.3 推理全链路(一)", 4.5 闪电索引器; "GLM-5.3 推理全链路(十一)",
 *      索引器缓存里存的是什么) -------------------------------------------------
 * For each of n new tokens: LayerNorm over the 128 dims of k (eps, optional
 * affine gamma/beta, fp32), interleaved RoPE on dims 0..63 (pairs (2i, 2i+1)
 * rotated by pos * rope_base^(-2i/64)), then FP8 E4M3 (round to nearest even)
 * with one scale 2^e per token, e the smallest integer with amax <= 448 * 2^e
 * (amax == 0 -> 1.0), stored as fp32.  Token goes to cache slot `slot`
 * (page slot/64, row slot%64); slot < 0 skips the token (padded rows).
 *   k          device bf16 [n,128], row-major
 *   pos        device int32 [n]
 *   slot       device int64 [n]
 *   gamma,beta device fp32 [128] or NULL (identity affine)
 *   idxk_cache device uint8 [num_pages * 8448], 16-byte aligned
 * A slot >= 64 * num_pages is skipped and recorded (DSA_DEVERR_SLOT_RANGE). */
dsa_status dsa_index_k_store(const void* k, const int32_t* pos, const int64_t* slot, int64_t n,
                             const float* gamma, const float* beta, float ln_eps, float rope_base,
                             uint8_t* idxk_cache, int64_t num_pages,
                             int32_t* dev_status, void* stream);

/* ---- Index-K store, MXFP4 variant --------------------------------------------
 * The same LayerNorm and RoPE as dsa_index_k_store, then per block of 32 dims
 * the OCP MX scale 2^e with e = floor(log2(amax)) - 2 (amax == 0 -> e = 0; e
 * clamped to [-127, 127]) and E2M1 elements rounded to nearest, ties to even,
 * saturated at +-6.  Arguments as dsa_index_k_store, except
 *   idxk_cache device uint8 [num_pages * 4352], 32-byte aligned.              */
dsa_status dsa_index_k_store_mxfp4(const void* k, const int32_t* pos, const int64_t* slot, int64_t n,
                                   const float* gamma, const float* beta, float ln_eps, float rope_base,
                                   uint8_t* idxk_cache, int64_t num_pages,
                                   int32_t* dev_status, void* stream);

/* ---- Latent KV store (writes the 656-B rows that sparse MLA gathers;
 *      "GLM-5.3 推理全链路(十一)", 主 KV 缓存里存的是什么) --------------------------
 * For each token: c (512 dims) -> four blocks of 128, each FP8 E4M3 with its own
 * scale (same rule as above); the 64 RoPE dims are copied as bf16.
 *   c        device bf16 [n,512];  rope  device bf16 [n,64]
 *   slot     device int64 [n] (slot < 0 skips the token)
 *   kv_cache device uint8 [num_pages * 41984], 16-byte aligned               */
dsa_status dsa_latent_kv_store(const void* c, const void* rope, const int64_t* slot, int64_t n,
                               uint8_t* kv_cache, int64_t num_pages,
                               int32_t* dev_status, void* stream);

/* ---- Latent store from the A-projection outputs ("GLM-5.3 推理全链路(一)", 4.3
 *      两个 RMSNorm 与 RoPE: the fused norm/RoPE kernel writes the KV pool and, on a
 *      layer with an indexer, the index cache) ----------------------------------
 * For each token: kv_c (512) -> RMSNorm x / sqrt(mean(x^2) + rms_eps), times
 * kv_gamma if given, fp32 -> the latent row of dsa_latent_kv_store (four FP8
 * blocks with their scales); k_pe (64) -> interleaved RoPE (pairs (2i, 2i+1)
 * rotated by pos * rope_base^(-2i/64)) -> bf16 (round to nearest even).
 * idx_k != NULL also stores the index key of each token exactly as
 * dsa_index_k_store does (LayerNorm idx_gamma/idx_beta/ln_eps, same RoPE) into
 * idxk_cache at the same slot; idx_k == NULL (a shared layer) writes no key.
 *   kv_c device bf16 [n,512], 16-byte aligned; k_pe device bf16 [n,64], 4-byte aligned
 *   pos  device int32 [n]; slot device int64 [n] (< 0 skips the token)
 *   kv_cache device uint8 [num_pages * 41984]; idx_k bf16 [n,128] or NULL;
 *   idxk_cache device uint8 [idx_num_pages * 8448] (when idx_k != NULL)
 * A slot beyond either cache is skipped and recorded (DSA_DEVERR_SLOT_RANGE). */
dsa_status dsa_latent_kv_store_fused(const void* kv_c, const void* k_pe, const int32_t* pos, const int64_t* slot,
                                     int64_t n, const float* kv_gamma, float rms_eps, float rope_base,
                                     uint8_t* kv_cache, int64_t num_pages,
                                     const void* idx_k, const float* idx_gamma, const float* idx_beta, float ln_eps,
                                     uint8_t* idxk_cache, int64_t idx_num_pages,
                                     int32_t* dev_status, void* stream);

/* ---- Indexer + top-2048 ("vLLM 推理链路概览", DSA Indexer; "GLM-5.3 推理全链路(十一)",
 *      优化二: 短上下文直接跳过打分) ------------------------------------------------
 * For every query row i (request r, position p): the query is quantised to
 * FP8 E4M3 with one scale per head (the scale rule above), scores
 * s_j = sum_m w_m ReLU(<q_m, k_j>) are formed on the dequantised values with
 * fp32 accumulation for j = 0..p, and topk[i] receives the 2048 positions with
 * the largest scores (ties -> lower position), in ascending order.  When
 * p + 1 <= 2048 no score is computed and topk[i] = [0, 1, ..., p, -1, ...].
 * Full score rows are never written to memory.
 *   q           device bf16 [T,32,128];  w  device fp32 [T,32]
 *   idxk_cache  device uint8 [num_pages * 8448], 16-byte aligned
 *   topk        device int32 [T,2048]
 *   topk_scores device fp32 [T,2048] or NULL: the score of each selected
 *               position (0 for -1 entries and for short contexts)
 *   share       NULL, or a share handle that receives (layer_id, topk, T)
 *   ws          device workspace of at least dsa_indexer_topk_workspace_size() bytes.
 *               A decode batch (one query row per request) needs O(T) bytes for
 *               any GPU; a batch with several rows per request needs row
 *               histograms plus candidate slots of 6144 entries per query row
 *               and CTA share, O(T x 6144), sized for the SM count of the device
 *               current at the size call (call both on the same device).       */
dsa_status dsa_indexer_topk_workspace_size(const dsa_batch* b, size_t* bytes);
dsa_status dsa_indexer_topk(const void* q, const float* w, const uint8_t* idxk_cache,
                            const dsa_batch* b, int32_t* topk, float* topk_scores,
                            dsa_topk_share* share, int32_t layer_id,
                            void* ws, size_t ws_bytes, int32_t* dev_status, void* stream);

/* ---- Indexer + top-2048 over an MXFP4 index-K cache --------------------------
 * dsa_indexer_topk for a cache written by dsa_index_k_store_mxfp4: the same
 * queries, selection rule, outputs, share handle and workspace (sized by
 * dsa_indexer_topk_workspace_size); scores are formed on the dequantised
 * values (E2M1 x 2^e per 32-dim block).  A batch with several query rows per
 * request (verify, prefill) runs each row as a decode row over its request's
 * keys up to its position: a request's keys are read once per row (the FP8
 * call reads them once per block of 8 rows); at most 65535 rows
 * (DSA_ERR_UNSUPPORTED beyond).
 *   idxk_cache device uint8 [num_pages * 4352], 32-byte aligned               */
dsa_status dsa_indexer_topk_mxfp4(const void* q, const float* w, const uint8_t* idxk_cache,
                                  const dsa_batch* b, int32_t* topk, float* topk_scores,
                                  dsa_topk_share* share, int32_t layer_id,
                                  void* ws, size_t ws_bytes, int32_t* dev_status, void* stream);

/* ---- Indexer + top-2048 without a workspace argument --------------------
 * The pages have no counterpart of this call.  It serves callers that cannot
 * allocate device memory per call and keep no workspace of their own: a plain
 * C host loop that owns no device allocator, or a runtime whose device memory
 * is fully reserved up front and forbids allocation on the serving path.
 * Inputs, outputs and kernels are those of dsa_indexer_topk, for decode
 * batches only (every request has q_len == 1; other shapes return
 * DSA_ERR_UNSUPPORTED).  The scratch is a fixed array of
 * DSA_NOALLOC_SCRATCH_BYTES inside this library, so no call allocates.  A batch
 * of T = B rows needs, on a GPU with S SMs,
 *   round_up(4224 T, 256) + 16384 T + (S + B) * 36884 + 12 (B + 1) + 8 S
 * bytes, plus up to 768 bytes of alignment (194 rows fit at S = 152, 195 do
 * not); a larger batch returns
 * DSA_ERR_SCRATCH_LIMIT and launches nothing.  Nothing in the scratch needs
 * to start at zero: the kernels clear the histogram bins and plan entries
 * before they read them.  The first call on a device performs set-up (it looks
 * up the scratch's device address); make that call before any stream capture
 * begins.  There is one scratch per device: calls that overlap in time (on
 * other streams or from other host threads) race on it, and the caller must
 * serialise them. */
#define DSA_NOALLOC_SCRATCH_BYTES (16u << 20)
dsa_status dsa_indexer_topk_noalloc(const void* q, const float* w, const uint8_t* idxk_cache,
                                    const dsa_batch* b, int32_t* topk, float* topk_scores,
                                    dsa_topk_share* share, int32_t layer_id,
                                    int32_t* dev_status, void* stream);

/* Debug / parity hook: the same scores as dsa_indexer_topk, written in full.
 *   scores device fp32 [T, ld]; entries j > p of row i (and every entry of a
 *   page whose id is out of range) are set to -inf.  Requires ld >= max_seq_len.
 *   ws: device workspace of dsa_indexer_scores_workspace_size() bytes.        */
dsa_status dsa_indexer_scores_workspace_size(const dsa_batch* b, size_t* bytes);
dsa_status dsa_indexer_scores(const void* q, const float* w, const uint8_t* idxk_cache,
                              const dsa_batch* b, float* scores, int64_t ld,
                              void* ws, size_t ws_bytes, int32_t* dev_status, void* stream);
/* The same score rows from a CUDA-core kernel (no tensor cores), for decode
 * batches only (one query row per request, at most 65535 of them; else
 * DSA_ERR_UNSUPPORTED): kept to measure the tensor-core path against.  Same
 * quantised queries, E4M3 products and fp32 sums, in another order, so its
 * scores meet the same tolerance.  Entries j >= seq_len of a row are not
 * written; pages out of range give -inf and are recorded.
 *   ws: device workspace of at least T * (4096 + 128) bytes, 16-byte aligned. */
dsa_status dsa_indexer_scores_cuda_core(const void* q, const float* w, const uint8_t* idxk_cache,
                                        const dsa_batch* b, float* scores, int64_t ld,
                                        void* ws, size_t ws_bytes, int32_t* dev_status, void* stream);

/* Parity hook: top-2048 of given fp32 score rows, same selection rule and
 * output order as dsa_indexer_topk.  Row r uses scores[r*ld + 0 .. valid_len[r]-1].
 *   scores device fp32 [rows, ld]; valid_len device int32 [rows] (<= max_len <= ld)
 *   topk   device int32 [rows, 2048]                                          */
dsa_status dsa_topk_from_scores_workspace_size(int32_t rows, int64_t max_len, size_t* bytes);
dsa_status dsa_topk_from_scores(const float* scores, int64_t ld, const int32_t* valid_len,
                                int32_t rows, int64_t max_len, int32_t* topk,
                                void* ws, size_t ws_bytes, void* stream);

/* ---- Sparse MLA ("vLLM 推理链路概览", Sparse MLA Attention) ---------------------
 * For every query row i (request r, position p) and head h < 64:
 *   S_hj = softmax_scale * <q_ih, k_j>,  k_j = [c_j * scale | rope_j] (576 dims)
 *   out_ih = sum_j softmax_j(S_hj) c_j   over the valid entries j of topk[i]
 * (entries -1 and entries > p are ignored; an entry >= seq_len[r] is skipped
 * and recorded).  Softmax statistics and accumulation are fp32.
 *   q        device bf16 [T,64,576]
 *   topk     device int32 [T,2048], or NULL to take the indices published in
 *            `share` (DSA_ERR_NO_TOPK_SOURCE when it holds none)
 *   kv_cache device uint8 [num_pages * 41984] of THIS layer, 16-byte aligned
 *   out      device [T,64,512], bf16 or fp32 per out_dtype
 *   lse      device fp32 [T,64] or NULL: natural-log sum of exp(S) (-inf when
 *            a row selects nothing, in which case out is 0)
 * decode: suited to few query rows per request (splits each row's 2048 keys
 * across CTAs); prefill: suited to many query rows.  Same results.           */
dsa_status dsa_sparse_mla_workspace_size(const dsa_batch* b, size_t* bytes);
dsa_status dsa_sparse_mla_decode(const void* q, const int32_t* topk, const dsa_topk_share* share,
                                 const uint8_t* kv_cache, const dsa_batch* b, float softmax_scale,
                                 void* out, int32_t out_dtype, float* lse,
                                 void* ws, size_t ws_bytes, int32_t* dev_status, void* stream);
dsa_status dsa_sparse_mla_prefill(const void* q, const int32_t* topk, const dsa_topk_share* share,
                                  const uint8_t* kv_cache, const dsa_batch* b, float softmax_scale,
                                  void* out, int32_t out_dtype, float* lse,
                                  void* ws, size_t ws_bytes, int32_t* dev_status, void* stream);

/* ---- Context-parallel split of long requests ("GLM-5.3 推理全链路(十一)", 两个框架的
 *      对照: with prefill context parallelism the indexer's reads are spread over
 *      the ranks; "Accelerating GLM-5.3-Flash on H200", prefill 的重点是少搬一次、少等
 *      一次: CP4 on the prefill side) ---------------------------------------------
 * A request's positions are cut into G <= 8 disjoint slices, one per rank; a
 * rank holds its slice in its own caches, as a request of seq_len = slice
 * length with local positions 0.., and runs the single-GPU calls on it.  Each
 * slice must be longer than 2048 tokens (a shorter one selects all its
 * positions without scores).  Per query row:
 *   1. dsa_indexer_topk on the slice gives the rank's top-2048 (local
 *      positions) and their scores (topk_scores);
 *   2. the caller gathers every rank's lists, [G, rows, 2048] int32 and fp32,
 *      and each slice's first global position, [G, rows] int64;
 *   3. dsa_cp_topk_merge: the global top-2048, which is the top-2048 of the
 *      union of the lists (a position selected over the whole context is
 *      also selected within its own slice); same order and ties as
 *      dsa_indexer_topk, global positions ascending, -1 padded;
 *   4. dsa_cp_topk_localize: the rank's share of the global list, as local
 *      positions compacted to the front of each row, -1 padded;
 *   5. sparse MLA on the slice with that list, fp32 output and lse;
 *   6. the caller gathers every rank's (out, lse), [G, rows, 64, 512] fp32 and
 *      [G, rows, 64] fp32;
 *   7. dsa_cp_attention_merge: softmax attention over the union,
 *      out = sum_g w_g out_g / sum_g w_g with w_g = exp(lse_g - max_g lse_g),
 *      lse = max_g lse_g + log(sum_g w_g) (a head empty on every rank: 0, -inf).
 * dsa_cp_topk_merge
 *   cand_pos    device int32 [G, rows, 2048]: local positions, -1 = none
 *   cand_scores device fp32 [G, rows, 2048]: their scores
 *   pos_offset  device int64 [G, rows]: global position of local position 0
 *   topk        device int32 [rows, 2048]; topk_scores device fp32 [rows, 2048]
 *               or NULL (0 for -1 entries)
 *   A global position outside [0, 2^31 - 1) is skipped and recorded
 *   (DSA_DEVERR_INDEX_RANGE).  Slices must not overlap.
 * dsa_cp_topk_localize
 *   topk        device int32 [rows, 2048] global positions
 *   slice_start device int64 [rows], slice_len device int64 [rows]: this rank's
 *               slice [start, start + len) of each row's request
 *   local_topk  device int32 [rows, 2048], not the same buffer as topk
 * dsa_cp_attention_merge
 *   o_parts     device fp32 [G, rows, 64, 512]; lse_parts device fp32 [G, rows, 64]
 *               (natural log, -inf for a rank with no selected position)
 *   out         device [rows, 64, 512] bf16 or fp32 per out_dtype
 *   lse         device fp32 [rows, 64] or NULL                                   */
dsa_status dsa_cp_topk_merge(const int32_t* cand_pos, const float* cand_scores, const int64_t* pos_offset,
                             int32_t ranks, int64_t rows, int32_t* topk, float* topk_scores,
                             int32_t* dev_status, void* stream);
dsa_status dsa_cp_topk_localize(const int32_t* topk, int64_t rows, const int64_t* slice_start,
                                const int64_t* slice_len, int32_t* local_topk, void* stream);
dsa_status dsa_cp_attention_merge(const float* o_parts, const float* lse_parts, int32_t ranks, int64_t rows,
                                  void* out, int32_t out_dtype, float* lse, void* stream);

/* ---- Full / shared layer schedule ("GLM-5.3 推理全链路(十一)", 配置里的 78 个字符) --
 * dsa_parse_indexer_types: types[l] is "full" or "shared"; is_full[l] = 1/0.
 *   An unknown string returns DSA_ERR_INVALID_ARGUMENT.
 * dsa_schedule_from_freq: the parameterised form, layer l is shared iff
 *   max(l - offset + 1, 0) % freq != 0 (GLM-5.3: freq 4, offset 3).           */
dsa_status dsa_parse_indexer_types(const char* const* types, int32_t n_layers, uint8_t* is_full);
dsa_status dsa_schedule_from_freq(int32_t n_layers, int32_t freq, int32_t offset, uint8_t* is_full);

/* ---- Schedule from whichever fields a model config carries ("GLM-5.3 推理全链路
 *      (十一)", 配置里的 78 个字符: the order SGLang's dsa_layer_skips_topk checks) ---
 * Layer l is shared (reuses the previous top-k) by the first rule that applies:
 *   1. indexer_types != NULL: types[l] == "shared" (layers past n_types: full;
 *      any entry other than "full" / "shared" -> DSA_ERR_INVALID_ARGUMENT);
 *   2. cli_factor > 1: l % cli_factor != 0;
 *   3. index_topk_pattern != NULL: pattern[l] == 'S' (past its end: full);
 *   4. max(l - offset + 1, 0) % index_topk_freq != 0 with offset =
 *      index_skip_topk_offset, or 2 when it is negative (absent): layers 0 and 1
 *      full, layer 2 shared, then one full layer in every index_topk_freq.
 * is_full[l] receives 0 / 1 for l < n_layers.                                  */
typedef struct dsa_schedule_config {
    const char* const* indexer_types;   /* n_types strings, or NULL            */
    int32_t n_types;
    int32_t cli_factor;                 /* <= 1: not set                       */
    const char* index_topk_pattern;     /* NUL-terminated, or NULL             */
    int32_t index_topk_freq;            /* >= 1                                */
    int32_t index_skip_topk_offset;     /* < 0: not set (2)                    */
} dsa_schedule_config;
dsa_status dsa_schedule_resolve(const dsa_schedule_config* cfg, int32_t n_layers, uint8_t* is_full);

/* ---- Share handle ("GLM-5.3 推理全链路(十一)", 一次前向里 topk 只算一遍) ------------
 * publish: record that `topk` (device int32 [rows,2048]) holds layer
 *   `layer_id`'s indices; the pointer is borrowed, not copied.
 * get: the last published indices; DSA_ERR_NO_TOPK_SOURCE if none.
 * reset: forget the published indices (e.g. at the start of a forward pass). */
dsa_status dsa_topk_share_create(dsa_topk_share** out);
dsa_status dsa_topk_share_destroy(dsa_topk_share* s);
dsa_status dsa_topk_share_reset(dsa_topk_share* s);
dsa_status dsa_topk_share_publish(dsa_topk_share* s, int32_t layer_id, const int32_t* topk, int64_t rows);
dsa_status dsa_topk_share_get(const dsa_topk_share* s, const int32_t** topk, int64_t* rows,
                              int32_t* layer_id);

/* ---- Top-k reuse across the draft steps of one MTP iteration
 *      ("GLM-5.3 推理全链路(十一)", sections 优化三: MTP 迭代内复用 topk and
 *      优化四: PD 分离下的 seed 传输) -----------------------------------------------
 * The MTP layer's draft steps can attend with the top-k of the iteration's
 * first step instead of running their own indexer.  A seed row is a plain copy
 * of one selected top-k row, index_topk + index_kpool - 1 int32 wide.
 *
 * dsa_mtp_topk_width: *width = index_topk + index_kpool - 1 (2048 for
 *   index_topk 2048, index_kpool 1).  Both must be >= 1.
 * dsa_mtp_seed_write: for r < n, seed[r, 0..2047] = topk[src_row[r], 0..2047]
 *   and seed[r, 2048..width-1] = -1 (the kpool tail slots).  src_row NULL means
 *   src_row[r] = r.  A src_row outside [0, topk_rows) yields a row of -1 and
 *   is recorded (DSA_DEVERR_INDEX_RANGE).
 *     topk    device int32 [topk_rows, 2048], 16-byte aligned
 *     src_row device int32 [n] or NULL
 *     seed    device int32 [n, width], width >= 2048, 16-byte aligned
 * dsa_topk_share_mtp_begin: start one MTP iteration on a share handle.  Reuse
 *   is on only when enabled != 0 and eagle_topk == 1; with several draft
 *   candidates per step the draft rows are reordered and a carried row no
 *   longer belongs to its request.  *reuse_on (optional) receives the decision.
 *   With reuse on, the handle's published indices are replaced by the carried
 *   seed when keep_carry_seed != 0 and seed != NULL (device int32 [rows, 2048];
 *   any other seed_width returns DSA_ERR_UNSUPPORTED), and forgotten
 *   otherwise.  With reuse off the published indices are left as they are.
 * dsa_topk_share_needs_scoring: *needs = 0 while an iteration with reuse on
 *   holds published indices: the draft step skips the indexer and passes
 *   topk = NULL plus the handle to sparse MLA.  *needs = 1 otherwise: the step
 *   runs dsa_indexer_topk with the handle, which publishes for the next steps.
 * dsa_topk_share_mtp_end: end the iteration: reuse off, published indices
 *   forgotten.
 * The three share calls are host-only and do not touch the device. */
dsa_status dsa_mtp_topk_width(int32_t index_topk, int32_t index_kpool, int32_t* width);
dsa_status dsa_mtp_seed_write(const int32_t* topk, int64_t topk_rows, const int32_t* src_row, int64_t n,
                              int32_t* seed, int32_t width, int32_t* dev_status, void* stream);
dsa_status dsa_topk_share_mtp_begin(dsa_topk_share* s, int32_t enabled, int32_t eagle_topk,
                                    int32_t keep_carry_seed, const int32_t* seed, int64_t rows,
                                    int32_t seed_width, int32_t* reuse_on);
dsa_status dsa_topk_share_needs_scoring(const dsa_topk_share* s, int32_t* needs);
dsa_status dsa_topk_share_mtp_end(dsa_topk_share* s);

#ifdef __cplusplus
}
#endif
#endif /* DSA_H_ */
