// Work plan of the fused tensor-core indexer (device buffers in the caller's
// workspace) and its host entry points.
#pragma once
#include <cuda.h>
#include "indexer_common.cuh"

namespace dsa {

// Tiles [lo, hi) (128 tokens each, relative to the request) of request r,
// scored by CTA `cta`; its candidates go to slot = segment index.
struct Seg {
    int32_t r, lo, hi, cta;
};

// Candidate slots of one segment (one query row's share of one CTA's tiles):
// the decode kernel's shared-memory buffer, and the multi-row kernel's larger
// workspace slots (a compaction there stalls the stream, so fewer of them pay).
constexpr int kSegCandidates = 4608;
constexpr int kRowSlotCandidates = 6144;

struct Plan {
    int64_t* tile_start;   // [B+1] tile prefix over requests that need scoring
    int32_t* seg_first;    // [B+1] first segment of each request
    int32_t* cta_range;    // [2G] segment range of each CTA
    Seg* segs;             // [G+B]
    uint32_t* cand_key;    // [G+B, segment candidate slots]
    int32_t* cand_pos;     // [G+B, segment candidate slots]
    int32_t* cand_cnt;     // [G+B]
    uint32_t* hist;        // [T, 4096] top-12-bit key histogram of every visible score, per query row
    // Row mode (batches with several query rows per request): the segments of
    // query row i are slots row_seg0[i] .. row_seg0[i] + row_segn[i] - 1, and
    // slot s belongs to row slot_row[s] (-1: unused); *nslots slots in use.
    // NULL in the decode layout, where request r's segments are seg_first[r] ...
    const int32_t* slot_row;
    const int32_t* row_seg0;
    const int32_t* row_segn;
    const int32_t* nslots;
    int64_t seg_stride;    // entries from one slot to the next (at most kSegCandidates of them in use)
};

// The two merge kernels of the decode indexer over a plan (decode or row
// mode): up to max_segs segment blocks, then one block per query row.
dsa_status launch_topk_merge(const dsa_batch* b, Plan p, int64_t max_segs, int32_t* topk, float* topk_scores,
                             cudaStream_t s);

size_t tc_plan_bytes(int64_t batch, int G);
// The decode indexer + top-2048 from the bf16 index queries q [T,32,128] and
// head weights w [T,32]: quantises q into q8 / wq (T x 4096 B, T x 32 fp32)
// and clears hist (T x 4096 words) in the launch that builds the plan, then
// scores and selects.  mx: the cache is the MXFP4 index-K layout
// (DSA_IDXK_MXFP4_PAGE_BYTES pages).
dsa_status launch_indexer_tc(const void* q, const float* w, uint8_t* q8, float* wq, uint32_t* hist,
                             const uint8_t* cache, const dsa_batch* b, int32_t* topk, float* topk_scores, void* plan_ws,
                             int G, int32_t* st, cudaStream_t s, bool mx = false);
int device_sm_count();

size_t mt_plan_bytes(int64_t batch, int64_t total_q);
size_t mt_topk_bytes(int64_t batch, int64_t total_q, int G);
dsa_status launch_indexer_rows_topk(const uint8_t* q8, const float* wq, uint32_t* hist, const uint8_t* cache,
                                    const dsa_batch* b, int32_t* topk, float* topk_scores, void* plan_ws, int G,
                                    int32_t* st, cudaStream_t s);
dsa_status launch_indexer_rows(const uint8_t* q8, const float* wq, const uint8_t* cache, const dsa_batch* b,
                               float* scores, int64_t ld, bool skip_short, bool full_rows, void* plan_ws, int G,
                               int32_t* st, cudaStream_t s);

}  // namespace dsa
