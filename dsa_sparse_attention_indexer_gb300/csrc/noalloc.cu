// Indexer + top-2048 for decode batches without a caller workspace: the
// quantised queries, row histograms and streaming plan live in a fixed-size
// device array of this library, so no call allocates device memory.  The
// kernels and their order are those of dsa_indexer_topk's decode path.
#include <mutex>

#include "dsa_internal.cuh"
#include "indexer_common.cuh"
#include "indexer_tc.cuh"

namespace dsa {

constexpr size_t kNoAllocScratchBytes = DSA_NOALLOC_SCRATCH_BYTES;

// The scratch.  Nothing in it needs to start at zero: the quantisation kernel
// clears the histogram bins and the plan kernel clears the plan entries that
// the later kernels read.
static __device__ __align__(256) uint8_t g_noalloc_scratch[kNoAllocScratchBytes];

namespace {

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mu;
void* g_scratch_ptr[kMaxDevices];

// Device address of the scratch on the current device, looked up on the first
// call per device.
dsa_status noalloc_scratch(void** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return DSA_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return DSA_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    if (!g_scratch_ptr[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) return DSA_ERR_CUDA;
        g_scratch_ptr[dev] = p;
    }
    *out = g_scratch_ptr[dev];
    return DSA_OK;
}

}  // namespace
}  // namespace dsa

using namespace dsa;

extern "C" dsa_status dsa_topk_share_publish(dsa_topk_share* s, int32_t layer_id, const int32_t* topk,
                                             int64_t rows);

extern "C" dsa_status dsa_indexer_topk_noalloc(const void* q, const float* w, const uint8_t* idxk_cache,
                                               const dsa_batch* b, int32_t* topk, float* topk_scores,
                                               dsa_topk_share* share, int32_t layer_id, int32_t* dev_status,
                                               void* stream) {
    dsa_status vs = validate_batch(b);
    if (vs != DSA_OK) return vs;
    if (b->total_q == 0) return share ? dsa_topk_share_publish(share, layer_id, topk, 0) : DSA_OK;   // no rows
    if (!q || !w || !idxk_cache || !topk) return DSA_ERR_INVALID_ARGUMENT;
    if (!aligned16(q) || !aligned16(idxk_cache) || !aligned16(topk)) return DSA_ERR_ALIGNMENT;
    if (b->total_q > 0) {
        if (b->max_q_len != 1 || b->total_q != b->batch) return DSA_ERR_UNSUPPORTED;   // decode batches only
        if (b->num_pages * 66 > 0x7fffffffLL) return DSA_ERR_UNSUPPORTED;
        const int G = device_sm_count();
        const size_t qbytes = (q8_workspace_bytes(b->total_q) + 255) / 256 * 256;
        const size_t need = qbytes + (size_t)b->total_q * 4096 * 4 + tc_plan_bytes(b->batch, G);
        if (need > kNoAllocScratchBytes) return DSA_ERR_SCRATCH_LIMIT;
        void* base = nullptr;
        dsa_status ss = noalloc_scratch(&base);
        if (ss != DSA_OK) return ss;
        cudaStream_t s = as_stream(stream);
        uint8_t* q8 = static_cast<uint8_t*>(base);
        float* wq = reinterpret_cast<float*>(q8 + (size_t)b->total_q * 4096);
        uint32_t* hist = reinterpret_cast<uint32_t*>(q8 + qbytes);
        void* plan = reinterpret_cast<uint8_t*>(hist) + (size_t)b->total_q * 4096 * 4;
        dsa_status rs = launch_indexer_tc(q, w, q8, wq, hist, idxk_cache, b, topk, topk_scores, plan, G, dev_status, s);
        if (rs != DSA_OK) return rs;
    }
    if (share) return dsa_topk_share_publish(share, layer_id, topk, b->total_q);
    return DSA_OK;
}
