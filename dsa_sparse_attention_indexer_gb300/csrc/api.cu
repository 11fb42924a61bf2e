// Host-only parts of the C ABI: status strings, the device status block, the
// full/shared layer schedule ("GLM-5.3 推理全链路(十一)", 配置里的 78 个字符)
// and the share handle that carries a full layer's indices to the shared
// layers after it ("GLM-5.3 推理全链路(十一)", 一次前向里 topk 只算一遍).
#include <atomic>
#include <cstring>
#include <mutex>
#include <new>
#include <vector>

#include "dsa_internal.cuh"

namespace dsa {

dsa_status ensure_smem_limit(const void* func, int bytes) {
    struct Applied {
        const void* func;
        int device;
        int bytes;
    };
    static std::mutex mu;
    static std::vector<Applied> applied;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return DSA_ERR_CUDA;
    std::lock_guard<std::mutex> lock(mu);
    for (const Applied& a : applied)
        if (a.func == func && a.device == dev && a.bytes >= bytes) return DSA_OK;
    if (cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes) != cudaSuccess)
        return DSA_ERR_CUDA;
    applied.push_back(Applied{func, dev, bytes});
    return DSA_OK;
}

void* tensor_map_encode_fn() {
    static void* const fn = [] {
        cudaDriverEntryPointQueryResult q;
        void* f = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) !=
                cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            return static_cast<void*>(nullptr);
        return f;
    }();
    return fn;
}

static std::atomic<uint64_t> g_wait_ns{2000000000ull};
uint64_t wait_limit_ns() { return g_wait_ns.load(std::memory_order_relaxed); }

}  // namespace dsa

extern "C" dsa_status dsa_debug_set_wait_limit_ns(uint64_t ns) {
    dsa::g_wait_ns.store(ns, std::memory_order_relaxed);
    return DSA_OK;
}

struct dsa_topk_share {
    const int32_t* topk;
    int64_t rows;
    int32_t layer_id;
    bool valid;
    bool mtp_reuse;      // inside an MTP iteration whose draft steps reuse the published indices
};

// layer id recorded for a seed carried into an MTP iteration (no layer made it)
constexpr int32_t kCarriedSeedLayer = -2;

extern "C" int32_t dsa_abi_version(void) { return 1; }

extern "C" const char* dsa_status_string(dsa_status s) {
    switch (s) {
        case DSA_OK: return "ok";
        case DSA_ERR_INVALID_ARGUMENT: return "invalid argument";
        case DSA_ERR_ALIGNMENT: return "buffer not 16-byte aligned";
        case DSA_ERR_UNSUPPORTED: return "unsupported shape";
        case DSA_ERR_WORKSPACE_TOO_SMALL: return "workspace too small";
        case DSA_ERR_NO_TOPK_SOURCE: return "shared layer without a published full-layer top-k";
        case DSA_ERR_CUDA: return "CUDA runtime error";
        case DSA_ERR_DEVICE: return "device-side errors recorded in the status block";
        case DSA_ERR_SCRATCH_LIMIT: return "batch too large for the fixed no-alloc scratch";
        default: return "unknown status";
    }
}

extern "C" dsa_status dsa_device_status_reset(int32_t* dev_status, void* stream) {
    if (!dev_status) return DSA_ERR_INVALID_ARGUMENT;
    if (cudaMemsetAsync(dev_status, 0, DSA_DEVICE_STATUS_WORDS * sizeof(int32_t),
                        dsa::as_stream(stream)) != cudaSuccess)
        return DSA_ERR_CUDA;
    return DSA_OK;
}

extern "C" dsa_status dsa_device_status_read(const int32_t* dev_status, void* stream, int32_t* host_out) {
    if (!dev_status || !host_out) return DSA_ERR_INVALID_ARGUMENT;
    cudaStream_t s = dsa::as_stream(stream);
    if (cudaMemcpyAsync(host_out, dev_status, DSA_DEVICE_STATUS_WORDS * sizeof(int32_t),
                        cudaMemcpyDeviceToHost, s) != cudaSuccess)
        return DSA_ERR_CUDA;
    if (cudaStreamSynchronize(s) != cudaSuccess) return DSA_ERR_CUDA;
    return host_out[0] != 0 ? DSA_ERR_DEVICE : DSA_OK;
}

extern "C" dsa_status dsa_parse_indexer_types(const char* const* types, int32_t n_layers, uint8_t* is_full) {
    if (!types || !is_full || n_layers < 0) return DSA_ERR_INVALID_ARGUMENT;
    for (int32_t l = 0; l < n_layers; ++l) {
        if (!types[l]) return DSA_ERR_INVALID_ARGUMENT;
        if (std::strcmp(types[l], "full") == 0) is_full[l] = 1;
        else if (std::strcmp(types[l], "shared") == 0) is_full[l] = 0;
        else return DSA_ERR_INVALID_ARGUMENT;
    }
    return DSA_OK;
}

extern "C" dsa_status dsa_schedule_from_freq(int32_t n_layers, int32_t freq, int32_t offset, uint8_t* is_full) {
    if (!is_full || n_layers < 0 || freq < 1) return DSA_ERR_INVALID_ARGUMENT;
    for (int32_t l = 0; l < n_layers; ++l) {
        int32_t v = l - offset + 1;
        if (v < 0) v = 0;
        is_full[l] = (v % freq != 0) ? 0 : 1;
    }
    return DSA_OK;
}

extern "C" dsa_status dsa_schedule_resolve(const dsa_schedule_config* cfg, int32_t n_layers, uint8_t* is_full) {
    if (!cfg || !is_full || n_layers < 0) return DSA_ERR_INVALID_ARGUMENT;
    if (cfg->indexer_types) {
        if (cfg->n_types < 0) return DSA_ERR_INVALID_ARGUMENT;
        for (int32_t l = 0; l < cfg->n_types; ++l) {
            const char* t = cfg->indexer_types[l];
            if (!t || (std::strcmp(t, "full") != 0 && std::strcmp(t, "shared") != 0)) return DSA_ERR_INVALID_ARGUMENT;
        }
        for (int32_t l = 0; l < n_layers; ++l)
            is_full[l] = (l < cfg->n_types && std::strcmp(cfg->indexer_types[l], "shared") == 0) ? 0 : 1;
        return DSA_OK;
    }
    if (cfg->cli_factor > 1) {
        for (int32_t l = 0; l < n_layers; ++l) is_full[l] = (l % cfg->cli_factor != 0) ? 0 : 1;
        return DSA_OK;
    }
    if (cfg->index_topk_pattern) {
        const size_t len = std::strlen(cfg->index_topk_pattern);
        for (int32_t l = 0; l < n_layers; ++l)
            is_full[l] = ((size_t)l < len && cfg->index_topk_pattern[l] == 'S') ? 0 : 1;
        return DSA_OK;
    }
    if (cfg->index_topk_freq < 1) return DSA_ERR_INVALID_ARGUMENT;
    const int32_t off = cfg->index_skip_topk_offset < 0 ? 2 : cfg->index_skip_topk_offset;
    return dsa_schedule_from_freq(n_layers, cfg->index_topk_freq, off, is_full);
}

extern "C" dsa_status dsa_topk_share_create(dsa_topk_share** out) {
    if (!out) return DSA_ERR_INVALID_ARGUMENT;
    dsa_topk_share* s = new (std::nothrow) dsa_topk_share{nullptr, 0, -1, false, false};
    if (!s) return DSA_ERR_INVALID_ARGUMENT;
    *out = s;
    return DSA_OK;
}

extern "C" dsa_status dsa_topk_share_destroy(dsa_topk_share* s) {
    delete s;
    return DSA_OK;
}

extern "C" dsa_status dsa_topk_share_reset(dsa_topk_share* s) {
    if (!s) return DSA_ERR_INVALID_ARGUMENT;
    s->topk = nullptr;
    s->rows = 0;
    s->layer_id = -1;
    s->valid = false;
    return DSA_OK;
}

extern "C" dsa_status dsa_topk_share_publish(dsa_topk_share* s, int32_t layer_id, const int32_t* topk,
                                             int64_t rows) {
    if (!s || rows < 0 || (!topk && rows > 0)) return DSA_ERR_INVALID_ARGUMENT;
    s->topk = topk;
    s->rows = rows;
    s->layer_id = layer_id;
    s->valid = true;
    return DSA_OK;
}

extern "C" dsa_status dsa_topk_share_get(const dsa_topk_share* s, const int32_t** topk, int64_t* rows,
                                         int32_t* layer_id) {
    if (!s || !topk) return DSA_ERR_INVALID_ARGUMENT;
    if (!s->valid) return DSA_ERR_NO_TOPK_SOURCE;
    *topk = s->topk;
    if (rows) *rows = s->rows;
    if (layer_id) *layer_id = s->layer_id;
    return DSA_OK;
}

// Top-k reuse across the draft steps of one MTP iteration ("GLM-5.3 推理全链路
// (十一)", 优化三: the iteration's context manager turns reuse on only for one
// draft candidate per step, keeps a carried seed on request, and clears the
// carried indices when the iteration ends).
extern "C" dsa_status dsa_topk_share_mtp_begin(dsa_topk_share* s, int32_t enabled, int32_t eagle_topk,
                                               int32_t keep_carry_seed, const int32_t* seed, int64_t rows,
                                               int32_t seed_width, int32_t* reuse_on) {
    if (!s || eagle_topk < 1 || rows < 0) return DSA_ERR_INVALID_ARGUMENT;
    const bool reuse = enabled != 0 && eagle_topk == 1;
    const bool carry = reuse && keep_carry_seed != 0 && seed != nullptr;
    if (carry && seed_width != DSA_TOPK) return DSA_ERR_UNSUPPORTED;
    if (reuse_on) *reuse_on = reuse ? 1 : 0;
    if (!reuse) return DSA_OK;
    s->mtp_reuse = true;
    if (carry) {
        s->topk = seed;
        s->rows = rows;
        s->layer_id = kCarriedSeedLayer;
        s->valid = true;
    } else {
        s->topk = nullptr;
        s->rows = 0;
        s->layer_id = -1;
        s->valid = false;
    }
    return DSA_OK;
}

extern "C" dsa_status dsa_topk_share_needs_scoring(const dsa_topk_share* s, int32_t* needs) {
    if (!s || !needs) return DSA_ERR_INVALID_ARGUMENT;
    *needs = (s->mtp_reuse && s->valid) ? 0 : 1;
    return DSA_OK;
}

extern "C" dsa_status dsa_topk_share_mtp_end(dsa_topk_share* s) {
    if (!s) return DSA_ERR_INVALID_ARGUMENT;
    s->mtp_reuse = false;
    s->topk = nullptr;
    s->rows = 0;
    s->layer_id = -1;
    s->valid = false;
    return DSA_OK;
}

extern "C" dsa_status dsa_mtp_topk_width(int32_t index_topk, int32_t index_kpool, int32_t* width) {
    if (!width || index_topk < 1 || index_kpool < 1) return DSA_ERR_INVALID_ARGUMENT;
    const int64_t w = (int64_t)index_topk + index_kpool - 1;
    if (w > INT32_MAX) return DSA_ERR_INVALID_ARGUMENT;
    *width = (int32_t)w;
    return DSA_OK;
}
