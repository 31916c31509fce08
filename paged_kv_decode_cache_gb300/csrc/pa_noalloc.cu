// pa_decode_splitkv_noalloc: split-KV decode attention whose scratch lives in
// a fixed device array compiled into the library, so the caller never has to
// provide (and therefore never has to allocate) a workspace.
//
// Who needs it: code that cannot call cudaMalloc or an allocator at the point
// where it runs decode -- for example a host runtime whose device memory is
// planned once up front by another component, a plugin that is only handed
// input and output buffers by its host framework, or a caller that must not
// enter an allocator between steps.  Such a caller still passes its own
// inputs and outputs; only the partial results of the split live here.
//
// The array below is a host-side stand-in in host code, not a device address:
// the device address is fetched with cudaGetSymbolAddress once per device
// (with that device current) and cached.
#include <atomic>
#include <mutex>

#include "pa_internal.h"

namespace {

constexpr size_t kScratchBytes = PA_NOALLOC_SCRATCH_BYTES;

// Partial outputs, LSEs and merge counters of the split (the same layout
// pa_decode_splitkv uses in its caller-provided workspace).  Each call clears
// the counters before its kernels run; the partials are written before read.
__device__ __align__(256) unsigned char g_splitkv_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mutex;
void *g_scratch_addr[kMaxDevices] = {};

// Device address of g_splitkv_scratch on the current device (cached).
int scratch_address(void **out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return PA_ECUDA;
    if (dev < 0 || dev >= kMaxDevices) return PA_EUNSUPPORTED;
    std::lock_guard<std::mutex> lock(g_scratch_mutex);
    if (!g_scratch_addr[dev]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_splitkv_scratch) != cudaSuccess || !p) return PA_ECUDA;
        g_scratch_addr[dev] = p;
    }
    *out = g_scratch_addr[dev];
    return PA_OK;
}

}  // namespace

extern "C" {

int pa_decode_splitkv_noalloc(void *out, float *lse, const void *q, const void *k_cache,
                              const void *v_cache, pa_cache_desc cache,
                              const int32_t *block_tables, int32_t max_blocks_per_seq,
                              const int32_t *seq_lens, int32_t B, int32_t Hq, float scale,
                              int32_t num_splits, int32_t *status, pa_stream_t stream) {
    if (num_splits < 0 || B < 0) return PA_EINVAL;
    if (B == 0) return PA_OK;
    if (cache.num_kv_heads <= 0 || cache.block_size <= 0 || max_blocks_per_seq <= 0 || Hq <= 0)
        return PA_EINVAL;
    int P = num_splits;
    if (P == 0) {
        P = pa_auto_num_splits(B, Hq, cache.num_kv_heads, cache.head_dim, max_blocks_per_seq,
                               cache.block_size);
        if (P < 0) return P;
    }
    // The split's partials must fit the built-in array.
    if (P > 1 && pa_splitkv_workspace_bytes(B, Hq, cache.head_dim, P) > kScratchBytes)
        return PA_EWORKSPACE;
    void *scratch = nullptr;
    if (P > 1) {
        int rc = scratch_address(&scratch);
        if (rc) return rc;
    }
    if (P > 1) {
        // The split's merge counters (after the partials) must start at zero; a
        // completed call leaves them at zero, this also covers one that did not.
        const int64_t rows = static_cast<int64_t>(B) * Hq * P;
        const size_t off = static_cast<size_t>(((rows * cache.head_dim * 4 + 255) / 256) * 256 +
                                               ((rows * 4 + 255) / 256) * 256);
        if (cudaMemsetAsync(static_cast<uint8_t *>(scratch) + off, 0,
                            static_cast<size_t>(B) * Hq * 8, stream) != cudaSuccess)
            return PA_ECUDA;
    }
    return pa_decode_splitkv(out, lse, q, k_cache, v_cache, cache, block_tables,
                             max_blocks_per_seq, seq_lens, B, Hq, scale, P, scratch,
                             P > 1 ? kScratchBytes : 0, status, stream);
}

}  // extern "C"
