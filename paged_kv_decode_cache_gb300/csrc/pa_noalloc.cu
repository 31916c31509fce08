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
// the device address is fetched with cudaGetSymbolAddress (with the device
// current) the first time a device is used, and again whenever the current
// context of that device has changed since (after cudaDeviceReset the module is
// loaded anew and the array may sit elsewhere).
#include <cudaTypedefs.h>

#include <mutex>

#include "pa_internal.h"

namespace {

constexpr size_t kScratchBytes = PA_NOALLOC_SCRATCH_BYTES;

// Partial outputs, LSEs and merge counters of the split (the same layout
// pa_decode_splitkv uses in its caller-provided workspace).  Each call clears
// the counters it uses before its kernel runs; the partials are written before
// they are read.
__device__ __align__(256) unsigned char g_splitkv_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;

struct ScratchSlot {
    CUcontext ctx = nullptr;  // the context the address was looked up in
    void *addr = nullptr;
};

std::mutex g_scratch_mutex;
ScratchSlot g_scratch[kMaxDevices];

PFN_cuCtxGetCurrent_v4000 ctx_get_current() {
    static PFN_cuCtxGetCurrent_v4000 fn = [] {
        void *f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 12000, cudaEnableDefault,
                                             &q) != cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            f = nullptr;
        return reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(f);
    }();
    return fn;
}

}  // namespace

namespace pa {

int noalloc_scratch(void **addr, size_t *bytes) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return PA_ECUDA;
    if (dev < 0 || dev >= kMaxDevices) return PA_EUNSUPPORTED;
    auto get_ctx = ctx_get_current();
    CUcontext ctx = nullptr;
    if (!get_ctx || get_ctx(&ctx) != CUDA_SUCCESS) return PA_ECUDA;
    std::lock_guard<std::mutex> lock(g_scratch_mutex);
    ScratchSlot &slot = g_scratch[dev];
    if (!ctx || !slot.addr || slot.ctx != ctx) {
        // (with no context current yet, this lookup makes the device's primary
        // context current; the context then keys the cached address)
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_splitkv_scratch) != cudaSuccess || !p) return PA_ECUDA;
        if (!ctx && (get_ctx(&ctx) != CUDA_SUCCESS || !ctx)) return PA_ECUDA;
        slot.addr = p;
        slot.ctx = ctx;
    }
    *addr = slot.addr;
    *bytes = kScratchBytes;
    return PA_OK;
}

}  // namespace pa

extern "C" {

int pa_decode_splitkv_noalloc(void *out, float *lse, const void *q, const void *k_cache,
                              const void *v_cache, pa_cache_desc cache,
                              const int32_t *block_tables, int32_t max_blocks_per_seq,
                              const int32_t *seq_lens, int32_t B, int32_t Hq, float scale,
                              int32_t num_splits, int32_t *status, pa_stream_t stream) {
    return pa::decode_splitkv_library_scratch(out, lse, q, k_cache, v_cache, cache, block_tables,
                                              max_blocks_per_seq, seq_lens, B, Hq, scale,
                                              num_splits, status, stream);
}

}  // extern "C"
