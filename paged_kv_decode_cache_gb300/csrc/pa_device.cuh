// Device-side building blocks shared by the decode kernels: mbarrier and
// TMA (cp.async.bulk.tensor) wrappers, bf16 unpacking, fast exp2, and the
// shared-memory addressing of the 128-byte-swizzled K/V tiles.
#pragma once

#include <atomic>

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/pa.h"

namespace pa {

// Tokens per TMA tile: 16 rows of one (block, KV head).  Every block size
// the library accepts is a multiple of this, so a tile never straddles two
// physical blocks.
constexpr int kTile = 16;
// A tile row is split into 64-element (128-byte) sub-rows so that each TMA
// box can use the 128-byte swizzle.
constexpr int kSubElems = 64;
constexpr int kSubBytes = 128;

// Bounded waits: a warp polls for at most about a second (the GPU's global
// nanosecond timer, read every 256 polls) and at most kWaitLimit polls, then
// gives up, flags PA_STATUS_TIMEOUT and stops consuming.  A healthy copy or
// merge completes in microseconds.
constexpr uint32_t kWaitLimit = 1u << 24;
constexpr uint64_t kWaitNs = 1000000000ull;

__device__ __forceinline__ uint64_t globaltimer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// True once poll i of a wait that started at t0 is past the time limit.
__device__ __forceinline__ bool wait_expired(uint32_t i, uint64_t t0) {
    return (i & 255u) == 255u && globaltimer_ns() - t0 > kWaitNs;
}

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
                 : "memory");
}

// Make mbarrier initialisation visible to the async (TMA) proxy.
__device__ __forceinline__ void fence_barrier_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Bulk copy (async proxy) of `bytes` from shared to global memory, tracked by
// this thread's bulk async-groups; both addresses 16-byte aligned, bytes a
// multiple of 16.
__device__ __forceinline__ void bulk_store_s2g(void *gdst, const void *ssrc, uint32_t bytes) {
    asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(gdst),
                 "r"(smem_u32(ssrc)), "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// Wait until all of this thread's bulk copies have completed (writes performed).
__device__ __forceinline__ void bulk_wait_all() {
    asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}
// Wait until all of this thread's bulk copies have read their sources (the
// writes may still be in flight; they complete before the kernel does).
__device__ __forceinline__ void bulk_wait_all_read() {
    asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
    asm volatile(
        "{\n\t.reg .b64 st;\n\t"
        "mbarrier.arrive.expect_tx.shared::cta.b64 st, [%0], %1;\n\t}" ::"r"(smem_u32(bar)),
        "r"(bytes)
        : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// Wait for phase `parity` of `bar` to complete; false after kWaitLimit tries.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t *bar, uint32_t parity) {
    const uint64_t t0 = globaltimer_ns();
    for (uint32_t i = 0; i < kWaitLimit; ++i) {
        if (mbar_try_wait(bar, parity)) return true;
        if (wait_expired(i, t0)) break;
    }
    return false;
}

// The polling part of a bounded wait that honours a CTA-wide abort flag:
// false once the flag is set (by another warp) or the wait has run out, in
// which case it sets the flag and PA_STATUS_TIMEOUT.  Kept out of line, so
// that the many wait sites of a warp-specialised kernel share one copy of
// the loop (callers try the barrier once inline first).
static __device__ __noinline__ bool mbar_wait_or_abort_slow(uint64_t *bar, uint32_t parity,
                                                           volatile int *abort_flag, int32_t *status);

// L2 policy for data read exactly once (the KV stream).
__device__ __forceinline__ uint64_t l2_evict_first_policy() {
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}

// L2 policy for data that other CTAs read again soon (no eviction preference).
__device__ __forceinline__ uint64_t l2_evict_normal_policy() {
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_normal.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}

// 4-D tiled TMA load of one box into shared memory, completing on `bar`.
__device__ __forceinline__ void tma_load_4d(void *dst, const CUtensorMap *map, int c0, int c1,
                                            int c2, int c3, uint64_t *bar, uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        ".L2::cache_hint [%0], [%1, {%2, %3, %4, %5}], [%6], %7;" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(c3),
        "r"(smem_u32(bar)), "l"(policy)
        : "memory");
}

// L2 prefetch of the box a tma_load_4d / tma_load_3d at these coordinates would
// copy (boxes past the tensor's bounds fetch nothing).
__device__ __forceinline__ void tma_prefetch_4d(const CUtensorMap *map, int c0, int c1, int c2, int c3) {
    asm volatile("cp.async.bulk.prefetch.tensor.4d.L2.global.tile [%0, {%1, %2, %3, %4}];" ::"l"(
                     reinterpret_cast<uint64_t>(map)),
                 "r"(c0), "r"(c1), "r"(c2), "r"(c3)
                 : "memory");
}
__device__ __forceinline__ void tma_prefetch_3d(const CUtensorMap *map, int c0, int c1, int c2) {
    asm volatile("cp.async.bulk.prefetch.tensor.3d.L2.global.tile [%0, {%1, %2, %3}];" ::"l"(
                     reinterpret_cast<uint64_t>(map)),
                 "r"(c0), "r"(c1), "r"(c2)
                 : "memory");
}
__device__ __forceinline__ void tma_load_3d(void *dst, const CUtensorMap *map, int c0, int c1,
                                            int c2, uint64_t *bar, uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        ".L2::cache_hint [%0], [%1, {%2, %3, %4}], [%5], %6;" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(smem_u32(bar)),
        "l"(policy)
        : "memory");
}

// 4-byte asynchronous global -> shared copy (cp.async), tracked per thread in
// commit groups: wait<N> returns once at most the N newest groups are pending.
__device__ __forceinline__ void cp_async_4(void *smem_dst, const void *gmem_src) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(smem_u32(smem_dst)), "l"(gmem_src)
                 : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// Hint: bring the line holding `p` into L2 (and its address translation into
// the TLBs) ahead of use.
__device__ __forceinline__ void prefetch_l2(const void *p) {
    asm volatile("prefetch.global.L2 [%0];" ::"l"(p));
}

__device__ __forceinline__ void prefetch_tensormap(const CUtensorMap *map) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// 2^x with the hardware approximation (ex2.approx, flush-to-zero).
__device__ __forceinline__ float fast_exp2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// Two bf16 packed in a 32-bit word -> two floats (exact: bf16 is the top half of fp32).
__device__ __forceinline__ float bf16lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

// FP8 pools: 8 bf16 values (one 16-byte chunk of a K or V row) to their e4m3
// codes (8 bytes, the same order): fp32(x) / scale, rounded to nearest even,
// saturating at the largest finite code (+-448), NaN kept.  The one
// definition of a stored code, for the cache write and the decode step's
// fused write alike.
__device__ __forceinline__ uint2 e4m3x8_from_bf16(const uint4 &in, float scale) {
    const uint32_t w[4] = {in.x, in.y, in.z, in.w};
    uint32_t out[2] = {0u, 0u};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const __nv_fp8_storage_t lo = __nv_cvt_float_to_fp8(bf16lo(w[k]) / scale, __NV_SATFINITE, __NV_E4M3);
        const __nv_fp8_storage_t hi = __nv_cvt_float_to_fp8(bf16hi(w[k]) / scale, __NV_SATFINITE, __NV_E4M3);
        out[k >> 1] |= (static_cast<uint32_t>(lo) | (static_cast<uint32_t>(hi) << 8)) << (16 * (k & 1));
    }
    return make_uint2(out[0], out[1]);
}

// Byte offset of 16-byte chunk `chunk` (0..7) of row `row` inside a tile of
// 128-byte rows written by TMA with CU_TENSOR_MAP_SWIZZLE_128B (the chunk
// index is XOR-ed with the row index modulo 8; tiles are 1024-byte aligned).
__device__ __forceinline__ uint32_t swz128(int row, int chunk) {
    return static_cast<uint32_t>(row * kSubBytes + ((chunk ^ (row & 7)) << 4));
}

// Four 8 x 8 matrices of 16-bit elements, transposed: lanes 8i .. 8i + 7 give
// the shared-memory addresses of rows 0..7 of matrix i (16 bytes each), and
// lane t receives in r[i] the elements (row 2 (t % 4), column t / 4) (low
// half) and (row 2 (t % 4) + 1, column t / 4) (high half) of matrix i.
__device__ __forceinline__ void ldsm_x4_trans(uint32_t saddr, uint32_t (&r)[4]) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(saddr)
                 : "memory");
}

// Plain arrive (count 1) on an mbarrier.
__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
    asm volatile("{\n\t.reg .b64 st;\n\tmbarrier.arrive.shared::cta.b64 st, [%0];\n\t}" ::"r"(
                     smem_u32(bar))
                 : "memory");
}

// Named barrier `id` over `nthreads` threads (a multiple of 32).
__device__ __forceinline__ void named_sync(int id, int nthreads) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// Named barrier that also returns whether any participating thread passed true.
__device__ __forceinline__ bool named_sync_or(int id, int nthreads, bool v) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred q, p;\n\t"
        "setp.ne.u32 q, %1, 0;\n\t"
        "bar.red.or.pred p, %2, %3, q;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(r)
        : "r"(static_cast<uint32_t>(v)), "r"(id), "r"(nthreads)
        : "memory");
    return r != 0;
}

__device__ __forceinline__ float ldcg(const float *p) { return __ldcg(p); }

// Thread-block clusters.  cluster_sync(): every thread of every CTA of the
// cluster arrives (release: its shared-memory writes become visible to the
// cluster) and waits for all the others (acquire).  Not the .aligned form, so
// the threads of a warp need not be converged.
__device__ __forceinline__ void cluster_sync() {
    asm volatile("barrier.cluster.arrive.release;\n\tbarrier.cluster.wait.acquire;" ::: "memory");
}
__device__ __forceinline__ uint32_t cluster_ctarank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
// The shared::cluster address of the same location in CTA `rank`'s shared memory.
__device__ __forceinline__ uint32_t map_shared_rank(uint32_t addr, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
    return r;
}
__device__ __forceinline__ float ld_shared_cluster(uint32_t addr) {
    float v;
    asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(addr) : "memory");
    return v;
}

// Order this thread's generic global writes before later async-proxy (TMA)
// reads of the same memory (by any thread that synchronises with it after).
__device__ __forceinline__ void fence_proxy_async_global() {
    asm volatile("fence.proxy.async.global;" ::: "memory");
}

// Fused cache write: does `slot` hold position L - 1 of the sequence whose
// block at that position is `phys`?  (The fused step only writes a token it
// will read itself.)
__device__ __forceinline__ bool slot_is_position(int64_t slot, int phys, int pos, int bs) {
    return slot >= 0 && phys >= 0 && slot == static_cast<int64_t>(phys) * bs + pos % bs;
}

__device__ __forceinline__ void set_status(int32_t *status, int bits) {
    if (status) atomicOr(status, bits);
}

static __device__ __noinline__ bool mbar_wait_or_abort_slow(uint64_t *bar, uint32_t parity,
                                                           volatile int *abort_flag, int32_t *status) {
    const uint64_t t0 = globaltimer_ns();
    for (uint32_t i = 0; i < kWaitLimit; ++i) {
        if (mbar_try_wait(bar, parity)) return true;
        if (*abort_flag) return false;
        if (wait_expired(i, t0)) break;
    }
    *abort_flag = 1;
    set_status(status, PA_STATUS_TIMEOUT);
    return false;
}

// Programmatic dependent launch.  griddep_wait(): returns once the grids this
// one depends on (the previous kernel in the stream, when this one was
// launched with programmatic stream serialization) have completed and their
// memory is visible; at once otherwise.  griddep_launch_dependents(): the next
// such launch may be scheduled once every CTA of this grid has executed it.
__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void griddep_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Launch `kern` normally, or cooperatively (all CTAs resident at once, as CTAs
// that wait for each other need) when `cooperative`; a cooperative grid larger
// than what fits at once fails with cudaErrorCooperativeLaunchTooLarge.  `pdl`:
// with programmatic stream serialization, for kernels that call griddep_wait()
// before any global memory access.
template <typename Kernel, typename... Args>
inline cudaError_t launch_maybe_cooperative(Kernel kern, dim3 grid, int threads, int smem,
                                            cudaStream_t stream, bool cooperative, bool pdl,
                                            Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = dim3(threads, 1, 1);
    cfg.dynamicSmemBytes = static_cast<size_t>(smem);
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    int na = 0;
    if (cooperative) {
        attr[na].id = cudaLaunchAttributeCooperative;
        attr[na++].val.cooperative = 1;
    }
    if (pdl) {
        attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[na++].val.programmaticStreamSerializationAllowed = 1;
    }
    cfg.attrs = attr;
    cfg.numAttrs = na;
    if (cooperative) {
        int per_sm = 0, dev = 0, sms = 0;
        cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, threads, smem);
        if (e == cudaSuccess) e = cudaGetDevice(&dev);
        if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess) return e;
        if (static_cast<int64_t>(grid.x) * grid.y * grid.z > static_cast<int64_t>(per_sm) * sms)
            return cudaErrorCooperativeLaunchTooLarge;
    }
    cudaError_t e = cudaLaunchKernelEx(&cfg, kern, args...);
    return e == cudaSuccess ? cudaGetLastError() : e;
}

// Launch `kern` with thread-block clusters of `cluster_x` CTAs along x (grid.x
// a multiple of it); `pdl` as for launch_maybe_cooperative.  Sizes above 8
// need the kernel's non-portable-size attribute, which max_active_clusters
// sets; callers ask it first whether (and how many) such clusters fit.
template <typename Kernel, typename... Args>
inline cudaError_t launch_clustered(Kernel kern, dim3 grid, int cluster_x, int threads, int smem,
                                    cudaStream_t stream, bool pdl, Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = dim3(threads, 1, 1);
    cfg.dynamicSmemBytes = static_cast<size_t>(smem);
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = static_cast<unsigned>(cluster_x);
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 2 : 1;
    cudaError_t e = cudaLaunchKernelEx(&cfg, kern, args...);
    return e == cudaSuccess ? cudaGetLastError() : e;
}

// How many clusters of `cluster_x` CTAs of `kern` (threads, smem per CTA) can
// be resident on device `dev` at once (0: none can be scheduled).  Asked once
// per (kernel, device, size) for sizes 1..31 and devices 0..63; the answers
// are kept in `cache` (count + 1 at [dev * 32 + size], 0 = not asked yet),
// which the caller owns (one per kernel).  Sizes above 8 are opted into first.
template <typename Kernel>
inline int max_active_clusters(Kernel kern, int cluster_x, int threads, int smem, int dev,
                               std::atomic<int> *cache) {
    if (cluster_x < 1 || cluster_x > 31 || dev < 0 || dev > 63) return 0;
    std::atomic<int> &slot = cache[dev * 32 + cluster_x];
    const int known = slot.load(std::memory_order_acquire);
    if (known > 0) return known - 1;
    int n = 0;
    bool ok = true;
    if (cluster_x > 8 &&
        cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) != cudaSuccess)
        ok = false;
    if (ok) {
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(static_cast<unsigned>(cluster_x), 1, 1);
        cfg.blockDim = dim3(threads, 1, 1);
        cfg.dynamicSmemBytes = static_cast<size_t>(smem);
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = static_cast<unsigned>(cluster_x);
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess) ok = false;
    }
    if (!ok) {
        cudaGetLastError();  // clear a refusal, so it does not surface later
        n = 0;
    }
    slot.store(n + 1, std::memory_order_release);
    return n;
}

}  // namespace pa
