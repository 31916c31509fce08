// End of a split-KV decode CTA: optionally merge the partial results of its
// (sequence, head group) inside the same launch.
//
// The split kernel is then launched cooperatively, so every CTA of the grid
// is resident at once and CTAs may wait for each other.  Protocol, per group
// of P CTAs (the P partitions of one sequence and head group):
//   1. each CTA writes its partials, fences them to device scope and
//      increments the group's arrival counter;
//   2. it waits (bounded) until the counter reads P: every partial exists;
//   3. the group's CTAs split the merge between them: merge task k = (output
//      row, 32-dim slice) goes to warp k of the group's P x nwarps warps; a
//      task computes the row's log-sum-exp over the P partial LSEs and sums
//      the weighted partial outputs of its slice (partials are read with
//      L1-bypassing loads);
//   4. each CTA increments the group's departure counter; the last one puts
//      both counters back to zero for the next call.
// A wait that runs out sets PA_STATUS_TIMEOUT and the CTA skips the merge.
#pragma once

#include <cuda_bf16.h>

#include "pa_device.cuh"
#include "pa_internal.h"

namespace pa {

__device__ __forceinline__ int ld_acquire_gpu(const int *p) {
    int v;
    asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

// One merge task: output row `row`, dims [32 * slice, 32 * slice + 32), by one warp.
template <int D>
__device__ __forceinline__ void merge_slice(const DecodeParams &p, int64_t row, int slice, int lane) {
    const int P = p.num_splits;
    const float *pl = p.part_lse + row * P;
    float M = -INFINITY;
    for (int i = lane; i < P; i += 32) M = fmaxf(M, __ldcg(pl + i));
#pragma unroll
    for (int off = 16; off; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
    float total = -INFINITY, acc = 0.f;
    if (M != -INFINITY) {
        float z = 0.f;
        for (int i = lane; i < P; i += 32) z += expf(__ldcg(pl + i) - M);
#pragma unroll
        for (int off = 16; off; off >>= 1) z += __shfl_xor_sync(0xffffffffu, z, off);
        total = M + logf(z);
        const float *po = p.part_o + row * P * D + slice * 32 + lane;
        for (int base = 0; base < P; base += 32) {
            const int i = base + lane;
            const float wl = i < P ? expf(__ldcg(pl + i) - total) : 0.f;
            const int n = min(32, P - base);
#pragma unroll 8
            for (int j = 0; j < n; ++j)
                acc = fmaf(__shfl_sync(0xffffffffu, wl, j),
                           __ldcg(po + static_cast<int64_t>(base + j) * D), acc);
        }
    }
    static_cast<__nv_bfloat16 *>(p.out)[row * D + slice * 32 + lane] = __float2bfloat16_rn(acc);
    if (slice == 0 && lane == 0 && p.lse) p.lse[row] = total;
}

// Merge tasks are spread over kMergeWarps warps per CTA, whatever the caller's
// thread count, so every CTA of a group agrees on who does which task.
constexpr int kMergeWarps = 4;

// Called by all `nt` threads (whole warps, index t, nt >= 32 * kMergeWarps)
// of a CTA after its partials for rows [row_first, row_first + nrows) are
// written; `sync` synchronises those threads; `flag` is a shared int.
template <int D, typename Sync>
__device__ void merge_split_group(const DecodeParams &p, int group, int part, int64_t row_first,
                                  int nrows, int *flag, int t, int nt, Sync sync) {
    if (!p.counters) return;
    int *arrive = p.counters + 2 * group, *depart = arrive + 1;
    const int P = p.num_splits;
    __threadfence();
    sync();
    if (t == 0) {
        atomicAdd(arrive, 1);
        bool ok = false;
        for (uint32_t i = 0; i < kWaitLimit; ++i) {
            if (ld_acquire_gpu(arrive) >= P) {
                ok = true;
                break;
            }
            __nanosleep(64);
        }
        if (!ok) set_status(p.status, PA_STATUS_TIMEOUT);
        *flag = ok;
    }
    sync();
    if (*flag) {
        __threadfence();
        const int warp = t >> 5, lane = t & 31;
        const int tasks = nrows * (D / 32);
        if (warp < kMergeWarps)
            for (int k = part * kMergeWarps + warp; k < tasks; k += P * kMergeWarps)
                merge_slice<D>(p, row_first + k / (D / 32), k % (D / 32), lane);
    }
    sync();
    if (t == 0 && atomicAdd(depart, 1) == P - 1) {
        *arrive = 0;
        *depart = 0;
    }
}

}  // namespace pa
