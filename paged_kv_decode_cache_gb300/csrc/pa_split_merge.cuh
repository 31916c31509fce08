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

// One merge task: output row `row`, dims [32 * slice, 32 * slice + 32), by one
// warp.  Lane i holds the LSEs of partitions i, i + 32, ... (read once); the
// row's log-sum-exp comes from two warp reductions, each lane turns its LSEs
// into weights, and the partial outputs are streamed with eight loads in
// flight per lane, each weight passed along by shuffle.
template <int D>
__device__ __forceinline__ void merge_slice(const DecodeParams &p, int64_t row, int slice, int lane) {
    constexpr int kMaxHeld = 8;  // LSEs per lane held in registers: P <= 256
    const int P = p.num_splits;
    const float *pl = p.part_lse + row * P;
    float lv[kMaxHeld];
    float M = -INFINITY;
#pragma unroll
    for (int k = 0; k < kMaxHeld; ++k) {
        const int i = lane + 32 * k;
        lv[k] = i < P ? __ldcg(pl + i) : -INFINITY;
        M = fmaxf(M, lv[k]);
    }
#pragma unroll
    for (int off = 16; off; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
    float total = -INFINITY, acc = 0.f;
    if (M != -INFINITY) {
        float z = 0.f;
#pragma unroll
        for (int k = 0; k < kMaxHeld; ++k) z += (lv[k] == -INFINITY) ? 0.f : expf(lv[k] - M);
#pragma unroll
        for (int off = 16; off; off >>= 1) z += __shfl_xor_sync(0xffffffffu, z, off);
        total = M + logf(z);
        const float *po = p.part_o + row * P * D + slice * 32 + lane;
#pragma unroll 1
        for (int k = 0; k < kMaxHeld && 32 * k < P; ++k) {
            const float wl = (lv[k] == -INFINITY) ? 0.f : expf(lv[k] - total);
            const int n = min(32, P - 32 * k);
            float part[8];
            for (int j0 = 0; j0 < n; j0 += 8) {
#pragma unroll
                for (int j = 0; j < 8; ++j)
                    part[j] = (j0 + j < n) ? __ldcg(po + static_cast<int64_t>(32 * k + j0 + j) * D) : 0.f;
#pragma unroll
                for (int j = 0; j < 8; ++j)
                    acc = fmaf(__shfl_sync(0xffffffffu, wl, (j0 + j) & 31), part[j], acc);
            }
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
