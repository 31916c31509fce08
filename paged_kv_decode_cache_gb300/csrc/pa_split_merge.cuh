// End of a split-KV decode CTA: optionally merge the partial results of its
// (sequence, head group) inside the same launch.
//
// The split kernel is then launched cooperatively, so every CTA of the grid
// is resident at once and CTAs may wait for each other.  Protocol, per group
// of P CTAs (the P partitions of one sequence and head group):
//   1. each CTA writes its partials; after a CTA barrier one thread
//      increments the group's arrival counter with release semantics;
//   2. the CTA whose arrival makes P resets the counter to zero at once; the
//      others wait (bounded) until it reads P or drops to at most their own
//      arrival value (the reset): every partial exists;
//   3. the group's CTAs split the merge between them: a merge task (output
//      row, dim slice) computes the row's log-sum-exp over the P partial LSEs
//      and sums the weighted partial outputs of its slice (partials are read
//      with L1-bypassing loads).  Up to 32 partitions task k goes to warp k of
//      the group's P x nwarps warps, a lane owning a dim of a 32-dim slice;
//      beyond, a task goes to ceil(P / 32) warps of one CTA, each taking 32
//      partitions with its lanes over a 32-dim slice, and their sums meet in
//      shared memory (the CUDA-core kernel: one warp, a lane owning
//      partitions of an 8-dim slice);
// A wait that runs out sets PA_STATUS_TIMEOUT and the CTA skips the merge.
// A task merges all part_stride partials of its row: part_stride = P for an
// ordinary call; a cascade's suffix pass (P CTAs per group) also merges the
// prefix pass's partials, which the previous launch left in the row's other
// slots.
#pragma once

#include <cuda_bf16.h>

#include "pa_device.cuh"
#include "pa_internal.h"

namespace pa {

// Release pattern: a gpu-scope fence, then a relaxed atomic add (the fence
// also acquires what this thread's earlier atomics read).
__device__ __forceinline__ void red_add_release_gpu(int *p, int v) {
    asm volatile("fence.acq_rel.gpu;\n\tred.relaxed.gpu.global.add.s32 [%0], %1;" ::"l"(p), "r"(v)
                 : "memory");
}
__device__ __forceinline__ int atom_add_release_gpu(int *p, int v) {
    int old;
    asm volatile("fence.acq_rel.gpu;\n\tatom.relaxed.gpu.global.add.s32 %0, [%1], %2;"
                 : "=r"(old)
                 : "l"(p), "r"(v)
                 : "memory");
    return old;
}

__device__ __forceinline__ int ld_acquire_gpu(const int *p) {
    int v;
    asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

// One merge task: output row `row`, dims [32 * slice, 32 * slice + 32), by one
// warp.  Lane i holds the LSEs of partitions i, i + 32, ... ; the LSEs and the
// first 32 partitions' outputs are loaded together (one round trip for
// P <= 32), the row's log-sum-exp comes from two warp reductions, and each
// further block of 32 partitions is loaded while the previous one is summed.
template <int D>
__device__ __forceinline__ void merge_slice(const DecodeParams &p, int64_t row, int slice, int lane) {
    constexpr int kMaxHeld = kMaxGridMerge / 32;  // LSEs per lane held in registers
    const int P = p.part_stride;                  // partials of the row
    const float *pl = p.part_lse + row * P;
    const float *po = p.part_o + row * P * D + slice * 32 + lane;
    float lv[kMaxHeld], cur[32];
#pragma unroll
    for (int k = 0; k < kMaxHeld; ++k) lv[k] = lane + 32 * k < P ? __ldcg(pl + lane + 32 * k) : -INFINITY;
#pragma unroll
    for (int j = 0; j < 32; ++j) cur[j] = j < P ? __ldcg(po + static_cast<int64_t>(j) * D) : 0.f;
    float M = -INFINITY;
#pragma unroll
    for (int k = 0; k < kMaxHeld; ++k) M = fmaxf(M, lv[k]);
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
#pragma unroll 1
        for (int k = 0; k < kMaxHeld && 32 * k < P; ++k) {
            const int next = 32 * (k + 1);
            float nxt[32];
            if (next < P) {
#pragma unroll
                for (int j = 0; j < 32; ++j)
                    nxt[j] = next + j < P ? __ldcg(po + static_cast<int64_t>(next + j) * D) : 0.f;
            }
            float lk = lv[0];
#pragma unroll
            for (int i = 1; i < kMaxHeld; ++i)
                if (i == k) lk = lv[i];
            const float wl = (lk == -INFINITY) ? 0.f : expf(lk - total);
#pragma unroll
            for (int j = 0; j < 32; ++j) acc = fmaf(__shfl_sync(0xffffffffu, wl, j), cur[j], acc);
            if (next < P) {
#pragma unroll
                for (int j = 0; j < 32; ++j) cur[j] = nxt[j];
            }
        }
    }
    static_cast<__nv_bfloat16 *>(p.out)[row * D + slice * 32 + lane] = __float2bfloat16_rn(acc);
    if (slice == 0 && lane == 0 && p.lse) p.lse[row] = total;
}

// Merge task for many partitions (P > 32): output row `row`, dims
// [8 * slice, 8 * slice + 8), by one warp whose lane i takes partitions i,
// i + 32, ... : every LSE and partial output the lane needs is loaded at once
// (one round trip), the lane sums its own weighted partials, and one warp
// reduction per dim adds the lanes' sums.
template <int D>
__device__ __forceinline__ void merge_slice_wide(const DecodeParams &p, int64_t row, int slice, int lane) {
    constexpr int kMaxHeld = kMaxGridMerge / 32;  // partitions per lane
    const int P = p.part_stride;                  // partials of the row
    const float *pl = p.part_lse + row * P;
    const float *po = p.part_o + row * P * D + slice * 8;
    float lv[kMaxHeld];
    float4 lo[kMaxHeld], hi[kMaxHeld];
#pragma unroll
    for (int k = 0; k < kMaxHeld; ++k) {
        const int i = lane + 32 * k;
        lv[k] = -INFINITY;
        lo[k] = hi[k] = make_float4(0.f, 0.f, 0.f, 0.f);
        if (i < P) {
            lv[k] = __ldcg(pl + i);
            lo[k] = __ldcg(reinterpret_cast<const float4 *>(po + static_cast<int64_t>(i) * D));
            hi[k] = __ldcg(reinterpret_cast<const float4 *>(po + static_cast<int64_t>(i) * D + 4));
        }
    }
    float M = -INFINITY;
#pragma unroll
    for (int k = 0; k < kMaxHeld; ++k) M = fmaxf(M, lv[k]);
#pragma unroll
    for (int off = 16; off; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
    float total = -INFINITY, acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    if (M != -INFINITY) {
        float z = 0.f;
#pragma unroll
        for (int k = 0; k < kMaxHeld; ++k) z += (lv[k] == -INFINITY) ? 0.f : expf(lv[k] - M);
#pragma unroll
        for (int off = 16; off; off >>= 1) z += __shfl_xor_sync(0xffffffffu, z, off);
        total = M + logf(z);
#pragma unroll
        for (int k = 0; k < kMaxHeld; ++k) {
            const float w = (lv[k] == -INFINITY) ? 0.f : expf(lv[k] - total);
            acc[0] = fmaf(w, lo[k].x, acc[0]);
            acc[1] = fmaf(w, lo[k].y, acc[1]);
            acc[2] = fmaf(w, lo[k].z, acc[2]);
            acc[3] = fmaf(w, lo[k].w, acc[3]);
            acc[4] = fmaf(w, hi[k].x, acc[4]);
            acc[5] = fmaf(w, hi[k].y, acc[5]);
            acc[6] = fmaf(w, hi[k].z, acc[6]);
            acc[7] = fmaf(w, hi[k].w, acc[7]);
        }
#pragma unroll
        for (int off = 16; off; off >>= 1)
#pragma unroll
            for (int j = 0; j < 8; ++j) acc[j] += __shfl_xor_sync(0xffffffffu, acc[j], off);
    }
    if (lane == 0) {
        __nv_bfloat162 o[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) o[j] = __floats2bfloat162_rn(acc[2 * j], acc[2 * j + 1]);
        *reinterpret_cast<uint4 *>(static_cast<__nv_bfloat16 *>(p.out) + row * D + slice * 8) =
            *reinterpret_cast<const uint4 *>(o);
        if (slice == 0 && p.lse) p.lse[row] = total;
    }
}

// Merge for many partitions with a shared-memory scratch: a task (output
// row, 32-dim slice) goes to nb = ceil(part_stride / 32) warps of one CTA,
// which merges kWarps / nb tasks at once; warp j of a task takes partitions
// 32j .. 32j + 31 with its lanes over the slice's dims, so every partial read
// is one whole 128-byte line.  Each warp loads all the row's LSEs and its 32
// partial lines at once (one round trip), computes the row's log-sum-exp
// itself and sums its weighted lines; the task's warps then add their sums
// in `scratch` (kWarps x 32 floats), in partition-block order.  The CTA's
// loop runs the same number of rounds in every thread (`sync` is a CTA
// barrier).  Needs nb <= kWarps.
template <int D, int kWarps, typename RowOf, typename Sync>
__device__ void merge_tasks_cta(const DecodeParams &p, RowOf row_of, int nrows, int part,
                                float *scratch, int t, Sync sync) {
    constexpr int kBlocks = kMaxGridMerge / 32;  // partition blocks of 32 at most
    const int PS = p.part_stride;
    const int nb = (PS + 31) / 32;
    const int per = kWarps / nb;                  // tasks one CTA merges at once
    const int warp = t >> 5, lane = t & 31, slot = warp / nb, blk = warp % nb;
    const int tasks = nrows * (D / 32);
    for (int base = part * per; base < tasks; base += p.num_splits * per) {
        const int k = base + slot;
        const bool active = slot < per && k < tasks;
        int64_t row = 0;
        int slice = 0;
        if (active) {
            row = row_of(k / (D / 32));
            slice = k % (D / 32);
            const float *pl = p.part_lse + row * PS;
            const float *po = p.part_o + (row * PS + 32 * blk) * D + slice * 32 + lane;
            float lv[kBlocks], ov[32];
#pragma unroll
            for (int i = 0; i < kBlocks; ++i) lv[i] = lane + 32 * i < PS ? __ldcg(pl + lane + 32 * i) : -INFINITY;
#pragma unroll
            for (int j = 0; j < 32; ++j) ov[j] = 32 * blk + j < PS ? __ldcg(po + static_cast<int64_t>(j) * D) : 0.f;
            float M = -INFINITY;
#pragma unroll
            for (int i = 0; i < kBlocks; ++i) M = fmaxf(M, lv[i]);
#pragma unroll
            for (int off = 16; off; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
            float total = -INFINITY, acc = 0.f;
            if (M != -INFINITY) {
                float z = 0.f;
#pragma unroll
                for (int i = 0; i < kBlocks; ++i) z += (lv[i] == -INFINITY) ? 0.f : expf(lv[i] - M);
#pragma unroll
                for (int off = 16; off; off >>= 1) z += __shfl_xor_sync(0xffffffffu, z, off);
                total = M + logf(z);
                float mine = lv[0];  // the LSE of partition 32 * blk + lane
#pragma unroll
                for (int i = 1; i < kBlocks; ++i)
                    if (i == blk) mine = lv[i];
                const float wl = (mine == -INFINITY) ? 0.f : expf(mine - total);
#pragma unroll
                for (int j = 0; j < 32; ++j) acc = fmaf(__shfl_sync(0xffffffffu, wl, j), ov[j], acc);
            }
            scratch[warp * 32 + lane] = acc;
            if (blk == 0 && slice == 0 && lane == 0 && p.lse) p.lse[row] = total;
        }
        sync();
        if (active && blk == 0) {
            float o = 0.f;
            for (int j = 0; j < nb; ++j) o += scratch[(warp + j) * 32 + lane];
            static_cast<__nv_bfloat16 *>(p.out)[row * D + slice * 32 + lane] = __float2bfloat16_rn(o);
        }
        sync();
    }
}

// Called by all 32 x kWarps threads (index t) of a CTA after its partials for
// its nrows rows are written: row j is row_first + (j / per_block) * stride +
// j % per_block (blocks of consecutive rows, e.g. one per query position).
// `sync` synchronises those threads; `flag` is a shared int.  Every CTA of a
// group launches the same kernel, so all agree on kWarps and hence on who does
// which task.
// (The host launches this merge only for P <= kMaxGridMerge.)
template <int D, int kWarps, typename Sync>
__device__ void merge_split_group(const DecodeParams &p, int group, int part, int64_t row_first,
                                  int nrows, int per_block, int64_t stride, int *flag, int t,
                                  Sync sync, float *scratch = nullptr) {
    auto row_of = [&](int j) -> int64_t { return row_first + (j / per_block) * stride + j % per_block; };
    if (!p.counters) return;
    int *arrive = p.counters + 2 * group;  // (the pair's second int is not used)
    const int P = p.num_splits;
    // Release: the barrier orders every thread's partial stores before thread
    // 0's gpu-scope release fence, which makes them visible before its arrival.
    sync();
    if (t == 0) {
        const int old = atom_add_release_gpu(arrive, 1);
        bool ok = false;
        if (old == P - 1) {
            // Last to arrive: acquire everyone's partials, then put the counter
            // back to zero (a release, so a waiter that reads zero acquires too).
            red_add_release_gpu(arrive, -P);
            ok = true;
        } else {
            // Done once the counter reads P, or reads at most this CTA's own
            // arrival value (it was reset, which happens only after the P-th).
            const uint64_t t0 = globaltimer_ns();
            for (uint32_t i = 0; i < kWaitLimit; ++i) {
                const int v = ld_acquire_gpu(arrive);
                if (v >= P || v <= old) {
                    ok = true;
                    break;
                }
                if (wait_expired(i, t0)) break;
            }
        }
        if (!ok) set_status(p.status, PA_STATUS_TIMEOUT);
        *flag = ok;
    }
    // Acquire: thread 0 saw all P arrivals with an acquire load (or as the last
    // arriver, after its fence); the barrier orders every thread's partial
    // loads after it.
    sync();
    if (*flag) {
        const int warp = t >> 5, lane = t & 31;
        if (p.part_stride <= 32) {  // lanes over dims: one round trip per 32-dim slice
            const int tasks = nrows * (D / 32);
            for (int k = part * kWarps + warp; k < tasks; k += P * kWarps)
                merge_slice<D>(p, row_of(k / (D / 32)), k % (D / 32), lane);
        } else if (scratch && (p.part_stride + 31) / 32 <= kWarps) {  // warps over partitions
            merge_tasks_cta<D, kWarps>(p, row_of, nrows, part, scratch, t, sync);
        } else {        // lanes over partitions: one round trip per 8-dim slice
            const int tasks = nrows * (D / 8);
            for (int k = part * kWarps + warp; k < tasks; k += P * kWarps)
                merge_slice_wide<D>(p, row_of(k / (D / 8)), k % (D / 8), lane);
        }
    }
}

// Cluster merge: the P CTAs of one (sequence, head group) are a thread-block
// cluster.  Each has left, in its own shared memory, its normalised partial
// output ostage[n][D] (fp32) and its log-sum-exp lse_s[n] (-inf: no key seen,
// then ostage is not read) for the n < ncols MMA columns; rel[n] is column
// n's output row relative to row0 (-1: padding), the same in every CTA of the
// cluster.  After a cluster barrier, CTA `rank` merges output elements
// e = (n, d) = rank * kThreads + t, then every P * kThreads-th one, reading
// each peer's stage through distributed shared memory (all 2P loads of an
// element are issued together), and writes the bf16 output (and the row's
// log-sum-exp).  A second barrier keeps every stage alive until all peers
// have read it.  Called by all kThreads threads of every CTA of the cluster.
template <int D, int kThreads>
__device__ void merge_cluster(const DecodeParams &p, const float *ostage, const float *lse_s,
                              const int *rel, int ncols, int64_t row0, int t) {
    cluster_sync();
    const int P = p.num_splits;
    const uint32_t rank = cluster_ctarank();
    const uint32_t o_loc = smem_u32(ostage), l_loc = smem_u32(lse_s);
    __nv_bfloat16 *out = static_cast<__nv_bfloat16 *>(p.out);
    for (int e = static_cast<int>(rank) * kThreads + t; e < ncols * D; e += P * kThreads) {
        const int n = e / D, d = e % D;
        const int r = rel[n];
        if (r < 0) continue;
        float lv[kMaxClusterMerge], ov[kMaxClusterMerge];
#pragma unroll
        for (int k = 0; k < kMaxClusterMerge; ++k) {
            lv[k] = -INFINITY;
            ov[k] = 0.f;
            if (k < P) {
                lv[k] = ld_shared_cluster(map_shared_rank(l_loc + 4u * n, k));
                ov[k] = ld_shared_cluster(map_shared_rank(o_loc + 4u * e, k));
            }
        }
        float M = -INFINITY;
#pragma unroll
        for (int k = 0; k < kMaxClusterMerge; ++k) M = fmaxf(M, lv[k]);
        float total = -INFINITY, acc = 0.f;
        if (M != -INFINITY) {
            float z = 0.f;
#pragma unroll
            for (int k = 0; k < kMaxClusterMerge; ++k) z += lv[k] == -INFINITY ? 0.f : expf(lv[k] - M);
            total = M + logf(z);
#pragma unroll
            for (int k = 0; k < kMaxClusterMerge; ++k)
                if (lv[k] != -INFINITY) acc = fmaf(expf(lv[k] - total), ov[k], acc);
        }
        out[(row0 + r) * D + d] = __float2bfloat16_rn(acc);
        if (d == 0 && p.lse) p.lse[row0 + r] = total;
    }
    cluster_sync();
}

}  // namespace pa
