// Paged decode attention on the CUDA cores, fed by TMA.
//
// One CTA per (partition p, KV head g, sequence b).  The CTA owns the G query
// heads that share KV head g (the GQA group), so every K/V tile of its token
// range is read from HBM exactly once.  Each of the NW warps streams its own
// interleaved subset of 16-token tiles through a private NST-stage ring in
// shared memory: lane 0 issues the TMA loads (block-table lookup, one 4-D box
// per 64-element sub-row and K or V) and every lane waits on the stage's
// mbarrier.  A warp keeps its own online-softmax state (running max, sum and
// output accumulator per head); the NW states are merged through shared
// memory at the end.
//
// Inside a warp, for one tile:
//   QK:  lane = (token t = lane % 16, half = lane / 16).  The lane takes the
//        dot product of K row t with the G pre-scaled query heads over its
//        half of D; one shuffle adds the halves.
//   softmax: tile max and sum per head by xor-shuffles over the 16 tokens;
//        scores are in the log2 domain (scale * log2 e folded into q), so
//        exp is a single ex2.approx.
//   PV:  lane owns D/32 output dims of every head; it walks the valid
//        tokens, reading V from the swizzled tile and p from a small
//        per-warp buffer (broadcast loads).
// Tokens past the sequence end inside the last tile are masked (score -inf)
// and skipped in PV, so stale pool rows never reach the result.
#pragma once

#include <atomic>

#include "pa_device.cuh"
#include "pa_internal.h"
#include "pa_split_merge.cuh"

namespace pa {

template <int D, int G, int NW, int NST>
struct CcCfg {
    static constexpr int kSub = D / kSubElems;                  // sub-rows per token row (1 or 2)
    static constexpr int kTileBytes = kTile * D * 2;            // one K (or V) tile
    static constexpr int kStageBytes = 2 * kTileBytes;          // K + V
    static constexpr int kQH = D / 2;                           // dims per lane half in QK
    static constexpr int kQHS = kQH + 4;                        // padded: halves land in different banks
    static constexpr int kQBytes = G * 2 * kQHS * 4;
    static constexpr int kPG = (G + 3) / 4 * 4;                 // p row padded to float4
    static constexpr int kPBytes = NW * kTile * kPG * 4;
    static constexpr int kRingBytes = NW * NST * kStageBytes;
    static constexpr int kMergeBytes = NW * G * (D + 2) * 4;    // acc + m + l per warp
    static constexpr int kRegion0 = kRingBytes > kMergeBytes ? kRingBytes : kMergeBytes;
    static constexpr int kQOff = kRegion0;
    static constexpr int kPOff = kQOff + kQBytes;
    static constexpr int kBarOff = (kPOff + kPBytes + 7) / 8 * 8;
    static constexpr int kTicketOff = kBarOff + NW * NST * 8;
    static constexpr int kSmemBytes = kTicketOff + 16 + 1024;  // + alignment slack
    static constexpr int kDPV = D / 32;                         // output dims per lane
};

template <int D, int G, int NW, int NST>
__global__ void __launch_bounds__(NW * 32)
decode_cc_kernel(const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap vmap,
                 const DecodeParams p) {
    using C = CcCfg<D, G, NW, NST>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                                ~uintptr_t(1023));
    float *qs = reinterpret_cast<float *>(smem + C::kQOff);
    float *pbuf_all = reinterpret_cast<float *>(smem + C::kPOff);
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + C::kBarOff);

    const int part = blockIdx.x, g = blockIdx.y, b = blockIdx.z;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int bs = p.block_size;

    int L = p.seq_lens[b];
    const int lmax = p.max_blocks * bs;
    if (L < 0 || L > lmax) {
        if (tid == 0 && part == 0 && g == 0) set_status(p.status, PA_STATUS_BAD_SEQLEN);
        L = L < 0 ? 0 : lmax;
    }
    const int t_begin = part * p.chunk;
    const int t_end = min(t_begin + p.chunk, L);
    const int ntiles = t_end > t_begin ? (t_end - t_begin + kTile - 1) / kTile : 0;
    const int32_t *bt = p.block_tables + static_cast<int64_t>(b) * p.max_blocks;

    // Query heads of this group, widened to fp32 and pre-scaled by scale*log2(e).
    const uint16_t *qg = p.q + (static_cast<int64_t>(b) * p.num_q_heads + g * G) * D;
    for (int i = tid; i < G * D; i += NW * 32) {
        const int h = i / D, d = i % D;
        const float v = __uint_as_float(static_cast<uint32_t>(qg[i]) << 16) * p.scale_log2;
        qs[h * 2 * C::kQHS + (d / C::kQH) * C::kQHS + (d % C::kQH)] = v;
    }
    if (tid < NW * NST) mbar_init(&bars[tid], 1);
    if (tid == 0) {
        prefetch_tensormap(&kmap);
        prefetch_tensormap(&vmap);
    }
    fence_barrier_init();
    __syncthreads();

    // ---- per-warp streaming loop -------------------------------------------------
    const int my_tiles = warp < ntiles ? (ntiles - warp + NW - 1) / NW : 0;
    uint8_t *ring = smem + warp * NST * C::kStageBytes;
    uint64_t *wbars = bars + warp * NST;
    float *pbuf = pbuf_all + warp * kTile * C::kPG;
    const uint64_t policy = l2_evict_first_policy();

    auto tile_phys = [&](int j) -> int {  // physical block of this warp's j-th tile
        const int tok0 = t_begin + (warp + j * NW) * kTile;
        return bt[tok0 / bs];
    };
    auto issue = [&](int j) {  // lane 0 only
        const int s = j % NST;
        const int tok0 = t_begin + (warp + j * NW) * kTile;
        const int phys = bt[tok0 / bs];
        if (phys < 0 || phys >= p.num_blocks) {
            set_status(p.status, PA_STATUS_BAD_BLOCK);
            mbar_arrive(&wbars[s]);
            return;
        }
        const int row0 = phys * bs + tok0 % bs;
        uint8_t *kt = ring + s * C::kStageBytes;
        uint8_t *vt = kt + C::kTileBytes;
        mbar_arrive_expect_tx(&wbars[s], C::kStageBytes);
#pragma unroll
        for (int sub = 0; sub < C::kSub; ++sub) {
            tma_load_4d(kt + sub * kTile * kSubBytes, &kmap, 0, sub, g, row0, &wbars[s], policy);
            tma_load_4d(vt + sub * kTile * kSubBytes, &vmap, 0, sub, g, row0, &wbars[s], policy);
        }
    };

    // Fused cache write: the warp whose tile holds position L - 1 writes that
    // token's K (lanes 0-15) and V (lanes 16-31) row of head g into the pool
    // just before loading the tile.  The row is fetched up front.
    const int last_pos = L - 1;
    const bool writes = p.k_new && last_pos >= t_begin && last_pos < t_end;
    const int64_t slot_b = writes ? p.slot_mapping[b] : -1;
    constexpr int kRowChunks = D / 8;  // 16-byte chunks of one head row
    const int wl = lane & 15;
    uint4 newrow = make_uint4(0u, 0u, 0u, 0u);
    if (writes && wl < kRowChunks)
        newrow = reinterpret_cast<const uint4 *>((lane < 16 ? p.k_new : p.v_new) +
                                                 (static_cast<int64_t>(b) * p.num_kv_heads + g) * D)[wl];
    auto write_if_holder = [&](int j) {  // whole warp, before tile j is issued
        const int tok0 = t_begin + (warp + j * NW) * kTile;
        if (!writes || last_pos < tok0 || last_pos >= tok0 + kTile) return;
        const int ph = bt[tok0 / bs];
        if (slot_is_position(slot_b, ph, last_pos, bs) && ph < p.num_blocks) {
            if (wl < kRowChunks)
                reinterpret_cast<uint4 *>((lane < 16 ? p.k_pool : p.v_pool) +
                                          (slot_b * p.num_kv_heads + g) * D)[wl] = newrow;
            fence_proxy_async_global();
        } else if (lane == 0 && slot_b >= 0) {
            set_status(p.status, PA_STATUS_BAD_SLOT);
        }
        __syncwarp();
    };

    int issued = 0;
    for (; issued < NST && issued < my_tiles; ++issued) {
        write_if_holder(issued);
        if (lane == 0) issue(issued);
    }

    float m_run[G], l_run[G], o[G][C::kDPV];
#pragma unroll
    for (int h = 0; h < G; ++h) {
        m_run[h] = -INFINITY;
        l_run[h] = 0.f;
#pragma unroll
        for (int k = 0; k < C::kDPV; ++k) o[h][k] = 0.f;
    }

    const int t = lane & 15, half = lane >> 4;
    // QK addressing: sub-row and first 16-byte chunk this lane reads.
    const int qk_sub = (D == 128) ? half : 0;
    const int qk_c0 = (D == 128) ? 0 : half * 4;
    constexpr int kNch = C::kQH / 8;  // chunks of 8 dims per lane half
    // PV addressing: the lane's D/32 output dims.
    const int pv_sub = (D == 128) ? (lane >> 4) : 0;
    const int pv_chunk = (D == 128) ? ((lane & 15) >> 1) : (lane >> 2);
    const int pv_byte = (D == 128) ? (lane & 1) * 8 : (lane & 3) * 4;

    int consumed = 0;
    bool aborted = false;
    for (int j = 0; j < my_tiles; ++j) {
        const int s = j % NST;
        const bool landed = mbar_wait_bounded(&wbars[s], (j / NST) & 1);
        if (!__all_sync(0xffffffffu, landed)) {
            if (lane == 0) set_status(p.status, PA_STATUS_TIMEOUT);
            aborted = true;
            break;
        }
        consumed = j + 1;
        const int tok0 = t_begin + (warp + j * NW) * kTile;
        const int phys = tile_phys(j);
        const int nvalid = (phys < 0 || phys >= p.num_blocks) ? 0 : min(kTile, t_end - tok0);
        if (nvalid > 0) {
            const uint8_t *kt = ring + s * C::kStageBytes;
            const uint8_t *vt = kt + C::kTileBytes;

            // ---- QK for token t over this lane's half of D
            float acc0[G], acc1[G];
#pragma unroll
            for (int h = 0; h < G; ++h) acc0[h] = acc1[h] = 0.f;
            const uint8_t *krow = kt + qk_sub * kTile * kSubBytes;
            const float *qh = qs + half * C::kQHS;
#pragma unroll
            for (int c = 0; c < kNch; ++c) {
                const uint4 kr = *reinterpret_cast<const uint4 *>(krow + swz128(t, qk_c0 + c));
                const float k0 = bf16lo(kr.x), k1 = bf16hi(kr.x), k2 = bf16lo(kr.y), k3 = bf16hi(kr.y);
                const float k4 = bf16lo(kr.z), k5 = bf16hi(kr.z), k6 = bf16lo(kr.w), k7 = bf16hi(kr.w);
#pragma unroll
                for (int h = 0; h < G; ++h) {
                    const float4 qa = *reinterpret_cast<const float4 *>(qh + h * 2 * C::kQHS + c * 8);
                    const float4 qb = *reinterpret_cast<const float4 *>(qh + h * 2 * C::kQHS + c * 8 + 4);
                    acc0[h] = fmaf(qa.x, k0, acc0[h]);
                    acc1[h] = fmaf(qa.y, k1, acc1[h]);
                    acc0[h] = fmaf(qa.z, k2, acc0[h]);
                    acc1[h] = fmaf(qa.w, k3, acc1[h]);
                    acc0[h] = fmaf(qb.x, k4, acc0[h]);
                    acc1[h] = fmaf(qb.y, k5, acc1[h]);
                    acc0[h] = fmaf(qb.z, k6, acc0[h]);
                    acc1[h] = fmaf(qb.w, k7, acc1[h]);
                }
            }
            float sc[G], alpha[G];
            const bool live = t < nvalid;
#pragma unroll
            for (int h = 0; h < G; ++h) {
                float v = acc0[h] + acc1[h];
                v += __shfl_xor_sync(0xffffffffu, v, 16);
                sc[h] = live ? v : -INFINITY;
            }
            // ---- online softmax over the 16 tokens (lanes 16..31 mirror 0..15)
#pragma unroll
            for (int h = 0; h < G; ++h) {
                float mt = sc[h];
                mt = fmaxf(mt, __shfl_xor_sync(0xffffffffu, mt, 1));
                mt = fmaxf(mt, __shfl_xor_sync(0xffffffffu, mt, 2));
                mt = fmaxf(mt, __shfl_xor_sync(0xffffffffu, mt, 4));
                mt = fmaxf(mt, __shfl_xor_sync(0xffffffffu, mt, 8));
                const float m_new = fmaxf(m_run[h], mt);
                alpha[h] = fast_exp2(m_run[h] - m_new);
                m_run[h] = m_new;
                const float pv = fast_exp2(sc[h] - m_new);
                sc[h] = pv;
                float lt = pv;
                lt += __shfl_xor_sync(0xffffffffu, lt, 1);
                lt += __shfl_xor_sync(0xffffffffu, lt, 2);
                lt += __shfl_xor_sync(0xffffffffu, lt, 4);
                lt += __shfl_xor_sync(0xffffffffu, lt, 8);
                l_run[h] = l_run[h] * alpha[h] + lt;
            }
            if (half == 0) {
#pragma unroll
                for (int h = 0; h < C::kPG; h += 4) {
                    float4 v;
                    v.x = sc[h];
                    v.y = (h + 1 < G) ? sc[(h + 1) % G] : 0.f;
                    v.z = (h + 2 < G) ? sc[(h + 2) % G] : 0.f;
                    v.w = (h + 3 < G) ? sc[(h + 3) % G] : 0.f;
                    *reinterpret_cast<float4 *>(pbuf + t * C::kPG + h) = v;
                }
            }
            __syncwarp();

            // ---- PV: rescale, then accumulate the valid tokens
#pragma unroll
            for (int h = 0; h < G; ++h)
#pragma unroll
                for (int k = 0; k < C::kDPV; ++k) o[h][k] *= alpha[h];
            const uint8_t *vrow = vt + pv_sub * kTile * kSubBytes + pv_byte;
            for (int tt = 0; tt < nvalid; ++tt) {
                float vv[C::kDPV];
                if constexpr (C::kDPV == 4) {
                    const uint2 w = *reinterpret_cast<const uint2 *>(vrow + swz128(tt, pv_chunk));
                    vv[0] = bf16lo(w.x); vv[1] = bf16hi(w.x); vv[2] = bf16lo(w.y); vv[3] = bf16hi(w.y);
                } else {
                    const uint32_t w = *reinterpret_cast<const uint32_t *>(vrow + swz128(tt, pv_chunk));
                    vv[0] = bf16lo(w); vv[1] = bf16hi(w);
                }
                float pr[C::kPG];
#pragma unroll
                for (int h = 0; h < C::kPG; h += 4) {
                    const float4 v4 = *reinterpret_cast<const float4 *>(pbuf + tt * C::kPG + h);
                    pr[h] = v4.x; pr[h + 1] = v4.y; pr[h + 2] = v4.z; pr[h + 3] = v4.w;
                }
#pragma unroll
                for (int h = 0; h < G; ++h)
#pragma unroll
                    for (int k = 0; k < C::kDPV; ++k) o[h][k] = fmaf(pr[h], vv[k], o[h][k]);
            }
        }
        __syncwarp();
        // Stage s is free again: refill it with this warp's tile j + NST.
        if (issued < my_tiles) {
            write_if_holder(issued);
            if (lane == 0) {
                fence_proxy_async_smem();
                issue(issued);
            }
            ++issued;
        }
    }
    if (aborted) {
        // Let this warp's copies in flight land before the CTA leaves (bounded).
        for (int j = consumed; j < issued; ++j) mbar_wait_bounded(&wbars[j % NST], (j / NST) & 1);
    }
    __syncthreads();  // ring no longer in use by any warp or copy: reuse it for the merge

    // ---- merge the NW warp states -------------------------------------------------
    float *macc = reinterpret_cast<float *>(smem);              // [NW][G][D]
    float *mm = macc + NW * G * D;                              // [NW][G]
    float *ml = mm + NW * G;                                    // [NW][G]
#pragma unroll
    for (int h = 0; h < G; ++h) {
#pragma unroll
        for (int k = 0; k < C::kDPV; ++k) {
            int d;
            if constexpr (D == 128) d = pv_sub * 64 + pv_chunk * 8 + (lane & 1) * 4 + k;
            else d = pv_chunk * 8 + (lane & 3) * 2 + k;
            macc[(warp * G + h) * D + d] = o[h][k];
        }
        if (lane == 0) {
            mm[warp * G + h] = m_run[h];
            ml[warp * G + h] = l_run[h];
        }
    }
    __syncthreads();

    const int hq0 = g * G;
    for (int i = tid; i < G * (D / 2); i += NW * 32) {
        const int h = i / (D / 2), d = (i % (D / 2)) * 2;
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < NW; ++w) M = fmaxf(M, mm[w * G + h]);
        float lsum = 0.f, o0 = 0.f, o1 = 0.f;
        if (M != -INFINITY) {
#pragma unroll
            for (int w = 0; w < NW; ++w) {
                const float f = fast_exp2(mm[w * G + h] - M);
                lsum = fmaf(ml[w * G + h], f, lsum);
                o0 = fmaf(macc[(w * G + h) * D + d], f, o0);
                o1 = fmaf(macc[(w * G + h) * D + d + 1], f, o1);
            }
            const float inv = 1.f / lsum;
            o0 *= inv;
            o1 *= inv;
        }
        const float lse_nat = (M == -INFINITY) ? -INFINITY : (M + log2f(lsum)) * 0.69314718055994531f;
        const int64_t row = static_cast<int64_t>(b) * p.num_q_heads + hq0 + h;
        if (p.split) {
            const int64_t prow = row * p.num_splits + part;
            *reinterpret_cast<float2 *>(p.part_o + prow * D + d) = make_float2(o0, o1);
            if (d == 0) p.part_lse[prow] = lse_nat;
        } else {
            __nv_bfloat162 v = __floats2bfloat162_rn(o0, o1);
            *reinterpret_cast<__nv_bfloat162 *>(static_cast<uint16_t *>(p.out) + row * D + d) = v;
            if (d == 0 && p.lse) p.lse[row] = lse_nat;
        }
    }
    if (p.split)
        merge_split_group<D, NW>(p, b * gridDim.y + g, part, static_cast<int64_t>(b) * p.num_q_heads + hq0,
                                 G, G, p.num_q_heads, reinterpret_cast<int *>(smem + C::kTicketOff),
                                 tid, [] { __syncthreads(); });
}

// Opt a kernel into more than 48 KB of dynamic shared memory, once per
// device.  `done` must be distinct for every kernel: callers pass a static
// that lives in their own (per-instantiation) function.
template <typename Kernel>
cudaError_t ensure_smem_attr(std::atomic<uint64_t> &done, Kernel kern, int bytes) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const uint64_t bit = 1ull << (dev & 63);
    if (done.load(std::memory_order_acquire) & bit) return cudaSuccess;
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e == cudaSuccess) done.fetch_or(bit, std::memory_order_release);
    return e;
}

template <int D, int G>
cudaError_t launch_cc_instance(const CUtensorMap &kmap, const CUtensorMap &vmap,
                               const DecodeParams &p, int B, cudaStream_t stream) {
    constexpr int NW = 4;
    constexpr int NST = (D == 128) ? 3 : 4;
    using C = CcCfg<D, G, NW, NST>;
    auto kern = decode_cc_kernel<D, G, NW, NST>;
    static std::atomic<uint64_t> smem_attr_done{0};
    cudaError_t e = ensure_smem_attr(smem_attr_done, kern, C::kSmemBytes);
    if (e != cudaSuccess) return e;
    return launch_maybe_cooperative(kern, dim3(p.num_splits, p.num_kv_heads, B), NW * 32,
                                    C::kSmemBytes, stream, p.counters != nullptr, false, kmap, vmap, p);
}

}  // namespace pa
