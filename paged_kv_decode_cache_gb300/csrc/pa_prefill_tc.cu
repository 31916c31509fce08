// Multi-query paged attention with the queries on the MMA's M side, for
// chunks of many new tokens per sequence (chunked prefill of a prompt, a
// long run of new tokens) and for many sequences' queries over one shared
// prefix (the cascade's prefix pass).  Head dim 128, tensor cores (tcgen05).
//
// One CTA per (partition p, query tile, KV head g, sequence b).  A query tile
// is 128 MMA rows r = (query position qi0 + r / G, group member r % G): up to
// 128 / G consecutive query positions with all G query heads of KV head g, so
// the CTA reads each KV block of its range once for 128 query rows (the decode
// kernel, with queries as MMA columns, holds at most 32 columns per head).
// The CTA streams its token range in chunks of T = 64 tokens (four 16-token
// tiles through the block table):
//
//   QK:  S[128 r, 64 t] = Q[128 r, 128 d] . K_chunk^T[128 d, 64 t]
//        A = the query tile (K-major, 128-byte swizzle), B = the K chunk as
//        TMA lands it ([64 t][128 d], K-major).
//   PV:  O[128 r, 128 d] += P[128 r, 64 t] . V_chunk[64 t, 128 d]
//        A = p written by the softmax threads (K-major), B = the V chunk as
//        TMA lands it, read MN-major (no transpose).  p is a bf16 pair
//        hi + lo carrying it to about 2^-17 relative (two MMAs per chunk).
//
// Two softmax warpgroups take alternate chunks: group g (warps 4g .. 4g + 3,
// thread = row r) handles chunks g, g + 2, ... with its own S buffer, P buffer
// and O accumulator in TMEM (lane = row r), so the two groups' exponentials
// overlap each other and the MMAs.  A thread loads its S row, masks keys past
// the range, past the row's causal position or in tiles not loaded, keeps a
// per-row reference max that moves only when a score exceeds it by more than
// 2^8 (the warp then rescales its rows of its group's O once the group's
// previous PV has finished), and writes the hi/lo rows of P.  The epilogue
// merges the two groups' (O, max, sum) like two partitions, normalises and
// writes bf16 rows (or fp32 partials with the range split) by bulk copies.
// Warp 8 issues QK, warp 11 issues PV; warps 9 and 10 stream K and V through
// 3-stage rings of 16 KB, one TMA box per 16-token tile and 64-element half.
// A tile past the range or with a bad block id is loaded from a coordinate
// past the pool, which fills the box with zeros.  Every wait is bounded.
#include <cuda_bf16.h>

#include <atomic>

#include "pa_device.cuh"
#include "pa_internal.h"
#include "pa_tcgen05.cuh"

namespace pa {
namespace {

constexpr int kPfRows = 128;                     // query rows per CTA (M of both MMAs)
constexpr int kPfT = 64;                         // tokens per chunk (N of QK, K of PV)
constexpr int kPfThreads = 384;                  // 2 softmax warpgroups, QK, K TMA, V TMA, PV
constexpr int kPfQkWarp = 8, kPfTmaKWarp = 9, kPfTmaVWarp = 10, kPfPvWarp = 11;
constexpr int kPfNK = 3, kPfNV = 3;              // K and V stages
constexpr int kPfNS = 2;                         // S buffers in TMEM (one per softmax group)
constexpr int kPfNP = 2;                         // P buffers (hi + lo) in shared memory (one per group)
constexpr int kPfTilesPerChunk = kPfT / kTile;   // 4
constexpr int kPfHalf = kPfT * kSubBytes;        // one 64-element half of a chunk: 8 KB
constexpr int kPfStage = 2 * kPfHalf;            // 16 KB
constexpr int kPfBox = kTile * kSubBytes;        // one TMA box: 16 rows x 128 B
constexpr int kPfQHalf = kPfRows * kSubBytes;    // 16 KB
constexpr int kPfPPart = kPfRows * kPfT * 2;     // [128 rows][64 tokens] bf16 = 16 KB
constexpr int kPfPBuf = 2 * kPfPPart;            // hi, then lo
constexpr float kPfLazyTau = 8.0f;               // log2 headroom before a row's reference max moves

constexpr int kPfKOff = 0;
constexpr int kPfVOff = kPfKOff + kPfNK * kPfStage;
constexpr int kPfQOff = kPfVOff + kPfNV * kPfStage;
constexpr int kPfPOff = kPfQOff + 2 * kPfQHalf;
constexpr int kPfRowsOff = kPfPOff + kPfNP * kPfPBuf;
constexpr int kPfBarOff = kPfRowsOff + kPrefillMaxTiles * 4;
// (+ 2: one per MMA issuer that an aborting CTA commits to, so that it frees
// TMEM only after every MMA it issued has completed)
constexpr int kPfNumBars = 2 * kPfNK + 2 * kPfNV + 2 * kPfNS + 2 * kPfNP + 2;
constexpr int kPfXOff = kPfBarOff + kPfNumBars * 8;   // group 1's row maxima and sums [2][128]
constexpr int kPfMiscOff = kPfXOff + 2 * kPfRows * 4;
constexpr int kPfSmemBytes = kPfMiscOff + 16 + 1024;   // + room to align the base to 1024
constexpr uint32_t kPfTmemCols = 512;                  // S: 2 x 64 columns, then O0, O1: 128 each
constexpr int kPfColO = kPfNS * kPfT;                  // O of group g at kPfColO + 128 g
static_assert(kPfColO + 2 * 128 <= static_cast<int>(kPfTmemCols), "TMEM columns");
static_assert(kPfSmemBytes <= 227 * 1024, "shared memory");
static_assert(kPfNP * kPfPBuf >= kPfRows * 128 * 4, "the epilogue stages fp32 rows in the P buffers");
static_assert(kPfStage % 1024 == 0 && kPfQHalf % 1024 == 0 && kPfPPart % 1024 == 0, "swizzle atoms");

__global__ void __launch_bounds__(kPfThreads, 1)
prefill_tc_kernel(const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap vmap,
                  const DecodeParams p, int G) {
    constexpr int D = 128;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                                ~uintptr_t(1023));
    uint8_t *kring = smem + kPfKOff;
    uint8_t *vring = smem + kPfVOff;
    uint8_t *qs = smem + kPfQOff;
    uint8_t *ps = smem + kPfPOff;
    int *tile_row = reinterpret_cast<int *>(smem + kPfRowsOff);  // pool row of each 16-token tile, -1: none
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + kPfBarOff);
    uint64_t *kfull = bars, *kempty = kfull + kPfNK, *vfull = kempty + kPfNK, *vempty = vfull + kPfNV;
    uint64_t *sdone = vempty + kPfNV, *sfree = sdone + kPfNS, *pready = sfree + kPfNS;
    uint64_t *pfree = pready + kPfNP;
    uint64_t *drain = pfree + kPfNP;  // [2]: QK issuer, PV issuer (abort only)
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + kPfMiscOff);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + kPfMiscOff + 4);

    // Launched with programmatic stream serialization: no global memory is
    // touched before the previous kernel in the stream has completed.
    griddep_wait();
    griddep_launch_dependents();

    const int part = blockIdx.x, b = blockIdx.z;
    const int Hkv = p.num_kv_heads, Hq = p.num_q_heads;
    const int g = blockIdx.y % Hkv;
    const int qi0 = static_cast<int>(blockIdx.y / Hkv) * p.q_per_cta;  // the tile's first query position
    const int nq = min(p.q_per_cta, p.q_len - qi0);
    const int nrows = nq * G;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int bs = p.block_size;
    const int lmax = p.max_blocks * bs;
    int L = p.seq_len_const >= 0 ? p.seq_len_const : p.seq_lens[b] - p.seq_len_offset;
    if (L < 0 || L > lmax) {
        if (tid == 0 && part == 0 && blockIdx.y == 0) set_status(p.status, PA_STATUS_BAD_SEQLEN);
        L = L < 0 ? 0 : lmax;
    }
    // Query qi0 + k sits at position qbase + k and sees keys up to it (causal);
    // without the causal rule every query sees all L keys.
    const int qbase = L - p.q_len + qi0;
    const int t_stop = p.causal ? min(L, qbase + nq) : L;
    const int t_begin = part * p.chunk;
    const int t_end = min(t_begin + p.chunk, max(0, t_stop));
    const int nch = t_end > t_begin ? (t_end - t_begin + kPfT - 1) / kPfT : 0;
    // output row of tile row r: ((b * q_len + position) * Hq + g * G + member)
    const int64_t orow0 = (static_cast<int64_t>(b) * p.q_len + qi0) * Hq + static_cast<int64_t>(g) * G;
    auto out_row = [&](int r) -> int64_t { return orow0 + static_cast<int64_t>(r / G) * Hq + r % G; };

    if (nch == 0) {  // no key in range: zero output, lse = -inf
        for (int i = tid; i < nrows * D; i += kPfThreads) {
            const int64_t o = out_row(i / D);
            if (p.split) p.part_o[(o * p.part_stride + p.part_offset + part) * D + i % D] = 0.f;
            else static_cast<__nv_bfloat16 *>(p.out)[o * D + i % D] = __float2bfloat16_rn(0.f);
        }
        for (int r = tid; r < nrows; r += kPfThreads) {
            if (p.split) p.part_lse[out_row(r) * p.part_stride + p.part_offset + part] = -INFINITY;
            else if (p.lse) p.lse[out_row(r)] = -INFINITY;
        }
        return;
    }

    // ---- set-up: the range's tile rows, the query tile, barriers, TMEM ----------------
    const int ntiles = (t_end - t_begin + kTile - 1) / kTile;  // <= kPrefillMaxTiles (host)
    const int32_t *bt = p.block_tables + static_cast<int64_t>(b) * p.table_stride;
    for (int i = tid; i < ntiles; i += kPfThreads) {
        const int tok = t_begin + i * kTile;
        const int phys = bt[tok / bs];
        int row = -1;
        if (phys >= 0 && phys < p.num_blocks) row = phys * bs + tok % bs;
        else set_status(p.status, PA_STATUS_BAD_BLOCK);
        tile_row[i] = row;
    }
    constexpr int kQChunks = kPfRows * (D / 8);                       // 16-byte chunks of the tile
    constexpr int kQLoads = (kQChunks + kPfThreads - 1) / kPfThreads;  // per thread
    uint4 qv[kQLoads];
#pragma unroll
    for (int j = 0; j < kQLoads; ++j) {
        const int i = tid + j * kPfThreads, r = i / (D / 8), c = i % (D / 8);
        qv[j] = make_uint4(0u, 0u, 0u, 0u);
        if (i < kQChunks && r < nrows) qv[j] = *reinterpret_cast<const uint4 *>(p.q + out_row(r) * D + c * 8);
    }
#pragma unroll
    for (int j = 0; j < kQLoads; ++j) {  // Q[r][d]: half d / 64, swizzled 16-byte chunk
        const int i = tid + j * kPfThreads, r = i / (D / 8), c = i % (D / 8);
        if (i < kQChunks) *reinterpret_cast<uint4 *>(qs + (c >> 3) * kPfQHalf + swz128(r, c & 7)) = qv[j];
    }
    if (warp == 0) tc5::tmem_alloc(tmem_slot, kPfTmemCols);
    if (tid == 0) {
        for (int i = 0; i < kPfNK; ++i) {
            mbar_init(&kfull[i], 1u);
            mbar_init(&kempty[i], 1u);
        }
        for (int i = 0; i < kPfNV; ++i) {
            mbar_init(&vfull[i], 1u);
            mbar_init(&vempty[i], 1u);
        }
        for (int i = 0; i < kPfNS; ++i) {
            mbar_init(&sdone[i], 1u);
            mbar_init(&sfree[i], 4u);  // the 4 warps of softmax group i release S buffer i
        }
        for (int i = 0; i < kPfNP; ++i) {
            mbar_init(&pready[i], 4u);  // ... and publish P buffer i
            mbar_init(&pfree[i], 1u);
        }
        mbar_init(&drain[0], 1u);
        mbar_init(&drain[1], 1u);
        *abort_flag = 0;
    }
    if (lane == 0 && warp == kPfTmaKWarp) prefetch_tensormap(&kmap);
    if (lane == 0 && warp == kPfTmaVWarp) prefetch_tensormap(&vmap);
    fence_proxy_async_smem();  // the query tile, written here, is read by the MMA
    fence_barrier_init();
    tc5::fence_before_sync();
    __syncthreads();
    tc5::fence_after_sync();
    const uint32_t tmem = *tmem_slot;

    auto wait_or_abort = [&](uint64_t *bar, uint32_t parity) -> bool {
        return mbar_try_wait(bar, parity) || mbar_wait_or_abort_slow(bar, parity, abort_flag, p.status);
    };

    if (warp == kPfTmaKWarp || warp == kPfTmaVWarp) {
        // ================= TMA producers: K (warp 9), V (warp 10) =================
        // lanes 0-7: lane = 2 * tile + half issues that box of each chunk
        const bool is_v = warp == kPfTmaVWarp;
        uint8_t *ring = is_v ? vring : kring;
        uint64_t *full = is_v ? vfull : kfull;
        uint64_t *empty = is_v ? vempty : kempty;
        const CUtensorMap *map = is_v ? &vmap : &kmap;
        const int nst = is_v ? kPfNV : kPfNK;
        const int tile = lane >> 1, half = lane & 1;
        const int oob_row = p.num_blocks * bs;  // a box starting here lies past the pool: zeros
        const uint64_t policy = l2_evict_normal_policy();  // other query tiles read these blocks too
        int issued = 0;
        for (int c = 0; c < nch; ++c) {
            const int s = c % nst;
            if (c >= nst) {
                const bool ok = wait_or_abort(&empty[s], ((c / nst) - 1) & 1);
                if (!__all_sync(0xffffffffu, ok)) break;
            }
            if (lane == 0) mbar_arrive_expect_tx(&full[s], 2u * kPfTilesPerChunk * kPfBox);
            __syncwarp();
            if (lane < 2 * kPfTilesPerChunk) {
                const int ti = c * kPfTilesPerChunk + tile;
                const int row = ti < ntiles ? tile_row[ti] : -1;
                tma_load_4d(ring + s * kPfStage + half * kPfHalf + tile * kPfBox, map, 0,
                            row >= 0 ? row : oob_row, g, half, &full[s], policy);
            }
            issued = c + 1;
        }
        if (*abort_flag && lane == 0)  // let this CTA's copies land before it leaves
            for (int c = max(0, issued - nst); c < issued; ++c) mbar_wait_bounded(&full[c % nst], (c / nst) & 1);
    } else if (warp == kPfQkWarp) {
        // ================= QK issuer =================
        if (lane == 0) {
            constexpr uint32_t kIdQK = tc5::idesc_bf16_f32(kPfRows, kPfT, false, false);
            int done = 0;
            for (int c = 0; c < nch; ++c) {
                // S buffer c % NS is free once softmax c - NS has read it; K c has landed
                if (c >= kPfNS && !wait_or_abort(&sfree[c % kPfNS], ((c / kPfNS) - 1) & 1)) break;
                if (!wait_or_abort(&kfull[c % kPfNK], (c / kPfNK) & 1)) break;
                tc5::fence_after_sync();
                const uint8_t *kt = kring + (c % kPfNK) * kPfStage;
                const uint32_t dcol = tmem + (c % kPfNS) * kPfT;
#pragma unroll
                for (int j = 0; j < D / 16; ++j) {  // K = 16 dims per MMA
                    const int hf = j >> 2, off = (j & 3) * 32;
                    tc5::mma_bf16(dcol, tc5::sw128_desc(qs + hf * kPfQHalf + off, 16, 1024),
                                  tc5::sw128_desc(kt + hf * kPfHalf + off, 16, 1024), kIdQK, j > 0);
                }
                tc5::commit(&sdone[c % kPfNS]);
                tc5::commit(&kempty[c % kPfNK]);
                done = c + 1;
            }
            if (*abort_flag && done > 0) {  // let issued MMAs finish before TMEM is freed
                tc5::commit(&drain[0]);
                mbar_wait_bounded(&drain[0], 0);
            }
        }
    } else if (warp == kPfPvWarp) {
        // ================= PV issuer =================
        if (lane == 0) {
            constexpr uint32_t kIdPV = tc5::idesc_bf16_f32(kPfRows, D, false, true);
            int done = 0;
            for (int c = 0; c < nch; ++c) {
                if (!wait_or_abort(&pready[c % kPfNP], (c / kPfNP) & 1)) break;
                if (!wait_or_abort(&vfull[c % kPfNV], (c / kPfNV) & 1)) break;
                tc5::fence_after_sync();
                const uint8_t *vt = vring + (c % kPfNV) * kPfStage;
                const uint8_t *pb = ps + (c % kPfNP) * kPfPBuf;
                const uint32_t ocol = tmem + kPfColO + (c % 2) * 128;  // the O of chunk c's group
#pragma unroll
                for (int hl = 0; hl < 2; ++hl) {  // hi part, then lo part of p
#pragma unroll
                    for (int j = 0; j < kPfT / 16; ++j)  // K = 16 tokens per MMA
                        tc5::mma_bf16(ocol, tc5::sw128_desc(pb + hl * kPfPPart + j * 32, 16, 1024),
                                      tc5::sw128_desc(vt + j * 16 * kSubBytes, kPfHalf, 1024), kIdPV,
                                      c >= 2 || hl > 0 || j > 0);
                }
                tc5::commit(&pfree[c % kPfNP]);
                tc5::commit(&vempty[c % kPfNV]);
                done = c + 1;
            }
            if (*abort_flag && done > 0) {
                tc5::commit(&drain[1]);
                mbar_wait_bounded(&drain[1], 0);
            }
        }
    } else {
        // ================= softmax groups: group grp = warp / 4, thread = query row r =================
        const int grp = warp >> 2, wq = warp & 3;  // wq: this warp's quarter of the TMEM lanes
        const int r = tid & (kPfRows - 1);
        const bool row_ok = r < nrows;
        const int pos = p.causal ? qbase + r / G : L - 1;  // the last key row r sees
        const float sl2 = p.scale_log2;
        const uint32_t ocol = tmem + kPfColO + grp * 128;   // this group's O
        uint8_t *prow = ps + grp * kPfPBuf + r * kSubBytes;   // this group's P row r
        float m_ref = -INFINITY, l = 0.f;
        for (int c = grp; c < nch; c += 2) {
            const bool ok = __all_sync(0xffffffffu, wait_or_abort(&sdone[grp], (c / 2) & 1));
            float sv[kPfT];
            if (ok) {
                tc5::fence_after_sync();
                uint32_t raw[kPfT];
#pragma unroll
                for (int k = 0; k < kPfT / 16; ++k)
                    tc5::ld_32x32b_x16_nowait(tc5::taddr(tmem, 32 * wq, grp * kPfT + 16 * k),
                                              *reinterpret_cast<uint32_t(*)[16]>(&raw[16 * k]));
                tc5::wait_ld();
#pragma unroll
                for (int k = 0; k < kPfT; ++k) sv[k] = __uint_as_float(raw[k]);
            }
            tc5::fence_before_sync();
            __syncwarp();  // (one arrival per warp, once all its lanes have read)
            if (lane == 0) mbar_arrive(&sfree[grp]);  // S buffer read: QK c + 2 may overwrite it
            if (!ok || *abort_flag) break;
            const int tok0 = t_begin + c * kPfT;
            bool tile_ok[kPfTilesPerChunk];
            bool all_tiles = true;
#pragma unroll
            for (int k = 0; k < kPfTilesPerChunk; ++k) {
                const int ti = c * kPfTilesPerChunk + k;
                tile_ok[k] = ti < ntiles && tile_row[ti] >= 0;
                all_tiles &= tile_ok[k];
            }
            // Most chunks are seen whole by every row of the warp: no mask then.
            const int tok_last = tok0 + kPfT - 1;
            const bool whole = __all_sync(0xffffffffu, row_ok && all_tiles && tok_last < t_end && tok_last <= pos);
            float mx = -INFINITY;
            if (whole) {
#pragma unroll
                for (int k = 0; k < kPfT; ++k) {
                    sv[k] *= sl2;
                    mx = fmaxf(mx, sv[k]);
                }
            } else {
#pragma unroll
                for (int k = 0; k < kPfT; ++k) {
                    const int t = tok0 + k;
                    const bool valid = row_ok && tile_ok[k / kTile] && t < t_end && t <= pos;
                    sv[k] = valid ? sv[k] * sl2 : -INFINITY;
                    mx = fmaxf(mx, sv[k]);
                }
            }
            // The group's previous PV (chunk c - 2) must be done before its O is
            // rescaled or its P buffer rewritten.
            const bool prev_done =
                c < 2 || __all_sync(0xffffffffu, wait_or_abort(&pfree[grp], ((c / 2) - 1) & 1));
            // Lazy rescaling: a row's reference max moves only when a score exceeds
            // it by more than 2^8; the warp then rescales its 32 rows of O together
            // (TMEM loads and stores are warp-wide).
            if (__any_sync(0xffffffffu, mx > m_ref + kPfLazyTau)) {
                const float mn = fmaxf(m_ref, mx);
                const float alpha = mn == -INFINITY ? 1.f : fast_exp2(m_ref - mn);
                l *= alpha;
                if (c >= 2 && prev_done) {
                    tc5::fence_after_sync();
#pragma unroll 1
                    for (int k = 0; k < D / 16; ++k) {
                        float ov[16];
                        const uint32_t ta = tc5::taddr(ocol, 32 * wq, 16 * k);
                        tc5::ld_32x32b_x16(ta, ov);
#pragma unroll
                        for (int i = 0; i < 16; ++i) ov[i] *= alpha;
                        tc5::st_32x32b_x16(ta, ov);
                    }
                }
                m_ref = mn;
            }
            // p = hi + lo, two bf16 values per word, written in two halves of 32
            // tokens.  A masked score is -inf and gives p = 0 (a row that has seen
            // no key yet subtracts 0, not -inf).  The row sum adds p itself: hi +
            // lo equals it to about 2^-17.
            const float m_use = m_ref == -INFINITY ? 0.f : m_ref;
#pragma unroll
            for (int hf = 0; hf < 2; ++hf) {
                uint32_t hw[kPfT / 4], lw[kPfT / 4];
#pragma unroll
                for (int k = 0; k < kPfT / 2; k += 2) {
                    const float p0 = fast_exp2(sv[hf * kPfT / 2 + k] - m_use);
                    const float p1 = fast_exp2(sv[hf * kPfT / 2 + k + 1] - m_use);
                    const __nv_bfloat162 h = __floats2bfloat162_rn(p0, p1);
                    const float2 hv = __bfloat1622float2(h);
                    const __nv_bfloat162 lo = __floats2bfloat162_rn(p0 - hv.x, p1 - hv.y);
                    hw[k / 2] = *reinterpret_cast<const uint32_t *>(&h);
                    lw[k / 2] = *reinterpret_cast<const uint32_t *>(&lo);
                    l += p0 + p1;
                }
#pragma unroll
                for (int j = 0; j < kPfT / 16; ++j) {  // 16-byte chunk 4 hf + j: tokens 8 (4 hf + j) ..
                    const int ch = 4 * hf + j;
                    const uint32_t off = static_cast<uint32_t>((ch ^ (r & 7)) << 4);
                    *reinterpret_cast<uint4 *>(prow + off) =
                        make_uint4(hw[4 * j], hw[4 * j + 1], hw[4 * j + 2], hw[4 * j + 3]);
                    *reinterpret_cast<uint4 *>(prow + kPfPPart + off) =
                        make_uint4(lw[4 * j], lw[4 * j + 1], lw[4 * j + 2], lw[4 * j + 3]);
                }
            }
            // V rows that were loaded from the pool but lie past the range (the
            // tail of the tile holding key t_end - 1) may hold anything, even
            // NaN: they are zeroed, so that 0 * V never reaches O.  (The wait on
            // the V stage is in chunk c's phase: PV c - 2 has finished, and the
            // one PV issuer works in chunk order, so PV c - 3, the stage's
            // previous user, was issued before it.)
            if (c == nch - 1) {
                const int z0 = t_end - tok0;
                const int z1 = min(kPfT, (t_end + kTile - 1) / kTile * kTile - tok0);
                if (z1 > z0 && wait_or_abort(&vfull[c % kPfNV], (c / kPfNV) & 1)) {
                    uint8_t *vt = vring + (c % kPfNV) * kPfStage;
                    for (int i = r; i < (z1 - z0) * 16; i += kPfRows) {
                        const int row = z0 + i / 16, hc = i % 16;
                        *reinterpret_cast<uint4 *>(vt + (hc >> 3) * kPfHalf + swz128(row, hc & 7)) =
                            make_uint4(0u, 0u, 0u, 0u);
                    }
                }
            }
            fence_proxy_async_smem();  // P (and zeroed V rows) are read by the MMA
            tc5::fence_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive(&pready[grp]);
        }

        // ---- epilogue: the two groups' rows merged, normalised, staged in the idle P
        //      buffers and bulk-copied out by group 0 ----
        float *xm = reinterpret_cast<float *>(smem + kPfXOff), *xl = xm + kPfRows;
        if (grp == 1) {
            xm[r] = m_ref;
            xl[r] = l;
        }
        named_sync(1, 2 * kPfRows);
        // every PV has completed once the last one has (one issuer, committed in order)
        const bool okf = grp == 0 && __all_sync(0xffffffffu, wait_or_abort(&pfree[(nch - 1) % 2],
                                                                           ((nch - 1) / 2) & 1)) &&
                         *abort_flag == 0;
        if (okf) {
            tc5::fence_after_sync();
            const bool has1 = nch >= 2;  // group 1 took a chunk: its O holds data
            const float m1 = has1 ? xm[r] : -INFINITY, l1 = has1 ? xl[r] : 0.f;
            const float M = fmaxf(m_ref, m1);
            const float a0 = m_ref == -INFINITY ? 0.f : fast_exp2(m_ref - M);
            const float a1 = m1 == -INFINITY ? 0.f : fast_exp2(m1 - M);
            const float lt = a0 * l + a1 * l1;
            const float inv = lt > 0.f ? p.v_scale / lt : 0.f;  // 0: no key seen
            const float w0 = a0 * inv, w1 = a1 * inv;
            const bool split = p.split != 0;
            uint8_t *stage = ps + r * (split ? D * 4 : D * 2);
#pragma unroll 1
            for (int k = 0; k < D / 16; ++k) {
                float ov[16], o1[16];
                tc5::ld_32x32b_x16(tc5::taddr(tmem + kPfColO, 32 * wq, 16 * k), ov);
                if (has1) {
                    tc5::ld_32x32b_x16(tc5::taddr(tmem + kPfColO + 128, 32 * wq, 16 * k), o1);
#pragma unroll
                    for (int i = 0; i < 16; ++i) ov[i] = ov[i] * w0 + o1[i] * w1;
                } else {
#pragma unroll
                    for (int i = 0; i < 16; ++i) ov[i] *= w0;
                }
                if (split) {
                    float4 *dst = reinterpret_cast<float4 *>(stage) + 4 * k;
#pragma unroll
                    for (int i = 0; i < 4; ++i)
                        dst[i] = make_float4(ov[4 * i], ov[4 * i + 1], ov[4 * i + 2], ov[4 * i + 3]);
                } else {
                    uint32_t w[8];
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        const __nv_bfloat162 h = __floats2bfloat162_rn(ov[2 * i], ov[2 * i + 1]);
                        w[i] = *reinterpret_cast<const uint32_t *>(&h);
                    }
                    uint4 *dst = reinterpret_cast<uint4 *>(stage) + 2 * k;
                    dst[0] = make_uint4(w[0], w[1], w[2], w[3]);
                    dst[1] = make_uint4(w[4], w[5], w[6], w[7]);
                }
            }
            fence_proxy_async_smem();  // the bulk copy (async proxy) reads the staged row
            if (row_ok) {
                const float lse = lt > 0.f ? (M + log2f(lt)) * 0.69314718055994531f : -INFINITY;
                const int64_t o = out_row(r);
                if (split) {
                    const int64_t slot = o * p.part_stride + p.part_offset + part;
                    bulk_store_s2g(p.part_o + slot * D, stage, D * 4);
                    bulk_commit();
                    p.part_lse[slot] = lse;
                } else {
                    bulk_store_s2g(static_cast<__nv_bfloat16 *>(p.out) + o * D, stage, D * 2);
                    bulk_commit();
                    if (p.lse) p.lse[o] = lse;
                }
                bulk_wait_all_read();
            }
        }
    }
    tc5::fence_before_sync();
    __syncthreads();
    if (warp == 0) tc5::tmem_free(tmem, kPfTmemCols);
}

}  // namespace

cudaError_t launch_prefill_tc(const CUtensorMap &kmap, const CUtensorMap &vmap, const DecodeParams &p,
                              int B, int G, cudaStream_t stream) {
    static std::atomic<uint64_t> smem_attr_done{0};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const uint64_t bit = 1ull << (dev & 63);
    if (!(smem_attr_done.load(std::memory_order_acquire) & bit)) {
        e = cudaFuncSetAttribute(prefill_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 kPfSmemBytes);
        if (e != cudaSuccess) return e;
        smem_attr_done.fetch_or(bit, std::memory_order_release);
    }
    const int qtiles = (p.q_len + p.q_per_cta - 1) / p.q_per_cta;
    const dim3 grid(p.num_splits, qtiles * p.num_kv_heads, B);
    return launch_maybe_cooperative(prefill_tc_kernel, grid, kPfThreads, kPfSmemBytes, stream, false,
                                    p.pdl != 0, kmap, vmap, p, G);
}

}  // namespace pa
