// Paged decode attention on the 5th-generation tensor cores (tcgen05), for
// head_dim 128.
//
// One CTA per (partition p, group of HC KV heads and of queries, sequence b)
// streams its token range in chunks of T = 128 / HC tokens, loading whole
// paged blocks: one TMA box per 16-token tile and 64-element half-row brings
// that tile for all HC heads (16 rows x HC heads x 128 bytes, head-major in
// shared memory), so the HBM reads of a block are contiguous bursts.  A chunk
// is therefore 128 rows m = (tile, head, row) of K (and of V), and both
// contractions are dense 128-row tiles:
//
//   QK:  S[128 m, N] = K_chunk[128 m, 128 d] . Q^T[128 d, N]
//        N = HC x GP columns n = (head', c): column c < Gq of KV head head'
//        is query position qi0 + c / G of group member c % G (one position
//        when q_len = 1), zero-padded to GP per head.  A = the K chunk as TMA
//        lands it (K-major, 128-byte swizzle), B = the packed queries.  Only
//        the columns with head' = head(m) are used.
//   PV:  O^T[128 d, 2N] += V_chunk^T[128 d, 128 m] . [P_hi | P_lo]^T[128 m, 2N]
//        A = the V chunk read transposed (MN-major descriptor, no copy).
//        p is split into a 16-bit part and the 16-bit rounding of its
//        remainder, so the pair carries p to about 2^-17 relative; one MMA
//        with N' = 2N accumulates both halves into adjacent TMEM columns,
//        which the epilogue adds.  B is block-diagonal by head: row m only
//        has its own head's GP columns, so O^T[d, (h, c)] sums over head h's
//        tokens only.
//
// S (NBS buffers of N columns) and O^T (2N columns) live in TMEM: lane = row m
// for S and lane = head dim d for O.  The CTA is warp-specialised:
//   warps 0-3 (softmax): thread t owns row m = t of each chunk and output dim
//        d = t.  It loads its S row (tcgen05.ld), keeps its head's GP scores
//        (masked where the token is past the range, its tile was not loaded,
//        or, with causal queries, past the column's position), forms
//        p = exp2(s - m_ref) against a per-column reference max, writes the
//        hi/lo pair into P^T and arrives on the chunk's "P ready" barrier.
//        m_ref only moves when some score exceeds it by more than 2^8 (a
//        CTA-wide vote, one barrier per chunk); then the chunk max is
//        reduced, O^T is rescaled in TMEM and the row sums with it.  Row sums
//        stay per thread and are reduced under the last PV; the epilogue reads
//        O^T, normalises it and stages it as rows in the idle P^T buffers
//        (bf16, or fp32 partials when the range is split), which one bulk
//        copy per row writes out (the cluster merge reads them in place).
//   warp 4 (QK issuer) and warp 7 (PV issuer): one thread each issues its
//        MMAs as soon as their inputs are ready (QK: K landed and the S buffer
//        released by the softmax threads; PV: P^T written and V landed) and
//        commits to the barriers that publish S, release the K stage, release
//        the P buffer and the V stage.
//   warps 5, 6 (TMA): stream K and V through separate rings (NK and NV
//        stages of 32 KB, 16 KB with FP8 pools).  Block ids arrive by cp.async into a small ring
//        kTcLook chunks ahead of use, so an issue never waits on a lookup
//        queued behind the KV stream.  Tiles past the range or with a bad
//        block id are not loaded; the K producer publishes, per chunk, a
//        tagged mask of the tiles it loaded, which the softmax threads read
//        (so they never touch a stage after its MMA has released it), and an
//        invalid row's V is zeroed.  With new K/V rows given, the producer
//        whose range holds position L - 1 writes them into the pool through
//        the slot mapping just before loading that tile.
//   warps 8-11 (FP8 pools only): the producers land the e4m3 codes in 16 KB
//        stages (so twice the token rows are in flight for the same shared
//        memory); warp 8 + q widens TMEM lanes 32 q .. 32 q + 31 of each
//        chunk's K and V^T into fp16 operand buffers in TMEM (two or three per tensor),
//        from which the QK and PV MMAs read their A operand.  k_scale is
//        folded into the softmax scale and v_scale into the epilogue.
// With the range split, the CTAs of one (sequence, head group) merge their
// partials in the same launch: once all P have arrived, they share the
// merge tasks, through global memory or, as one thread-block cluster,
// through distributed shared memory (pa_split_merge.cuh).  The kernel waits
// for the previous kernel in the stream (programmatic dependent launch)
// before it touches global memory.  Every mbarrier wait and spin is bounded in polls and
// in time and honours a CTA-wide abort flag; the softmax warps agree on an
// abort at their per-chunk vote.
#pragma once

#include <cuda_fp16.h>
#include <cuda_fp8.h>

#include <atomic>

#include "pa_device.cuh"
#include "pa_internal.h"
#include "pa_split_merge.cuh"
#include "pa_tcgen05.cuh"

namespace pa {

constexpr int kTcRows = 128;           // rows m per chunk (M of QK)
constexpr int kTcThreads = 256;        // 4 softmax warps + 2 MMA warps + 2 TMA warps
constexpr int kTcCvtWarp = 8;          // FP8 pools: first of the warps that widen the e4m3 codes
constexpr int kTcQkWarp = 4;
constexpr int kTcTmaKWarp = 5;
constexpr int kTcTmaVWarp = 6;
constexpr int kTcPvWarp = 7;
constexpr int kTcNBS = 4;              // S buffers in TMEM
constexpr float kTcLazyTau = 8.0f;     // log2 headroom before a reference max moves
constexpr int kTcLook = 4;             // chunks a producer's block-id lookups run ahead
constexpr int kTcMaskRing = 8;         // chunk validity masks the K producer publishes

constexpr int kTcSmemLimit = 227 * 1024;
// room to round the dynamic shared memory base (at least 16-byte aligned) up
// to the 1024-byte swizzle-atom boundary
constexpr int kAlignSlack = 1024 - 16;

template <int HC, int GP, bool F8 = false>
struct TcCfg {
    static constexpr int kN = HC * GP;                          // MMA N
    // FP8 converter warps: 8 (warps 8-11 widen K, 12-15 V) where the softmax
    // fits the 128 registers a thread of 512 gets (GP <= 8), else 4 (each
    // widens K, then V, of its TMEM lane quarter)
    static constexpr int kCvtWarps = !F8 ? 0 : GP <= 8 ? 8 : 4;
    static constexpr int kThreads = kTcThreads + 32 * kCvtWarps;
    static_assert(kN % 16 == 0 && kN >= 16 && kN <= 64, "MMA N");
    static constexpr int kT = kTcRows / HC;                     // tokens per chunk
    static constexpr int kTiles = kT / kTile;                   // 16-token tiles per chunk
    static_assert(kTiles >= 1 && kTiles * HC * kTile == kTcRows, "tiles");
    static constexpr int kSubTile = kTcRows * kSubBytes;        // [128 m][64 d] bf16 = 16 KB
    static constexpr int kTileBytes = 2 * kSubTile;             // K (or V) of one chunk: 32 KB
    static constexpr int kBoxBytes = HC * kTile * kSubBytes;    // one TMA box: HC heads x 16 rows
    static constexpr int kQBytes = 2 * kN * kSubBytes;          // [N][64] x 2 halves
    static constexpr int kPBytes = 2 * kN * kSubBytes;          // 2 atoms of [N][64 m]
    // P^T buffer: the hi (columns n' = 0..N-1) and lo (n' = N..2N-1) bf16
    // parts of p; one MMA with N' = 2N accumulates both into adjacent TMEM
    // column ranges.  Layout, 128-byte swizzle: for N = 32 and 64 MN-major,
    // [2N / 64 atoms][128 m][64 n'] (a row's 2GP values are whole 16-byte
    // chunks, written with vector stores); for N = 16 (64-byte rows) K-major,
    // 2 atoms of [2N][64 m].
    static constexpr bool kPMn = kN == 32 || kN == 64;
    static constexpr int kPBufBytes = 2 * kPBytes;
    static_assert(!kPMn || kPBufBytes == (2 * kN / 64) * kSubTile, "MN-major P^T: whole atoms");
    // (a cluster merge stages the partial O^T, kN x 128 fp32, in the P^T buffers)
    static_assert(kPBufBytes >= kN * 128 * 4, "cluster merge stage");
    // red[128 rows][GPr], col[N], m_ref[N], alpha[N], rel[N] (output row of
    // column n relative to the CTA's first row, -1: padding), abort flag,
    // TMEM slot, merge ticket.  Thread t writes its row t of red, so rows are
    // GP + 1 floats apart where that fits (a warp's stores then fall in 32
    // different banks; GP apart they share 32 / GP banks).
    static constexpr int red_bytes(int gpr) { return (kTcRows * gpr + 4 * kN) * 4 + 16; }
    // S buffers in TMEM (FP8 pools with N >= 32 keep 2, to leave room for the
    // widened operands: three buffers of each at N = 32 beat 4 S buffers and
    // two of each, 17.3 against 17.5 us on the 7B layer)
    static constexpr int kNBS = (F8 && kN >= 32) ? 2 : kTcNBS;
    // chunk validity masks the producers publish (ring slots)
    static constexpr int kMaskRing = F8 ? 16 : kTcMaskRing;
    // TMEM: S buffers (NBS x N columns), O^T (hi part N, lo part N), then with
    // FP8 pools the widened K and V^T operands, NOB buffers of 64 columns each
    // (128 rows x 128 16-bit values) starting on a 64-column boundary: three
    // where they fit in the 512 columns (N = 16), else two
    static constexpr int kColO = kNBS * kN;
    static constexpr int kColK = (kColO + 2 * kN + 63) / 64 * 64;
    static constexpr int kNOB = (F8 && kColK + 6 * 64 <= 512) ? 3 : 2;
    static constexpr int kColV = kColK + 64 * kNOB;
    static constexpr int kColsUsed = F8 ? kColV + 64 * kNOB : kColO + 2 * kN;
    // A K (V) stage in shared memory: a bf16 chunk (32 KB), or with FP8 pools
    // the chunk's one-byte codes (16 KB), which the converter warps widen into
    // TMEM (the MMAs read their A operands there).
    static constexpr int kStageBytes = F8 ? kTcRows * 128 : kTileBytes;
    // shared memory for nk K stages, nv V stages and nbp P^T buffers, laid out
    // as below (rings, Q, P^T, scratch, barriers, masks, block-id rings, align)
    // (FP8: the operand buffers' "widened" and "released" barriers, NOB each for
    // K and V, and the V producer's mask ring)
    static constexpr int smem_for(int nk, int nv, int nbp, int gpr = GP) {
        return ((nk + nv) * kStageBytes + kQBytes + nbp * kPBufBytes + red_bytes(gpr) + 7) / 8 * 8 +
               (2 * nk + 2 * nv + 2 * kNBS + 2 * nbp + (F8 ? 4 * kNOB : 0) + 2) * 8 +
               kMaskRing * 8 * (F8 ? 2 : 1) + 2 * (kTcLook + 1) * 32 * 4 + kAlignSlack;
    }
    // bf16: the deepest pipeline that fits: K and V stages first, then P^T buffers
    static constexpr int choice_for(int gpr) {
        return smem_for(3, 3, 2, gpr) <= kTcSmemLimit ? 0
               : smem_for(3, 3, 1, gpr) <= kTcSmemLimit ? 1
               : smem_for(2, 3, 2, gpr) <= kTcSmemLimit ? 2
               : smem_for(2, 2, 2, gpr) <= kTcSmemLimit ? 3 : 4;
    }
    // FP8: the most code stages (as many K as V) that fit beside two P^T buffers
    static constexpr int f8_stages(int gpr) {
        return smem_for(6, 6, 2, gpr) <= kTcSmemLimit ? 6
               : smem_for(5, 5, 2, gpr) <= kTcSmemLimit ? 5
               : smem_for(4, 4, 2, gpr) <= kTcSmemLimit ? 4 : 3;
    }
    static constexpr int depth_for(int gpr) { return F8 ? f8_stages(gpr) : choice_for(gpr); }
    // the padded scratch only where it costs no pipeline depth
    static constexpr int kGPr = depth_for(GP + 1) == depth_for(GP) ? GP + 1 : GP;
    static constexpr int kRedBytes = red_bytes(kGPr);
    static constexpr int kChoice = choice_for(kGPr);
    static constexpr int kNK = F8 ? f8_stages(kGPr) : kChoice <= 1 ? 3 : 2;  // K stages
    static constexpr int kNV = F8 ? f8_stages(kGPr) : kChoice <= 2 ? 3 : 2;  // V stages
    static constexpr int kNBP = F8 ? 2 : (kChoice == 1 || kChoice == 4) ? 1 : 2;  // P^T buffers
    static constexpr int kVOff = kNK * kStageBytes;
    static constexpr int kQOff = (kNK + kNV) * kStageBytes;
    static constexpr int kPOff = kQOff + kQBytes;
    static constexpr int kRedOff = kPOff + kNBP * kPBufBytes;
    static constexpr int kBarOff = (kRedOff + kRedBytes + 7) / 8 * 8;
    // (+ 2: the MMA issuers' drain barriers, committed to only by an aborting CTA)
    static constexpr int kNumBars = 2 * kNK + 2 * kNV + 2 * kNBS + 2 * kNBP + (F8 ? 4 * kNOB : 0) + 2;
    // validity masks [kMaskRing] (u64: chunk << 32 | lane mask), then the two
    // producers' block-id rings [2][kTcLook + 1][32 lanes]
    static constexpr int kMaskOff = kBarOff + kNumBars * 8;
    static constexpr int kVMaskOff = kMaskOff + kMaskRing * 8;   // FP8 only
    static constexpr int kLookOff = kVMaskOff + (F8 ? kMaskRing * 8 : 0);
    static constexpr int kSmemBytes = kLookOff + 2 * (kTcLook + 1) * 32 * 4 + kAlignSlack;
    static_assert(kSmemBytes == smem_for(kNK, kNV, kNBP, kGPr), "layout");
    // the K producer rewrites mask slot c % ring only once softmax c has read it
    // (FP8: the producer runs at most NK stages, NOB + 1 chunks of converter
    // and operand buffers and NBS S buffers ahead of the softmax)
    static_assert(kNK + kNBS + (F8 ? kNOB + 1 : 0) <= kMaskRing, "mask ring");
    static_assert(kSmemBytes <= kTcSmemLimit, "shared memory");

    static constexpr uint32_t kTmemCols = kColsUsed <= 128 ? 128u : kColsUsed <= 256 ? 256u : 512u;
    static_assert(kColsUsed <= 512, "TMEM columns");
};

// Max (or sum) over the rows of column n's head of a [128 rows][GPr] array:
// row m = (tile * HC + head) * 16 + r holds the GP values of its own head.
template <int HC, int GP, int GPr, bool kMax>
__device__ __forceinline__ float column_reduce(const float *red, int n) {
    const int hh = n / GP, q = n % GP;
    float acc = kMax ? -INFINITY : 0.f;
#pragma unroll 1
    for (int t = 0; t < kTcRows / (kTile * HC); ++t) {
        const float *base = red + ((t * HC + hh) * kTile) * GPr + q;
#pragma unroll
        for (int r = 0; r < kTile; ++r) acc = kMax ? fmaxf(acc, base[r * GPr]) : acc + base[r * GPr];
    }
    return acc;
}

// 16-bit operand values of p for the PV MMA: bf16, or fp16 with FP8 pools
// (whose K/V tiles are widened to fp16).
template <bool F8>
__device__ __forceinline__ float p16_value(uint16_t b) {
    if constexpr (F8) return __half2float(__ushort_as_half(b));
    else return __bfloat162float(__ushort_as_bfloat16(b));
}
// Two values at once (one packed conversion): a in the low 16 bits, b in the high.
template <bool F8>
__device__ __forceinline__ uint32_t p16x2_bits(float a, float b) {
    if constexpr (F8) {
        const __half2 h = __floats2half2_rn(a, b);
        return *reinterpret_cast<const uint32_t *>(&h);
    } else {
        const __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
        return *reinterpret_cast<const uint32_t *>(&h);
    }
}

// Widens 16 e4m3 codes to 16 fp16 values (exact: e4m3 is a subset of fp16),
// one cvt per pair of codes: the low byte of each 16-bit pair becomes the low
// half of the result.
__device__ __forceinline__ uint2 e4m3x4_to_f16x4(uint32_t w) {
    uint2 r;
    asm("{\n\t.reg .b16 lo, hi;\n\t"
        "mov.b32 {lo, hi}, %2;\n\t"
        "cvt.rn.f16x2.e4m3x2 %0, lo;\n\t"
        "cvt.rn.f16x2.e4m3x2 %1, hi;\n\t}"
        : "=r"(r.x), "=r"(r.y)
        : "r"(w));
    return r;
}
__device__ __forceinline__ void e4m3x16_to_f16(const uint4 &in, uint4 &lo, uint4 &hi) {
    const uint2 a = e4m3x4_to_f16x4(in.x), b = e4m3x4_to_f16x4(in.y);
    const uint2 c = e4m3x4_to_f16x4(in.z), d = e4m3x4_to_f16x4(in.w);
    lo = make_uint4(a.x, a.y, b.x, b.y);
    hi = make_uint4(c.x, c.y, d.x, d.y);
}

// FP8 pools: the widened V^T operand in TMEM.  Its lanes are 16-lane groups
// of 16 head dims, 8 x 8 transposed loads giving each thread dims 2 i and
// 2 i + 1 of a group, which 16-lane stores put in lanes i and i + 8: lane L
// holds dim vt_dim(L).  Its columns pair rows of 16-row groups the same way
// (rows 2 j, 2 j + 1 and 8 + 2 j, 9 + 2 j of a group share the thread, and
// land in adjacent columns): row m is index vt_row_k(m) of the contraction.
__host__ __device__ constexpr int vt_dim(int L) { return (L & ~15) | ((L & 7) << 1) | ((L >> 3) & 1); }
__host__ __device__ constexpr int vt_row_k(int m) {
    return (m & ~15) | (((m >> 1) & 3) << 2) | (((m >> 3) & 1) << 1) | (m & 1);
}

template <int HC, int GP, bool F8>
__global__ void __launch_bounds__((TcCfg<HC, GP, F8>::kThreads), 1)
decode_tc_kernel(const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap vmap,
                 const DecodeParams p, int G) {
    constexpr int D = 128;
    using C = TcCfg<HC, GP, F8>;
    constexpr int kThreads = C::kThreads;
    constexpr int N = C::kN, NK = C::kNK, NV = C::kNV, NBP = C::kNBP, NBS = C::kNBS;
    extern __shared__ __align__(16) uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                                ~uintptr_t(1023));
    uint8_t *kring = smem;
    uint8_t *vring = smem + C::kVOff;
    uint8_t *qs = smem + C::kQOff;
    uint8_t *ps = smem + C::kPOff;
    float *red = reinterpret_cast<float *>(smem + C::kRedOff);      // [128 rows][GPr] scratch
    float *col = red + kTcRows * C::kGPr;                           // [N] per-column result
    float *m_ref = col + N;                                         // [N] reference max
    float *alpha_s = m_ref + N;                                     // [N] rescale factors
    int *rel_s = reinterpret_cast<int *>(alpha_s + N);               // [N] output row offsets
    volatile int *abort_flag = reinterpret_cast<volatile int *>(alpha_s + 2 * N);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(alpha_s + 2 * N + 1);
    int *ticket = reinterpret_cast<int *>(alpha_s + 2 * N + 2);
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + C::kBarOff);
    uint64_t *kfull = bars, *kempty = bars + NK, *vfull = bars + 2 * NK, *vempty = vfull + NV;
    uint64_t *sdone = vempty + NV, *sfree = sdone + NBS, *pready = sfree + NBS;
    uint64_t *pfree = pready + NBP;
    // FP8: operand buffer (chunk c % NOB) widened into TMEM, and released by its MMAs
    constexpr int NOB = C::kNOB;
    uint64_t *kconv = pfree + NBP, *kopfree = kconv + NOB, *vconv = kopfree + NOB, *vopfree = vconv + NOB;
    // QK and PV issuers: an aborting CTA commits here, so that it frees TMEM
    // only once every MMA it issued has completed
    uint64_t *drain = bars + C::kNumBars - 2;
    volatile uint64_t *mask_ring = reinterpret_cast<volatile uint64_t *>(smem + C::kMaskOff);
    volatile uint64_t *vmask_ring = reinterpret_cast<volatile uint64_t *>(smem + C::kVMaskOff);
    int *look_ring = reinterpret_cast<int *>(smem + C::kLookOff);  // [2][kTcLook + 1][32]

    // Launched after another kernel with programmatic stream serialization,
    // this CTA may be running before that kernel has finished: nothing above
    // this wait writes global memory or uses what it reads for a result.  The
    // next such launch may be scheduled once every CTA of this grid is past
    // it (it then waits in turn).
    //
    // Meanwhile the PV issuer's warp (idle until the first P) warms L2 with
    // this CTA's first 2 chunks of K and V (4 of codes with FP8 pools), so
    // that those copies are served from L2 once the wait is over (the 7B
    // layer's step: 18.0 -> 16.6 us, 18.5 -> 17.6 us with FP8 pools; one
    // chunk more or less was slower for either).  The
    // length and block ids it reads may still be the previous kernel's to
    // write: they only pick which boxes to warm (an id outside the pool warms
    // nothing), and every load after the wait reads the current values.
    if (threadIdx.x >= 32 * kTcPvWarp && threadIdx.x < 32 * (kTcPvWarp + 1)) {
        constexpr int kPre = F8 ? 4 : 2;  // chunks
        const int ln = threadIdx.x & 31;
        if (ln < kPre * C::kTiles) {
            const int c = ln / C::kTiles, tl = ln % C::kTiles;
            const int bz = blockIdx.z, hg0 = (blockIdx.y % p.head_groups) * HC;
            const int t0 = static_cast<int>(blockIdx.x) * p.chunk;
            const int tok = t0 + c * C::kT + tl * kTile;
            const int lp = p.seq_len_const >= 0 ? p.seq_len_const
                                                : *reinterpret_cast<const volatile int32_t *>(p.seq_lens + bz) -
                                                      p.seq_len_offset;
            const int lim = min(t0 + p.chunk, min(lp, p.max_blocks * p.block_size));
            if (tok < lim) {
                const int phys = *reinterpret_cast<const volatile int32_t *>(
                    p.block_tables + static_cast<int64_t>(bz) * p.table_stride + tok / p.block_size);
                if (phys >= 0 && phys < p.num_blocks) {
                    const int row = phys * p.block_size + tok % p.block_size;
                    if constexpr (F8) {
                        tma_prefetch_3d(&kmap, 0, row, hg0);
                        tma_prefetch_3d(&vmap, 0, row, hg0);
                    } else {
#pragma unroll
                        for (int sub = 0; sub < 2; ++sub) {
                            tma_prefetch_4d(&kmap, 0, row, hg0, sub);
                            tma_prefetch_4d(&vmap, 0, row, hg0, sub);
                        }
                    }
                }
            }
        }
    }
    griddep_wait();
    griddep_launch_dependents();

    const int part = blockIdx.x, b = blockIdx.z;
    const int g0 = (blockIdx.y % p.head_groups) * HC;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int bs = p.block_size;
    // This CTA's queries: positions qi0 .. qi0 + nq - 1 of the q_len new ones
    // (q_len = 1: plain decode).  Per head, MMA column c < Gq is query
    // qi0 + c / G of group member c % G; its output row is col_row(head, c).
    const int qi0 = static_cast<int>(blockIdx.y / p.head_groups) * p.q_per_cta;
    const int nq = min(p.q_per_cta, p.q_len - qi0);
    const int Gq = nq * G;
    const int Hq = p.num_q_heads;

    // Global reads that do not depend on the sequence length go out first, so
    // their latencies overlap: the length, this CTA's queries, and (producer
    // lanes) the block ids of the first kTcLook chunks.
    const int lmax = p.max_blocks * bs;
    const int t_begin = part * p.chunk;
    const int t_lim = min(t_begin + p.chunk, lmax);  // range end before the length is known
    const int64_t row0 = (static_cast<int64_t>(b) * p.q_len + qi0) * Hq + static_cast<int64_t>(g0) * G;
    auto col_row = [&](int hh, int c) -> int64_t {
        return row0 + static_cast<int64_t>(c / G) * Hq + hh * G + c % G;
    };
    const int32_t *bt = p.block_tables + static_cast<int64_t>(b) * p.table_stride;
    int L = p.seq_len_const >= 0 ? p.seq_len_const : p.seq_lens[b] - p.seq_len_offset;
    constexpr int kQLoads = (N * (D / 8) + kThreads - 1) / kThreads;
    uint4 qv[kQLoads];
#pragma unroll
    for (int j = 0; j < kQLoads; ++j) {
        const int i = tid + j * kThreads, n = i / (D / 8), c = i % (D / 8);
        qv[j] = make_uint4(0u, 0u, 0u, 0u);
        if (i < N * (D / 8) && n % GP < Gq)
            qv[j] = *reinterpret_cast<const uint4 *>(p.q + col_row(n / GP, n % GP) * D + c * 8);
    }
    // Block ids reach the TMA producers through cp.async copies into a small
    // ring, kTcLook chunks ahead of use, so no issue waits on a lookup that is
    // queued behind the KV stream.  Lanes 2 * tile + sub of a producer carry
    // tile `tile` of a chunk; both lanes of a tile look its block up.
    const bool producer = warp == kTcTmaKWarp || warp == kTcTmaVWarp;
    const bool is_v = warp == kTcTmaVWarp;
    const int tile = lane >> 1, sub = lane & 1;
    const bool carrier = producer && lane < 2 * C::kTiles;
    int *my_look = look_ring + (is_v ? (kTcLook + 1) * 32 : 0) + lane;  // slot j at my_look[32 * j]
    auto look_ahead = [&](int c, int t_stop) {  // copy chunk c's block id; one commit group per chunk
        const int tok0 = t_begin + c * C::kT + tile * kTile;
        if (carrier && tok0 < t_stop) cp_async_4(my_look + 32 * (c % (kTcLook + 1)), bt + tok0 / bs);
        cp_async_commit();
    };
    if (producer) {
#pragma unroll
        for (int c = 0; c < kTcLook; ++c) look_ahead(c, t_lim);
    }
    if (warp == kTcPvWarp && lane < 4) {
        // The epilogue and the merge first touch the outputs after the KV
        // stream has filled the memory queues; touching them now takes their
        // address translations off that path.
        const void *touch = nullptr;
        const int64_t last = col_row(HC - 1, Gq - 1);
        const __nv_bfloat16 *out_rows = static_cast<const __nv_bfloat16 *>(p.out) + row0 * D;
        if (p.split) {
            if (lane == 0) touch = p.part_o + (row0 * p.part_stride + p.part_offset + part) * D;
            if (lane == 1) touch = p.part_o + (last * p.part_stride + p.part_offset + part) * D;
            if (lane == 2) touch = p.part_lse + row0 * p.part_stride + p.part_offset + part;
            if (lane == 3 && p.counters && p.out) touch = out_rows;  // the merge writes out
        } else {
            if (lane == 0) touch = out_rows;
            if (lane == 1 && p.lse) touch = p.lse + row0;
        }
        if (touch) prefetch_l2(touch);
    }
    if (L < 0 || L > lmax) {
        if (tid == 0 && part == 0 && g0 == 0) set_status(p.status, PA_STATUS_BAD_SEQLEN);
        L = L < 0 ? 0 : lmax;
    }
    // Query qi0 + k sits at position qbase + k and sees tokens up to it
    // (causal); no key past this CTA's last query is read.  Non-causal
    // (cascade prefix pass): every query sees all L keys.
    const int qbase = p.causal ? L - p.q_len + qi0 : L;
    const int t_end = min(t_begin + p.chunk, max(0, min(L, p.causal ? qbase + nq : L)));
    const int nch = t_end > t_begin ? (t_end - t_begin + C::kT - 1) / C::kT : 0;

    if (nch == 0) {  // empty range: zero output, lse = -inf
        cp_async_wait<0>();
        if (p.cluster_merge) {  // a stage with no key seen (its O^T is never read)
            if (tid < N) {
                rel_s[tid] = tid % GP < Gq ? static_cast<int>(col_row(tid / GP, tid % GP) - row0) : -1;
                col[tid] = -INFINITY;
            }
            merge_cluster<D, kThreads>(p, reinterpret_cast<const float *>(ps), col, rel_s, N, row0, tid);
            return;
        }
        for (int i = tid; i < HC * Gq * D; i += kThreads) {
            const int j = i / D, d = i % D;
            const int64_t r = col_row(j / Gq, j % Gq);
            if (p.split) p.part_o[(r * p.part_stride + p.part_offset + part) * D + d] = 0.f;
            else static_cast<__nv_bfloat16 *>(p.out)[r * D + d] = __float2bfloat16_rn(0.f);
        }
        if (tid < HC * Gq) {
            const int64_t r = col_row(tid / Gq, tid % Gq);
            if (p.split) p.part_lse[r * p.part_stride + p.part_offset + part] = -INFINITY;
            else if (p.lse) p.lse[r] = -INFINITY;
        }
        if (p.split)
            merge_split_group<D, kThreads / 32>(p, b * gridDim.y + blockIdx.y, part, row0, HC * Gq,
                                                  HC * G, Hq, ticket, tid, [] { __syncthreads(); },
                                                  reinterpret_cast<float *>(ps));
        return;
    }

    auto wait_or_abort = [&](uint64_t *bar, uint32_t parity) -> bool {
        return mbar_try_wait(bar, parity) || mbar_wait_or_abort_slow(bar, parity, abort_flag, p.status);
    };

    // ---- TMA producers: K ring (warp 5), V ring (warp 6) ----------------------------------
    // Each producer initialises its own ring's barriers and issues its first
    // stages before the CTA-wide set-up barrier (those need no "empty" wait),
    // so the first tiles are in flight while TMEM, Q and the other barriers
    // are set up.
    const int nst = is_v ? NV : NK;
    uint8_t *ring = is_v ? vring : kring;
    uint64_t *full = is_v ? vfull : kfull;
    uint64_t *empty = is_v ? vempty : kempty;
    const CUtensorMap *map = is_v ? &vmap : &kmap;
    // Fused cache write: the CTA whose range holds position L - 1 writes that
    // token's K (warp 5) or V (warp 6) rows of its HC heads into the pool just
    // before loading the tile that holds it.  The rows are fetched up front.
    const int last_pos = L - 1;
    const bool writes = producer && p.k_new && last_pos >= t_begin && last_pos < t_end;
    constexpr int kNewChunks = HC * D / 8;                 // 16-byte chunks of HC rows
    constexpr int kNewPerLane = (kNewChunks + 31) / 32;
    uint4 newrow[kNewPerLane];   // (FP8 pools: newcode, its e4m3 codes)
    uint2 newcode[F8 ? kNewPerLane : 1];
    int64_t slot_b = -1;
    if (writes) {
        slot_b = p.slot_mapping[b];
        const uint4 *src = reinterpret_cast<const uint4 *>(
            (is_v ? p.v_new : p.k_new) + (static_cast<int64_t>(b) * p.num_kv_heads + g0) * D);
#pragma unroll
        for (int j = 0; j < kNewPerLane; ++j)
            if (lane + 32 * j < kNewChunks) newrow[j] = src[lane + 32 * j];
        if constexpr (F8) {  // quantised here, out of the issue loop
            const float wscale = is_v ? p.v_scale : p.k_scale;
#pragma unroll
            for (int j = 0; j < kNewPerLane; ++j)
                if (lane + 32 * j < kNewChunks) newcode[j] = e4m3x8_from_bf16(newrow[j], wscale);
        }
    }
    int issued = 0;
    // Issues chunks [c_from, c_to) of this producer's ring; false once it aborts.
    auto produce = [&](int c_from, int c_to, uint64_t policy) -> bool {
        for (int c = c_from; c < c_to; ++c) {
            const int s = c % nst;
            look_ahead(c + kTcLook, t_end);  // (an empty group past the range)
            cp_async_wait<kTcLook>();        // chunk c's copy has landed
            const int phys = carrier ? my_look[32 * (c % (kTcLook + 1))] : -1;
            if (c >= nst) {
                const bool ok = wait_or_abort(&empty[s], ((c / nst) - 1) & 1);
                if (!__all_sync(0xffffffffu, ok)) return false;
            }
            const int tok0 = t_begin + c * C::kT + tile * kTile;
            bool valid = false;
            if (carrier && tok0 < t_end) {
                if (phys >= 0 && phys < p.num_blocks) valid = true;
                else if (!is_v && sub == 0) set_status(p.status, PA_STATUS_BAD_BLOCK);
            }
            const uint32_t vm = __ballot_sync(0xffffffffu, valid);
            // publish which tiles of chunk c are loaded (bit 2 * tile) for the softmax
            // (and, FP8, for the V converter, which zeroes the V rows not loaded)
            if (lane == 0 && !is_v) mask_ring[c % C::kMaskRing] = (static_cast<uint64_t>(c) << 32) | vm;
            if (F8 && lane == 0 && is_v) vmask_ring[c % C::kMaskRing] = (static_cast<uint64_t>(c) << 32) | vm;
            const int chunk0 = t_begin + c * C::kT;
            if (writes && last_pos >= chunk0 && last_pos < chunk0 + C::kT) {  // holds position L - 1
                const int ph = __shfl_sync(0xffffffffu, phys, 2 * ((last_pos - chunk0) / kTile));
                if (slot_is_position(slot_b, ph, last_pos, bs) && ph < p.num_blocks) {
                    if constexpr (F8) {  // one byte per value, quantised with the pool's scale
                        uint2 *dst = reinterpret_cast<uint2 *>(
                            reinterpret_cast<uint8_t *>(is_v ? p.v_pool : p.k_pool) +
                            (slot_b * p.num_kv_heads + g0) * D);
#pragma unroll
                        for (int j = 0; j < kNewPerLane; ++j)
                            if (lane + 32 * j < kNewChunks) dst[lane + 32 * j] = newcode[j];
                    } else {
                        uint4 *dst = reinterpret_cast<uint4 *>((is_v ? p.v_pool : p.k_pool) +
                                                               (slot_b * p.num_kv_heads + g0) * D);
#pragma unroll
                        for (int j = 0; j < kNewPerLane; ++j)
                            if (lane + 32 * j < kNewChunks) dst[lane + 32 * j] = newrow[j];
                    }
                    fence_proxy_async_global();
                } else if (lane == 0 && !is_v && slot_b >= 0) {
                    set_status(p.status, PA_STATUS_BAD_SLOT);
                }
                __syncwarp();
            }
            if constexpr (F8) {
                // one box per tile (16 rows x HC heads x 128 one-byte codes) into the
                // code stage, from which the converter warps widen it into TMEM
                if (lane == 0)
                    mbar_arrive_expect_tx(&full[s], static_cast<uint32_t>(__popc(vm & 0x55555555u)) * C::kBoxBytes);
                __syncwarp();
                if (valid && sub == 0)
                    tma_load_3d(ring + s * C::kStageBytes + tile * C::kBoxBytes, map, 0,
                                phys * bs + tok0 % bs, g0, &full[s], policy);
            } else {
                if (lane == 0) mbar_arrive_expect_tx(&full[s], static_cast<uint32_t>(__popc(vm)) * C::kBoxBytes);
                __syncwarp();
                if (valid)
                    tma_load_4d(ring + s * C::kStageBytes + sub * C::kSubTile + tile * C::kBoxBytes, map, 0,
                                phys * bs + tok0 % bs, g0, sub, &full[s], policy);
            }
            issued = c + 1;
        }
        return true;
    };
    const int c_pre = min(nch, nst);
    if (producer) {
        if (lane == 0) {
            for (int i = 0; i < nst; ++i) {
                mbar_init(&full[i], 1u);
                // released by the MMA's commit, or (FP8) by the four converter warps
                mbar_init(&empty[i], F8 ? 4u : 1u);
            }
            for (int i = 0; i < C::kMaskRing; ++i) {  // no chunk's tag yet
                if (!is_v) mask_ring[i] = ~uint64_t(0);
                else if (F8) vmask_ring[i] = ~uint64_t(0);
            }
            fence_barrier_init();
            prefetch_tensormap(map);
        }
        __syncwarp();
        produce(0, c_pre, l2_evict_first_policy());
    }

    // ---- set-up: TMEM, barriers, the Q operand, zeroed P^T buffers ---------------------
    if (warp == 0) tc5::tmem_alloc(tmem_slot, C::kTmemCols);
    if (tid == 0) {
        // the MMA / softmax barriers (the rings' are the producers'): every one
        // completes on one arrival except "S free" and "P ready", which each of
        // the 4 softmax warps arrives on once
        for (uint64_t *bar = sdone; bar < pfree + NBP; ++bar)
            mbar_init(bar, (bar >= sfree && bar < pready + NBP) ? 4u : 1u);
        mbar_init(&drain[0], 1u);
        mbar_init(&drain[1], 1u);
        if (F8)  // operand buffers: "widened" by the four converter warps, "released" by a commit
            for (int i = 0; i < NOB; ++i) {
                mbar_init(&kconv[i], 4u);
                mbar_init(&vconv[i], 4u);
                mbar_init(&kopfree[i], 1u);
                mbar_init(&vopfree[i], 1u);
            }
        *abort_flag = 0;
    }
    if (tid < N) m_ref[tid] = -INFINITY;
#pragma unroll
    for (int j = 0; j < kQLoads; ++j) {  // Q operand row n = (head', q), 16-byte chunk c
        const int i = tid + j * kThreads, n = i / (D / 8), c = i % (D / 8);
        if (i < N * (D / 8)) {
            uint4 v = qv[j];
            if constexpr (F8) {  // the MMA takes fp16 operands with FP8 pools
                uint32_t *w = reinterpret_cast<uint32_t *>(&v);
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    const __half2 h = __floats2half2_rn(bf16lo(w[k]), bf16hi(w[k]));
                    w[k] = *reinterpret_cast<const uint32_t *>(&h);
                }
            }
            *reinterpret_cast<uint4 *>(qs + (c >> 3) * (N * kSubBytes) + swz128(n, c & 7)) = v;
        }
    }
    for (int i = tid; i < NBP * C::kPBufBytes / 16; i += kThreads)
        reinterpret_cast<uint4 *>(ps)[i] = make_uint4(0u, 0u, 0u, 0u);
    fence_proxy_async_smem();
    fence_barrier_init();
    tc5::fence_before_sync();
    __syncthreads();
    tc5::fence_after_sync();
    const uint32_t tmem = *tmem_slot;

    if (producer) {
        const bool done = produce(c_pre, nch, l2_evict_first_policy());
        cp_async_wait<0>();
        if (!done || *abort_flag) {
            if (lane == 0)  // let this CTA's copies land before it leaves
                for (int c = max(0, issued - nst); c < issued; ++c)
                    mbar_wait_bounded(&full[c % nst], (c / nst) & 1);
        }
    } else if (warp == kTcQkWarp) {
        // ================= QK issuer =================
        if (lane == 0) {
            constexpr uint32_t kIdQK = tc5::idesc_bf16_f32(kTcRows, N, false, false, F8);
            int done = 0;
            for (int c = 0; c < nch; ++c) {
                // S buffer c % NBS is free once softmax c - NBS has read it; K c has
                // landed (FP8: has been widened into TMEM operand buffer c % NOB)
                if (c >= NBS && !wait_or_abort(&sfree[c % NBS], ((c / NBS) - 1) & 1)) break;
                if (!wait_or_abort(F8 ? &kconv[c % NOB] : &kfull[c % NK], F8 ? (c / NOB) & 1 : (c / NK) & 1)) break;
                tc5::fence_after_sync();
                const uint8_t *kt = kring + (c % NK) * C::kStageBytes;
                const uint32_t dcol = tmem + (c % NBS) * N;
#pragma unroll
                for (int j = 0; j < D / 16; ++j) {  // K = 16 dims d per MMA
                    const int half = j >> 2, off = (j & 3) * 32;
                    const uint64_t qdesc = tc5::sw128_desc(qs + half * (N * kSubBytes) + off, 16, 1024);
                    if constexpr (F8)  // A: lane m, column d / 2 of the widened chunk
                        tc5::mma_f16_tmem_a(dcol, tmem + C::kColK + 64 * (c % NOB) + 8 * j, qdesc, kIdQK, j > 0);
                    else
                        tc5::mma_bf16(dcol, tc5::sw128_desc(kt + half * C::kSubTile + off, 16, 1024), qdesc,
                                      kIdQK, j > 0);
                }
                tc5::commit(&sdone[c % NBS]);
                tc5::commit(F8 ? &kopfree[c % NOB] : &kempty[c % NK]);
                done = c + 1;
            }
            if (*abort_flag && done > 0) {  // let issued MMAs finish before TMEM is freed
                tc5::commit(&drain[0]);
                mbar_wait_bounded(&drain[0], 0);
            }
        }
    } else if (warp == kTcPvWarp) {
        // ================= PV issuer =================
        if (lane == 0) {
            // (V^T read transposed from shared memory, or FP8: from TMEM, K-major)
            constexpr uint32_t kIdPV = tc5::idesc_bf16_f32(kTcRows, 2 * N, !F8, C::kPMn, F8);
            int done = 0;
            for (int c = 0; c < nch; ++c) {
                if (!wait_or_abort(&pready[c % NBP], (c / NBP) & 1)) break;
                if (!wait_or_abort(F8 ? &vconv[c % NOB] : &vfull[c % NV], F8 ? (c / NOB) & 1 : (c / NV) & 1)) break;
                tc5::fence_after_sync();
                const uint8_t *vt = vring + (c % NV) * C::kStageBytes;
                const uint8_t *pt = ps + (c % NBP) * C::kPBufBytes;
#pragma unroll
                for (int j = 0; j < kTcRows / 16; ++j) {  // K = 16 rows of P^T per MMA
                    const uint64_t bdesc =
                        C::kPMn ? tc5::sw128_desc(pt + j * 16 * kSubBytes, C::kSubTile, 1024)
                                : tc5::sw128_desc(pt + (j >> 2) * (2 * N * kSubBytes) + (j & 3) * 32, 16, 1024);
                    if constexpr (F8)  // A: V^T widened into TMEM, 16 rows of P^T = 8 columns
                        tc5::mma_f16_tmem_a(tmem + C::kColO, tmem + C::kColV + 64 * (c % NOB) + 8 * j, bdesc,
                                            kIdPV, c > 0 || j > 0);
                    else
                        tc5::mma_bf16(tmem + C::kColO, tc5::sw128_desc(vt + j * 16 * kSubBytes, C::kSubTile, 1024),
                                      bdesc, kIdPV, c > 0 || j > 0);
                }
                tc5::commit(&pfree[c % NBP]);
                tc5::commit(F8 ? &vopfree[c % NOB] : &vempty[c % NV]);
                done = c + 1;
            }
            if (*abort_flag && done > 0) {
                tc5::commit(&drain[1]);
                mbar_wait_bounded(&drain[1], 0);
            }
        }
    } else if (F8 && warp >= kTcCvtWarp) {
        // ================= FP8 converters: widen each chunk's e4m3 codes into TMEM =================
        // Warp 8 + q4 writes TMEM lanes 32 q4 .. 32 q4 + 31 of both operand
        // buffers (c % NOB) of chunk c:
        //   K (QK's A): lane m = row m of the chunk, column d / 2 = fp16 pair
        //     (d, d + 1): thread = row, its 128 codes read whole.
        //   V^T (PV's A): lane L holds head dim vt_dim(L) of the V rows, column
        //     = pair of rows, in the order that transposed 8 x 8 loads of byte
        //     pairs and 16-lane stores give (vt_row_k maps row m to its index
        //     along the contraction; the P^T rows follow the same order).
        //   Rows the V producer did not load, or past the range, widen to zeros,
        //   so 0 * (stale bytes) never reaches O^T.
        // An operand buffer is rewritten once the MMAs of chunk c - NOB have read
        // it; the code stage is released once its codes are widened.  The
        // passes are loops, not unrolled: the warp roles of a CTA run different
        // code at once, and compact loops stay in the instruction cache.
        const int q4 = warp & 3;
        const bool do_k = C::kCvtWarps == 4 || warp < kTcCvtWarp + 4;
        const bool do_v = C::kCvtWarps == 4 || warp >= kTcCvtWarp + 4;
        const int m = 32 * q4 + lane;  // this thread's K row
        for (int c = 0; c < nch; ++c) {
            const int ob = c % NOB;
            // ---- K: 32 columns (64 codes of row m) per pass ----
            if (do_k) {
                if (!wait_or_abort(&kfull[c % NK], (c / NK) & 1)) break;
                if (c >= NOB && !wait_or_abort(&kopfree[ob], ((c / NOB) - 1) & 1)) break;
                tc5::fence_after_sync();
                const uint8_t *krow = kring + (c % NK) * C::kStageBytes + m * kSubBytes;
                const uint32_t kcol = tc5::taddr(tmem, 32 * q4, C::kColK + 64 * ob);
#pragma unroll 1
                for (int hf = 0; hf < 2; ++hf) {
                    uint32_t w[32];
#pragma unroll
                    for (int j = 0; j < 4; ++j) {  // codes 16 (4 hf + j) .. + 15 -> columns 8 (4 hf + j) ..
                        uint4 a, b;
                        e4m3x16_to_f16(*reinterpret_cast<const uint4 *>(krow + (((4 * hf + j) ^ (m & 7)) << 4)), a, b);
                        w[8 * j + 0] = a.x, w[8 * j + 1] = a.y, w[8 * j + 2] = a.z, w[8 * j + 3] = a.w;
                        w[8 * j + 4] = b.x, w[8 * j + 5] = b.y, w[8 * j + 6] = b.z, w[8 * j + 7] = b.w;
                    }
                    tc5::st_32x32b_x32_nowait(kcol + 32 * hf, w);
                }
                __syncwarp();  // the stage's codes are read (the stores took them)
                if (lane == 0) mbar_arrive(&kempty[c % NK]);
                tc5::wait_st();
                tc5::fence_before_sync();
                __syncwarp();
                if (lane == 0) mbar_arrive(&kconv[ob]);
            }

            // ---- V^T: 16 dims x 128 rows (four transposed 4-matrix loads) per pass ----
            if (!do_v) continue;
            uint64_t mk = 0;
            {  // the V producer wrote chunk c's mask before its loads
                uint32_t i = 0;
                const uint64_t t0 = globaltimer_ns();
                for (; i < kWaitLimit; ++i) {
                    mk = vmask_ring[c % C::kMaskRing];
                    if (static_cast<uint32_t>(mk >> 32) == static_cast<uint32_t>(c) || *abort_flag) break;
                    if (wait_expired(i, t0)) {
                        i = kWaitLimit;
                        break;
                    }
                }
                if (static_cast<uint32_t>(mk >> 32) != static_cast<uint32_t>(c)) {
                    if (i == kWaitLimit) {
                        *abort_flag = 1;
                        set_status(p.status, PA_STATUS_TIMEOUT);
                    }
                    break;
                }
            }
            if (!wait_or_abort(&vfull[c % NV], (c / NV) & 1)) break;
            if (c >= NOB && !wait_or_abort(&vopfree[ob], ((c / NOB) - 1) & 1)) break;
            tc5::fence_after_sync();
            const uint32_t vm = static_cast<uint32_t>(mk);
            const int tok_c = t_begin + c * C::kT;
            constexpr uint32_t kAllTiles = 0x55555555u & ((1u << (2 * C::kTiles)) - 1u);
            const bool whole = (vm & kAllTiles) == kAllTiles && tok_c + C::kT <= t_end;
            // pass u: dims 16 dc .. 16 dc + 15 (dc = 2 q4 + u); load k takes row groups
            // g = 2 k, 2 k + 1, lane t giving the address of row t % 8 of matrix
            // t / 8 = 2 (g - 2 k) + h (rows 16 g + 8 h .. + 7)
            const int mi = lane >> 3, r8 = lane & 7;
            const uint32_t vsrc = smem_u32(vring + (c % NV) * C::kStageBytes) +
                                  (16 * (mi >> 1) + 8 * (mi & 1) + r8) * kSubBytes;
            const uint32_t vcol = tc5::taddr(tmem, 32 * q4, C::kColV + 64 * ob);
#pragma unroll 1
            for (int u = 0; u < 2; ++u) {
                uint32_t w[32];
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    uint32_t r[4];
                    ldsm_x4_trans(vsrc + 32 * k * kSubBytes + (((2 * q4 + u) ^ r8) << 4), r);
#pragma unroll
                    for (int gg = 0; gg < 2; ++gg) {
                        // lane t holds rows 16 g + 8 h + 2 (t % 4) and + 1 of dims 16 dc + 2 (t / 4) and + 1
                        const uint2 a = e4m3x4_to_f16x4(__byte_perm(r[2 * gg], 0u, 0x3120));      // h = 0
                        const uint2 b = e4m3x4_to_f16x4(__byte_perm(r[2 * gg + 1], 0u, 0x3120));  // h = 1
                        uint32_t ka = 0xffffffffu, kb = 0xffffffffu;
                        if (!whole) {
                            const int tl = (2 * k + gg) / HC;
                            const bool tile_ok = (vm >> (2 * tl)) & 1u;
                            const int r0 = tok_c + tl * kTile + 2 * (lane & 3);
                            ka = (tile_ok && r0 < t_end ? 0x0000ffffu : 0u) | (tile_ok && r0 + 1 < t_end ? 0xffff0000u : 0u);
                            kb = (tile_ok && r0 + 8 < t_end ? 0x0000ffffu : 0u) | (tile_ok && r0 + 9 < t_end ? 0xffff0000u : 0u);
                        }
                        // repetition g = 2 k + gg of the store: columns 8 g + 2 (t % 4) (+ 1)
                        w[8 * k + 4 * gg + 0] = a.x & ka;  // dim 2 (t / 4): lane t / 4, rows of h = 0
                        w[8 * k + 4 * gg + 1] = b.x & kb;  //               rows of h = 1
                        w[8 * k + 4 * gg + 2] = a.y & ka;  // dim 2 (t / 4) + 1: lane t / 4 + 8
                        w[8 * k + 4 * gg + 3] = b.y & kb;
                    }
                }
                tc5::st_16x256b_x8_nowait(vcol + ((16 * u) << 16), w);
            }
            __syncwarp();  // the stage's codes are read
            if (lane == 0) mbar_arrive(&vempty[c % NV]);
            tc5::wait_st();
            tc5::fence_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive(&vconv[ob]);
        }
    } else {
        // ================= softmax warps: thread = row m of a chunk, and output dim d =================
        const int my_head = (tid >> 4) % HC;                // head of row m = tid
        float l_thr[GP];
#pragma unroll
        for (int q = 0; q < GP; ++q) l_thr[q] = 0.f;
        const float sl2 = p.scale_log2;
        bool dead = false;
        const int my_tile = tid / (kTile * HC);              // tile of row m = tid
        const int my_tok = my_tile * kTile + (tid & 15);     // its token's offset in a chunk
        // The 16-row groups of warp w's rows are heads (2 w) % HC (lanes 0-15)
        // and that + 1 (lanes 16-31): the warp loads those two heads' GP
        // columns of S, each lane keeps its own.
        const int head_a = HC == 1 ? 0 : (2 * warp) % HC;
        // this row's head's reference maxima (m_ref only moves after a vote)
        float mr[GP];
#pragma unroll
        for (int q = 0; q < GP; ++q) mr[q] = -INFINITY;
        for (int c = 0; c < nch; ++c) {
            const int sbuf = c % NBS, pbuf = c % NBP;
            bool ok = wait_or_abort(&sdone[sbuf], (c / NBS) & 1);
            // the K producer wrote chunk c's mask before its loads, hence before S c
            uint64_t mk = 0;
            if (ok) {
                uint32_t i = 0;
                const uint64_t t0 = globaltimer_ns();
                for (; i < kWaitLimit; ++i) {
                    mk = mask_ring[c % C::kMaskRing];
                    if (static_cast<uint32_t>(mk >> 32) == static_cast<uint32_t>(c) || *abort_flag) break;
                    if (wait_expired(i, t0)) {
                        i = kWaitLimit;
                        break;
                    }
                }
                if (static_cast<uint32_t>(mk >> 32) != static_cast<uint32_t>(c)) {
                    ok = false;
                    if (i == kWaitLimit) {
                        *abort_flag = 1;
                        set_status(p.status, PA_STATUS_TIMEOUT);
                    }
                }
            }
            ok = __all_sync(0xffffffffu, ok);
            const bool in_pool =
                t_begin + c * C::kT + my_tok < t_end && ((static_cast<uint32_t>(mk) >> (2 * my_tile)) & 1u);
            float sv[GP];  // this row's head's GP scores
            if (ok) {
                tc5::fence_after_sync();
                const uint32_t scol = tc5::taddr(tmem, 32 * warp, sbuf * N + head_a * GP);
                if constexpr (GP >= 16) {
                    static_assert(HC == 1 || GP == 16, "S columns");
                    uint32_t ra[GP], rb[HC == 1 ? 1 : GP];
#pragma unroll
                    for (int k = 0; k < GP / 16; ++k)
                        tc5::ld_32x32b_x16_nowait(scol + 16 * k, *reinterpret_cast<uint32_t(*)[16]>(&ra[16 * k]));
                    if constexpr (HC > 1) tc5::ld_32x32b_x16_nowait(scol + GP, *reinterpret_cast<uint32_t(*)[16]>(&rb[0]));
                    tc5::wait_ld();
#pragma unroll
                    for (int q = 0; q < GP; ++q)
                        sv[q] = __uint_as_float(HC == 1 || lane < 16 ? ra[q] : rb[HC == 1 ? 0 : q]);
                } else {
                    uint32_t ra[GP], rb[GP];
                    tc5::ld_32x32b_nowait<GP>(scol, ra);
                    tc5::ld_32x32b_nowait<GP>(scol + GP, rb);
                    tc5::wait_ld();
#pragma unroll
                    for (int q = 0; q < GP; ++q) sv[q] = __uint_as_float(lane < 16 ? ra[q] : rb[q]);
                }
            }
            tc5::fence_before_sync();
            __syncwarp();  // (one arrival per warp, once all its lanes have read)
            if (lane == 0) mbar_arrive(&sfree[sbuf]);  // S buffer read: QK c + NBS may overwrite it
            const bool valid = ok && in_pool;
            // causal: column q (query qi0 + q / G) sees this row's token only if
            // the token is not past the query's position
            const int cmin = max(0, t_begin + c * C::kT + my_tok - qbase) * G;
            float sc[GP];
            bool over = false;
#pragma unroll
            for (int q = 0; q < GP; ++q) {
                sc[q] = (valid && q < Gq && q >= cmin) ? sv[q] * sl2 : -INFINITY;
                over |= sc[q] > mr[q] + kTcLazyTau;
            }
            // one vote per chunk: does any reference max have to move (or is the CTA aborting)?
            const bool bad = !ok || *abort_flag != 0;
            if (named_sync_or(1, 128, over || bad)) {
                if (named_sync_or(1, 128, bad)) {
                    dead = true;
                    break;
                }
                // chunk max of every column (head, q) over that head's rows, via shared memory
#pragma unroll
                for (int q = 0; q < GP; ++q) red[tid * C::kGPr + q] = sc[q];
                named_sync(1, 128);
                if (tid < N) {
                    const float cm = column_reduce<HC, GP, C::kGPr, true>(red, tid);
                    const float old = m_ref[tid];
                    const float mn = fmaxf(old, cm);
                    alpha_s[tid] = (mn == -INFINITY) ? 1.f : fast_exp2(old - mn);
                    m_ref[tid] = mn;
                }
                named_sync(1, 128);
#pragma unroll
                for (int q = 0; q < GP; ++q) {
                    mr[q] = m_ref[my_head * GP + q];
                    l_thr[q] *= alpha_s[my_head * GP + q];
                }
                if (c >= 1) {  // O^T (all chunks so far) is rescaled once PV c-1 is done
                    bool ok3 = wait_or_abort(&pfree[(c - 1) % NBP], ((c - 1) / NBP) & 1);
                    if (__all_sync(0xffffffffu, ok3)) {
                        tc5::fence_after_sync();
#pragma unroll 1
                        for (int k = 0; k < 2 * N / 16; ++k) {  // hi and lo parts
                            float ov[16];
                            const uint32_t ta = tc5::taddr(tmem, 32 * warp, C::kColO + 16 * k);
                            tc5::ld_32x32b_x16(ta, ov);
                            const float *al = alpha_s + 16 * (k % (N / 16));
#pragma unroll
                            for (int i = 0; i < 16; ++i) ov[i] *= al[i];
                            tc5::st_32x32b_x16(ta, ov);
                        }
                    }
                }
                named_sync(1, 128);  // alpha_s / red read by all before any later reuse
            }
            // p = hi + lo, both bf16 (the PV MMA takes bf16 operands): the pair
            // carries p to about 2^-17 relative, where hi alone would be 2^-9
            // bf16 (fp16 with FP8 pools) bit patterns, two columns per word
            uint32_t hw[GP / 2], lw[GP / 2];
#pragma unroll
            for (int q = 0; q < GP; q += 2) {  // two columns per packed conversion
                const float p0 = sc[q] != -INFINITY ? fast_exp2(sc[q] - mr[q]) : 0.f;
                const float p1 = sc[q + 1] != -INFINITY ? fast_exp2(sc[q + 1] - mr[q + 1]) : 0.f;
                const uint32_t hi = p16x2_bits<F8>(p0, p1);
                const float h0 = p16_value<F8>(static_cast<uint16_t>(hi));
                const float h1 = p16_value<F8>(static_cast<uint16_t>(hi >> 16));
                const uint32_t lo = p16x2_bits<F8>(p0 - h0, p1 - h1);
                hw[q / 2] = hi;
                lw[q / 2] = lo;
                l_thr[q] += h0 + p16_value<F8>(static_cast<uint16_t>(lo));
                l_thr[q + 1] += h1 + p16_value<F8>(static_cast<uint16_t>(lo >> 16));
            }
            if (c >= NBP) wait_or_abort(&pfree[pbuf], ((c / NBP) - 1) & 1);  // PV c - NBP done
            // row k of P^T along the PV contraction: row m = tid (FP8: in the
            // order of the widened V^T's columns)
            const int prow = F8 ? vt_row_k(tid) : tid;
            if constexpr (C::kPMn) {
                // row k of P^T, this row's own head's columns (hi, then lo at
                // N + n); the other heads' columns stay zero
                uint8_t *row = ps + pbuf * C::kPBufBytes + prow * kSubBytes;
                auto at = [&](int n) -> uint32_t {  // byte offset of column n of the row
                    return (n >> 6) * C::kSubTile + ((((n & 63) >> 3) ^ (prow & 7)) << 4) + (n & 7) * 2;
                };
                const int n0 = my_head * GP;
                if constexpr (GP >= 8) {
#pragma unroll
                    for (int g = 0; g < GP / 8; ++g) {
                        *reinterpret_cast<uint4 *>(row + at(n0 + 8 * g)) =
                            make_uint4(hw[4 * g], hw[4 * g + 1], hw[4 * g + 2], hw[4 * g + 3]);
                        *reinterpret_cast<uint4 *>(row + at(N + n0 + 8 * g)) =
                            make_uint4(lw[4 * g], lw[4 * g + 1], lw[4 * g + 2], lw[4 * g + 3]);
                    }
                } else {  // GP = 4: half a chunk
                    *reinterpret_cast<uint2 *>(row + at(n0)) = make_uint2(hw[0], hw[1]);
                    *reinterpret_cast<uint2 *>(row + at(N + n0)) = make_uint2(lw[0], lw[1]);
                }
            } else {
                // P^T[n][k] for this row's own head block; the other heads' columns stay zero
                uint8_t *pt = ps + pbuf * C::kPBufBytes + (prow >> 6) * (2 * N * kSubBytes);
                const int tt = prow & 63;
#pragma unroll
                for (int q = 0; q < GP; ++q) {
                    const int n = my_head * GP + q;   // lo row N + n swizzles as n (N % 8 == 0)
                    const uint32_t at = n * kSubBytes + (((tt >> 3) ^ (n & 7)) << 4) + (tt & 7) * 2;
                    const uint32_t sh = (q & 1) * 16;
                    *reinterpret_cast<uint16_t *>(pt + at) = static_cast<uint16_t>(hw[q / 2] >> sh);
                    *reinterpret_cast<uint16_t *>(pt + N * kSubBytes + at) = static_cast<uint16_t>(lw[q / 2] >> sh);
                }
            }
            // an invalid row zeroes its V row, so 0 * (stale or NaN) never reaches O^T
            // (with FP8 pools the V converter writes those rows as zeros)
            if (!F8 && !valid && wait_or_abort(&vfull[c % NV], (c / NV) & 1)) {
                uint8_t *vrow = vring + (c % NV) * C::kStageBytes + tid * kSubBytes;
#pragma unroll
                for (int sub = 0; sub < 2; ++sub)
#pragma unroll
                    for (int k = 0; k < 8; ++k)
                        *reinterpret_cast<uint4 *>(vrow + sub * C::kSubTile + k * 16) =
                            make_uint4(0u, 0u, 0u, 0u);
            }
            fence_proxy_async_smem();
            tc5::fence_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive(&pready[pbuf]);
        }

        // ---- epilogue: row sums, O^T, normalise, store ----------------------------------
        // The row sums are final once the last chunk's p is written, so they are
        // reduced (through shared memory) while its PV still runs.
#pragma unroll
        for (int q = 0; q < GP; ++q) red[tid * C::kGPr + q] = l_thr[q];
        named_sync(1, 128);
        if (tid < N) {  // row sum of column n, its reciprocal (alpha_s is free now), its row
            const float lsum = column_reduce<HC, GP, C::kGPr, false>(red, tid);
            col[tid] = lsum;
            alpha_s[tid] = lsum > 0.f ? p.v_scale / lsum : 0.f;  // 0: no key seen (causal)
            const int c = tid % GP;
            rel_s[tid] = c < Gq ? static_cast<int>(col_row(tid / GP, c) - row0) : -1;
        }
        bool okf = !dead && wait_or_abort(&pfree[(nch - 1) % NBP], ((nch - 1) / NBP) & 1);
        // (this barrier also publishes col[], alpha_s and rel_s)
        okf = named_sync_or(1, 128, !okf) ? false : true;
        if (okf) {
            tc5::fence_after_sync();
            // O^T row d = tid, 16 columns at a time, normalised and staged in the
            // idle P^T buffers as rows ostage[n][d] (fp32 partials when split,
            // else bf16), column n = (head hh, query q) being output row
            // row0 + rel_s[n].  The cluster merge reads the stage in place;
            // otherwise each column's row is copied out by one bulk copy.
            // (FP8: lane tid of O^T is head dim vt_dim(tid))
            const bool split = p.split != 0;
            float *ostage0 = reinterpret_cast<float *>(ps);
            __nv_bfloat16 *ostage16_0 = reinterpret_cast<__nv_bfloat16 *>(ps);
            float *ostage = ostage0 + (F8 ? vt_dim(tid) : tid);
            __nv_bfloat16 *ostage16 = ostage16_0 + (F8 ? vt_dim(tid) : tid);
#pragma unroll 1
            for (int k = 0; k < N / 16; ++k) {
                float ov[16], lo[16], al[16];
                int rel[16];
#pragma unroll
                for (int i = 0; i < 16; ++i) {  // the columns' rows and scales, ahead of the stores
                    rel[i] = rel_s[16 * k + i];
                    al[i] = alpha_s[16 * k + i];
                }
                tc5::ld_32x32b_x16(tc5::taddr(tmem, 32 * warp, C::kColO + 16 * k), ov);
                tc5::ld_32x32b_x16(tc5::taddr(tmem, 32 * warp, C::kColO + N + 16 * k), lo);
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                    if (rel[i] < 0) continue;
                    const float o = (ov[i] + lo[i]) * al[i];
                    if (split) ostage[(16 * k + i) * D] = o;
                    else ostage16[(16 * k + i) * D] = __float2bfloat16_rn(o);
                }
            }
            const bool copy_out = !p.cluster_merge;
            if (copy_out) {  // the stage is complete before any row of it is copied
                fence_proxy_async_smem();
                named_sync(1, 128);
            }
            if (tid < N && rel_s[tid] >= 0) {
                const int n = tid;
                const float lse = (m_ref[n] + log2f(col[n])) * 0.69314718055994531f;
                const int64_t r = row0 + rel_s[n];
                if (p.cluster_merge) {
                    col[n] = lse;
                } else if (split) {
                    const int64_t slot = r * p.part_stride + p.part_offset + part;
                    bulk_store_s2g(p.part_o + slot * D, ostage0 + n * D, D * 4);
                    bulk_commit();
                    p.part_lse[slot] = lse;
                    bulk_wait_all();              // the row is written ...
                    fence_proxy_async_global();   // ... and ordered before the merge's release
                } else {
                    bulk_store_s2g(static_cast<__nv_bfloat16 *>(p.out) + r * D, ostage16_0 + n * D, D * 2);
                    bulk_commit();
                    if (p.lse) p.lse[r] = lse;
                    bulk_wait_all_read();  // the stage is read before the CTA moves on
                }
            }
        } else if (p.cluster_merge && tid < N) {
            col[tid] = -INFINITY;  // aborted: this partition drops out of the merge
        }
    }
    tc5::fence_before_sync();
    __syncthreads();
    if (warp == 0) tc5::tmem_free(tmem, C::kTmemCols);
    if (p.cluster_merge)  // all warps of all the cluster's CTAs share the merge
        merge_cluster<D, kThreads>(p, reinterpret_cast<const float *>(ps), col, rel_s, N, row0, tid);
    else if (p.split)  // all eight warps share the merge
        merge_split_group<D, kThreads / 32>(p, b * gridDim.y + blockIdx.y, part, row0, HC * Gq,
                                              HC * G, Hq, ticket, tid, [] { __syncthreads(); },
                                              reinterpret_cast<float *>(ps));
}

template <int HC, int GP, bool F8>
cudaError_t launch_tc_instance(const CUtensorMap &kmap, const CUtensorMap &vmap,
                               const DecodeParams &p, int B, int G, cudaStream_t stream) {
    using C = TcCfg<HC, GP, F8>;
    auto kern = decode_tc_kernel<HC, GP, F8>;
    static std::atomic<uint64_t> smem_attr_done{0};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const uint64_t bit = 1ull << (dev & 63);
    if (!(smem_attr_done.load(std::memory_order_acquire) & bit)) {
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
        if (e != cudaSuccess) return e;
        smem_attr_done.fetch_or(bit, std::memory_order_release);
    }
    const int qgroups = (p.q_len + p.q_per_cta - 1) / p.q_per_cta;
    const dim3 grid(p.num_splits, p.head_groups * qgroups, B);
    const int threads = C::kThreads;
    if (p.cluster_merge) {
        // One cluster per (sequence, head group, query group), all resident at
        // once (a second wave of clusters would cost more than the merge saves).
        static std::atomic<int> cap[64 * 32];
        const int64_t clusters = static_cast<int64_t>(grid.y) * grid.z;
        if (p.num_splits >= 2 && p.num_splits <= kMaxClusterMerge &&
            clusters <= max_active_clusters(kern, p.num_splits, threads, C::kSmemBytes, dev, cap))
            return launch_clustered(kern, grid, p.num_splits, threads, C::kSmemBytes, stream, p.pdl != 0,
                                    kmap, vmap, p, G);
        DecodeParams q = p;  // merge through global memory instead
        q.cluster_merge = 0;
        return launch_maybe_cooperative(kern, grid, threads, C::kSmemBytes, stream, q.counters != nullptr,
                                        q.pdl != 0, kmap, vmap, q, G);
    }
    return launch_maybe_cooperative(kern, grid, threads, C::kSmemBytes, stream, p.counters != nullptr,
                                    p.pdl != 0, kmap, vmap, p, G);
}

}  // namespace pa
