// C ABI of libpagedattn (declared in include/pa.h): host-side argument
// checks, TMA descriptor encoding, split-count policy and kernel dispatch.
// Nothing here allocates device memory or synchronises the stream.
#include <cudaTypedefs.h>

#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdint>
#include <cstdlib>
#include <cstring>
#include <mutex>

#include "pa_internal.h"

namespace pa {
cudaError_t launch_decode_cc_d64(int G, const CUtensorMap &kmap, const CUtensorMap &vmap,
                                 const DecodeParams &p, int B, cudaStream_t stream);
cudaError_t launch_decode_cc_d128(int G, const CUtensorMap &kmap, const CUtensorMap &vmap,
                                  const DecodeParams &p, int B, cudaStream_t stream);

cudaError_t launch_decode_tc(int HC, int GP, int G, const CUtensorMap &kmap,
                             const CUtensorMap &vmap, const DecodeParams &p, int B,
                             cudaStream_t stream);
cudaError_t launch_decode_tc_f8(int HC, int GP, int G, const CUtensorMap &kmap,
                                const CUtensorMap &vmap, const DecodeParams &p, int B,
                                cudaStream_t stream);

cudaError_t launch_decode_cc(int D, int G, const CUtensorMap &kmap, const CUtensorMap &vmap,
                             const DecodeParams &p, int B, cudaStream_t stream) {
    if (D == 128) return launch_decode_cc_d128(G, kmap, vmap, p, B, stream);
    if (D == 64) return launch_decode_cc_d64(G, kmap, vmap, p, B, stream);
    return cudaErrorInvalidValue;
}

}  // namespace pa

namespace {

constexpr int kMaxGroupCc = 8;    // query heads per KV head, CUDA-core kernel
constexpr int kMaxGroupTc = 32;   // MMA columns per KV head (query heads x positions), tensor cores
constexpr int kMaxGridZ = 65535;  // sequences per launch (gridDim.z)
constexpr int kMinTilesPerSplit = 2;  // 32 tokens: one MMA chunk of four KV heads
constexpr int kNarrowMergeSplits = 32;  // partitions the one-warp-per-task merge holds
constexpr int kMultiWaveTiles = 48;   // tiles per partition of a batch that takes several waves
constexpr int64_t kMaxRowsQ = 1 << 24;  // B x q_len of one multi-query call
constexpr int kMaxSplits = 256;
constexpr int PA_ETOOLARGE = -100;  // internal: the cooperative grid does not fit at once


enum class Kernel { kCudaCore, kTensorCore };

// Resident decode CTAs per SM (shared memory bound): 2 for the CUDA-core
// kernel (~104 KB each), 1 for the tensor-core kernel (~210 KB).
int ctas_per_sm(Kernel k) { return k == Kernel::kTensorCore ? 1 : 2; }

int next_pow2(int x) {
    int p = 1;
    while (p < x) p <<= 1;
    return p;
}

// Shape of the tensor-core kernel for Hkv KV heads of G columns each (query
// heads, times query positions for multi-query calls): HC KV heads share a
// CTA (a power of two dividing Hkv, at most 8: a chunk is 128 rows = 128 / HC
// tokens x HC heads) and every head's columns are padded to GP, with HC * GP
// (the MMA N) between 16 and 64; more than 16 columns take a CTA per head.
bool tc_shape(int G, int Hkv, int *HC, int *GP) {
    if (G < 1 || G > kMaxGroupTc || Hkv < 1) return false;
    int hc = 1;
    while (hc < 8 && Hkv % (hc * 2) == 0) hc *= 2;
    if (G > 16) hc = 1;
    int gp = 1;
    for (;;) {
        gp = next_pow2(G);
        if (gp * hc < 16) gp = 16 / hc;
        if (gp * hc <= 64) break;
        hc /= 2;
    }
    *HC = hc;
    *GP = gp;
    return true;
}

// CTAs per split of the decode grid: one per (sequence, KV head) for the
// CUDA-core kernel, one per (sequence, group of HC KV heads) for the
// tensor-core kernel.
int64_t units_per_split(Kernel k, int B, int G, int Hkv, int qpc = 1, int qgroups = 1) {
    if (k == Kernel::kTensorCore) {
        int hc = 1, gp = 1;
        tc_shape(G * qpc, Hkv, &hc, &gp);
        return static_cast<int64_t>(B) * (Hkv / hc) * qgroups;
    }
    return static_cast<int64_t>(B) * Hkv;
}

// Process-wide switches (pa_set_option), each initialised once from its
// environment variable the first time any of them is read.
std::atomic<int> g_options[4];
std::once_flag g_options_once;

int option(int which) {
    std::call_once(g_options_once, [] {
        const char *k = std::getenv("PA_DECODE_KERNEL");
        g_options[PA_OPT_DECODE_KERNEL].store(
            k && std::strcmp(k, "cuda_core") == 0     ? PA_KERNEL_CUDA_CORE
            : k && std::strcmp(k, "tensor_core") == 0 ? PA_KERNEL_TENSOR_CORE
                                                      : PA_KERNEL_AUTO);
        const char *m = std::getenv("PA_SPLIT_MERGE");
        g_options[PA_OPT_SPLIT_MERGE].store(m && std::strcmp(m, "grid") == 0 ? PA_MERGE_GRID
                                                                            : PA_MERGE_AUTO);
        const char *d = std::getenv("PA_PDL");
        g_options[PA_OPT_PDL].store(d && std::strcmp(d, "0") == 0 ? 0 : 1);
        const char *cs = std::getenv("PA_CASCADE");
        g_options[PA_OPT_CASCADE].store(cs && std::strcmp(cs, "always") == 0  ? PA_CASCADE_ALWAYS
                                        : cs && std::strcmp(cs, "never") == 0 ? PA_CASCADE_NEVER
                                                                              : PA_CASCADE_AUTO);
    });
    return g_options[which].load(std::memory_order_relaxed);
}

// Which decode kernel runs for a GQA group of G heads of dimension D.  The
// tensor-core kernel needs D = 128 and G <= 32; the CUDA-core kernel takes
// D in {64, 128} and G <= 8.  By default the tensor cores take every shape
// they can; the PA_OPT_DECODE_KERNEL option can force one of them (a shape the
// forced kernel cannot run is rejected).
int pick_kernel(int G, int D, Kernel *k) {
    const bool tc_ok = D == 128 && G >= 1 && G <= kMaxGroupTc;
    const bool cc_ok = (D == 64 || D == 128) && G >= 1 && G <= kMaxGroupCc;
    const int forced = option(PA_OPT_DECODE_KERNEL);
    if (forced == PA_KERNEL_CUDA_CORE) {
        if (!cc_ok) return PA_EUNSUPPORTED;
        *k = Kernel::kCudaCore;
        return PA_OK;
    }
    if (forced == PA_KERNEL_TENSOR_CORE) {
        if (!tc_ok) return PA_EUNSUPPORTED;
        *k = Kernel::kTensorCore;
        return PA_OK;
    }
    if (tc_ok) {
        *k = Kernel::kTensorCore;
        return PA_OK;
    }
    if (cc_ok) {
        *k = Kernel::kCudaCore;
        return PA_OK;
    }
    return PA_EUNSUPPORTED;
}

// How the partitions of an in-launch split merge meet: by default the
// tensor-core kernel makes the P CTAs of a (sequence, head group) one
// thread-block cluster when P <= 16 and all the launch's clusters can be
// resident at once, and merges through distributed shared memory; otherwise
// (and with PA_OPT_SPLIT_MERGE = PA_MERGE_GRID) the grid is launched
// cooperatively and the partials meet in global memory.
bool merge_forced_grid() { return option(PA_OPT_SPLIT_MERGE) == PA_MERGE_GRID; }

// The tensor-core kernel is launched with programmatic stream serialization
// (programmatic dependent launch) unless PA_OPT_PDL is 0: it may then become
// resident while the previous kernel in the stream finishes, and waits for it
// before touching global memory.
bool pdl_enabled() { return option(PA_OPT_PDL) != 0; }

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    std::call_once(g_encode_once, [] {
        void *fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    });
    return g_encode;
}

bool aligned(const void *p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

int64_t round_up(int64_t x, int64_t a) { return (x + a - 1) / a * a; }

// K or V pool [num_blocks, bs, Hkv, D] viewed as a 4-D tensor
// (64 elements, D/64 sub-rows, Hkv heads, num_blocks*bs token rows); one box
// is 16 token rows of one 64-element sub-row of one head, 128-byte swizzled.
int make_kv_map(CUtensorMap *map, const void *base, const pa_cache_desc &c) {
    auto enc = encode_fn();
    if (!enc) return PA_ECUDA;
    const cuuint64_t dims[4] = {64u, static_cast<cuuint64_t>(c.head_dim / 64),
                                static_cast<cuuint64_t>(c.num_kv_heads),
                                static_cast<cuuint64_t>(c.num_blocks) * c.block_size};
    const cuuint64_t strides[3] = {128u, static_cast<cuuint64_t>(c.head_dim) * 2,
                                   static_cast<cuuint64_t>(c.num_kv_heads) * c.head_dim * 2};
    const cuuint32_t box[4] = {64u, 1u, 1u, 16u};
    const cuuint32_t estr[4] = {1u, 1u, 1u, 1u};
    CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void *>(base), dims,
                     strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? PA_OK : PA_ECUDA;
}

// The same pool for the tensor-core kernel: a 4-D view (64 elements, token
// rows, heads, D/64 sub-rows) whose box is 16 token rows of HC heads of one
// 64-element sub-row; in shared memory the box is head-major, so a block's
// rows for all HC heads arrive in one copy.  (The head stride, D * 2 bytes, is
// smaller than the row stride: the dimensions are deliberately not in
// increasing stride order.)
int make_kv_map_heads(CUtensorMap *map, const void *base, const pa_cache_desc &c, int HC) {
    auto enc = encode_fn();
    if (!enc) return PA_ECUDA;
    const cuuint64_t dims[4] = {64u, static_cast<cuuint64_t>(c.num_blocks) * c.block_size,
                                static_cast<cuuint64_t>(c.num_kv_heads),
                                static_cast<cuuint64_t>(c.head_dim / 64)};
    const cuuint64_t strides[3] = {static_cast<cuuint64_t>(c.num_kv_heads) * c.head_dim * 2,
                                   static_cast<cuuint64_t>(c.head_dim) * 2, 128u};
    const cuuint32_t box[4] = {64u, 16u, static_cast<cuuint32_t>(HC), 1u};
    const cuuint32_t estr[4] = {1u, 1u, 1u, 1u};
    CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void *>(base), dims,
                     strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? PA_OK : PA_ECUDA;
}

// An FP8 pool (one-byte e4m3 codes) for the tensor-core kernel: a 3-D view
// (128 codes = one token row of one head, token rows, heads); one box is 16
// token rows of HC heads, head-major, 128-byte swizzled.
int make_kv_map_fp8(CUtensorMap *map, const void *base, const pa_cache_desc &c, int HC) {
    auto enc = encode_fn();
    if (!enc) return PA_ECUDA;
    const cuuint64_t dims[3] = {static_cast<cuuint64_t>(c.head_dim),
                                static_cast<cuuint64_t>(c.num_blocks) * c.block_size,
                                static_cast<cuuint64_t>(c.num_kv_heads)};
    const cuuint64_t strides[2] = {static_cast<cuuint64_t>(c.num_kv_heads) * c.head_dim,
                                   static_cast<cuuint64_t>(c.head_dim)};
    const cuuint32_t box[3] = {static_cast<cuuint32_t>(c.head_dim), 16u, static_cast<cuuint32_t>(HC)};
    const cuuint32_t estr[3] = {1u, 1u, 1u};
    CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void *>(base), dims, strides,
                     box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? PA_OK : PA_ECUDA;
}

int check_cache_desc(const pa_cache_desc &c) {
    if (c.num_blocks <= 0 || c.block_size <= 0 || c.num_kv_heads <= 0 || c.head_dim <= 0)
        return PA_EINVAL;
    if (c.head_dim != 64 && c.head_dim != 128) return PA_EUNSUPPORTED;
    if (c.block_size % 16 != 0) return PA_EUNSUPPORTED;
    if (static_cast<int64_t>(c.num_blocks) * c.block_size > INT32_MAX) return PA_EUNSUPPORTED;
    return PA_OK;
}

int check_decode_args(const void *q, const void *k_cache, const void *v_cache,
                      const pa_cache_desc &c, const int32_t *block_tables,
                      int32_t max_blocks_per_seq, const int32_t *seq_lens, int32_t B, int32_t Hq,
                      float scale) {
    if (B < 0) return PA_EINVAL;
    if (!q || !k_cache || !v_cache || !block_tables || !seq_lens) return PA_EINVAL;
    int rc = check_cache_desc(c);
    if (rc) return rc;
    if (Hq <= 0 || Hq % c.num_kv_heads != 0) return PA_EINVAL;
    Kernel k;
    rc = pick_kernel(Hq / c.num_kv_heads, c.head_dim, &k);
    if (rc) return rc;
    if (c.num_kv_heads > 65535) return PA_EUNSUPPORTED;
    if (B > kMaxGridZ) return PA_EUNSUPPORTED;
    if (max_blocks_per_seq <= 0) return PA_EINVAL;
    if (static_cast<int64_t>(max_blocks_per_seq) * c.block_size > (INT32_MAX / 2))
        return PA_EUNSUPPORTED;
    if (!aligned(q, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16) ||
        !aligned(block_tables, 4) || !aligned(seq_lens, 4))
        return PA_EINVAL;
    if (!std::isfinite(scale)) return PA_EINVAL;
    return PA_OK;
}

pa::DecodeParams base_params(const void *q, const pa_cache_desc &c, const int32_t *block_tables,
                             int32_t max_blocks, const int32_t *seq_lens, int32_t Hq, float scale,
                             int32_t *status) {
    pa::DecodeParams p{};
    p.q = static_cast<const uint16_t *>(q);
    p.block_tables = block_tables;
    p.seq_lens = seq_lens;
    p.status = status;
    p.num_blocks = c.num_blocks;
    p.block_size = c.block_size;
    p.num_kv_heads = c.num_kv_heads;
    p.num_q_heads = Hq;
    p.max_blocks = max_blocks;
    p.scale_log2 = scale * 1.4426950408889634f;
    p.q_len = 1;
    p.q_per_cta = 1;
    p.head_groups = c.num_kv_heads;
    p.v_scale = 1.f;
    p.k_scale = 1.f;
    p.causal = 1;
    p.seq_len_const = -1;
    p.seq_len_offset = 0;
    p.part_stride = 0;   // run_decode: the partition count
    p.part_offset = 0;
    p.table_stride = max_blocks;
    return p;
}

// Multi-query calls with more query columns per KV head than the decode
// kernel holds in one CTA (q_len * G > 32) run the prefill-shaped kernel,
// whose CTAs take 128 query rows each and read each KV block once per tile.
bool prefill_shape(int G, int q_len) {
    return q_len > 1 && static_cast<int64_t>(q_len) * G > kMaxGroupTc;
}
int prefill_positions_per_tile(int G) { return pa::kPrefillRows / G; }
int64_t prefill_tiles(int G, int q_len) {
    const int qpt = prefill_positions_per_tile(G);
    return (q_len + qpt - 1) / qpt;
}

// Query positions per tensor-core CTA for q_len queries of G heads each: as
// many as fit the kernel's column limit (G * positions <= 32).
int queries_per_cta(int G, int q_len) {
    if (q_len <= 1) return 1;
    return std::min(q_len, std::max(1, kMaxGroupTc / G));
}

int sm_count_current() {
    static std::atomic<int> cache[64];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return -1;
    if (dev >= 0 && dev < 64) {
        int v = cache[dev].load(std::memory_order_relaxed);
        if (v > 0) return v;
    }
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return -1;
    if (dev >= 0 && dev < 64) cache[dev].store(n, std::memory_order_relaxed);
    return n;
}

// Settings of one pass of a cascade decode (defaults: an ordinary call).
struct PassOpts {
    int32_t causal = 1;
    int32_t seq_len_const = -1;   // >= 0: every sequence has this length
    int32_t seq_len_offset = 0;   // subtracted from seq_lens[b]
    int32_t part_stride = 0;      // 0: the pass's own partition count
    int32_t part_offset = 0;
    int32_t table_stride = 0;     // 0: max_blocks
};

// Scales of FP8 (e4m3) pools: a stored code c means c * scale.
struct Fp8Scales {
    float k_scale, v_scale;
};

// This step's new K/V for the fused write of pa_decode_step (all null: none).
struct NewTokens {
    const void *k_new = nullptr;
    const void *v_new = nullptr;
    const int64_t *slot_mapping = nullptr;
};

int run_decode(bool split, void *out, float *lse, float *part_o, float *part_lse, const void *q,
               const void *k_cache, const void *v_cache, const pa_cache_desc &c,
               const int32_t *block_tables, int32_t max_blocks, const int32_t *seq_lens,
               int32_t B, int32_t Hq, float scale, int32_t P, int32_t *status,
               cudaStream_t stream, int32_t *counters = nullptr, const NewTokens &nt = NewTokens(),
               int32_t q_len = 1, const Fp8Scales *f8 = nullptr, const PassOpts &po = PassOpts()) {
    const int G = Hq / c.num_kv_heads;
    const int qpc = queries_per_cta(G, q_len);
    Kernel k;
    int rc = pick_kernel(G * qpc, c.head_dim, &k);
    if (rc) return rc;
    if ((q_len > 1 || f8) && k != Kernel::kTensorCore) return PA_EUNSUPPORTED;  // tensor cores only
    pa::DecodeParams p = base_params(q, c, block_tables, max_blocks, seq_lens, Hq, scale, status);
    p.q_len = q_len;
    p.q_per_cta = qpc;
    p.out = out;
    p.lse = lse;
    p.part_o = part_o;
    p.part_lse = part_lse;
    p.split = split ? 1 : 0;
    p.num_splits = P;
    p.part_stride = po.part_stride ? po.part_stride : P;
    p.part_offset = po.part_offset;
    p.causal = po.causal;
    p.seq_len_const = po.seq_len_const;
    p.seq_len_offset = po.seq_len_offset;
    if (po.table_stride) p.table_stride = po.table_stride;
    if ((po.table_stride || po.seq_len_const >= 0 || po.seq_len_offset || !po.causal ||
         po.part_offset) && k != Kernel::kTensorCore)
        return PA_EUNSUPPORTED;  // cascade passes: tensor cores only
    p.chunk = pa_partition_tokens(max_blocks, c.block_size, P);
    p.counters = counters;
    // (a cluster merges its own P partials only: not a pass that shares its
    // rows' partial slots with another pass)
    p.cluster_merge = split && counters && k == Kernel::kTensorCore && P >= 2 &&
                      P <= pa::kMaxClusterMerge && p.part_stride == P && !merge_forced_grid();
    p.pdl = k == Kernel::kTensorCore && pdl_enabled();
    p.k_new = static_cast<const uint16_t *>(nt.k_new);
    p.v_new = static_cast<const uint16_t *>(nt.v_new);
    p.slot_mapping = nt.slot_mapping;
    p.k_pool = static_cast<uint16_t *>(const_cast<void *>(k_cache));
    p.v_pool = static_cast<uint16_t *>(const_cast<void *>(v_cache));
    CUtensorMap kmap, vmap;
    cudaError_t e;
    if (k == Kernel::kTensorCore && !f8 && !nt.k_new && prefill_shape(G, q_len) &&
        p.chunk <= pa::kPrefillMaxTiles * 16) {
        // queries on the MMA's M side; split partials are merged by the combine kernel
        if (counters) return PA_ETOOLARGE;
        p.q_per_cta = prefill_positions_per_tile(G);
        p.cluster_merge = 0;
        if (prefill_tiles(G, q_len) * c.num_kv_heads > 65535) return PA_EUNSUPPORTED;
        rc = make_kv_map_heads(&kmap, k_cache, c, 1);
        if (!rc) rc = make_kv_map_heads(&vmap, v_cache, c, 1);
        if (rc) return rc;
        e = pa::launch_prefill_tc(kmap, vmap, p, B, G, stream);
    } else if (k == Kernel::kTensorCore) {
        int HC = 1, GP = 1;
        if (!tc_shape(G * qpc, c.num_kv_heads, &HC, &GP)) return PA_EUNSUPPORTED;
        p.head_groups = c.num_kv_heads / HC;
        if (static_cast<int64_t>(p.head_groups) * ((q_len + qpc - 1) / qpc) > 65535) return PA_EUNSUPPORTED;
        if (f8) {
            p.scale_log2 = scale * f8->k_scale * 1.4426950408889634f;
            p.v_scale = f8->v_scale;
            p.k_scale = f8->k_scale;
            rc = make_kv_map_fp8(&kmap, k_cache, c, HC);
            if (!rc) rc = make_kv_map_fp8(&vmap, v_cache, c, HC);
            if (rc) return rc;
            e = pa::launch_decode_tc_f8(HC, GP, G, kmap, vmap, p, B, stream);
        } else {
            rc = make_kv_map_heads(&kmap, k_cache, c, HC);
            if (!rc) rc = make_kv_map_heads(&vmap, v_cache, c, HC);
            if (rc) return rc;
            e = pa::launch_decode_tc(HC, GP, G, kmap, vmap, p, B, stream);
        }
    } else {
        rc = make_kv_map(&kmap, k_cache, c);
        if (!rc) rc = make_kv_map(&vmap, v_cache, c);
        if (rc) return rc;
        e = pa::launch_decode_cc(c.head_dim, G, kmap, vmap, p, B, stream);
    }
    if (e == cudaErrorCooperativeLaunchTooLarge && counters) return PA_ETOOLARGE;
    return e == cudaSuccess ? PA_OK : PA_ECUDA;
}

}  // namespace

extern "C" {

int pa_version(void) { return 200; }

int pa_set_option(int32_t which, int32_t value) {
    switch (which) {
        case PA_OPT_DECODE_KERNEL:
            if (value < PA_KERNEL_AUTO || value > PA_KERNEL_TENSOR_CORE) return PA_EINVAL;
            break;
        case PA_OPT_SPLIT_MERGE:
            if (value != PA_MERGE_AUTO && value != PA_MERGE_GRID) return PA_EINVAL;
            break;
        case PA_OPT_PDL:
            if (value != 0 && value != 1) return PA_EINVAL;
            break;
        case PA_OPT_CASCADE:
            if (value < PA_CASCADE_AUTO || value > PA_CASCADE_NEVER) return PA_EINVAL;
            break;
        default:
            return PA_EINVAL;
    }
    option(which);  // the environment's defaults first, so they cannot overwrite this
    g_options[which].store(value, std::memory_order_relaxed);
    return PA_OK;
}

int pa_get_option(int32_t which) {
    if (which < PA_OPT_DECODE_KERNEL || which > PA_OPT_CASCADE) return PA_EINVAL;
    return option(which);
}

const char *pa_strerror(int code) {
    switch (code) {
        case PA_OK: return "success";
        case PA_EINVAL: return "invalid argument (null or misaligned pointer, inconsistent sizes)";
        case PA_EUNSUPPORTED: return "unsupported shape (head_dim, block_size or GQA group size)";
        case PA_EWORKSPACE: return "split-KV workspace missing or too small";
        case PA_ECUDA: return "CUDA call or kernel launch failed";
        default: return "unknown error code";
    }
}

int pa_cache_write(const void *k_new, const void *v_new, const int64_t *slot_mapping,
                   int64_t n_tokens, void *k_cache, void *v_cache, pa_cache_desc cache,
                   int32_t *status, pa_stream_t stream) {
    if (n_tokens < 0) return PA_EINVAL;
    int rc = check_cache_desc(cache);
    if (rc) return rc;
    if (n_tokens == 0) return PA_OK;
    if (!k_new || !v_new || !slot_mapping || !k_cache || !v_cache) return PA_EINVAL;
    if (!aligned(k_new, 16) || !aligned(v_new, 16) || !aligned(k_cache, 16) ||
        !aligned(v_cache, 16) || !aligned(slot_mapping, 8))
        return PA_EINVAL;
    const int row_bytes = cache.num_kv_heads * cache.head_dim * 2;
    cudaError_t e = pa::launch_cache_write(
        k_new, v_new, slot_mapping, n_tokens, k_cache, v_cache,
        static_cast<int64_t>(cache.num_blocks) * cache.block_size, row_bytes, status, stream);
    return e == cudaSuccess ? PA_OK : PA_ECUDA;
}

int pa_decode(void *out, float *lse, const void *q, const void *k_cache, const void *v_cache,
              pa_cache_desc cache, const int32_t *block_tables, int32_t max_blocks_per_seq,
              const int32_t *seq_lens, int32_t B, int32_t Hq, float scale, int32_t *status,
              pa_stream_t stream) {
    int rc = check_decode_args(q, k_cache, v_cache, cache, block_tables, max_blocks_per_seq,
                               seq_lens, B, Hq, scale);
    if (rc) return rc;
    if (!out || !aligned(out, 16) || (lse && !aligned(lse, 4))) return PA_EINVAL;
    if (B == 0) return PA_OK;
    return run_decode(false, out, lse, nullptr, nullptr, q, k_cache, v_cache, cache, block_tables,
                      max_blocks_per_seq, seq_lens, B, Hq, scale, 1, status, stream);
}

int pa_partition_tokens(int32_t max_blocks_per_seq, int32_t block_size, int32_t num_splits) {
    if (max_blocks_per_seq <= 0 || block_size <= 0 || num_splits <= 0) return PA_EINVAL;
    const int64_t lmax = static_cast<int64_t>(max_blocks_per_seq) * block_size;
    const int64_t per = (lmax + num_splits - 1) / num_splits;
    return static_cast<int>(round_up(per, 16));
}

int pa_choose_num_splits(int32_t B, int32_t Hq, int32_t Hkv, int32_t D,
                         int32_t max_blocks_per_seq, int32_t block_size, int32_t sm_count) {
    return pa_choose_num_splits_mq(B, 1, Hq, Hkv, D, max_blocks_per_seq, block_size, sm_count);
}

int pa_choose_num_splits_mq(int32_t B, int32_t q_len, int32_t Hq, int32_t Hkv, int32_t D,
                            int32_t max_blocks_per_seq, int32_t block_size, int32_t sm_count) {
    if (B < 0 || q_len <= 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv != 0 || max_blocks_per_seq <= 0 ||
        block_size <= 0 || sm_count <= 0)
        return PA_EINVAL;
    if (B == 0) return 1;
    const int G = Hq / Hkv;
    const int qpc = queries_per_cta(G, q_len);
    Kernel k;
    int rc = pick_kernel(G * qpc, D, &k);
    if (rc) return rc;
    if (q_len > 1 && k != Kernel::kTensorCore) return PA_EUNSUPPORTED;
    const bool prefill = k == Kernel::kTensorCore && prefill_shape(G, q_len);
    const int64_t units = prefill ? static_cast<int64_t>(B) * Hkv * prefill_tiles(G, q_len)
                                  : units_per_split(k, B, G, Hkv, qpc, (q_len + qpc - 1) / qpc);
    const int64_t slots = static_cast<int64_t>(sm_count) * ctas_per_sm(k);
    const int64_t lmax = static_cast<int64_t>(max_blocks_per_seq) * block_size;
    const int64_t tiles = (lmax + 15) / 16;
    int64_t P = slots / units;  // largest P whose grid still fits one wave
    if (P < 1 && !prefill) {
        // More units than CTA slots: the grid runs in waves, and sequences of
        // different lengths end at different times.  Partitions of about 48
        // tiles even the waves out (a Qwen3 batch of 256 sequences of
        // U[129, 2048] tokens: 1.1x faster with 3 partitions than unsplit);
        // their partials are merged by a combine launch.
        P = (tiles + kMultiWaveTiles - 1) / kMultiWaveTiles;
    }
    const int64_t p_by_tiles = (tiles + kMinTilesPerSplit - 1) / kMinTilesPerSplit;
    if (P > p_by_tiles) P = p_by_tiles;
    // Past 32 partitions the in-launch merge gives each task several warps of
    // one CTA (about 1 us more per step); that pays only where partitions of
    // 4 tiles would already be more than 32 (one sequence of 4k tokens:
    // P = 128 beats 64), not where the smaller floor alone crosses the line
    // (one sequence of 2k tokens: P = 32 beats 64).
    const int64_t p_by_4_tiles = (tiles + 3) / 4;
    if (P > kNarrowMergeSplits && p_by_4_tiles <= kNarrowMergeSplits) P = kNarrowMergeSplits;
    if (P > kMaxSplits) P = kMaxSplits;
    if (P < 1) P = 1;
    // the prefill-shaped kernel keeps a partition's tiles in shared memory
    if (prefill) P = std::max<int64_t>(P, (tiles + pa::kPrefillMaxTiles - 1) / pa::kPrefillMaxTiles);
    // Drop partitions that the rounding of the chunk to whole tiles leaves empty.
    const int chunk = pa_partition_tokens(max_blocks_per_seq, block_size, static_cast<int>(P));
    P = (lmax + chunk - 1) / chunk;
    return static_cast<int>(P);
}

int pa_auto_num_splits(int32_t B, int32_t Hq, int32_t Hkv, int32_t D, int32_t max_blocks_per_seq,
                       int32_t block_size) {
    const int sms = sm_count_current();
    if (sms <= 0) return PA_ECUDA;
    return pa_choose_num_splits(B, Hq, Hkv, D, max_blocks_per_seq, block_size, sms);
}

size_t pa_splitkv_workspace_bytes(int32_t B, int32_t Hq, int32_t D, int32_t num_splits) {
    if (B <= 0 || Hq <= 0 || D <= 0 || num_splits <= 1) return 0;
    const int64_t rows = static_cast<int64_t>(B) * Hq * num_splits;
    return static_cast<size_t>(round_up(rows * D * 4, 256) + round_up(rows * 4, 256) +
                               round_up(static_cast<int64_t>(B) * Hq * 8, 256));
}

int pa_decode_partial(float *part_o, float *part_lse, const void *q, const void *k_cache,
                      const void *v_cache, pa_cache_desc cache, const int32_t *block_tables,
                      int32_t max_blocks_per_seq, const int32_t *seq_lens, int32_t B, int32_t Hq,
                      float scale, int32_t num_splits, int32_t *status, pa_stream_t stream) {
    int rc = check_decode_args(q, k_cache, v_cache, cache, block_tables, max_blocks_per_seq,
                               seq_lens, B, Hq, scale);
    if (rc) return rc;
    if (num_splits <= 0) return PA_EINVAL;
    if (num_splits > 65535) return PA_EUNSUPPORTED;
    if (!part_o || !part_lse || !aligned(part_o, 16) || !aligned(part_lse, 4)) return PA_EINVAL;
    if (B == 0) return PA_OK;
    return run_decode(true, nullptr, nullptr, part_o, part_lse, q, k_cache, v_cache, cache,
                      block_tables, max_blocks_per_seq, seq_lens, B, Hq, scale, num_splits, status,
                      stream);
}

int pa_combine(void *out, float *lse, const float *part_o, const float *part_lse, int32_t B,
               int32_t Hq, int32_t num_splits, int32_t D, pa_stream_t stream) {
    if (B < 0 || Hq <= 0 || num_splits <= 0) return PA_EINVAL;
    if (D != 64 && D != 128) return PA_EUNSUPPORTED;
    if (B == 0) return PA_OK;
    if (!out || !part_o || !part_lse || !aligned(out, 16) || !aligned(part_o, 16) ||
        !aligned(part_lse, 4) || (lse && !aligned(lse, 4)))
        return PA_EINVAL;
    const int64_t rows = static_cast<int64_t>(B) * Hq;
    if (rows > INT32_MAX / 2) return PA_EUNSUPPORTED;
    cudaError_t e = pa::launch_combine(out, lse, part_o, part_lse, static_cast<int>(rows),
                                       num_splits, D, stream);
    return e == cudaSuccess ? PA_OK : PA_ECUDA;
}

namespace {
// Whether a split call (P partitions) merges its partials in the same launch:
// its cooperative grid must fit on the GPU at once (sm_count x the kernel's
// CTAs per SM) and a merge task must hold every partition; the prefill-shaped
// kernel never does.  Otherwise partials, then pa_combine.
bool merge_in_launch(int32_t B, int32_t q_len, int32_t Hq, int32_t Hkv, int32_t D, int32_t P,
                     int sm_count) {
    if (P < 2 || P > pa::kMaxGridMerge || sm_count <= 0) return false;
    const int G = Hq / Hkv;
    const int qpc = queries_per_cta(G, q_len);
    Kernel k;
    if (pick_kernel(G * qpc, D, &k)) return false;
    if (k == Kernel::kTensorCore && prefill_shape(G, q_len)) return false;
    const int64_t units = units_per_split(k, B, G, Hkv, qpc, (q_len + qpc - 1) / qpc);
    return units * P <= static_cast<int64_t>(sm_count) * ctas_per_sm(k);
}

// Split-KV decode shared by pa_decode_splitkv, pa_decode_step, pa_decode_mq,
// pa_decode_splitkv_fp8 and pa_decode_splitkv_noalloc.  With library_scratch
// the workspace is the library's own array (pa::noalloc_scratch), looked up
// only after every argument check has passed, and the merge counters in it
// are cleared on `stream` before the kernel runs (a caller's workspace keeps
// its counters at zero between calls instead).
int splitkv_common(void *out, float *lse, const void *q, const void *k_cache, const void *v_cache,
                   const pa_cache_desc &cache, const int32_t *block_tables,
                   int32_t max_blocks_per_seq, const int32_t *seq_lens, int32_t B, int32_t Hq,
                   float scale, int32_t num_splits, void *workspace, size_t workspace_bytes,
                   int32_t *status, cudaStream_t stream, const NewTokens &nt, int32_t q_len = 1,
                   const Fp8Scales *f8 = nullptr, bool library_scratch = false) {
    int rc = check_decode_args(q, k_cache, v_cache, cache, block_tables, max_blocks_per_seq,
                               seq_lens, B, Hq, scale);
    if (rc) return rc;
    if (!out || !aligned(out, 16) || (lse && !aligned(lse, 4))) return PA_EINVAL;
    if (num_splits < 0 || q_len < 1) return PA_EINVAL;
    if (static_cast<int64_t>(B) * q_len > kMaxRowsQ) return PA_EUNSUPPORTED;
    if (B == 0) return PA_OK;
    int P = num_splits;
    if (P == 0) {
        const int sms = sm_count_current();
        if (sms <= 0) return PA_ECUDA;
        P = pa_choose_num_splits_mq(B, q_len, Hq, cache.num_kv_heads, cache.head_dim,
                                    max_blocks_per_seq, cache.block_size, sms);
        if (P < 0) return P;
    }
    if (P > 65535) return PA_EUNSUPPORTED;
    if (P == 1)
        return run_decode(false, out, lse, nullptr, nullptr, q, k_cache, v_cache, cache,
                          block_tables, max_blocks_per_seq, seq_lens, B, Hq, scale, 1, status,
                          stream, nullptr, nt, q_len, f8);
    // rows of the partials: (sequence, query position, head)
    const int32_t Bq = B * q_len;
    const size_t need = pa_splitkv_workspace_bytes(Bq, Hq, cache.head_dim, P);
    if (library_scratch) {
        rc = pa::noalloc_scratch(&workspace, &workspace_bytes);
        if (rc) return rc;
    }
    if (!workspace || workspace_bytes < need || !aligned(workspace, 256)) return PA_EWORKSPACE;
    const int64_t rows = static_cast<int64_t>(Bq) * Hq * P;
    uint8_t *ws = static_cast<uint8_t *>(workspace);
    float *part_o = reinterpret_cast<float *>(ws);
    float *part_lse = reinterpret_cast<float *>(ws + round_up(rows * cache.head_dim * 4, 256));
    int32_t *counters = reinterpret_cast<int32_t *>(ws + round_up(rows * cache.head_dim * 4, 256) +
                                                    round_up(rows * 4, 256));
    // One cooperative launch that merges its own partials when the whole grid
    // fits on the GPU at once and its merge tasks can hold every partition;
    // otherwise partials, then pa_combine.
    if (merge_in_launch(B, q_len, Hq, cache.num_kv_heads, cache.head_dim, P, sm_count_current())) {
        if (library_scratch &&
            cudaMemsetAsync(counters, 0, static_cast<size_t>(Bq) * Hq * 8, stream) != cudaSuccess)
            return PA_ECUDA;
        rc = run_decode(true, out, lse, part_o, part_lse, q, k_cache, v_cache, cache, block_tables,
                        max_blocks_per_seq, seq_lens, B, Hq, scale, P, status, stream, counters, nt,
                        q_len, f8);
        if (rc != PA_ETOOLARGE) return rc;
    }
    rc = run_decode(true, nullptr, nullptr, part_o, part_lse, q, k_cache, v_cache, cache,
                    block_tables, max_blocks_per_seq, seq_lens, B, Hq, scale, P, status, stream,
                    nullptr, nt, q_len, f8);
    if (rc) return rc;
    cudaError_t e = pa::launch_combine(out, lse, part_o, part_lse, static_cast<int>(Bq * Hq), P,
                                       cache.head_dim, stream);
    return e == cudaSuccess ? PA_OK : PA_ECUDA;
}
}  // namespace

}  // extern "C"

namespace pa {
int decode_splitkv_library_scratch(void *out, float *lse, const void *q, const void *k_cache,
                                   const void *v_cache, const pa_cache_desc &cache,
                                   const int32_t *block_tables, int32_t max_blocks_per_seq,
                                   const int32_t *seq_lens, int32_t B, int32_t Hq, float scale,
                                   int32_t num_splits, int32_t *status, cudaStream_t stream) {
    return splitkv_common(out, lse, q, k_cache, v_cache, cache, block_tables, max_blocks_per_seq,
                          seq_lens, B, Hq, scale, num_splits, nullptr, 0, status, stream,
                          NewTokens(), 1, nullptr, true);
}
}  // namespace pa

extern "C" {

int pa_decode_mq(void *out, float *lse, const void *q, int32_t q_len, const void *k_cache,
                 const void *v_cache, pa_cache_desc cache, const int32_t *block_tables,
                 int32_t max_blocks_per_seq, const int32_t *seq_lens, int32_t B, int32_t Hq,
                 float scale, int32_t num_splits, void *workspace, size_t workspace_bytes,
                 int32_t *status, pa_stream_t stream) {
    if (q_len < 1 || q_len > 65535) return PA_EINVAL;
    return splitkv_common(out, lse, q, k_cache, v_cache, cache, block_tables, max_blocks_per_seq,
                          seq_lens, B, Hq, scale, num_splits, workspace, workspace_bytes, status,
                          stream, NewTokens(), q_len);
}

int pa_cache_write_fp8(const void *k_new, const void *v_new, const int64_t *slot_mapping,
                       int64_t n_tokens, void *k_cache, void *v_cache, pa_cache_desc cache,
                       float k_scale, float v_scale, int32_t *status, pa_stream_t stream) {
    if (n_tokens < 0) return PA_EINVAL;
    int rc = check_cache_desc(cache);
    if (rc) return rc;
    if (!(k_scale > 0.f) || !(v_scale > 0.f) || !std::isfinite(k_scale) || !std::isfinite(v_scale))
        return PA_EINVAL;
    if (n_tokens == 0) return PA_OK;
    if (!k_new || !v_new || !slot_mapping || !k_cache || !v_cache) return PA_EINVAL;
    if (!aligned(k_new, 16) || !aligned(v_new, 16) || !aligned(k_cache, 16) ||
        !aligned(v_cache, 16) || !aligned(slot_mapping, 8))
        return PA_EINVAL;
    const int row_elems = cache.num_kv_heads * cache.head_dim;
    cudaError_t e = pa::launch_cache_write_fp8(
        k_new, v_new, slot_mapping, n_tokens, k_cache, v_cache,
        static_cast<int64_t>(cache.num_blocks) * cache.block_size, row_elems, k_scale, v_scale,
        status, stream);
    return e == cudaSuccess ? PA_OK : PA_ECUDA;
}

int pa_decode_step_fp8(void *out, float *lse, const void *q, const void *k_new, const void *v_new,
                       const int64_t *slot_mapping, void *k_cache, void *v_cache,
                       pa_cache_desc cache, float k_scale, float v_scale,
                       const int32_t *block_tables, int32_t max_blocks_per_seq,
                       const int32_t *seq_lens, int32_t B, int32_t Hq, float scale,
                       int32_t num_splits, void *workspace, size_t workspace_bytes,
                       int32_t *status, pa_stream_t stream) {
    if (!(k_scale > 0.f) || !(v_scale > 0.f) || !std::isfinite(k_scale) || !std::isfinite(v_scale))
        return PA_EINVAL;
    if (cache.head_dim != 128) return PA_EUNSUPPORTED;
    if (B == 0) return PA_OK;
    if (!k_new || !v_new || !slot_mapping) return PA_EINVAL;
    if (!aligned(k_new, 16) || !aligned(v_new, 16) || !aligned(slot_mapping, 8)) return PA_EINVAL;
    NewTokens nt;
    nt.k_new = k_new;
    nt.v_new = v_new;
    nt.slot_mapping = slot_mapping;
    const Fp8Scales f8{k_scale, v_scale};
    return splitkv_common(out, lse, q, k_cache, v_cache, cache, block_tables, max_blocks_per_seq,
                          seq_lens, B, Hq, scale, num_splits, workspace, workspace_bytes, status,
                          stream, nt, 1, &f8);
}

int pa_decode_splitkv_fp8(void *out, float *lse, const void *q, const void *k_cache,
                          const void *v_cache, pa_cache_desc cache, float k_scale, float v_scale,
                          const int32_t *block_tables, int32_t max_blocks_per_seq,
                          const int32_t *seq_lens, int32_t B, int32_t Hq, float scale,
                          int32_t num_splits, void *workspace, size_t workspace_bytes,
                          int32_t *status, pa_stream_t stream) {
    if (!(k_scale > 0.f) || !(v_scale > 0.f) || !std::isfinite(k_scale) || !std::isfinite(v_scale))
        return PA_EINVAL;
    if (cache.head_dim != 128) return PA_EUNSUPPORTED;
    const Fp8Scales f8{k_scale, v_scale};
    return splitkv_common(out, lse, q, k_cache, v_cache, cache, block_tables, max_blocks_per_seq,
                          seq_lens, B, Hq, scale, num_splits, workspace, workspace_bytes, status,
                          stream, NewTokens(), 1, &f8);
}

// Cascade decode: partition counts of the prefix pass (all B sequences' queries
// as one multi-query call over the shared blocks) and of the suffix pass.
static int cascade_splits_on(int32_t B, int32_t Hq, int32_t Hkv, int32_t D, int32_t n_prefix_blocks,
                             int32_t max_blocks_per_seq, int32_t block_size, int sms, int *P1, int *P2) {
    *P1 = pa_choose_num_splits_mq(1, B, Hq, Hkv, D, n_prefix_blocks, block_size, sms);
    if (*P1 < 0) return *P1;
    *P2 = pa_choose_num_splits(B, Hq, Hkv, D, max_blocks_per_seq - n_prefix_blocks, block_size, sms);
    if (*P2 < 0) return *P2;
    return PA_OK;
}

static int cascade_splits(int32_t B, int32_t Hq, int32_t Hkv, int32_t D, int32_t n_prefix_blocks,
                          int32_t max_blocks_per_seq, int32_t block_size, int *P1, int *P2) {
    const int sms = sm_count_current();
    if (sms <= 0) return PA_ECUDA;
    return cascade_splits_on(B, Hq, Hkv, D, n_prefix_blocks, max_blocks_per_seq, block_size, sms, P1,
                             P2);
}

// Whether the cascade's suffix pass (P2 partitions) merges the P1 + P2
// partials of its rows in its own launch.
static bool cascade_suffix_merges(int32_t B, int32_t Hq, int32_t Hkv, int32_t D, int P1, int P2, int sms) {
    return P1 + P2 <= pa::kMaxGridMerge && merge_in_launch(B, 1, Hq, Hkv, D, P2, sms);
}

// Does attending the shared prefix once for the whole batch pay?  Without the
// cascade every sequence attends the prefix again: B - 1 extra passes over its
// K/V.  Those passes mostly hit L2 (the sequences' CTAs of one partition read
// the same blocks at about the same time, even for a prefix larger than L2),
// so what they cost is L2 traffic and the SMs' work on the extra rows, against
// the cascade's extra launch and merge.  Calibrated on this GPU: the cascade
// pays once the extra reads reach 256 MiB (256 sequences behind a 2048-token
// prefix of 8 KV heads, 2.1 GB: 3.4x faster; 4 sequences behind 65536
// tokens, 805 MB: 68.4 against 76.4 us; 8 behind 16384, 470 MB: 36.3
// against 44.2 us; plain decode is faster for 256 behind 8 blocks, 134 MB:
// 162.4 against 171.4 us).
static bool cascade_pays(int32_t B, int32_t Hkv, int32_t D, int32_t n_prefix_blocks,
                         int32_t block_size) {
    const int mode = option(PA_OPT_CASCADE);
    if (mode != PA_CASCADE_AUTO) return mode == PA_CASCADE_ALWAYS;
    const double prefix_bytes = static_cast<double>(n_prefix_blocks) * block_size * Hkv * D * 2 * 2;
    return (B - 1) * prefix_bytes >= 256.0 * (1 << 20);
}

int pa_cascade_launches(int32_t B, int32_t Hq, int32_t Hkv, int32_t D, int32_t n_prefix_blocks,
                        int32_t max_blocks_per_seq, int32_t block_size, int32_t sm_count) {
    if (B < 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv != 0 || D <= 0 || n_prefix_blocks < 0 ||
        n_prefix_blocks >= max_blocks_per_seq || block_size <= 0 || sm_count <= 0)
        return PA_EINVAL;
    if (B == 0) return 0;
    if (n_prefix_blocks == 0 || !cascade_pays(B, Hkv, D, n_prefix_blocks, block_size))
        return pa_decode_launches(B, 1, Hq, Hkv, D, max_blocks_per_seq, block_size, 0, sm_count);
    int P1 = 0, P2 = 0;
    const int rc = cascade_splits_on(B, Hq, Hkv, D, n_prefix_blocks, max_blocks_per_seq, block_size,
                                     sm_count, &P1, &P2);
    if (rc) return rc;
    return cascade_suffix_merges(B, Hq, Hkv, D, P1, P2, sm_count) ? 2 : 3;
}

int pa_cascade_pays(int32_t B, int32_t Hkv, int32_t D, int32_t n_prefix_blocks, int32_t block_size) {
    if (B <= 0 || Hkv <= 0 || D <= 0 || n_prefix_blocks < 0 || block_size <= 0) return PA_EINVAL;
    return n_prefix_blocks > 0 && cascade_pays(B, Hkv, D, n_prefix_blocks, block_size) ? 1 : 0;
}

size_t pa_cascade_workspace_bytes(int32_t B, int32_t Hq, int32_t Hkv, int32_t D,
                                  int32_t n_prefix_blocks, int32_t max_blocks_per_seq,
                                  int32_t block_size) {
    if (B <= 0 || Hq <= 0 || Hkv <= 0 || n_prefix_blocks <= 0 ||
        n_prefix_blocks >= max_blocks_per_seq)
        return 0;
    int P1 = 0, P2 = 0;
    if (cascade_splits(B, Hq, Hkv, D, n_prefix_blocks, max_blocks_per_seq, block_size, &P1, &P2))
        return 0;
    // enough for either path (the plain split decode when the cascade does not pay)
    const int P = pa_auto_num_splits(B, Hq, Hkv, D, max_blocks_per_seq, block_size);
    return std::max(pa_splitkv_workspace_bytes(B, Hq, D, P1 + P2 < 2 ? 2 : P1 + P2),
                    P > 0 ? pa_splitkv_workspace_bytes(B, Hq, D, P) : 0);
}

int pa_decode_cascade(void *out, float *lse, const void *q, const void *k_cache,
                      const void *v_cache, pa_cache_desc cache, int32_t n_prefix_blocks,
                      const int32_t *block_tables, int32_t max_blocks_per_seq,
                      const int32_t *seq_lens, int32_t B, int32_t Hq, float scale,
                      void *workspace, size_t workspace_bytes, int32_t *status,
                      pa_stream_t stream) {
    int rc = check_decode_args(q, k_cache, v_cache, cache, block_tables, max_blocks_per_seq,
                               seq_lens, B, Hq, scale);
    if (rc) return rc;
    if (!out || !aligned(out, 16) || (lse && !aligned(lse, 4))) return PA_EINVAL;
    if (n_prefix_blocks < 0 || n_prefix_blocks >= max_blocks_per_seq) return PA_EINVAL;
    if (B == 0) return PA_OK;
    // nothing shared, or too little to pay for the cascade's launches: plain split decode
    if (n_prefix_blocks == 0 ||
        !cascade_pays(B, cache.num_kv_heads, cache.head_dim, n_prefix_blocks, cache.block_size))
        return splitkv_common(out, lse, q, k_cache, v_cache, cache, block_tables,
                              max_blocks_per_seq, seq_lens, B, Hq, scale, 0, workspace,
                              workspace_bytes, status, stream, NewTokens());
    int P1 = 0, P2 = 0;
    rc = cascade_splits(B, Hq, cache.num_kv_heads, cache.head_dim, n_prefix_blocks,
                        max_blocks_per_seq, cache.block_size, &P1, &P2);
    if (rc) return rc;
    const int PT = P1 + P2;
    const size_t need = pa_splitkv_workspace_bytes(B, Hq, cache.head_dim, PT);
    if (!workspace || workspace_bytes < need || !aligned(workspace, 256)) return PA_EWORKSPACE;
    const int64_t rows = static_cast<int64_t>(B) * Hq;
    uint8_t *ws = static_cast<uint8_t *>(workspace);
    float *part_o = reinterpret_cast<float *>(ws);
    float *part_lse = reinterpret_cast<float *>(ws + round_up(rows * PT * cache.head_dim * 4, 256));
    const int32_t prefix_len = n_prefix_blocks * cache.block_size;
    // 1. the shared prefix, once: every sequence's queries as the q_len = B
    //    queries of one non-causal call over table row 0's first blocks
    PassOpts pre;
    pre.causal = 0;
    pre.seq_len_const = prefix_len;
    pre.part_stride = PT;
    pre.part_offset = 0;
    rc = run_decode(true, nullptr, nullptr, part_o, part_lse, q, k_cache, v_cache, cache,
                    block_tables, n_prefix_blocks, seq_lens, 1, Hq, scale, P1, status, stream,
                    nullptr, NewTokens(), B, nullptr, pre);
    if (rc) return rc;
    // 2. each sequence's own blocks: the table from entry n_prefix_blocks on,
    //    lengths less the prefix.  Where the suffix is split (P2 >= 2: its
    //    grid fits on the GPU at once, and the merge tasks spread over P2
    //    CTAs per group) and a merge task can hold every partition, this
    //    launch also merges the P1 + P2 partials of every row (the prefix
    //    pass's are complete: the launch waits for the previous one before it
    //    reads anything).  An unsplit suffix leaves the merge to the combine
    //    kernel, which spreads it over the whole GPU.
    PassOpts suf;
    suf.seq_len_offset = prefix_len;
    suf.part_stride = PT;
    suf.part_offset = P1;
    suf.table_stride = max_blocks_per_seq;
    if (cascade_suffix_merges(B, Hq, cache.num_kv_heads, cache.head_dim, P1, P2, sm_count_current())) {
        int32_t *counters = reinterpret_cast<int32_t *>(
            ws + round_up(rows * PT * cache.head_dim * 4, 256) + round_up(rows * PT * 4, 256));
        rc = run_decode(true, out, lse, part_o, part_lse, q, k_cache, v_cache, cache,
                        block_tables + n_prefix_blocks, max_blocks_per_seq - n_prefix_blocks,
                        seq_lens, B, Hq, scale, P2, status, stream, counters, NewTokens(), 1,
                        nullptr, suf);
        if (rc != PA_ETOOLARGE) return rc;
    }
    rc = run_decode(true, nullptr, nullptr, part_o, part_lse, q, k_cache, v_cache, cache,
                    block_tables + n_prefix_blocks, max_blocks_per_seq - n_prefix_blocks, seq_lens,
                    B, Hq, scale, P2, status, stream, nullptr, NewTokens(), 1, nullptr, suf);
    if (rc) return rc;
    // 3. one log-sum-exp merge of the P1 + P2 partials of every row
    cudaError_t e = pa::launch_combine(out, lse, part_o, part_lse, static_cast<int>(rows), PT,
                                       cache.head_dim, stream);
    return e == cudaSuccess ? PA_OK : PA_ECUDA;
}

int pa_decode_splitkv(void *out, float *lse, const void *q, const void *k_cache,
                      const void *v_cache, pa_cache_desc cache, const int32_t *block_tables,
                      int32_t max_blocks_per_seq, const int32_t *seq_lens, int32_t B, int32_t Hq,
                      float scale, int32_t num_splits, void *workspace, size_t workspace_bytes,
                      int32_t *status, pa_stream_t stream) {
    return splitkv_common(out, lse, q, k_cache, v_cache, cache, block_tables, max_blocks_per_seq,
                          seq_lens, B, Hq, scale, num_splits, workspace, workspace_bytes, status,
                          stream, NewTokens());
}

int pa_decode_step(void *out, float *lse, const void *q, const void *k_new, const void *v_new,
                   const int64_t *slot_mapping, void *k_cache, void *v_cache, pa_cache_desc cache,
                   const int32_t *block_tables, int32_t max_blocks_per_seq,
                   const int32_t *seq_lens, int32_t B, int32_t Hq, float scale,
                   int32_t num_splits, void *workspace, size_t workspace_bytes, int32_t *status,
                   pa_stream_t stream) {
    if (B == 0) return PA_OK;
    if (!k_new || !v_new || !slot_mapping) return PA_EINVAL;
    if (!aligned(k_new, 16) || !aligned(v_new, 16) || !aligned(slot_mapping, 8)) return PA_EINVAL;
    NewTokens nt;
    nt.k_new = k_new;
    nt.v_new = v_new;
    nt.slot_mapping = slot_mapping;
    return splitkv_common(out, lse, q, k_cache, v_cache, cache, block_tables, max_blocks_per_seq,
                          seq_lens, B, Hq, scale, num_splits, workspace, workspace_bytes, status,
                          stream, nt);
}


int pa_decode_launches(int32_t B, int32_t q_len, int32_t Hq, int32_t Hkv, int32_t D,
                       int32_t max_blocks_per_seq, int32_t block_size, int32_t num_splits,
                       int32_t sm_count) {
    if (B < 0 || q_len <= 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv != 0 || D <= 0 ||
        max_blocks_per_seq <= 0 || block_size <= 0 || num_splits < 0 || sm_count <= 0)
        return PA_EINVAL;
    if (B == 0) return 0;
    int P = num_splits;
    if (P == 0) {
        P = pa_choose_num_splits_mq(B, q_len, Hq, Hkv, D, max_blocks_per_seq, block_size, sm_count);
        if (P < 0) return P;
    }
    if (P == 1) return 1;
    return merge_in_launch(B, q_len, Hq, Hkv, D, P, sm_count) ? 1 : 2;
}

}  // extern "C"
