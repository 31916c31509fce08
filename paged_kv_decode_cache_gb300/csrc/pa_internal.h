// Host-side declarations shared by the library's translation units.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/pa.h"

namespace pa {

// Most partitions a split merge takes through one thread-block cluster.
constexpr int kMaxClusterMerge = 16;
// Multi-query calls whose query positions times group size exceed the decode
// kernel's 32 MMA columns per KV head take the prefill-shaped kernel
// (pa_prefill_tc.cu): 128 query rows (position, group member) per CTA, each
// CTA's token range at most kPrefillMaxTiles 16-token tiles.
constexpr int kPrefillRows = 128;
constexpr int kPrefillMaxTiles = 2048;

// Most partitions the in-launch grid merge takes (its tasks hold up to 8 LSEs
// per lane of a warp); a split with more partitions writes partials and is
// merged by the separate combine kernel, which takes any count.
constexpr int kMaxGridMerge = 256;

// Everything a decode CTA needs besides the two tensor maps.
struct DecodeParams {
    void *out;              // bf16 [B, Hq, D]            (unsplit)
    float *lse;             // fp32 [B, Hq] or null      (unsplit)
    float *part_o;          // fp32 [B, Hq, P, D]         (split)
    float *part_lse;        // fp32 [B, Hq, P]            (split)
    const uint16_t *q;      // bf16 [B, Hq, D]
    const int32_t *block_tables;
    const int32_t *seq_lens;
    int32_t *status;
    int32_t num_blocks;
    int32_t block_size;
    int32_t num_kv_heads;
    int32_t num_q_heads;
    int32_t max_blocks;
    int32_t num_splits;     // P (gridDim.x)
    int32_t chunk;          // tokens per partition, multiple of 16
    int32_t split;          // 1: write partials, 0: write out/lse
    float scale_log2;       // scale * log2(e)
    // Fused combine (split only): the last CTA of each (sequence, head group)
    // to finish merges the group's partials into out/lse.  counters has one
    // int per (sequence, head group), zero on entry and left zero on exit.
    int32_t *counters;      // null: partials only
    // Cluster merge (split only, tensor-core kernel): the P CTAs of a
    // (sequence, head group) are one thread-block cluster and merge their
    // partials through distributed shared memory; counters, part_o and
    // part_lse are then unused.
    int32_t cluster_merge;
    // Host side only: launch with programmatic stream serialization (the
    // kernel waits for the previous kernel in the stream before it touches
    // global memory, but may become resident while that kernel finishes).
    int32_t pdl;
    // Fused cache write (pa_decode_step): sequence b's new token, the one at
    // position L_b - 1, is written into the pools by the CTA that reads that
    // position, right before its TMA load of that tile.  null: no write.
    const uint16_t *k_new;  // bf16 [B, Hkv, D]
    const uint16_t *v_new;
    const int64_t *slot_mapping;  // [B]
    uint16_t *k_pool;       // the pools, writable
    uint16_t *v_pool;
    // Multi-query decode: the last q_len positions of each sequence are
    // queries (q, out: [B, q_len, Hq, D]; rows (b * q_len + i) * Hq + h), query
    // i at position L - q_len + i attending causally.  A CTA takes q_per_cta
    // consecutive query positions; gridDim.y = head_groups x query groups.
    int32_t q_len;          // 1: plain decode
    int32_t q_per_cta;
    int32_t head_groups;    // CTAs across the KV heads (Hkv / heads per CTA)
    // FP8 pools (e4m3 codes): scale_log2 already includes k_scale; the output
    // is multiplied by v_scale.  1 for bf16 pools.  The fused write quantises
    // the new rows with the pools' scales (k_scale, v_scale).
    float v_scale;
    float k_scale;
    // Cascade passes (tensor-core kernel): causal = 0 lets every query see all
    // L keys; L is seq_len_const when >= 0, else seq_lens[b] - seq_len_offset;
    // partials of row r, partition p go to [r * part_stride + part_offset + p].
    int32_t causal;
    int32_t seq_len_const;
    int32_t seq_len_offset;
    int32_t part_stride;
    int32_t part_offset;
    int32_t table_stride;   // entries between block-table rows (>= max_blocks)
};

// CUDA-core decode kernel launch (pa_decode_cc_d*.cu).  Returns a cudaError_t.
cudaError_t launch_decode_cc(int D, int G, const CUtensorMap &kmap, const CUtensorMap &vmap,
                             const DecodeParams &p, int B, cudaStream_t stream);

// Prefill-shaped multi-query kernel (pa_prefill_tc.cu): grid (num_splits,
// query tiles x Hkv, B); p.q_per_cta query positions per tile; writes out/lse,
// or fp32 partials when p.split (no in-launch merge).
cudaError_t launch_prefill_tc(const CUtensorMap &kmap, const CUtensorMap &vmap, const DecodeParams &p,
                              int B, int G, cudaStream_t stream);

cudaError_t launch_combine(void *out, float *lse, const float *part_o, const float *part_lse,
                           int rows, int P, int D, cudaStream_t stream);

cudaError_t launch_cache_write(const void *k_new, const void *v_new, const int64_t *slots,
                               int64_t n, void *k_cache, void *v_cache, int64_t n_slots,
                               int row_bytes, int32_t *status, cudaStream_t stream);

// Split-KV decode on the library's own scratch array (pa_decode_splitkv_noalloc):
// the device address and size of that array on the current device and
// context, looked up on first use (pa_noalloc.cu).  Returns PA_OK or a PA_E* code.
int noalloc_scratch(void **addr, size_t *bytes);

// pa_decode_splitkv with the library's scratch array as its workspace
// (pa_api.cu): every argument is checked first, then the array is looked up and
// the merge counters the call uses are cleared on `stream`.
int decode_splitkv_library_scratch(void *out, float *lse, const void *q, const void *k_cache,
                                   const void *v_cache, const pa_cache_desc &cache,
                                   const int32_t *block_tables, int32_t max_blocks_per_seq,
                                   const int32_t *seq_lens, int32_t B, int32_t Hq, float scale,
                                   int32_t num_splits, int32_t *status, cudaStream_t stream);

cudaError_t launch_cache_write_fp8(const void *k_new, const void *v_new, const int64_t *slots,
                                   int64_t n, void *k_cache, void *v_cache, int64_t n_slots,
                                   int row_elems, float k_scale, float v_scale, int32_t *status,
                                   cudaStream_t stream);

}  // namespace pa
