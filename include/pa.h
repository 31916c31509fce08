/*
 * pa.h -- C ABI of libpagedattn: decode attention over a paged KV cache on
 * NVIDIA GB300 (sm_103a).
 *
 * The operations are the hot path of one decode step of an LLM server, as the
 * "mini-infer" pages describe it:
 *   - a physical pool of fixed-size KV blocks (16 tokens per block; 256-token
 *     pages for the FlashAttention-2 backend) and a per-sequence
 *     virtual-to-physical block table ("mini-infer" docs by prajwal7-2002,
 *     section "Systems Architecture"; "MiniInfer" by tom-jerr, table
 *     "Attention Backend");
 *   - the [B, 1] decode step that writes each sequence's new K/V through a
 *     slot mapping and gathers physical K/V rows for attention (prajwal7-2002
 *     docs, table "Core Capabilities at a Glance", row "Batched Paged
 *     Decode");
 *   - split-K "flash decoding" for long contexts, which partitions each
 *     sequence's tokens and merges the partial results (psmarter "mini-infer"
 *     forum write-up, feature list item 7 and benchmark list item
 *     "Flash Decoding"; tom-jerr "Attention Backend" table, "split-KV").
 *
 * Layouts (all row-major, contiguous):
 *   q          [B, Hq, D]                       bf16
 *   k_cache    [num_blocks, block_size, Hkv, D] bf16   (v_cache identical)
 *   block_tables [B, max_blocks_per_seq]        int32, entry j of row b is the
 *                                               physical block holding tokens
 *                                               [j*block_size, (j+1)*block_size)
 *                                               of sequence b; entries past
 *                                               ceil(L_b / block_size) are
 *                                               never read
 *   seq_lens   [B]                              int32, L_b = tokens attended,
 *                                               including the one written this
 *                                               step
 *   slot_mapping [N]                            int64, slot = block * block_size
 *                                               + offset; a negative slot is
 *                                               padding and is skipped
 *   out        [B, Hq, D]                       bf16 (round to nearest even)
 *   lse        [B, Hq]                          fp32, natural-log log-sum-exp
 *                                               of the scaled scores; -inf for
 *                                               L_b = 0
 * Query head h reads KV head h / (Hq / Hkv).  bf16 arguments are passed as
 * untyped pointers to 16-bit storage.
 *
 * Conventions for every entry point:
 *   - Pointers marked "device" are device (or managed) memory owned by the
 *     caller; the library keeps no reference after the call returns.  It
 *     allocates no memory and never synchronises: work is enqueued on
 *     `stream` (NULL = the legacy default stream) and the call returns.
 *   - Device pointers to bf16/fp32 tensors must be 16-byte aligned.
 *   - Return value: PA_OK, or a negative PA_E* code when the arguments are
 *     rejected on the host (nothing is enqueued then) or a launch fails.
 *   - `status` (nullable, device int32): the kernels OR PA_STATUS_* bits
 *     into it when they meet bad data that the host cannot see (a block id
 *     outside the pool, a slot outside the pool, a sequence length larger
 *     than the table allows).  The offending element is skipped, never
 *     dereferenced.  The caller zeroes it and reads it back when convenient.
 *   - A call writes every element of its outputs.
 *   - Stream order holds for every call.  The head_dim-128 (tensor-core)
 *     decode kernel is launched with programmatic stream serialization: it
 *     may become resident while the previous kernel in the stream finishes,
 *     but waits for that kernel's completion (griddepcontrol.wait) before it
 *     reads or writes any global memory, and lets the next such launch queue
 *     once all of its CTAs run.  pa_set_option(PA_OPT_PDL, 0) launches it
 *     plainly.
 */
#ifndef PA_H_
#define PA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same handle as cudaStream_t / CUstream. */
typedef struct CUstream_st *pa_stream_t;

/* Shape of the physical K (and V) pool: [num_blocks, block_size, num_kv_heads, head_dim]. */
typedef struct {
    int32_t num_blocks;
    int32_t block_size;   /* tokens per block; a multiple of 16 */
    int32_t num_kv_heads; /* Hkv */
    int32_t head_dim;     /* D: 64 or 128 */
} pa_cache_desc;

/* Host-side return codes. */
enum {
    PA_OK = 0,
    PA_EINVAL = -1,       /* null or misaligned pointer, inconsistent sizes */
    PA_EUNSUPPORTED = -2, /* valid request outside what the kernels implement */
    PA_EWORKSPACE = -3,   /* workspace missing or smaller than required */
    PA_ECUDA = -4         /* a CUDA call or kernel launch failed */
};

/*
 * Process-wide switches, for tests and measurements (the defaults are what the
 * library is tuned for).  Each starts from the environment variable named
 * beside it, read once, the first time the library needs any of them; after
 * that only pa_set_option changes them.  A call uses the values current when it
 * is made; the switches are shared by all host threads and devices.
 */
enum {
    PA_OPT_DECODE_KERNEL = 0, /* which decode kernel runs: PA_KERNEL_* below
                                 (PA_DECODE_KERNEL=cuda_core|tensor_core) */
    PA_OPT_SPLIT_MERGE = 1,   /* PA_MERGE_AUTO, or PA_MERGE_GRID: never merge split
                                 partials through a thread-block cluster
                                 (PA_SPLIT_MERGE=grid) */
    PA_OPT_PDL = 2,           /* 1: programmatic stream serialization for the
                                 tensor-core kernel; 0: plain launches (PA_PDL=0) */
    PA_OPT_CASCADE = 3        /* pa_decode_cascade: PA_CASCADE_AUTO (the cascade
                                 where it pays), _ALWAYS or _NEVER
                                 (PA_CASCADE=always|never) */
};
enum { PA_CASCADE_AUTO = 0, PA_CASCADE_ALWAYS = 1, PA_CASCADE_NEVER = 2 };
enum {
    PA_KERNEL_AUTO = 0,        /* tensor cores wherever they can run the shape */
    PA_KERNEL_CUDA_CORE = 1,   /* force the CUDA-core kernel */
    PA_KERNEL_TENSOR_CORE = 2  /* force the tensor-core kernel */
};
enum { PA_MERGE_AUTO = 0, PA_MERGE_GRID = 1 };

/* Set a switch; PA_EINVAL for an unknown switch or value. */
int pa_set_option(int32_t option, int32_t value);
/* Current value of a switch, or PA_EINVAL. */
int pa_get_option(int32_t option);

/* Device status bits (OR-ed into *status). */
enum {
    PA_STATUS_BAD_BLOCK = 1,  /* block table entry outside [0, num_blocks) */
    PA_STATUS_BAD_SLOT = 2,   /* slot_mapping entry >= num_blocks * block_size */
    PA_STATUS_BAD_SEQLEN = 4, /* seq_len < 0 or > max_blocks_per_seq * block_size */
    PA_STATUS_TIMEOUT = 8     /* a bounded wait (an async copy, an MMA, the
                                 split merge's arrival) gave up after about a
                                 second; that call's outputs are not valid */
};

/*
 * Slot-mapping scatter of this step's new K and V (prajwal7-2002 docs, table
 * "Core Capabilities at a Glance", row "Batched Paged Decode": "zero-overhead
 * slot mapping").  For every i < n_tokens with s = slot_mapping[i] >= 0:
 *   k_cache[s / bs, s % bs, :, :] = k_new[i, :, :]   (bit copy), same for V.
 * k_new, v_new: device [n_tokens, Hkv, D] bf16.  slot_mapping: device int64.
 * Slots must be distinct (a repeated slot leaves one of the writers' rows;
 * which one is unspecified).  A slot >= num_blocks * bs is skipped and
 * reported through `status`.  n_tokens == 0 is a no-op.
 */
int pa_cache_write(const void *k_new, const void *v_new, const int64_t *slot_mapping,
                   int64_t n_tokens, void *k_cache, void *v_cache, pa_cache_desc cache,
                   int32_t *status, pa_stream_t stream);

/*
 * Batched single-token decode attention over the paged cache, one pass over
 * each sequence's KV (psmarter write-up, feature 1: PagedAttention with
 * block tables; prajwal7-2002 docs, row "Batched Paged Decode").  For every
 * sequence b and query head h:
 *   s_t = scale * <q[b,h,:], K[b, t, h / (Hq/Hkv), :]>,  t < L_b (through the table)
 *   out[b,h,:] = sum_t softmax(s)_t V[b, t, h/(Hq/Hkv), :]
 *   lse[b,h]   = ln sum_t exp(s_t)
 * out: device bf16 [B, Hq, D]; lse: device fp32 [B, Hq] or NULL.
 * q: device bf16 [B, Hq, D].  block_tables: device int32 [B, max_blocks_per_seq].
 * seq_lens: device int32 [B].  B == 0 is a no-op.
 * Supported: Hq % Hkv == 0, block_size a multiple of 16, and either D = 128
 * with G = Hq / Hkv <= 32 or D = 64 with G <= 8.  One CTA per (sequence, KV
 * head) holds the G query heads, so each KV tile is read once; use
 * pa_decode_splitkv when B * Hkv is small next to the SM count.
 * Two kernels implement the step: a tensor-core one (tcgen05, chosen
 * whenever D = 128) and a CUDA-core one (D = 64).  The switch
 * PA_OPT_DECODE_KERNEL forces one of them (a shape the forced kernel cannot
 * run is PA_EUNSUPPORTED).  Both are checked against the same oracle.
 */
int pa_decode(void *out, float *lse, const void *q, const void *k_cache, const void *v_cache,
              pa_cache_desc cache, const int32_t *block_tables, int32_t max_blocks_per_seq,
              const int32_t *seq_lens, int32_t B, int32_t Hq, float scale, int32_t *status,
              pa_stream_t stream);

/*
 * Split-KV partition count for a decode batch (psmarter benchmark list,
 * "Flash Decoding": splitting lifts SM utilisation at seq 4096).  Picks the
 * largest P for which the B * Hkv * P CTAs fit one wave of the decode kernel
 * that the group size Hq / Hkv and head_dim D select (2 CTAs per SM for the
 * CUDA-core kernel, 1 for the tensor-core kernel), capped so that every
 * partition keeps at least two 16-token tiles, and at 32 partitions where
 * partitions of four tiles would number 32 or fewer (more than 32 partitions
 * take a costlier merge).  A batch with more CTAs than
 * one wave holds runs in waves: its sequences are split into partitions of
 * about 48 tiles (of max_blocks_per_seq * block_size tokens), which evens the
 * waves out when the lengths differ.  Host-only; depends only on its
 * arguments and the PA_OPT_DECODE_KERNEL switch.
 * Returns P >= 1, or PA_EINVAL / PA_EUNSUPPORTED.
 */
int pa_choose_num_splits(int32_t B, int32_t Hq, int32_t Hkv, int32_t D,
                         int32_t max_blocks_per_seq, int32_t block_size, int32_t sm_count);

/*
 * Split-K partitioning of each sequence's tokens (psmarter "mini-infer" forum
 * write-up, feature list item 7: flash decoding splits the KV of a long
 * sequence into partitions that are attended in parallel and then merged).
 * Tokens per partition for P splits: ceil(ceil(max_blocks_per_seq*bs / P) / 16) * 16.
 * Partition p of sequence b covers tokens [p * chunk, min((p + 1) * chunk, L_b)).
 * Returns the chunk, or PA_EINVAL.
 */
int pa_partition_tokens(int32_t max_blocks_per_seq, int32_t block_size, int32_t num_splits);

/*
 * Bytes of workspace pa_decode_splitkv needs: fp32 partial outputs
 * [B, Hq, P, D], fp32 partial LSEs [B, Hq, P] and two int32 merge counters
 * per (sequence, head group) (at most 2 * B * Hq), each region 256-byte
 * aligned.
 * 0 when num_splits <= 1.
 */
size_t pa_splitkv_workspace_bytes(int32_t B, int32_t Hq, int32_t D, int32_t num_splits);

/*
 * Per-partition decode attention, the first half of split-K flash decoding
 * (psmarter write-up, feature list item 7: each partition of a sequence's KV
 * is attended on its own).
 * part_o: device fp32 [B, Hq, P, D], each partial normalised over its own
 * token range; part_lse: device fp32 [B, Hq, P], natural-log LSE of the
 * range, -inf for an empty range (and then part_o = 0).  Partition ranges as
 * in pa_partition_tokens.  num_splits >= 1.  Other arguments as pa_decode.
 */
int pa_decode_partial(float *part_o, float *part_lse, const void *q, const void *k_cache,
                      const void *v_cache, pa_cache_desc cache, const int32_t *block_tables,
                      int32_t max_blocks_per_seq, const int32_t *seq_lens, int32_t B,
                      int32_t Hq, float scale, int32_t num_splits, int32_t *status,
                      pa_stream_t stream);

/*
 * Log-sum-exp merge of P partials per (b, h), the second half of split-K
 * flash decoding (psmarter write-up, feature list item 7: the partitions'
 * partial results are merged into the exact output):
 *   lse = M + ln sum_p exp(lse_p - M),  M = max_p lse_p
 *   out = sum_p exp(lse_p - lse) * o_p           (bf16, round to nearest even)
 * A partial with lse_p = -inf has weight 0; if all are -inf, out = 0 and
 * lse = -inf.  part_o: device fp32 [B, Hq, P, D]; part_lse: device fp32
 * [B, Hq, P]; out: device bf16 [B, Hq, D]; lse: device fp32 [B, Hq] or NULL.
 */
int pa_combine(void *out, float *lse, const float *part_o, const float *part_lse, int32_t B,
               int32_t Hq, int32_t num_splits, int32_t D, pa_stream_t stream);

/*
 * Split-KV ("flash decoding") decode attention: per-partition partials into
 * the caller's workspace, merged by log-sum-exp into out/lse, all on
 * `stream`.  The decode kernel merges its own partials in the same launch
 * where it can:
 *   - tensor-core kernel, P <= 16, and all B x (Hkv / heads per CTA) x
 *     (query groups) clusters of P CTAs resident at once: the P partitions
 *     of each sequence and head group form a thread-block cluster and merge
 *     through distributed shared memory (the workspace's partial and counter
 *     regions are not touched);
 *   - otherwise, when the split grid fits on the GPU at once: a cooperative
 *     launch whose CTAs of each sequence and head group meet at a counter in
 *     the workspace, then share the merge;
 *   - otherwise pa_combine runs after the decode kernel.
 * Partitions beyond 256 are always merged by pa_combine.
 * pa_set_option(PA_OPT_SPLIT_MERGE, PA_MERGE_GRID) skips the cluster merge.
 * num_splits == 0 picks P with pa_auto_num_splits; P == 1 runs pa_decode
 * directly and needs no workspace.  workspace: device, at least
 * pa_splitkv_workspace_bytes(B, Hq, D, P) bytes, 256-byte aligned, else
 * PA_EWORKSPACE.  It must be zero-filled before its first use (cudaMemset):
 * the merge counters in it start at zero and every completed call leaves
 * them at zero again, so a workspace can be reused call after call (not by
 * calls that overlap on the GPU).  A call that reported PA_STATUS_TIMEOUT
 * may leave them non-zero: zero the workspace again before reusing it.
 * Results equal pa_decode's up to fp32 rounding order.
 */
int pa_decode_splitkv(void *out, float *lse, const void *q, const void *k_cache,
                      const void *v_cache, pa_cache_desc cache, const int32_t *block_tables,
                      int32_t max_blocks_per_seq, const int32_t *seq_lens, int32_t B,
                      int32_t Hq, float scale, int32_t num_splits, void *workspace,
                      size_t workspace_bytes, int32_t *status, pa_stream_t stream);

/* Size of the scratch array built into the library for pa_decode_splitkv_noalloc. */
#define PA_NOALLOC_SCRATCH_BYTES ((size_t)4 << 20)

/*
 * Split-KV decode attention that needs no workspace from the caller and
 * allocates nothing.  There is no counterpart on the pages: it exists for
 * callers that cannot call cudaMalloc (or any allocator) where they run
 * decode -- for instance code whose device memory is planned up front by
 * another component, or a plugin that is handed only its inputs and outputs.
 * Arguments and results are those of pa_decode_splitkv without the
 * workspace.  The split's partials live in a file-scope device array of
 * PA_NOALLOC_SCRATCH_BYTES (4 MiB) inside the library, which every GPU that
 * loads the library holds until the process exits.
 *   - The first call on a device looks up that array's device address
 *     (cudaGetSymbolAddress, with the device current) and caches it; make
 *     that first call before any stream capture.  The address is looked up
 *     again when the device's current context has changed (after
 *     cudaDeviceReset the library's module is loaded anew); make the first
 *     call after such a reset before any capture too.
 *   - Arguments are checked exactly as pa_decode_splitkv checks them before
 *     the array is touched; a rejected call enqueues nothing.
 *   - Returns PA_EWORKSPACE when the split's partials,
 *     pa_splitkv_workspace_bytes(B, Hq, D, P), exceed the array.
 *   - Every call shares the one array: calls whose kernels overlap on the
 *     GPU (other streams, other host threads) race on it and must be
 *     serialised by the caller.  Each call clears the merge counters it
 *     uses (cudaMemsetAsync on `stream`, no allocation) and writes every
 *     partial before reading it.  num_splits == 1 does not use the array.
 */
int pa_decode_splitkv_noalloc(void *out, float *lse, const void *q, const void *k_cache,
                              const void *v_cache, pa_cache_desc cache,
                              const int32_t *block_tables, int32_t max_blocks_per_seq,
                              const int32_t *seq_lens, int32_t B, int32_t Hq, float scale,
                              int32_t num_splits, int32_t *status, pa_stream_t stream);

/*
 * One whole decode step in one launch: the slot-mapping write of this step's
 * new K/V and split-KV decode attention (prajwal7-2002 docs, row "Batched
 * Paged Decode": the [B, 1] step writes the new token through the slot
 * mapping and attends over the gathered blocks).  The same result as
 *   pa_cache_write(k_new, v_new, slot_mapping, B, ...) then pa_decode_splitkv(...)
 * when slot_mapping[b] is the slot of position seq_lens[b] - 1 of sequence b
 * (write-then-attend), but without the separate write launch: the CTA that
 * reads that position writes the token's rows just before loading them.
 * k_new, v_new: device bf16 [B, Hkv, D] (row b is sequence b's new token);
 * slot_mapping: device int64 [B], a negative slot means no write for that
 * sequence.  A non-negative slot that is not position seq_lens[b] - 1 of
 * sequence b is not written and sets PA_STATUS_BAD_SLOT (a slot this step
 * does not read could be read by another sequence in the same launch).
 * Every other argument, the workspace contract included, as
 * pa_decode_splitkv; num_splits == 1 needs no workspace.
 */
int pa_decode_step(void *out, float *lse, const void *q, const void *k_new, const void *v_new,
                   const int64_t *slot_mapping, void *k_cache, void *v_cache, pa_cache_desc cache,
                   const int32_t *block_tables, int32_t max_blocks_per_seq,
                   const int32_t *seq_lens, int32_t B, int32_t Hq, float scale,
                   int32_t num_splits, void *workspace, size_t workspace_bytes, int32_t *status,
                   pa_stream_t stream);

/*
 * Multi-query decode: several new tokens per sequence attend at once, causally
 * -- speculative verification of drafted tokens, or a small chunk of new
 * tokens ("mini-infer" psmarter write-up, feature list items 3 and 5;
 * prajwal7-2002 docs, table "Core Capabilities at a Glance", row "Prompt
 * Ingestion", and the speculative-decoding overview: the target model
 * verifies a draft's tokens in one pass).  The last q_len positions of every
 * sequence are queries, their K/V already in the pool (pa_cache_write first):
 * query i of sequence b sits at position seq_lens[b] - q_len + i and attends
 * to positions [0, seq_lens[b] - q_len + i] (a negative position sees
 * nothing: out = 0, lse = -inf).
 * q: device bf16 [B, q_len, Hq, D]; out: device bf16 [B, q_len, Hq, D];
 * lse: device fp32 [B, q_len, Hq] or NULL.  1 <= q_len <= 65535.
 * Supported: D = 128, G = Hq / Hkv <= 32 (the tensor-core kernels; q_len > 1
 * with the CUDA-core kernel forced, or D = 64, is PA_EUNSUPPORTED).  Two
 * kernels serve it: with q_len * G <= 32 (verification of a few drafted
 * tokens) the decode kernel holds the q_len positions of a KV head's G query
 * heads as MMA columns in one CTA; with more (a chunked-prefill chunk, e.g.
 * 512 tokens) a prefill-shaped kernel holds 128 query rows (128 / G
 * positions x G heads) per CTA on the MMA's M side and reads each KV block
 * once per such tile (split partials are then merged by the combine step).
 * num_splits: 0 = pa_choose_num_splits_mq on the current device, 1 = no
 * split (no workspace), P > 1 = split with the workspace contract of
 * pa_decode_splitkv for pa_splitkv_workspace_bytes(B * q_len, Hq, D, P)
 * bytes.  q_len = 1 is exactly pa_decode_splitkv.  Other arguments as
 * pa_decode_splitkv.
 */
int pa_decode_mq(void *out, float *lse, const void *q, int32_t q_len, const void *k_cache,
                 const void *v_cache, pa_cache_desc cache, const int32_t *block_tables,
                 int32_t max_blocks_per_seq, const int32_t *seq_lens, int32_t B, int32_t Hq,
                 float scale, int32_t num_splits, void *workspace, size_t workspace_bytes,
                 int32_t *status, pa_stream_t stream);

/*
 * Decode over a shared prefix, as a cascade where that pays: the first n_prefix_blocks entries of
 * every sequence's block table name the same physical blocks (a prefix-cache
 * hit shared by the batch: "mini-infer" prajwal7-2002 docs, table "Core
 * Capabilities at a Glance", row "Prompt Caching", radix-tree prefix cache;
 * psmarter write-up, feature list item 4, prefix caching).  The result is
 * pa_decode_splitkv's.  The cascade computes it in two or three launches:
 * (1) the prefix once, all B sequences' queries attending it together (128
 * query rows, i.e. 128 / G sequences, per CTA of the prefill-shaped kernel
 * when B * G > 32); (2) every sequence's remaining positions,
 * [n_prefix_blocks * block_size, seq_lens[b]), which, when that pass is split
 * (at least two partitions per sequence) and both passes have at most 256
 * partitions together, also merges both passes' fp32 partials; else (3) a
 * log-sum-exp combine of them.  It pays when attending the prefix once per
 * sequence would cost more than that: with PA_OPT_CASCADE at
 * PA_CASCADE_AUTO the call runs the cascade when (B - 1) x the prefix's K/V
 * bytes reach 256 MiB, and pa_decode_splitkv otherwise (the same result).  Requires seq_lens[b] >= n_prefix_blocks *
 * block_size (a shorter sequence sets PA_STATUS_BAD_SEQLEN and its result is
 * undefined); 0 <= n_prefix_blocks < max_blocks_per_seq (0: plain
 * pa_decode_splitkv).  The library reads the prefix's block ids from table
 * row 0.  workspace: pa_cascade_workspace_bytes(...) bytes (fp32 partials,
 * enough for either path), 256-byte aligned, zero-filled before its first use
 * (the pa_decode_splitkv contract).  Tensor-core kernel only: head_dim 128, Hq / Hkv <= 32.
 */
int pa_decode_cascade(void *out, float *lse, const void *q, const void *k_cache,
                      const void *v_cache, pa_cache_desc cache, int32_t n_prefix_blocks,
                      const int32_t *block_tables, int32_t max_blocks_per_seq,
                      const int32_t *seq_lens, int32_t B, int32_t Hq, float scale,
                      void *workspace, size_t workspace_bytes, int32_t *status,
                      pa_stream_t stream);

/* 1 when pa_decode_cascade runs the cascade for this shape under the current
 * PA_OPT_CASCADE switch, 0 when it runs pa_decode_splitkv; PA_EINVAL on bad
 * arguments.  Host-only. */
int pa_cascade_pays(int32_t B, int32_t Hkv, int32_t D, int32_t n_prefix_blocks, int32_t block_size);

/* Kernel launches pa_decode_cascade makes for this shape on sm_count SMs
 * under the current PA_OPT_CASCADE switch: 2 or 3 when it runs the cascade
 * (prefix pass, suffix pass, and the combine unless the suffix launch merges
 * both passes' partials), else pa_decode_launches of the plain split decode
 * with the automatic P.  0 for B = 0; PA_EINVAL on bad arguments.
 * Host-only. */
int pa_cascade_launches(int32_t B, int32_t Hq, int32_t Hkv, int32_t D, int32_t n_prefix_blocks,
                        int32_t max_blocks_per_seq, int32_t block_size, int32_t sm_count);

/* Workspace bytes pa_decode_cascade needs on the current device (0 on bad arguments). */
size_t pa_cascade_workspace_bytes(int32_t B, int32_t Hq, int32_t Hkv, int32_t D,
                                  int32_t n_prefix_blocks, int32_t max_blocks_per_seq,
                                  int32_t block_size);

/*
 * FP8 KV cache.  The pages say only that the KV-cache manager supports several
 * quantisation schemes ("Mini-Infer: A High-Performance LLM Inference
 * Acceleration Engine for Production Environments", section "Memory
 * Optimization and KV Cache Management").  Here: pools of one-byte OCP e4m3
 * codes (4 exponent bits, bias 7; 3 mantissa bits; no infinities; 0x7F/0xFF
 * NaN; largest finite 448), [num_blocks, block_size, Hkv, D] uint8, with one
 * fp32 scale per pool: a code c stands for e4m3(c) * scale.  Half the bytes
 * of a bf16 pool per token.
 */

/*
 * Slot-mapping write into FP8 pools: as pa_cache_write, each new bf16 row
 * stored as round_to_nearest_even_e4m3(fp32(x) / scale), saturating at +-448
 * (NaN stays NaN).  k_scale, v_scale: finite and > 0, else PA_EINVAL.
 * k_cache, v_cache: device uint8 pools described by `cache`.
 */
int pa_cache_write_fp8(const void *k_new, const void *v_new, const int64_t *slot_mapping,
                       int64_t n_tokens, void *k_cache, void *v_cache, pa_cache_desc cache,
                       float k_scale, float v_scale, int32_t *status, pa_stream_t stream);

/*
 * Split-KV decode attention over FP8 pools: pa_decode_splitkv's arguments and
 * results (num_splits 0 = pa_auto_num_splits, 1 = no split and no workspace,
 * the same workspace contract otherwise), with k_cache / v_cache e4m3 pools
 * and their scales.  The result is attention over the dequantised values
 * (code * scale); the tensor-core kernel keeps the codes one byte wide in
 * shared memory, widens each chunk to fp16 exactly into tensor memory and runs
 * its MMAs in fp16 (q is rounded to fp16: |q| must stay below 65504).  Supported: head_dim 128, Hq / Hkv <= 32 (PA_EUNSUPPORTED
 * otherwise, and with the CUDA-core kernel forced).
 */
int pa_decode_splitkv_fp8(void *out, float *lse, const void *q, const void *k_cache,
                          const void *v_cache, pa_cache_desc cache, float k_scale, float v_scale,
                          const int32_t *block_tables, int32_t max_blocks_per_seq,
                          const int32_t *seq_lens, int32_t B, int32_t Hq, float scale,
                          int32_t num_splits, void *workspace, size_t workspace_bytes,
                          int32_t *status, pa_stream_t stream);

/*
 * One whole decode step over FP8 pools in one launch: pa_decode_step's
 * fused write, quantised as pa_cache_write_fp8 quantises (the same codes,
 * byte for byte), and pa_decode_splitkv_fp8's attention.  The same result as
 *   pa_cache_write_fp8(k_new, v_new, slot_mapping, B, ...) then
 *   pa_decode_splitkv_fp8(...)
 * when slot_mapping[b] is the slot of position seq_lens[b] - 1 of sequence b;
 * a non-negative slot that is not is not written and sets
 * PA_STATUS_BAD_SLOT.  k_new, v_new: device bf16 [B, Hkv, D]; every other
 * argument as pa_decode_step and pa_decode_splitkv_fp8.
 */
int pa_decode_step_fp8(void *out, float *lse, const void *q, const void *k_new, const void *v_new,
                       const int64_t *slot_mapping, void *k_cache, void *v_cache,
                       pa_cache_desc cache, float k_scale, float v_scale,
                       const int32_t *block_tables, int32_t max_blocks_per_seq,
                       const int32_t *seq_lens, int32_t B, int32_t Hq, float scale,
                       int32_t num_splits, void *workspace, size_t workspace_bytes,
                       int32_t *status, pa_stream_t stream);

/*
 * Split count for pa_decode_mq, by the rule of pa_choose_num_splits with the
 * CTAs of every query-position group counted.  q_len = 1 gives
 * pa_choose_num_splits.  Returns P >= 1, or PA_EINVAL / PA_EUNSUPPORTED.
 */
int pa_choose_num_splits_mq(int32_t B, int32_t q_len, int32_t Hq, int32_t Hkv, int32_t D,
                            int32_t max_blocks_per_seq, int32_t block_size, int32_t sm_count);

/* P that pa_decode_splitkv uses for num_splits == 0 on the current device (PA_ECUDA on error). */
int pa_auto_num_splits(int32_t B, int32_t Hq, int32_t Hkv, int32_t D, int32_t max_blocks_per_seq,
                       int32_t block_size);

/*
 * Kernel launches that pa_decode_splitkv, pa_decode_step, pa_decode_mq,
 * pa_decode_splitkv_fp8 and pa_decode_step_fp8 make for this shape with num_splits partitions (0:
 * the automatic choice for sm_count SMs): 1 unsplit, or split with the
 * partials merged inside the launch (its grid fits on the GPU at once and
 * P <= 256); 2 otherwise (partials, then the combine kernel).  0 for B = 0;
 * PA_EINVAL on bad arguments.  Host-only.
 */
int pa_decode_launches(int32_t B, int32_t q_len, int32_t Hq, int32_t Hkv, int32_t D,
                       int32_t max_blocks_per_seq, int32_t block_size, int32_t num_splits,
                       int32_t sm_count);

/* Static description of a return code. */
const char *pa_strerror(int code);

/* Library ABI version (major * 10000 + minor * 100 + patch). */
int pa_version(void);

#ifdef __cplusplus
}
#endif

#endif /* PA_H_ */
