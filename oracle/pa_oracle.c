/*
 * Paged-KV decode attention: fp64 CPU oracle.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the slow, obviously-correct
 * statement of what the GPU library computes.  Only the tests, the smoke
 * check and the benchmark's CPU-baseline leg load it; the product path never
 * does, and it shares no code, header or constant with the CUDA sources.
 *
 * What it follows (web pages on the "mini-infer" LLM engines):
 *   - "mini-infer" (prajwal7-2002 docs page), section "Systems Architecture":
 *     a fixed pool of physical KV blocks of 16 tokens and a per-request
 *     virtual-to-physical block table.
 *   - same page, table "Core Capabilities at a Glance", row "Batched Paged
 *     Decode": the [B, 1] decode step gathers physical K/V rows directly
 *     and writes the new token through a slot mapping; the model then runs
 *     plain scaled-dot-product attention (row "Model Architecture": "SDPA").
 *   - "mini-infer" (psmarter, zingnex forum write-up), feature list item 1
 *     (PagedAttention with flash_attn block tables) and item 7 (split-K
 *     flash decoding).
 *   - "MiniInfer" (tom-jerr), table "Attention Backend": FA2 paged decode
 *     with split-KV and page_size = 256.
 *
 * The pages never write the attention formula out.  Split-K flash decoding
 * is an exact re-association of softmax attention, so the oracle is the
 * plain definition, evaluated in double precision:
 *
 *   s[t]   = scale * sum_d q[b,h,d] * K[p(t), t mod bs, g, d],  p(t) = bt[b][t / bs]
 *   out    = sum_t exp(s[t] - m) V[p(t), t mod bs, g, :] / sum_t exp(s[t] - m)
 *   lse    = m + ln sum_t exp(s[t] - m),   m = max_t s[t]
 *
 * with the query-head group reading g = h / (Hq / Hkv) (consecutive query
 * heads share one KV head; the pages are silent, this is the plainest
 * reading).  L = 0 gives out = 0, lse = -inf.
 *
 * Element type conventions: bf16 values arrive as their uint16 bit
 * patterns and are widened exactly (bits << 16 is the fp32 value).
 */
#include <math.h>
#include <stdint.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORACLE_OK 0
#define ORACLE_EBADARG (-1)
#define ORACLE_EBLOCK (-2)
#define ORACLE_ESLOT (-3)

static double bf16_to_f64(uint16_t bits) {
    uint32_t u = ((uint32_t)bits) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* Team size for one call: nthreads > 0 asks for exactly that many threads,
 * otherwise the OpenMP default (OMP_NUM_THREADS or the core count).  The
 * global OpenMP setting is never modified. */
static int team_size(int nthreads) {
#ifdef _OPENMP
    return nthreads > 0 ? nthreads : omp_get_max_threads();
#else
    (void)nthreads;
    return 1;
#endif
}

int oracle_max_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/*
 * Slot-mapping scatter ("Batched Paged Decode" row: the new token's K/V go
 * to slot s = physical_block * bs + offset).  Slot < 0 marks padding and is
 * skipped.  A pure byte copy of Hkv*D elements per token and per K or V.
 * Returns ORACLE_ESLOT when a slot is out of the pool or repeated (the pages
 * do not define a repeated slot; the oracle refuses it).
 */
int oracle_cache_write(const uint16_t *k_new, const uint16_t *v_new,
                       const int64_t *slot_mapping, int64_t n_tokens,
                       uint16_t *k_cache, uint16_t *v_cache,
                       int num_blocks, int block_size, int num_kv_heads, int head_dim) {
    if (n_tokens < 0 || num_blocks <= 0 || block_size <= 0 || num_kv_heads <= 0 || head_dim <= 0)
        return ORACLE_EBADARG;
    const int64_t n_slots = (int64_t)num_blocks * block_size;
    const int64_t row = (int64_t)num_kv_heads * head_dim;
    for (int64_t i = 0; i < n_tokens; ++i) {
        const int64_t s = slot_mapping[i];
        if (s < 0) continue;
        if (s >= n_slots) return ORACLE_ESLOT;
        for (int64_t j = 0; j < i; ++j)
            if (slot_mapping[j] == s) return ORACLE_ESLOT;
    }
    for (int64_t i = 0; i < n_tokens; ++i) {
        const int64_t s = slot_mapping[i];
        if (s < 0) continue;
        const int64_t blk = s / block_size, off = s % block_size;
        const int64_t dst = (blk * block_size + off) * row;
        memcpy(k_cache + dst, k_new + i * row, (size_t)row * sizeof(uint16_t));
        memcpy(v_cache + dst, v_new + i * row, (size_t)row * sizeof(uint16_t));
    }
    return ORACLE_OK;
}

/*
 * FP8 KV cache.  The pages say only that the KV-cache manager supports
 * several quantisation schemes ("Mini-Infer: A High-Performance LLM Inference
 * Acceleration Engine for Production Environments", section "Memory
 * Optimization and KV Cache Management"); the plainest
 * reading for a KV cache is OCP FP8 E4M3 ("e4m3fn": 1 sign bit, 4 exponent
 * bits with bias 7, 3 mantissa bits, no infinities, S.1111.111 = NaN, largest
 * finite value 448) with one fp32 scale per pool: a stored code c means the
 * value e4m3(c) * scale.  Writing a bf16 value x stores
 *     c = round_to_nearest_even_e4m3(fp32(x) / scale)   (fp32 IEEE division),
 * saturating at +-448 (the largest finite code) and keeping NaN as NaN.
 */
static double e4m3_value(uint8_t c) {
    const int e = (c >> 3) & 15, m = c & 7;
    double mag;
    if (e == 15 && m == 7) mag = NAN;
    else if (e == 0) mag = ldexp((double)m, -9);          /* subnormal: m/8 * 2^-6 */
    else mag = ldexp((double)(8 + m), e - 10);            /* (1 + m/8) * 2^(e-7) */
    return (c & 0x80) ? -mag : mag;
}

static uint8_t f32_to_e4m3_sat(float f) {
    if (isnan(f)) return 0x7F;
    const uint8_t sign = signbit(f) ? 0x80 : 0x00;
    const double a = fabs((double)f);
    if (a >= 448.0) return sign | 0x7E;
    /* codes 0x00..0x7E are increasing in value: bracket a, take the nearer,
     * ties to the even code (the code's last bit is the mantissa's) */
    int lo = 0, hi = 0x7E;
    while (hi - lo > 1) {
        const int mid = (lo + hi) / 2;
        if (e4m3_value((uint8_t)mid) <= a) lo = mid;
        else hi = mid;
    }
    const double dl = a - e4m3_value((uint8_t)lo), dh = e4m3_value((uint8_t)hi) - a;
    const int code = dl < dh ? lo : dh < dl ? hi : ((lo & 1) ? hi : lo);
    return sign | (uint8_t)code;
}

/* Widen e4m3 codes to bf16 bit patterns (exact: every e4m3 value is a bf16 value). */
int oracle_e4m3_to_bf16(uint16_t *out, const uint8_t *in, int64_t n) {
    if (n < 0) return ORACLE_EBADARG;
    for (int64_t i = 0; i < n; ++i) {
        const float f = (float)e4m3_value(in[i]);
        uint32_t bits;
        memcpy(&bits, &f, sizeof bits);
        out[i] = isnan(f) ? (uint16_t)(0x7FC0 | ((in[i] & 0x80) << 8)) : (uint16_t)(bits >> 16);
    }
    return ORACLE_OK;
}

/* Quantise bf16 values to e4m3 codes with one scale, as defined above. */
int oracle_bf16_to_e4m3(uint8_t *out, const uint16_t *in, int64_t n, float scale) {
    if (n < 0 || !(scale > 0.0f)) return ORACLE_EBADARG;
    for (int64_t i = 0; i < n; ++i) {
        const float x = (float)bf16_to_f64(in[i]);
        out[i] = f32_to_e4m3_sat(x / scale);
    }
    return ORACLE_OK;
}

/* Slot-mapping write into e4m3 pools: the cache write above, with each new
 * K (V) row quantised with k_scale (v_scale). */
int oracle_cache_write_fp8(const uint16_t *k_new, const uint16_t *v_new,
                           const int64_t *slot_mapping, int64_t n_tokens,
                           uint8_t *k_cache, uint8_t *v_cache,
                           int num_blocks, int block_size, int num_kv_heads, int head_dim,
                           float k_scale, float v_scale) {
    if (n_tokens < 0 || num_blocks <= 0 || block_size <= 0 || num_kv_heads <= 0 || head_dim <= 0 ||
        !(k_scale > 0.0f) || !(v_scale > 0.0f))
        return ORACLE_EBADARG;
    const int64_t n_slots = (int64_t)num_blocks * block_size;
    const int64_t row = (int64_t)num_kv_heads * head_dim;
    for (int64_t i = 0; i < n_tokens; ++i) {
        const int64_t s = slot_mapping[i];
        if (s < 0) continue;
        if (s >= n_slots) return ORACLE_ESLOT;
        for (int64_t j = 0; j < i; ++j)
            if (slot_mapping[j] == s) return ORACLE_ESLOT;
    }
    for (int64_t i = 0; i < n_tokens; ++i) {
        const int64_t s = slot_mapping[i];
        if (s < 0) continue;
        oracle_bf16_to_e4m3(k_cache + s * row, k_new + i * row, row, k_scale);
        oracle_bf16_to_e4m3(v_cache + s * row, v_new + i * row, row, v_scale);
    }
    return ORACLE_OK;
}

/* Pointer to K or V row (token t of sequence b, KV head g) through the block table. */
static const uint16_t *gather_row(const uint16_t *cache, const int32_t *bt_row, int t,
                                  int block_size, int num_kv_heads, int head_dim, int g) {
    const int64_t phys = bt_row[t / block_size];
    const int64_t off = t % block_size;
    return cache + ((phys * block_size + off) * num_kv_heads + g) * (int64_t)head_dim;
}

static int check_tables(const int32_t *block_tables, int max_blocks, const int32_t *seq_lens,
                        int B, int num_blocks, int block_size) {
    for (int b = 0; b < B; ++b) {
        const int L = seq_lens[b];
        if (L < 0 || (int64_t)L > (int64_t)max_blocks * block_size) return ORACLE_EBADARG;
        const int nb = (L + block_size - 1) / block_size;
        for (int j = 0; j < nb; ++j) {
            const int32_t p = block_tables[(int64_t)b * max_blocks + j];
            if (p < 0 || p >= num_blocks) return ORACLE_EBLOCK;
        }
    }
    return ORACLE_OK;
}

/*
 * Attention of query head h of sequence b over tokens [t0, t1): writes the
 * normalised output row (D doubles) and returns its log-sum-exp (natural
 * log).  An empty range gives a zero row and -inf.
 */
static double attend_range(double *out_row, const uint16_t *q_row,
                           const uint16_t *k_cache, const uint16_t *v_cache,
                           const int32_t *bt_row, int t0, int t1,
                           int block_size, int num_kv_heads, int head_dim, int g,
                           double scale, double *scores) {
    for (int d = 0; d < head_dim; ++d) out_row[d] = 0.0;
    if (t1 <= t0) return -INFINITY;
    double m = -INFINITY;
    for (int t = t0; t < t1; ++t) {
        const uint16_t *k = gather_row(k_cache, bt_row, t, block_size, num_kv_heads, head_dim, g);
        double dot = 0.0;
        for (int d = 0; d < head_dim; ++d) dot += bf16_to_f64(q_row[d]) * bf16_to_f64(k[d]);
        const double s = scale * dot;
        scores[t - t0] = s;
        if (s > m) m = s;
    }
    double z = 0.0;
    for (int t = t0; t < t1; ++t) {
        const double w = exp(scores[t - t0] - m);
        z += w;
        const uint16_t *v = gather_row(v_cache, bt_row, t, block_size, num_kv_heads, head_dim, g);
        for (int d = 0; d < head_dim; ++d) out_row[d] += w * bf16_to_f64(v[d]);
    }
    for (int d = 0; d < head_dim; ++d) out_row[d] /= z;
    return m + log(z);
}

/*
 * Decode attention for an explicit list of (b, h) rows.  out is
 * [n_rows, D], lse is [n_rows] (nullable).  `scale` multiplies every dot
 * product in double precision: the library's fp32 softmax scale, widened
 * exactly (or, over FP8 pools, that scale times the pool's k_scale, the
 * product formed in double).  `scores` is caller-provided work
 * memory of [team size, max_blocks * block_size] doubles: each OpenMP thread
 * keeps the scores of its current row in its own slice.
 */
int oracle_decode_rows(double *out, double *lse,
                       const int32_t *rows_b, const int32_t *rows_h, int n_rows,
                       const uint16_t *q, const uint16_t *k_cache, const uint16_t *v_cache,
                       int num_blocks, int block_size, int num_kv_heads, int head_dim,
                       const int32_t *block_tables, int max_blocks, const int32_t *seq_lens,
                       int B, int Hq, double scale, double *scores, int nthreads) {
    if (B <= 0 || Hq <= 0 || num_kv_heads <= 0 || Hq % num_kv_heads != 0 || head_dim <= 0 ||
        block_size <= 0 || max_blocks <= 0 || n_rows < 0)
        return ORACLE_EBADARG;
    int rc = check_tables(block_tables, max_blocks, seq_lens, B, num_blocks, block_size);
    if (rc) return rc;
    for (int i = 0; i < n_rows; ++i)
        if (rows_b[i] < 0 || rows_b[i] >= B || rows_h[i] < 0 || rows_h[i] >= Hq) return ORACLE_EBADARG;
    const int group = Hq / num_kv_heads;
    const int64_t lmax = (int64_t)max_blocks * block_size;
    const int nt = team_size(nthreads);
#pragma omp parallel num_threads(nt)
    {
        int tid = 0;
#ifdef _OPENMP
        tid = omp_get_thread_num();
#endif
        double *my_scores = scores + (int64_t)tid * lmax;
#pragma omp for schedule(dynamic, 1)
        for (int i = 0; i < n_rows; ++i) {
            const int b = rows_b[i], h = rows_h[i];
            const int g = h / group;
            const double l = attend_range(out + (int64_t)i * head_dim,
                                          q + ((int64_t)b * Hq + h) * head_dim, k_cache, v_cache,
                                          block_tables + (int64_t)b * max_blocks, 0, seq_lens[b],
                                          block_size, num_kv_heads, head_dim, g, scale,
                                          my_scores);
            if (lse) lse[i] = l;
        }
    }
    return ORACLE_OK;
}

/*
 * Multi-query decode: the last q_len tokens of each sequence are this step's
 * queries (speculative verification of drafted tokens, or a chunk of new
 * tokens), already written into the pool.  The pages name both uses
 * ("mini-infer" psmarter write-up, feature list items 3 and 5: chunked
 * prefill, speculative decoding; "mini-infer" prajwal7-2002 docs, table
 * "Core Capabilities at a Glance", row "Prompt Ingestion": 512-token chunks,
 * and its overview of a draft model's tokens verified in parallel by the
 * target) without giving the masking rule; the plainest reading is causal
 * attention: query i of sequence b sits at position
 * L - q_len + i (L = seq_lens[b]) and attends to tokens [0, L - q_len + i].
 * A query at a negative position (L < q_len) sees no token: out = 0,
 * lse = -inf.  q and out are [B, q_len, Hq, D]; lse is [B, q_len, Hq]
 * (nullable).
 */
int oracle_decode_mq(double *out, double *lse,
                     const uint16_t *q, int q_len, const uint16_t *k_cache, const uint16_t *v_cache,
                     int num_blocks, int block_size, int num_kv_heads, int head_dim,
                     const int32_t *block_tables, int max_blocks, const int32_t *seq_lens,
                     int B, int Hq, double scale, double *scores, int nthreads) {
    if (B <= 0 || q_len <= 0 || Hq <= 0 || num_kv_heads <= 0 || Hq % num_kv_heads != 0 ||
        head_dim <= 0 || block_size <= 0 || max_blocks <= 0)
        return ORACLE_EBADARG;
    int rc = check_tables(block_tables, max_blocks, seq_lens, B, num_blocks, block_size);
    if (rc) return rc;
    const int group = Hq / num_kv_heads;
    const int64_t lmax = (int64_t)max_blocks * block_size;
    const int64_t n_rows = (int64_t)B * q_len * Hq;
    const int nt = team_size(nthreads);
#pragma omp parallel num_threads(nt)
    {
        int tid = 0;
#ifdef _OPENMP
        tid = omp_get_thread_num();
#endif
        double *my_scores = scores + (int64_t)tid * lmax;
#pragma omp for schedule(dynamic, 1)
        for (int64_t r = 0; r < n_rows; ++r) {  /* r = (b * q_len + i) * Hq + h */
            const int h = (int)(r % Hq);
            const int i = (int)((r / Hq) % q_len);
            const int b = (int)(r / ((int64_t)Hq * q_len));
            int visible = seq_lens[b] - q_len + i + 1;  /* tokens [0, position] */
            if (visible < 0) visible = 0;
            const double l = attend_range(out + r * head_dim, q + r * head_dim, k_cache, v_cache,
                                          block_tables + (int64_t)b * max_blocks, 0, visible,
                                          block_size, num_kv_heads, head_dim, h / group,
                                          scale, my_scores);
            if (lse) lse[r] = l;
        }
    }
    return ORACLE_OK;
}

/*
 * Split-K / split-KV partials (psmarter write-up, feature 7; tom-jerr
 * "Attention Backend" table).  Partition p of sequence b covers tokens
 * [p*chunk, min((p+1)*chunk, L)); part_o is [B, Hq, P, D] and part_lse is
 * [B, Hq, P].  Each partial is normalised within its own range.
 */
int oracle_decode_partial(double *part_o, double *part_lse,
                          const uint16_t *q, const uint16_t *k_cache, const uint16_t *v_cache,
                          int num_blocks, int block_size, int num_kv_heads, int head_dim,
                          const int32_t *block_tables, int max_blocks, const int32_t *seq_lens,
                          int B, int Hq, double scale, int num_parts, int chunk,
                          double *scores, int nthreads) {
    if (B <= 0 || Hq <= 0 || num_kv_heads <= 0 || Hq % num_kv_heads != 0 || head_dim <= 0 ||
        block_size <= 0 || max_blocks <= 0 || num_parts <= 0 || chunk <= 0)
        return ORACLE_EBADARG;
    int rc = check_tables(block_tables, max_blocks, seq_lens, B, num_blocks, block_size);
    if (rc) return rc;
    const int group = Hq / num_kv_heads;
    const int64_t lmax = (int64_t)max_blocks * block_size;
    const int nt = team_size(nthreads);
#pragma omp parallel num_threads(nt)
    {
        int tid = 0;
#ifdef _OPENMP
        tid = omp_get_thread_num();
#endif
        double *my_scores = scores + (int64_t)tid * lmax;
#pragma omp for schedule(dynamic, 1) collapse(2)
        for (int b = 0; b < B; ++b) {
            for (int h = 0; h < Hq; ++h) {
                const int L = seq_lens[b];
                for (int p = 0; p < num_parts; ++p) {
                    int64_t t0 = (int64_t)p * chunk, t1 = t0 + chunk;
                    if (t0 > L) t0 = L;
                    if (t1 > L) t1 = L;
                    const int64_t row = ((int64_t)b * Hq + h) * num_parts + p;
                    part_lse[row] = attend_range(part_o + row * head_dim,
                                                 q + ((int64_t)b * Hq + h) * head_dim, k_cache, v_cache,
                                                 block_tables + (int64_t)b * max_blocks, (int)t0, (int)t1,
                                                 block_size, num_kv_heads, head_dim, h / group,
                                                 scale, my_scores);
                }
            }
        }
    }
    return ORACLE_OK;
}

/*
 * Log-sum-exp combine of P partials per row:
 *   lse = M + ln sum_p exp(lse_p - M),  M = max_p lse_p
 *   out = sum_p exp(lse_p - lse) * o_p
 * A partial with lse_p = -inf carries weight 0; all -inf gives out = 0,
 * lse = -inf.  part_o is [rows, P, D], part_lse is [rows, P].
 */
int oracle_combine(double *out, double *lse, const double *part_o, const double *part_lse,
                   int64_t rows, int num_parts, int head_dim) {
    if (rows < 0 || num_parts <= 0 || head_dim <= 0) return ORACLE_EBADARG;
    for (int64_t r = 0; r < rows; ++r) {
        const double *pl = part_lse + r * num_parts;
        double m = -INFINITY;
        for (int p = 0; p < num_parts; ++p)
            if (pl[p] > m) m = pl[p];
        double *o = out + r * head_dim;
        for (int d = 0; d < head_dim; ++d) o[d] = 0.0;
        if (m == -INFINITY) {
            if (lse) lse[r] = -INFINITY;
            continue;
        }
        double z = 0.0;
        for (int p = 0; p < num_parts; ++p) z += exp(pl[p] - m);
        const double total = m + log(z);
        for (int p = 0; p < num_parts; ++p) {
            const double w = exp(pl[p] - total);
            if (w == 0.0) continue;
            const double *op = part_o + (r * num_parts + p) * head_dim;
            for (int d = 0; d < head_dim; ++d) o[d] += w * op[d];
        }
        if (lse) lse[r] = total;
    }
    return ORACLE_OK;
}
