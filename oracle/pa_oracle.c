/*
 * Paged-KV decode attention: plain fp64 CPU oracle.
 *
 * TEST INFRASTRUCTURE ONLY. This file is the independent checker for the CUDA
 * path. Only the test suite, the smoke check and the benchmark's CPU-baseline
 * leg may load it. It shares no code, header, table or helper with the CUDA
 * library, and it does none of the CUDA path's blocking, splitting or fusion:
 * it gathers each sequence's context into a contiguous buffer and runs dense
 * masked attention over it, one query row at a time.
 *
 * What it computes, and where each step comes from:
 *
 *  - Cache layout. The caches are head-major, [kv_heads, num_blocks,
 *    block_size, head_dim], so one index over a sequence's slots returns its
 *    context in order ("From 183 ms to 19 ms per decode step", section
 *    "2. Head-major KV cache"). Token t of sequence b lives in physical block
 *    block_tables[b][t / block_size] at row t % block_size.
 *
 *  - Cache write (slot-mapping scatter). Each step's per-token inputs include
 *    the cache slots of the new tokens ("From 183 ms to 19 ms per decode
 *    step", section "4. CUDA graphs per batch bucket"). Slot s is block
 *    s / block_size, row s % block_size. The new K/V are written before the
 *    step attends ("Anatomy of a Decode-Step Stall", the engine's Model._layer
 *    writes K[l, positions[i]] and then attends over [:end]). A negative slot
 *    is skipped (reading: a padded token with no slot). Writes are applied in
 *    token order, so with duplicate slots the last write wins.
 *
 *  - Attention. The plain per-row softmax of the stall article's
 *    Model._layer: scores = K q * scale, subtract the max, exponentiate,
 *    normalise, weight V. Grouped-query: query head hq reads KV head
 *    hq / (q_heads / kv_heads), the contiguous grouping that repeat_kv
 *    expansion implies ("A Rust inference server for Qwen2 on Apple Silicon",
 *    Day 3 "Throughput against concurrency", cost 2; "From 183 ms to 19 ms per
 *    decode step", section "1. Grouped attention").
 *
 *  - Verify rows. A verify step carries num_queries new tokens per sequence
 *    with a causal mask among them ("From 183 ms to 19 ms per decode step",
 *    section "Then speculative decoding got slower"). context_lens includes
 *    the new tokens, so query i sits at position L - num_queries + i and
 *    attends to positions t <= L - num_queries + i. Decode is num_queries = 1.
 *
 *  - A row with no key to attend to (L = 0, or a verify row whose position is
 *    negative) returns zeros (reading: the pages are silent; zeros and no NaN).
 *
 * Everything is done in double precision. bf16 and fp32 inputs convert to
 * double exactly.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORACLE_F32 0
#define ORACLE_BF16 1

static size_t elem_bytes(int dtype) { return dtype == ORACLE_F32 ? 4u : 2u; }

/* Exact widening of one stored element to double. bf16 is the top half of
 * an IEEE binary32 pattern. */
static double load_elem(const void *base, int dtype, int64_t index) {
    if (dtype == ORACLE_F32) {
        return (double)((const float *)base)[index];
    }
    uint32_t bits = ((uint32_t)((const uint16_t *)base)[index]) << 16;
    float f;
    memcpy(&f, &bits, sizeof f);
    return (double)f;
}

int oracle_max_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

void oracle_set_threads(int n) {
#ifdef _OPENMP
    if (n > 0) omp_set_num_threads(n);
#else
    (void)n;
#endif
}

/*
 * Slot-mapping scatter: cache[h, s / bs, s % bs, :] = new[i, h, :] for every
 * token i with slot s = slot_mapping[i] >= 0, copied bit for bit.
 * k_new / v_new: [num_tokens, kv_heads, head_dim] in the cache dtype.
 * Returns the number of slots that were out of range (>= num_blocks * bs);
 * those tokens are skipped.
 */
int oracle_cache_write(void *k_cache, void *v_cache, int dtype, int kv_heads,
                       int num_blocks, int block_size, int head_dim,
                       const void *k_new, const void *v_new,
                       const int32_t *slot_mapping, int num_tokens) {
    const size_t es = elem_bytes(dtype);
    const size_t row_bytes = (size_t)head_dim * es;
    const int64_t num_slots = (int64_t)num_blocks * block_size;
    int out_of_range = 0;
    for (int i = 0; i < num_tokens; ++i) {
        const int64_t slot = slot_mapping[i];
        if (slot < 0) continue;
        if (slot >= num_slots) {
            ++out_of_range;
            continue;
        }
        const int64_t block = slot / block_size;
        const int64_t row = slot % block_size;
        for (int h = 0; h < kv_heads; ++h) {
            const int64_t dst = (((int64_t)h * num_blocks + block) * block_size + row) * head_dim;
            const int64_t src = ((int64_t)i * kv_heads + h) * head_dim;
            memcpy((char *)k_cache + dst * es, (const char *)k_new + src * es, row_bytes);
            memcpy((char *)v_cache + dst * es, (const char *)v_new + src * es, row_bytes);
        }
    }
    return out_of_range;
}

/*
 * Dense masked grouped-query attention over each sequence's gathered context.
 *
 * q:   [batch, num_queries, q_heads, head_dim] in the cache dtype.
 * out: [batch, num_queries, q_heads, head_dim] doubles; only sequences in
 *      [b_begin, b_end) are written.
 * block_tables: [batch, max_blocks_per_seq]; context_lens: [batch].
 *
 * Returns 0, or the number of sequences whose length or block ids were out of
 * range (their rows are set to zero and nothing out of range is read).
 */
int oracle_attend(const void *k_cache, const void *v_cache, int dtype,
                  int kv_heads, int num_blocks, int block_size, int head_dim,
                  const void *q, double *out, const int32_t *block_tables,
                  int max_blocks_per_seq, const int32_t *context_lens,
                  int batch, int q_heads, int num_queries, double scale,
                  int b_begin, int b_end) {
    if (kv_heads <= 0 || q_heads % kv_heads != 0) return -1;
    if (b_begin < 0) b_begin = 0;
    if (b_end > batch) b_end = batch;
    const int group = q_heads / kv_heads;
    int bad = 0;

#pragma omp parallel for schedule(dynamic, 1) reduction(+ : bad)
    for (int b = b_begin; b < b_end; ++b) {
        const int64_t L = context_lens[b];
        const int64_t row_elems = (int64_t)num_queries * q_heads * head_dim;
        double *out_b = out + (int64_t)b * row_elems;

        /* Validate this sequence's length and the block ids it uses. */
        int ok = (L >= 0 && L <= (int64_t)max_blocks_per_seq * block_size);
        for (int64_t j = 0; ok && j < (L + block_size - 1) / block_size; ++j) {
            const int32_t pb = block_tables[(int64_t)b * max_blocks_per_seq + j];
            if (pb < 0 || pb >= num_blocks) ok = 0;
        }
        if (!ok) {
            for (int64_t e = 0; e < row_elems; ++e) out_b[e] = 0.0;
            bad += 1;
            continue;
        }

        /* Gather the context into contiguous [kv_heads, L, head_dim] buffers. */
        const int64_t ctx_elems = (int64_t)kv_heads * (L > 0 ? L : 1) * head_dim;
        double *Kc = (double *)malloc((size_t)ctx_elems * sizeof(double));
        double *Vc = (double *)malloc((size_t)ctx_elems * sizeof(double));
        double *s = (double *)malloc((size_t)(L > 0 ? L : 1) * sizeof(double));
        for (int h = 0; h < kv_heads; ++h) {
            for (int64_t t = 0; t < L; ++t) {
                const int32_t pb = block_tables[(int64_t)b * max_blocks_per_seq + t / block_size];
                const int64_t src = (((int64_t)h * num_blocks + pb) * block_size + t % block_size) * head_dim;
                const int64_t dst = ((int64_t)h * L + t) * head_dim;
                for (int d = 0; d < head_dim; ++d) {
                    Kc[dst + d] = load_elem(k_cache, dtype, src + d);
                    Vc[dst + d] = load_elem(v_cache, dtype, src + d);
                }
            }
        }

        for (int i = 0; i < num_queries; ++i) {
            /* Query i sits at position L - num_queries + i and sees t <= that. */
            const int64_t visible = L - num_queries + i + 1;
            for (int hq = 0; hq < q_heads; ++hq) {
                const int h = hq / group;
                const int64_t qoff = (((int64_t)b * num_queries + i) * q_heads + hq) * head_dim;
                double *o = out + qoff;
                for (int d = 0; d < head_dim; ++d) o[d] = 0.0;
                if (visible <= 0) continue;

                double m = -INFINITY;
                for (int64_t t = 0; t < visible; ++t) {
                    const double *k = Kc + ((int64_t)h * L + t) * head_dim;
                    double dot = 0.0;
                    for (int d = 0; d < head_dim; ++d) dot += load_elem(q, dtype, qoff + d) * k[d];
                    s[t] = dot * scale;
                    if (s[t] > m) m = s[t];
                }
                double denom = 0.0;
                for (int64_t t = 0; t < visible; ++t) {
                    s[t] = exp(s[t] - m);
                    denom += s[t];
                }
                for (int64_t t = 0; t < visible; ++t) {
                    const double *v = Vc + ((int64_t)h * L + t) * head_dim;
                    const double w = s[t] / denom;
                    for (int d = 0; d < head_dim; ++d) o[d] += w * v[d];
                }
            }
        }
        free(Kc);
        free(Vc);
        free(s);
    }
    return bad;
}

/*
 * int8 KV cache ("A Rust inference server for Qwen2 on Apple Silicon",
 * Day 4 measurements, sections "int8 KV", "Grouping is the whole question"
 * and "Partial blocks").
 *
 *  - Codes. Symmetric int8 values q in [-127, 127], stored as the byte
 *    q + 128 (the page keeps u8 with a +128 offset).
 *  - Groups. K is scaled per channel within a block: one scale per (kv head,
 *    block, channel), spanning the block's rows. V is scaled per token: one
 *    scale per (kv head, block, row). This is the KIVI grouping the page
 *    adopts.
 *  - Quantising a group is done in fp32, the precision of the page's
 *    tensors. The stored scale is s = max |x| / 127, and q = x * (127 / max|x|)
 *    rounded to nearest, clamped to [-127, 127]. (Reading: the page fixes
 *    the scale by the group's largest magnitude but not how a code is
 *    rounded; this takes the usual quantiser form, one inverse scale per
 *    group and a multiply per element, rounded with IEEE's default, ties to
 *    even.) An all-zero group gets s = 0 and bytes 128 (reading: the page is
 *    silent on it).
 *  - Dequantising is one fp32 multiply: x = (byte - 128) * s.
 *  - Writing rows ("Partial blocks"). For each block that receives rows in a
 *    call, the block's K rows are dequantised, the incoming rows overwrite
 *    theirs, every channel's scale is recomputed over the block's rows, and
 *    all rows are requantised. Each incoming V row is quantised on its own.
 *    Rows never written hold byte 128 (zero), so they cannot raise a maximum.
 *    (Reading: all rows one call writes into a block are overwritten
 *    together before the block's single requantisation; with duplicate slots
 *    the later token wins, as in the plain write.)
 *
 * New rows arrive as bf16 bit patterns and widen to fp32 exactly.
 */

static float q8_widen_bf16(uint16_t bits) {
    const uint32_t u = (uint32_t)bits << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

/* Scale of a group whose largest magnitude is maxabs. */
static float q8_scale(float maxabs) { return maxabs / 127.0f; }

/* Inverse scale used to quantise that group (0 for an all-zero group). */
static float q8_inverse(float maxabs) { return maxabs == 0.0f ? 0.0f : 127.0f / maxabs; }

/* Stored byte of value x in a group of inverse scale inv. */
static uint8_t q8_code(float x, float inv) {
    if (inv == 0.0f) return 128;
    float r = rintf(x * inv);
    if (r > 127.0f) r = 127.0f;
    if (r < -127.0f) r = -127.0f;
    return (uint8_t)((int)r + 128);
}

static float q8_value(uint8_t byte, float s) { return (float)((int)byte - 128) * s; }

/*
 * Quantised slot-mapping write. Codes: [kv_heads, num_blocks, block_size,
 * head_dim] bytes; k_scale: [kv_heads, num_blocks, head_dim] fp32; v_scale:
 * [kv_heads, num_blocks, block_size] fp32. k_new / v_new: [num_tokens,
 * kv_heads, head_dim] bf16 bits. Negative slots are skipped; out-of-range
 * slots are skipped and counted (the return value).
 */
int oracle_cache_write_q8(uint8_t *k_codes, uint8_t *v_codes, float *k_scale, float *v_scale,
                          int kv_heads, int num_blocks, int block_size, int head_dim,
                          const uint16_t *k_new, const uint16_t *v_new,
                          const int32_t *slot_mapping, int num_tokens) {
    const int64_t num_slots = (int64_t)num_blocks * block_size;
    int out_of_range = 0;
    float *x = (float *)malloc((size_t)block_size * head_dim * sizeof(float));
    for (int i = 0; i < num_tokens; ++i) {
        const int64_t slot = slot_mapping[i];
        if (slot < 0) continue;
        if (slot >= num_slots) {
            ++out_of_range;
            continue;
        }
        const int64_t block = slot / block_size;
        /* The block is handled once, at the first token of this call that lands in it. */
        int seen = 0;
        for (int j = 0; j < i; ++j) {
            const int64_t sj = slot_mapping[j];
            if (sj >= 0 && sj < num_slots && sj / block_size == block) seen = 1;
        }
        if (seen) continue;
        for (int h = 0; h < kv_heads; ++h) {
            const int64_t blk = (int64_t)h * num_blocks + block;
            uint8_t *kc = k_codes + blk * block_size * head_dim;
            float *ks = k_scale + blk * head_dim;
            /* K: dequantise the block, overwrite the incoming rows, requantise per channel. */
            for (int r = 0; r < block_size; ++r)
                for (int d = 0; d < head_dim; ++d)
                    x[r * head_dim + d] = q8_value(kc[r * head_dim + d], ks[d]);
            for (int j = i; j < num_tokens; ++j) {
                const int64_t sj = slot_mapping[j];
                if (sj < 0 || sj >= num_slots || sj / block_size != block) continue;
                const int r = (int)(sj % block_size);
                const uint16_t *src = k_new + ((int64_t)j * kv_heads + h) * head_dim;
                for (int d = 0; d < head_dim; ++d) x[r * head_dim + d] = q8_widen_bf16(src[d]);
            }
            for (int d = 0; d < head_dim; ++d) {
                float m = 0.0f;
                for (int r = 0; r < block_size; ++r) {
                    const float a = fabsf(x[r * head_dim + d]);
                    if (a > m) m = a;
                }
                ks[d] = q8_scale(m);
                const float inv = q8_inverse(m);
                for (int r = 0; r < block_size; ++r) kc[r * head_dim + d] = q8_code(x[r * head_dim + d], inv);
            }
            /* V: each incoming row on its own scale. */
            for (int j = i; j < num_tokens; ++j) {
                const int64_t sj = slot_mapping[j];
                if (sj < 0 || sj >= num_slots || sj / block_size != block) continue;
                const int r = (int)(sj % block_size);
                const uint16_t *src = v_new + ((int64_t)j * kv_heads + h) * head_dim;
                float m = 0.0f;
                for (int d = 0; d < head_dim; ++d) {
                    const float a = fabsf(q8_widen_bf16(src[d]));
                    if (a > m) m = a;
                }
                v_scale[blk * block_size + r] = q8_scale(m);
                const float inv = q8_inverse(m);
                uint8_t *vc = v_codes + (blk * block_size + r) * head_dim;
                for (int d = 0; d < head_dim; ++d) vc[d] = q8_code(q8_widen_bf16(src[d]), inv);
            }
        }
    }
    free(x);
    return out_of_range;
}

/* Dequantise a whole pool into fp32 caches of the plain layout. */
void oracle_dequant_q8(const uint8_t *k_codes, const uint8_t *v_codes, const float *k_scale,
                       const float *v_scale, int kv_heads, int num_blocks, int block_size,
                       int head_dim, float *k_out, float *v_out) {
    for (int64_t blk = 0; blk < (int64_t)kv_heads * num_blocks; ++blk)
        for (int r = 0; r < block_size; ++r)
            for (int d = 0; d < head_dim; ++d) {
                const int64_t e = (blk * block_size + r) * head_dim + d;
                k_out[e] = q8_value(k_codes[e], k_scale[blk * head_dim + d]);
                v_out[e] = q8_value(v_codes[e], v_scale[blk * block_size + r]);
            }
}
