/*
 * Plain CPU oracle for paged single-token decode attention and for the KV
 * append scatter.  TEST INFRASTRUCTURE ONLY: it is loaded by the tests, by the
 * package's smoke check and by the benchmark's CPU-baseline leg, never by the
 * CUDA library, and it shares no code with it.
 *
 * What it computes (fp64 throughout, no blocking, no reordering):
 *
 *   Paged layout.  "PagedAttention" section of the third page (bbs.pinggu.org
 *   thread 16345627): the KV cache of every sequence is cut into fixed-size
 *   physical blocks that need not be contiguous, a per-sequence block table maps
 *   logical block j to a physical block, and the attention kernel reaches K/V by
 *   looking the block up in that table (indirect addressing).  Here the cache
 *   is k_cache[num_blocks][num_kv_heads][block_size][head_dim] and token t of
 *   sequence i lives in physical block block_tables[i][t / block_size] at row
 *   t % block_size.
 *
 *   Attention.  Section 3.1 of the second page (intelligence-paradigm "model
 *   executor" article, scaled_dot_product_attention): scores = q . k^T * scale,
 *   weights = softmax(scores), out = weights . v.  A decode step has one query
 *   per sequence that attends to all context_lens[i] tokens, so no mask.
 *
 *   Grouped-query heads: query head h reads kv head h / (Hq / Hkv).
 *
 *   Block copy: block pairs[2i] of a source pool is copied to block
 *   pairs[2i+1] of a destination pool, every kv head, K and V (the swap and
 *   copy-on-write moves of the tiered block manager, section 4.2 of the first
 *   page).
 *
 *   KV append: each new token's K/V row is written into slot s of the cache,
 *   block s / block_size, row s % block_size (block manager allocation,
 *   section 4.2 of the first page, 0539edu.com news 6031734; per-iteration
 *   metadata update, "continuous batching" section of the third page).  A
 *   negative slot means "no write".
 *
 * Element storage is the 16-bit pattern of IEEE binary16 (dtype 0) or bfloat16
 * (dtype 1); both are widened exactly to double by converters written from the
 * two format definitions below.
 */
#include <math.h>
#include <stdint.h>
#include <stddef.h>
#include <stdlib.h>
#include <string.h>

/* IEEE 754 binary16: 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits.
 * Normal: (-1)^s * 2^(e-15) * (1 + f/1024).  Subnormal (e == 0):
 * (-1)^s * 2^(-14) * (f/1024).  e == 31: infinity (f == 0) or NaN. */
double pkv_oracle_half_to_double(uint16_t h) {
    int s = (h >> 15) & 1;
    int e = (h >> 10) & 0x1f;
    int f = h & 0x3ff;
    double mag;
    if (e == 0) {
        mag = ldexp((double)f, -24);            /* f/1024 * 2^-14 */
    } else if (e == 31) {
        mag = (f == 0) ? INFINITY : NAN;
    } else {
        mag = ldexp((double)(1024 + f), e - 25); /* (1024+f)/1024 * 2^(e-15) */
    }
    return s ? -mag : mag;
}

/* bfloat16: 1 sign bit, 8 exponent bits (bias 127), 7 fraction bits.
 * Normal: (-1)^s * 2^(e-127) * (1 + f/128).  Subnormal (e == 0):
 * (-1)^s * 2^(-126) * (f/128).  e == 255: infinity (f == 0) or NaN. */
double pkv_oracle_bf16_to_double(uint16_t b) {
    int s = (b >> 15) & 1;
    int e = (b >> 7) & 0xff;
    int f = b & 0x7f;
    double mag;
    if (e == 0) {
        mag = ldexp((double)f, -133);            /* f/128 * 2^-126 */
    } else if (e == 255) {
        mag = (f == 0) ? INFINITY : NAN;
    } else {
        mag = ldexp((double)(128 + f), e - 134); /* (128+f)/128 * 2^(e-127) */
    }
    return s ? -mag : mag;
}

static double widen(uint16_t bits, int dtype) {
    return dtype == 0 ? pkv_oracle_half_to_double(bits)
                      : pkv_oracle_bf16_to_double(bits);
}

/* One (sequence i, query head h) row of decode attention, written to out[0..D).
 * Returns 0, or -1 when the row's inputs break the contract (context length
 * outside [1, max_blocks_per_seq * block_size], or a physical block id outside
 * [0, num_blocks)); out is then left untouched. */
static int attend_one(int i, int h,
                      int Hq, int Hkv, int D, int bs, int NB, int MB, int dtype,
                      const uint16_t* q, const uint16_t* k_cache,
                      const uint16_t* v_cache, const int32_t* block_tables,
                      const int32_t* context_lens, double scale, double* out) {
    int G = Hq / Hkv;
    int g = h / G;                       /* kv head shared by the group */
    int L = context_lens[i];
    if (L < 1 || L > MB * bs) return -1;

    const uint16_t* qrow = q + ((size_t)i * Hq + h) * D;
    double* s = (double*)malloc(sizeof(double) * (size_t)L);
    if (!s) return -1;

    /* scores s_t = scale * sum_d q[d] * k_t[d], tokens gathered by table lookup */
    for (int t = 0; t < L; ++t) {
        int p = block_tables[(size_t)i * MB + t / bs];
        int off = t % bs;
        if (p < 0 || p >= NB) { free(s); return -1; }
        const uint16_t* krow =
            k_cache + (((size_t)p * Hkv + g) * bs + off) * D;
        double acc = 0.0;
        for (int d = 0; d < D; ++d)
            acc += widen(qrow[d], dtype) * widen(krow[d], dtype);
        s[t] = scale * acc;
    }

    /* softmax: m = max_t s_t, w_t = exp(s_t - m), Z = sum_t w_t */
    double m = s[0];
    for (int t = 1; t < L; ++t)
        if (s[t] > m) m = s[t];
    double Z = 0.0;
    for (int t = 0; t < L; ++t) {
        s[t] = exp(s[t] - m);
        Z += s[t];
    }

    /* out[d] = sum_t w_t * v_t[d] / Z */
    for (int d = 0; d < D; ++d) out[d] = 0.0;
    for (int t = 0; t < L; ++t) {
        int p = block_tables[(size_t)i * MB + t / bs];
        int off = t % bs;
        const uint16_t* vrow =
            v_cache + (((size_t)p * Hkv + g) * bs + off) * D;
        for (int d = 0; d < D; ++d) out[d] += s[t] * widen(vrow[d], dtype);
    }
    for (int d = 0; d < D; ++d) out[d] /= Z;
    free(s);
    return 0;
}

/* Whole batch: out[B][Hq][D] in double.  Returns the number of rows that broke
 * the contract (0 when every row was computed). */
int pkv_oracle_decode(int B, int Hq, int Hkv, int D, int bs, int NB, int MB,
                      int dtype, const uint16_t* q, const uint16_t* k_cache,
                      const uint16_t* v_cache, const int32_t* block_tables,
                      const int32_t* context_lens, double scale, double* out) {
    if (B < 0 || Hq < 1 || Hkv < 1 || Hq % Hkv != 0 || D < 1 || bs < 1) return -1;
    int bad = 0;
    for (int i = 0; i < B; ++i)
        for (int h = 0; h < Hq; ++h)
            bad += attend_one(i, h, Hq, Hkv, D, bs, NB, MB, dtype, q, k_cache,
                              v_cache, block_tables, context_lens, scale,
                              out + ((size_t)i * Hq + h) * D) != 0;
    return bad;
}

/* Selected rows only: rows[2r] = sequence, rows[2r+1] = query head, result in
 * out[r][D].  Used to check sampled outputs of full-size batches. */
int pkv_oracle_decode_rows(int Hq, int Hkv, int D, int bs, int NB, int MB,
                           int dtype, const uint16_t* q, const uint16_t* k_cache,
                           const uint16_t* v_cache, const int32_t* block_tables,
                           const int32_t* context_lens, double scale,
                           const int32_t* rows, int nrows, double* out) {
    if (Hq < 1 || Hkv < 1 || Hq % Hkv != 0 || D < 1 || bs < 1) return -1;
    int bad = 0;
    for (int r = 0; r < nrows; ++r)
        bad += attend_one(rows[2 * r], rows[2 * r + 1], Hq, Hkv, D, bs, NB, MB,
                          dtype, q, k_cache, v_cache, block_tables, context_lens,
                          scale, out + (size_t)r * D) != 0;
    return bad;
}

/* KV append: for each token t and kv head h with slot s = slot_mapping[t] >= 0,
 * copy the D 16-bit patterns of k[t][h] and v[t][h] into row s % bs of block
 * s / bs.  Returns the number of slots outside [0, NB * bs) (those are
 * skipped) — negative slots are not errors, they mean "do not write". */
int pkv_oracle_append(int T, int Hkv, int D, int bs, int NB,
                      const uint16_t* k, const uint16_t* v,
                      const int32_t* slot_mapping,
                      uint16_t* k_cache, uint16_t* v_cache) {
    int bad = 0;
    for (int t = 0; t < T; ++t) {
        int s = slot_mapping[t];
        if (s < 0) continue;
        if ((long long)s >= (long long)NB * bs) { ++bad; continue; }
        int blk = s / bs, off = s % bs;
        for (int h = 0; h < Hkv; ++h) {
            size_t dst = (((size_t)blk * Hkv + h) * bs + off) * D;
            size_t src = ((size_t)t * Hkv + h) * D;
            for (int d = 0; d < D; ++d) {
                k_cache[dst + d] = k[src + d];
                v_cache[dst + d] = v[src + d];
            }
        }
    }
    return bad;
}

/* Block copy: for each pair i, block pairs[2i] of src (a pool of src_nb blocks
 * of Hkv * bs * D elements) is copied to block pairs[2i+1] of dst (dst_nb
 * blocks).  Returns the number of pairs with an id outside its pool (those are
 * skipped). */
int pkv_oracle_copy_blocks(int n_pairs, int Hkv, int bs, int D, int src_nb, int dst_nb,
                           const uint16_t* src, uint16_t* dst, const int32_t* pairs) {
    size_t per = (size_t)Hkv * bs * D;
    int bad = 0;
    for (int i = 0; i < n_pairs; ++i) {
        int s = pairs[2 * i], d = pairs[2 * i + 1];
        if (s < 0 || s >= src_nb || d < 0 || d >= dst_nb) { ++bad; continue; }
        for (size_t e = 0; e < per; ++e) dst[(size_t)d * per + e] = src[(size_t)s * per + e];
    }
    return bad;
}
