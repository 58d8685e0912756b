/*
 * Paged-attention decode oracle: a slow, plain, fp64 restatement of what the
 * decode step computes.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may call, link or
 * load this file: only the tests, the smoke check and the benchmark's CPU
 * baseline leg use it.  It shares no code, header, table or constant with the
 * CUDA library; it is written from the pages' statement of the problem.
 *
 * What it follows:
 *   - "benchmark_decoding.py", function reference_output: for each sequence b
 *     and query head h, gather the logical sequence of keys/values through the
 *     block table, then out[b,h] = softmax(q[b,h] . K^T * scale) . V.
 *   - MiniVLLM docs "Decoding Benchmark", section "Block table lookup
 *     mechanics": logical token t of sequence b lives in physical block
 *     block_tables[b][t // block_size] at slot t % block_size; -1 marks an
 *     unallocated slot.
 *   - "benchmark_decoding.py", Triton (new) kernel: query head h reads kv head
 *     h // (num_heads / num_kv_heads); the cache is laid out
 *     [num_blocks, block_size, num_kv_heads, head_dim], contiguous.
 *
 * Readings taken where the pages are silent or disagree (each is a choice the
 * CUDA path must make identically, and each is pinned by a test):
 *   - A table entry that is -1, or outside [0, num_blocks), inside the used
 *     range excludes that token from the softmax (the Triton (new) kernel's
 *     masking); it is never dereferenced.
 *   - Tokens at or beyond max_blocks * block_size are not reachable through a
 *     table row and are excluded; a negative context length counts as 0.
 *   - A sequence with no attended token (context length 0, or every entry
 *     masked) yields an all-zero output row instead of the pages' 0/0.
 *
 * Arithmetic: every input element is widened exactly to double; scores,
 * max, exp (libm) and the weighted sum are all in double.  The walk does one
 * block-table lookup per token, as the pages' per-token gather does.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define PAO_F16 0
#define PAO_BF16 1

/* IEEE 754 binary16 -> double, from the format's definition:
 * 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits. */
static double pao_half_to_double(uint16_t h) {
    int sign = (h >> 15) & 1;
    int e = (h >> 10) & 0x1f;
    int f = h & 0x3ff;
    double v;
    if (e == 0) {
        v = ldexp((double)f, -24); /* subnormal: f * 2^-14 * 2^-10 */
    } else if (e == 31) {
        v = (f == 0) ? INFINITY : NAN;
    } else {
        v = ldexp((double)(1024 + f), e - 25); /* (1 + f/1024) * 2^(e-15) */
    }
    return sign ? -v : v;
}

/* bfloat16 -> double: bf16 is the upper half of an IEEE binary32. */
static double pao_bf16_to_double(uint16_t h) {
    uint32_t bits = ((uint32_t)h) << 16;
    float f;
    memcpy(&f, &bits, sizeof f);
    return (double)f;
}

static double pao_elem(const uint16_t* base, size_t idx, int dtype) {
    return dtype == PAO_BF16 ? pao_bf16_to_double(base[idx]) : pao_half_to_double(base[idx]);
}

/* Number of tokens of sequence b that a table row can reach. */
static int64_t pao_reachable(const int32_t* context_lens, int b, int block_size, int max_blocks) {
    int64_t t = context_lens[b];
    int64_t cap = (int64_t)max_blocks * block_size;
    if (t < 0) t = 0;
    if (t > cap) t = cap;
    return t;
}

/* Physical block of logical token t of sequence b, or -1 if masked. */
static int64_t pao_lookup(const int32_t* block_tables, int b, int64_t t, int block_size,
                          int max_blocks, int64_t num_blocks) {
    int64_t j = t / block_size;
    int64_t e = block_tables[(int64_t)b * max_blocks + j];
    if (e < 0 || e >= num_blocks) return -1;
    return e;
}

/* Attention of one query row against tokens t < n of sequence b, kv head
 * `kvh`, into out[0..head_dim).  `qoff` is the row's element offset in q.
 * Returns 0, or -1 if scratch memory could not be had. */
static int pao_attend(double* out, const uint16_t* q, size_t qoff, const uint16_t* k_cache,
                      const uint16_t* v_cache, const int32_t* block_tables, int b, int kvh,
                      int64_t n, int num_kv_heads, int head_dim, int block_size, int max_blocks,
                      int64_t num_blocks, int dtype, double scale) {
    size_t row_stride = (size_t)num_kv_heads * head_dim;          /* one token slot */
    size_t block_stride = (size_t)block_size * row_stride;        /* one physical block */

    for (int d = 0; d < head_dim; ++d) out[d] = 0.0;
    if (n <= 0) return 0;

    double* s = (double*)malloc(sizeof(double) * (size_t)n);
    unsigned char* keep = (unsigned char*)malloc((size_t)n);
    if (!s || !keep) {
        free(s);
        free(keep);
        return -1;
    }

    /* scores s_t = scale * sum_d q[d] K_t[d] over the attended tokens */
    double smax = -INFINITY;
    int64_t kept = 0;
    for (int64_t t = 0; t < n; ++t) {
        int64_t phys = pao_lookup(block_tables, b, t, block_size, max_blocks, num_blocks);
        keep[t] = phys >= 0;
        if (!keep[t]) continue;
        size_t koff = (size_t)phys * block_stride + (size_t)(t % block_size) * row_stride +
                      (size_t)kvh * head_dim;
        double acc = 0.0;
        for (int d = 0; d < head_dim; ++d)
            acc += pao_elem(q, qoff + d, dtype) * pao_elem(k_cache, koff + d, dtype);
        s[t] = scale * acc;
        if (s[t] > smax) smax = s[t];
        ++kept;
    }

    if (kept > 0) {
        /* softmax weights w_t = exp(s_t - max) and out = sum_t w_t V_t / sum_t w_t */
        double wsum = 0.0;
        for (int64_t t = 0; t < n; ++t) {
            if (!keep[t]) continue;
            int64_t phys = pao_lookup(block_tables, b, t, block_size, max_blocks, num_blocks);
            size_t voff = (size_t)phys * block_stride + (size_t)(t % block_size) * row_stride +
                          (size_t)kvh * head_dim;
            double w = exp(s[t] - smax);
            wsum += w;
            for (int d = 0; d < head_dim; ++d) out[d] += w * pao_elem(v_cache, voff + d, dtype);
        }
        for (int d = 0; d < head_dim; ++d) out[d] /= wsum;
    }
    free(s);
    free(keep);
    return 0;
}

/* Attention output of one (b, h) pair of a one-token decode. */
static int pao_one(double* out, const uint16_t* q, const uint16_t* k_cache,
                   const uint16_t* v_cache, const int32_t* block_tables,
                   const int32_t* context_lens, int b, int h, int num_heads, int num_kv_heads,
                   int head_dim, int block_size, int max_blocks, int64_t num_blocks, int dtype,
                   double scale) {
    int group = num_heads / num_kv_heads;
    int kvh = h / group;
    int64_t n = pao_reachable(context_lens, b, block_size, max_blocks);
    const size_t qoff = ((size_t)b * num_heads + h) * head_dim;
    return pao_attend(out, q, qoff, k_cache, v_cache, block_tables, b, kvh, n, num_kv_heads,
                      head_dim, block_size, max_blocks, num_blocks, dtype, scale);
}

static int pao_shape_ok(int batch, int num_heads, int num_kv_heads, int head_dim, int block_size,
                        int max_blocks, int64_t num_blocks, int dtype) {
    if (batch < 0 || num_heads <= 0 || num_kv_heads <= 0 || head_dim <= 0) return 0;
    if (block_size <= 0 || max_blocks < 0 || num_blocks < 0) return 0;
    if (num_heads % num_kv_heads != 0) return 0;
    if (dtype != PAO_F16 && dtype != PAO_BF16) return 0;
    return 1;
}

/* Full decode: out[b][h][d] (double), for every b < batch and h < num_heads.
 * q: [batch, num_heads, head_dim]; k_cache, v_cache:
 * [num_blocks, block_size, num_kv_heads, head_dim]; block_tables:
 * [batch, max_blocks] int32; context_lens: [batch] int32; elements are raw
 * 16-bit patterns of the given dtype (0 = fp16, 1 = bf16).
 * Returns 0 on success, -1 on a bad shape or out of host memory. */
int pao_decode(double* out, const uint16_t* q, const uint16_t* k_cache, const uint16_t* v_cache,
               const int32_t* block_tables, const int32_t* context_lens, int batch,
               int num_heads, int num_kv_heads, int head_dim, int block_size, int max_blocks,
               int64_t num_blocks, int dtype, double scale) {
    if (!pao_shape_ok(batch, num_heads, num_kv_heads, head_dim, block_size, max_blocks,
                      num_blocks, dtype))
        return -1;
    for (int b = 0; b < batch; ++b)
        for (int h = 0; h < num_heads; ++h)
            if (pao_one(out + ((size_t)b * num_heads + h) * head_dim, q, k_cache, v_cache,
                        block_tables, context_lens, b, h, num_heads, num_kv_heads, head_dim,
                        block_size, max_blocks, num_blocks, dtype, scale))
                return -1;
    return 0;
}

/* Selected rows only: rows[2*i] = b, rows[2*i+1] = h; out[i][d].  Used to
 * check sampled outputs of workloads too large to walk whole. */
int pao_decode_rows(double* out, const uint16_t* q, const uint16_t* k_cache,
                    const uint16_t* v_cache, const int32_t* block_tables,
                    const int32_t* context_lens, int batch, int num_heads, int num_kv_heads,
                    int head_dim, int block_size, int max_blocks, int64_t num_blocks, int dtype,
                    double scale, const int32_t* rows, int nrows) {
    if (!pao_shape_ok(batch, num_heads, num_kv_heads, head_dim, block_size, max_blocks,
                      num_blocks, dtype))
        return -1;
    for (int i = 0; i < nrows; ++i) {
        int b = rows[2 * i], h = rows[2 * i + 1];
        if (b < 0 || b >= batch || h < 0 || h >= num_heads) return -1;
        if (pao_one(out + (size_t)i * head_dim, q, k_cache, v_cache, block_tables, context_lens,
                    b, h, num_heads, num_kv_heads, head_dim, block_size, max_blocks, num_blocks,
                    dtype, scale))
            return -1;
    }
    return 0;
}

/* The physical block each (b, logical block j) resolves to on the token walk:
 * out_phys[b][j] = the block read for tokens of page j, or -1 where page j holds
 * no attended token (beyond the context, or a masked entry). */
int pao_resolve_blocks(int32_t* out_phys, const int32_t* block_tables, const int32_t* context_lens,
                       int batch, int block_size, int max_blocks, int64_t num_blocks) {
    if (batch < 0 || block_size <= 0 || max_blocks < 0 || num_blocks < 0) return -1;
    for (int b = 0; b < batch; ++b) {
        for (int j = 0; j < max_blocks; ++j) out_phys[(size_t)b * max_blocks + j] = -1;
        int64_t n = pao_reachable(context_lens, b, block_size, max_blocks);
        for (int64_t t = 0; t < n; ++t) {
            int64_t phys = pao_lookup(block_tables, b, t, block_size, max_blocks, num_blocks);
            out_phys[(size_t)b * max_blocks + t / block_size] = (int32_t)phys;
        }
    }
    return 0;
}

/* Append of one new token per sequence to the paged cache (MiniVLLM docs
 * "Decoding Benchmark", "What paged attention decode does": each decode step
 * adds one token whose keys/values are stored in the block the table assigns,
 * at slot position % block_size).  For each b with 0 <= positions[b] <
 * max_blocks * block_size and table entry e = block_tables[b][positions[b] /
 * block_size] in [0, num_blocks): k_cache[e][positions[b] % block_size][:][:] =
 * k_new[b][:][:] (all kv heads), and likewise for v.  Other sequences write
 * nothing.  Elements are copied as raw 16-bit patterns.  Returns 0, or -1 on a
 * bad shape. */
int pao_append_kv(uint16_t* k_cache, uint16_t* v_cache, const uint16_t* k_new,
                  const uint16_t* v_new, const int32_t* block_tables, const int32_t* positions,
                  int batch, int num_kv_heads, int head_dim, int block_size, int max_blocks,
                  int64_t num_blocks) {
    if (batch < 0 || num_kv_heads <= 0 || head_dim <= 0 || block_size <= 0 || max_blocks < 0 ||
        num_blocks < 0)
        return -1;
    size_t row = (size_t)num_kv_heads * head_dim; /* one token slot, all kv heads */
    for (int b = 0; b < batch; ++b) {
        int64_t pos = positions[b];
        if (pos < 0 || pos >= (int64_t)max_blocks * block_size) continue;
        int64_t e = block_tables[(int64_t)b * max_blocks + pos / block_size];
        if (e < 0 || e >= num_blocks) continue;
        size_t dst = ((size_t)e * block_size + (size_t)(pos % block_size)) * row;
        for (size_t i = 0; i < row; ++i) {
            k_cache[dst + i] = k_new[(size_t)b * row + i];
            v_cache[dst + i] = v_new[(size_t)b * row + i];
        }
    }
    return 0;
}

/* Several query tokens per sequence (a multi-token decode step, e.g. the
 * verification of drafted tokens): q and out are [batch, q_len, num_heads,
 * head_dim]; context_lens[b] counts the q_len new tokens, which are already
 * in the cache at positions T - q_len .. T - 1.  Query token i sits at
 * position p = T - q_len + i and attends causally to the tokens t <= p that a
 * table row reaches (the same masking as the one-token decode); a query with
 * no attended token gets zeros.  With q_len = 1 this is pao_decode. */
int pao_decode_multi(double* out, const uint16_t* q, const uint16_t* k_cache,
                     const uint16_t* v_cache, const int32_t* block_tables,
                     const int32_t* context_lens, int batch, int q_len, int num_heads,
                     int num_kv_heads, int head_dim, int block_size, int max_blocks,
                     int64_t num_blocks, int dtype, double scale) {
    if (!pao_shape_ok(batch, num_heads, num_kv_heads, head_dim, block_size, max_blocks,
                      num_blocks, dtype) || q_len <= 0)
        return -1;
    int group = num_heads / num_kv_heads;
    for (int b = 0; b < batch; ++b) {
        int64_t reach = pao_reachable(context_lens, b, block_size, max_blocks);
        int64_t T = context_lens[b];
        for (int i = 0; i < q_len; ++i) {
            int64_t n = T - q_len + i + 1; /* tokens 0 .. p */
            if (n > reach) n = reach;
            for (int h = 0; h < num_heads; ++h) {
                size_t row = ((size_t)b * q_len + i) * num_heads + h;
                if (pao_attend(out + row * head_dim, q, row * head_dim, k_cache, v_cache,
                               block_tables, b, h / group, n, num_kv_heads, head_dim, block_size,
                               max_blocks, num_blocks, dtype, scale))
                    return -1;
            }
        }
    }
    return 0;
}
