/*
 * Exact scaled-dot-product attention oracle: plain fp64 C, CPU only.
 *
 * TEST INFRASTRUCTURE.  Only the tests, the smoke check and the benchmark's
 * CPU-baseline leg may load this library.  The CUDA library never links,
 * includes or calls anything here, and nothing here comes from it.
 *
 * What it computes (the plain definition, not the tiled algorithm):
 *   "FlashAttention complete summary" (cell-devlog), section "Attention이 뭔가":
 *       Attention(Q, K, V) = softmax(Q K^T / sqrt(d_k)) V
 *   "FlashAttention complete summary", section "문제": the standard computation
 *       materialises the score row, applies softmax, then multiplies by V.
 *   "Flash Attention ... complete guide" (holysheep), section "Online Softmax
 *       알고리즘": the numerically safe softmax subtracts the maximum m, sums the
 *       exponentials into l and divides by l.
 *   "FlashAttention complete summary", section "FlashAttention 1": the tiled
 *       result is exact ("not an approximation"), so the oracle for the tiled
 *       kernels is the untiled definition.
 *
 * For one query row i of head h in batch b, with J_i the visible keys
 * (all keys; or, causal, keys j <= i + (Nk - Nq), i.e. j <= i when Nq == Nk):
 *     s_j   = scale * sum_c q[c] * k_j[c]                (fp64, bf16 inputs upcast exactly)
 *     m     = max_{j in J_i} s_j
 *     l     = sum_{j in J_i} exp(s_j - m)                (pass 1)
 *     P_j   = exp(s_j - m) / l                           (pass 2)
 *     o[c]  = sum_{j in J_i} P_j * v_j[c]
 *     lse   = m + ln(l)                                  (natural log of the scaled scores)
 * Decode is the same row formula with one query per sequence, J = {0..L_s-1},
 * and key t of sequence s found either at kcache[s][t] (contiguous cache) or at
 * pool[page_table[s][t / page_size]][t % page_size] (paged cache).
 *
 * Layouts (all row-major, bf16 stored as its 16 raw bits):
 *   q  [B, Nq, H, d]   k, v [B, Nk, H, d]   o [B, Nq, H, d] fp64   lse [B, H, Nq] fp64
 * Every entry point returns 0 on success and -1 on a bad argument.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* bf16 -> fp64: the 16 bits are the top half of an IEEE binary32; exact. */
static double bf16_to_f64(uint16_t bits) {
    uint32_t u = ((uint32_t)bits) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

static void set_threads(int nthreads) {
#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
#else
    (void)nthreads;
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
 * One attention row.  q_row: d bf16 values.  keys/vals: pointers to the d
 * bf16 values of each visible key, gathered by the caller.  s: scratch of n
 * doubles that holds the materialised score row.  Writes o_row[d], *lse.
 */
static void attention_row(const uint16_t *q_row, const uint16_t *const *keys,
                          const uint16_t *const *vals, long n, int d, double scale,
                          double *s, double *o_row, double *lse) {
    /* the score row S_i = scale * q_i . k_j, materialised */
    for (long j = 0; j < n; ++j) {
        double acc = 0.0;
        for (int c = 0; c < d; ++c) acc += bf16_to_f64(q_row[c]) * bf16_to_f64(keys[j][c]);
        s[j] = scale * acc;
    }
    /* safe softmax: m = max, pass 1: l = sum exp(s - m) */
    double m = -INFINITY;
    for (long j = 0; j < n; ++j)
        if (s[j] > m) m = s[j];
    double l = 0.0;
    for (long j = 0; j < n; ++j) l += exp(s[j] - m);
    /* pass 2: P_j = exp(s_j - m) / l ; o = sum_j P_j v_j */
    for (int c = 0; c < d; ++c) o_row[c] = 0.0;
    for (long j = 0; j < n; ++j) {
        double p = exp(s[j] - m) / l;
        for (int c = 0; c < d; ++c) o_row[c] += p * bf16_to_f64(vals[j][c]);
    }
    *lse = m + log(l);
}

/* number of keys visible to query row i */
static long visible_keys(int causal, long i, long Nq, long Nk) {
    if (!causal) return Nk;
    long n = i + (Nk - Nq) + 1; /* bottom-right aligned; j <= i when Nq == Nk */
    if (n < 0) n = 0;
    if (n > Nk) n = Nk;
    return n;
}

static int check_shape(int B, int H, long Nq, long Nk, int d) {
    return (B < 0 || H < 0 || Nq < 0 || Nk < 0 || d <= 0) ? -1 : 0;
}

/* scratch for one row: key/value pointer tables and the score row */
typedef struct {
    const uint16_t **keys;
    const uint16_t **vals;
    double *s;
} row_scratch;

static int scratch_alloc(row_scratch *w, long n) {
    size_t cnt = (size_t)(n > 0 ? n : 1);
    w->keys = (const uint16_t **)malloc(cnt * sizeof(*w->keys));
    w->vals = (const uint16_t **)malloc(cnt * sizeof(*w->vals));
    w->s = (double *)malloc(cnt * sizeof(double));
    return (w->keys && w->vals && w->s) ? 0 : -1;
}

static void scratch_free(row_scratch *w) {
    free((void *)w->keys);
    free((void *)w->vals);
    free(w->s);
}

/* one (b, h, i) row of the prefill problem */
static void prefill_row(const uint16_t *q, const uint16_t *k, const uint16_t *v, int H,
                        long Nq, long Nk, int d, int causal, double scale, int b, int h,
                        long i, row_scratch *w, double *o_row, double *lse) {
    long n = visible_keys(causal, i, Nq, Nk);
    const uint16_t *q_row = q + (((size_t)b * Nq + i) * H + h) * d;
    for (long j = 0; j < n; ++j) {
        size_t off = (((size_t)b * Nk + j) * H + h) * d;
        w->keys[j] = k + off;
        w->vals[j] = v + off;
    }
    if (n == 0) { /* no visible key: defined here as O = 0, LSE = -inf */
        for (int c = 0; c < d; ++c) o_row[c] = 0.0;
        *lse = -INFINITY;
        return;
    }
    attention_row(q_row, w->keys, w->vals, n, d, scale, w->s, o_row, lse);
}

/*
 * Full forward: o [B, Nq, H, d] fp64, lse [B, H, Nq] fp64 (lse may be NULL).
 */
int oracle_attn_fwd(const uint16_t *q, const uint16_t *k, const uint16_t *v, int B, int H,
                    long Nq, long Nk, int d, int causal, double scale, double *o, double *lse,
                    int nthreads) {
    if (check_shape(B, H, Nq, Nk, d) || !q || !k || !v || !o) return -1;
    set_threads(nthreads);
    long rows = (long)B * H * Nq;
    int err = 0;
#pragma omp parallel reduction(| : err)
    {
        row_scratch w;
        if (scratch_alloc(&w, Nk)) {
            err = 1;
        } else {
#pragma omp for schedule(dynamic, 16)
            for (long r = 0; r < rows; ++r) {
                int b = (int)(r / ((long)H * Nq));
                int h = (int)((r / Nq) % H);
                long i = r % Nq;
                double l_out;
                prefill_row(q, k, v, H, Nq, Nk, d, causal, scale, b, h, i, &w,
                            o + (((size_t)b * Nq + i) * H + h) * d, &l_out);
                if (lse) lse[((size_t)b * H + h) * Nq + i] = l_out;
            }
        }
        scratch_free(&w);
    }
    return err ? -1 : 0;
}

/*
 * Selected rows only.  rows: nrows triples (b, h, i) as int64.  o_rows
 * [nrows, d] fp64, lse_rows [nrows] fp64.  Same row formula as above.
 */
int oracle_attn_rows(const uint16_t *q, const uint16_t *k, const uint16_t *v, int B, int H,
                     long Nq, long Nk, int d, int causal, double scale, const int64_t *rows,
                     long nrows, double *o_rows, double *lse_rows, int nthreads) {
    if (check_shape(B, H, Nq, Nk, d) || !q || !k || !v || !rows || !o_rows || !lse_rows)
        return -1;
    for (long r = 0; r < nrows; ++r) {
        int64_t b = rows[3 * r], h = rows[3 * r + 1], i = rows[3 * r + 2];
        if (b < 0 || b >= B || h < 0 || h >= H || i < 0 || i >= Nq) return -1;
    }
    set_threads(nthreads);
    int err = 0;
#pragma omp parallel reduction(| : err)
    {
        row_scratch w;
        if (scratch_alloc(&w, Nk)) {
            err = 1;
        } else {
#pragma omp for schedule(dynamic, 1)
            for (long r = 0; r < nrows; ++r)
                prefill_row(q, k, v, H, Nq, Nk, d, causal, scale, (int)rows[3 * r],
                            (int)rows[3 * r + 1], (long)rows[3 * r + 2], &w, o_rows + (size_t)r * d,
                            lse_rows + r);
        }
        scratch_free(&w);
    }
    return err ? -1 : 0;
}

/*
 * The probability matrix P [B, H, Nq, Nk] fp64 (zero where a key is not
 * visible), for checking the softmax itself on small inputs.
 */
int oracle_attn_probs(const uint16_t *q, const uint16_t *k, int B, int H, long Nq, long Nk,
                      int d, int causal, double scale, double *P) {
    if (check_shape(B, H, Nq, Nk, d) || !q || !k || !P) return -1;
    double *s = (double *)malloc((size_t)(Nk > 0 ? Nk : 1) * sizeof(double));
    if (!s) return -1;
    for (int b = 0; b < B; ++b)
        for (int h = 0; h < H; ++h)
            for (long i = 0; i < Nq; ++i) {
                double *prow = P + (((size_t)b * H + h) * Nq + i) * Nk;
                long n = visible_keys(causal, i, Nq, Nk);
                const uint16_t *q_row = q + (((size_t)b * Nq + i) * H + h) * d;
                for (long j = 0; j < n; ++j) {
                    const uint16_t *k_row = k + (((size_t)b * Nk + j) * H + h) * d;
                    double acc = 0.0;
                    for (int c = 0; c < d; ++c) acc += bf16_to_f64(q_row[c]) * bf16_to_f64(k_row[c]);
                    s[j] = scale * acc;
                }
                double m = -INFINITY, l = 0.0;
                for (long j = 0; j < n; ++j)
                    if (s[j] > m) m = s[j];
                for (long j = 0; j < n; ++j) l += exp(s[j] - m);
                for (long j = 0; j < Nk; ++j) prow[j] = (j < n) ? exp(s[j] - m) / l : 0.0;
            }
    free(s);
    return 0;
}

/*
 * Decode: one query token per sequence against its KV cache.
 *   q [S, H, d] bf16; o [S, H, d] fp64; lse [S, H] fp64 (may be NULL).
 *   seqlens [S] int32, each in [0, max_seqlen]; a sequence with no key gets
 *   O = 0 and LSE = -inf.
 *   page_table == NULL: kcache/vcache are [S, max_seqlen, H, d].
 *   page_table != NULL: kcache/vcache are pools [num_pages, page_size, H, d] and
 *   page_table is [S, max_pages_per_seq] int32; key t of sequence s lives in
 *   page page_table[s][t / page_size], slot t % page_size.
 */
int oracle_decode(const uint16_t *q, const uint16_t *kcache, const uint16_t *vcache,
                  const int32_t *seqlens, const int32_t *page_table, int S, int H, int d,
                  long max_seqlen, int page_size, long max_pages_per_seq, long num_pages,
                  double scale, double *o, double *lse, int nthreads) {
    if (S < 0 || H < 0 || d <= 0 || max_seqlen < 0 || !q || !kcache || !vcache || !seqlens || !o)
        return -1;
    if (page_table && (page_size <= 0 || max_pages_per_seq <= 0 || num_pages <= 0)) return -1;
    for (int s = 0; s < S; ++s) {
        if (seqlens[s] < 0 || seqlens[s] > max_seqlen) return -1;
        if (page_table) {
            long need = ((long)seqlens[s] + page_size - 1) / page_size;
            if (need > max_pages_per_seq) return -1;
            for (long p = 0; p < need; ++p) {
                int32_t pg = page_table[(size_t)s * max_pages_per_seq + p];
                if (pg < 0 || pg >= num_pages) return -1;
            }
        }
    }
    set_threads(nthreads);
    long rows = (long)S * H;
    int err = 0;
#pragma omp parallel reduction(| : err)
    {
        row_scratch w;
        if (scratch_alloc(&w, max_seqlen)) {
            err = 1;
        } else {
#pragma omp for schedule(dynamic, 1)
            for (long r = 0; r < rows; ++r) {
                int s = (int)(r / H), h = (int)(r % H);
                long n = seqlens[s];
                for (long t = 0; t < n; ++t) {
                    size_t off;
                    if (page_table) {
                        int32_t pg = page_table[(size_t)s * max_pages_per_seq + t / page_size];
                        off = (((size_t)pg * page_size + (size_t)(t % page_size)) * H + h) * d;
                    } else {
                        off = (((size_t)s * max_seqlen + t) * H + h) * d;
                    }
                    w.keys[t] = kcache + off;
                    w.vals[t] = vcache + off;
                }
                double *o_row = o + (size_t)r * d;
                double l_out;
                if (n == 0) {
                    for (int c = 0; c < d; ++c) o_row[c] = 0.0;
                    l_out = -INFINITY;
                } else {
                    attention_row(q + (size_t)r * d, w.keys, w.vals, n, d, scale, w.s, o_row, &l_out);
                }
                if (lse) lse[r] = l_out;
            }
        }
        scratch_free(&w);
    }
    return err ? -1 : 0;
}
