/*
 * plmla_oracle.c -- plain double-precision CPU oracle for paged gated-MLA decode.
 *
 * TEST INFRASTRUCTURE ONLY.  Only tests/, the smoke check in __graft_entry__ and
 * the CPU-baseline leg of bench.py may load this library.  It shares no code,
 * header, table or constant with the CUDA library under
 * paged_latent_attention_gb300/csrc, and it is written to be read against the
 * definition, not to be fast.
 *
 * What it computes (per request r, query token j, head h):
 *
 *   L'  = seq_lens[r] - (n_q - 1 - j)          causal limit among the n_q draft
 *                                              tokens; the speculative verifier
 *                                              checks four drafted tokens per
 *                                              request (TokenSpeed AgentX post,
 *                                              section "Use TP4 selectively for
 *                                              projections and shared experts")
 *   x_t = slab[page_table[r][t / P] * page_stride + (t % P) * row_elems + 0..]
 *                                              flat page pool, one global page ID
 *                                              per page (TokenSpeed Kimi K3 post,
 *                                              section "A Generic, Unified Flat KV
 *                                              Layout for Cache Management")
 *   c_t = x_t[0 : dc]   (compressed latent),  k_t = x_t[dc : dc + dr] (rope key)
 *   s_t = scale * ( sum_d qn[d] c_t[d] + sum_d qr[d] k_t[d] )
 *   m   = max_t s_t,   Z = sum_t exp(s_t - m)
 *   o   = sum_t exp(s_t - m) / Z * c_t          full softmax attention whose values
 *                                              are the stored compressed latent
 *                                              rows (TokenSpeed Kimi K3 post,
 *                                              architecture list, Gated MLA)
 *   lse = m + ln Z
 *
 * for t in [t_lo, min(t_hi, L')).  With t_lo = 0 and t_hi = INT64_MAX this is
 * the whole history; a narrower [t_lo, t_hi) gives the partial state of one KV
 * chunk, which a second kernel merges with the other chunks' states (TokenSpeed
 * Kimi K3 post, section "Gluon kernels on AMD GPUs", Gated MLA decode
 * paragraph).  An empty range gives o = 0 and lse = -inf.
 * The sigmoid output gate is applied by the Python side of the oracle.
 *
 * All arithmetic is in double; bf16 inputs are widened exactly.
 *
 * FP8 pages: the deployment keeps its MLA cache in FP8 (TokenSpeed AgentX post,
 * memory-budget paragraph: "FP8 target/drafter KV cache").  With kv_fp8 set,
 * every slab element is one OCP E4M3 byte (1 sign bit, 4 exponent bits with
 * bias 7, 3 mantissa bits; exponent 0 is subnormal, S.1111.111 is NaN, there is
 * no infinity) and the stored value is kv_scale times the decoded number.
 * The query is passed in double and used as given: the definition takes the
 * bf16 query exactly, whatever the cache format.
 *
 * Sensitivity outputs (optional, for error bounds derived by the caller): the
 * largest softmax weight w_max = 1 / Z, the unweighted absolute latent sum
 * sum_t |c_t[d]|, and, given a per-element bound eps[d] on the error of a query
 * element, the largest bound on a score's error over the row's tokens,
 * D = max_t |scale| * sum_d eps[d] * |x_t[d]| (latent and rope elements).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

static double bf16_to_double(uint16_t bits)
{
    uint32_t u = ((uint32_t)bits) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* OCP E4M3: value = (-1)^s * 2^(e-7) * (1 + m/8) for e >= 1, (-1)^s * 2^-6 * m/8
 * for e = 0; e = 15 with m = 7 is NaN. */
static double e4m3_to_double(uint8_t b)
{
    int sign = b >> 7, e = (b >> 3) & 0xF, m = b & 7;
    double v;
    if (e == 15 && m == 7)
        return NAN;
    if (e == 0)
        v = ldexp((double)m / 8.0, -6);
    else
        v = ldexp(1.0 + (double)m / 8.0, e - 7);
    return sign ? -v : v;
}

/* Element `idx` of the slab as a double: a bf16 value, or kv_scale times an
 * E4M3 value. */
static double kv_elem(const void *slab, int64_t idx, int kv_fp8, double kv_scale)
{
    if (kv_fp8)
        return kv_scale * e4m3_to_double(((const uint8_t *)slab)[idx]);
    return bf16_to_double(((const uint16_t *)slab)[idx]);
}

/* Attention for one output row.  Returns 0 on success, -1 if a page index read
 * from the page table lies outside [0, num_pages).  o_abs (may be NULL)
 * receives sum_t w_t |c_t[d]|, the probability-weighted absolute latent; the
 * sensitivity outputs abs_sum, w_max and d_max (each may be NULL; d_max needs
 * eps) are described in the file header. */
static int attend_one_row(const double *qn, const double *qr, const void *slab, int kv_fp8,
                          double kv_scale, int64_t num_pages, int64_t page_stride,
                          int64_t page_tokens, int64_t row_elems, const int32_t *table_row,
                          int64_t L_eff, int64_t t_lo, int64_t t_hi, int64_t dc, int64_t dr,
                          double scale, double *o_out, double *o_abs, double *lse_out,
                          double *scores, const double *eps, double *abs_sum, double *w_max,
                          double *d_max)
{
    int64_t lo = t_lo < 0 ? 0 : t_lo;
    int64_t hi = t_hi < L_eff ? t_hi : L_eff;
    for (int64_t d = 0; d < dc; ++d) {
        o_out[d] = 0.0;
        if (o_abs)
            o_abs[d] = 0.0;
        if (abs_sum)
            abs_sum[d] = 0.0;
    }
    if (w_max)
        *w_max = 0.0;
    if (d_max)
        *d_max = 0.0;
    if (hi <= lo) {
        *lse_out = -INFINITY;
        return 0;
    }
    /* pass 1: scores and their maximum */
    double m = -INFINITY;
    double dm = 0.0;
    for (int64_t t = lo; t < hi; ++t) {
        int64_t page = table_row[t / page_tokens];
        if (page < 0 || page >= num_pages)
            return -1;
        int64_t x = page * page_stride + (t % page_tokens) * row_elems;
        double dot = 0.0;
        for (int64_t d = 0; d < dc; ++d)
            dot += qn[d] * kv_elem(slab, x + d, kv_fp8, kv_scale);
        for (int64_t d = 0; d < dr; ++d)
            dot += qr[d] * kv_elem(slab, x + dc + d, kv_fp8, kv_scale);
        double s = scale * dot;
        scores[t - lo] = s;
        if (s > m)
            m = s;
        if (eps && d_max) {
            double delta = 0.0;
            for (int64_t d = 0; d < dc + dr; ++d)
                if (eps[d] != 0.0)
                    delta += eps[d] * fabs(kv_elem(slab, x + d, kv_fp8, kv_scale));
            delta *= fabs(scale);
            if (delta > dm)
                dm = delta;
        }
    }
    /* pass 2: normaliser and the probability-weighted latent sum */
    double Z = 0.0;
    for (int64_t t = lo; t < hi; ++t)
        Z += exp(scores[t - lo] - m);
    for (int64_t t = lo; t < hi; ++t) {
        int64_t page = table_row[t / page_tokens];
        int64_t x = page * page_stride + (t % page_tokens) * row_elems;
        double p = exp(scores[t - lo] - m) / Z;
        for (int64_t d = 0; d < dc; ++d) {
            double c = kv_elem(slab, x + d, kv_fp8, kv_scale);
            o_out[d] += p * c;
            if (o_abs)
                o_abs[d] += p * fabs(c);
            if (abs_sum)
                abs_sum[d] += fabs(c);
        }
    }
    *lse_out = m + log(Z);
    if (w_max)
        *w_max = 1.0 / Z;   /* the weight of a token at the maximum score */
    if (d_max)
        *d_max = dm;
    return 0;
}

/*
 * oracle_attend_rows -- ungated attention output and log-sum-exp for a list of
 * output rows.
 *
 * q_nope   [R*n_q, H, dc] double (absorbed query, latent part)
 * q_rope   [R*n_q, H, dr] double
 * slab     num_pages pages, page p at element offset p*page_stride; token i of a
 *          page at i*row_elems; row = dc latent values then dr rope values;
 *          bf16 elements, or E4M3 bytes times kv_scale when kv_fp8 != 0
 * page_table [R, table_ld] int32 global page IDs
 * seq_lens [R] int32 (includes the n_q draft tokens)
 * rows     [n_rows] flat row ids ((r*n_q + j)*H + h); NULL means all rows
 * t_lo, t_hi  token window applied to every row (partial-state evaluation)
 * o        [n_rows, dc] double, lse [n_rows] double (outputs); o_abs [n_rows, dc]
 *          (NULL allowed) the probability-weighted absolute latent
 * eps      [R*n_q*H, dc + dr] per-element query error bounds, or NULL
 * abs_sum  [n_rows, dc], w_max [n_rows], d_max [n_rows]: sensitivity outputs
 *          (each NULL allowed; d_max is written only with eps)
 *
 * Returns 0, or -1 if a page ID is out of range, or -2 on allocation failure.
 */
int oracle_attend_rows(const double *q_nope, const double *q_rope, const void *slab, int kv_fp8,
                       double kv_scale, int64_t num_pages, int64_t page_stride,
                       int64_t page_tokens, int64_t row_elems, const int32_t *page_table,
                       int64_t table_ld, const int32_t *seq_lens, int64_t R, int64_t n_q,
                       int64_t H, int64_t dc, int64_t dr, double scale, const int64_t *rows,
                       int64_t n_rows, int64_t t_lo, int64_t t_hi, double *o, double *o_abs,
                       double *lse, const double *eps, double *abs_sum, double *w_max,
                       double *d_max, int num_threads)
{
    int64_t total_rows = R * n_q * H;
    if (rows == NULL)
        n_rows = total_rows;
    int64_t max_len = 0;
    for (int64_t r = 0; r < R; ++r)
        if (seq_lens[r] > max_len)
            max_len = seq_lens[r];
    int status = 0;
#pragma omp parallel num_threads(num_threads > 0 ? num_threads : 1)
    {
        double *scores = (double *)malloc(sizeof(double) * (size_t)(max_len > 0 ? max_len : 1));
#pragma omp for schedule(dynamic, 1)
        for (int64_t i = 0; i < n_rows; ++i) {
            if (scores == NULL) {
#pragma omp atomic write
                status = -2;
                continue;
            }
            int64_t row = rows ? rows[i] : i;
            int64_t tok = row / H; /* r*n_q + j */
            int64_t r = tok / n_q;
            int64_t j = tok % n_q;
            int64_t L_eff = (int64_t)seq_lens[r] - (n_q - 1 - j);
            int rc = attend_one_row(q_nope + row * dc, q_rope + row * dr, slab, kv_fp8, kv_scale,
                                    num_pages, page_stride, page_tokens, row_elems,
                                    page_table + r * table_ld, L_eff, t_lo, t_hi, dc, dr, scale,
                                    o + i * dc, o_abs ? o_abs + i * dc : NULL, lse + i, scores,
                                    eps ? eps + row * (dc + dr) : NULL,
                                    abs_sum ? abs_sum + i * dc : NULL, w_max ? w_max + i : NULL,
                                    (eps && d_max) ? d_max + i : NULL);
            if (rc != 0) {
#pragma omp atomic write
                status = rc;
            }
        }
        free(scores);
    }
    return status;
}
