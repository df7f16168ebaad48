/*
 * fa_ref.c -- FP64 CPU oracle for the exact attention forward and backward
 * passes.
 *
 * TEST INFRASTRUCTURE ONLY (see fa_ref.h).  Plain loops in double precision,
 * no blocking beyond what the blocked form itself states, no fusion.
 */
#include "fa_ref.h"

#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* ---- exact decoding of the input encodings ------------------------------ */

/* IEEE 754 binary16: 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits. */
static double decode_binary16(uint16_t h)
{
    int sign = (h >> 15) & 1;
    int e = (h >> 10) & 0x1f;
    int f = h & 0x3ff;
    double mag;
    if (e == 0)
        mag = ldexp((double)f, -24);                 /* zero / subnormal */
    else if (e == 31)
        mag = f ? NAN : INFINITY;
    else
        mag = ldexp((double)(1024 + f), e - 25);     /* (1.f) * 2^(e-15) */
    return sign ? -mag : mag;
}

/* bfloat16 is the upper half of an IEEE 754 binary32. */
static double decode_bfloat16(uint16_t b)
{
    uint32_t w = (uint32_t)b << 16;
    float x;
    memcpy(&x, &w, sizeof x);
    return (double)x;
}

/* Every 16-bit pattern decoded once by the functions above; the inner loops
 * then look values up instead of decoding them again. */
static double g_dec_f16[65536], g_dec_bf16[65536];
static int g_dec_ready = 0;

static void build_decode_tables(void)
{
    if (g_dec_ready) return;
#pragma omp critical(fa_ref_decode_tables)
    {
        if (!g_dec_ready) {
            for (uint32_t h = 0; h < 65536u; ++h) {
                g_dec_f16[h] = decode_binary16((uint16_t)h);
                g_dec_bf16[h] = decode_bfloat16((uint16_t)h);
            }
#pragma omp flush
            g_dec_ready = 1;
        }
    }
}

static double load(const void* p, int enc, size_t idx)
{
    switch (enc) {
    case FA_REF_ENC_F16:  return g_dec_f16[((const uint16_t*)p)[idx]];
    case FA_REF_ENC_BF16: return g_dec_bf16[((const uint16_t*)p)[idx]];
    default:              return ((const double*)p)[idx];
    }
}

static int bad_args(const void* q, const void* k, const void* v, int enc,
                    long B, long H, long N, long D)
{
    if (!q || !k || !v) return 1;
    if (B < 1 || H < 1 || N < 1 || D < 1) return 1;
    if (enc != FA_REF_ENC_F64 && enc != FA_REF_ENC_F16 && enc != FA_REF_ENC_BF16) return 1;
    build_decode_tables();
    return 0;
}

int fa_ref_max_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

static void set_threads(int nthreads)
{
#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
    else omp_set_num_threads(omp_get_num_procs());
#else
    (void)nthreads;
#endif
}

/* ---- naive safe softmax, one row ---------------------------------------- */

/* Scores of row i against every key, the row max, the exponentials shifted
 * by that max, their sum, the weighted sum of values, and the log-sum-exp.
 * s is scratch of length N. */
static void naive_row(const void* q, const void* k, const void* v, int enc,
                      long N, long D, double scale, int causal,
                      size_t q_base, size_t head_base, long i, double* s,
                      double* o_row, double* lse_out)
{
    long nvis = causal ? (i + 1 < N ? i + 1 : N) : N;
    size_t qrow = q_base + (size_t)i * (size_t)D;
    for (long d = 0; d < D; ++d) o_row[d] = 0.0;
    if (nvis <= 0) {
        *lse_out = -INFINITY;
        return;
    }
    double m = -INFINITY;
    for (long j = 0; j < nvis; ++j) {
        size_t krow = head_base + (size_t)j * (size_t)D;
        double dot = 0.0;
        for (long d = 0; d < D; ++d)
            dot += load(q, enc, qrow + d) * load(k, enc, krow + d);
        s[j] = scale * dot;
        if (s[j] > m) m = s[j];
    }
    double l = 0.0;
    for (long j = 0; j < nvis; ++j) {
        double p = exp(s[j] - m);
        size_t vrow = head_base + (size_t)j * (size_t)D;
        l += p;
        for (long d = 0; d < D; ++d)
            o_row[d] += p * load(v, enc, vrow + d);
    }
    for (long d = 0; d < D; ++d) o_row[d] /= l;
    *lse_out = m + log(l);
}

int fa_ref_naive(const void* q, const void* k, const void* v, int enc,
                 double* o, double* lse,
                 long B, long H, long N, long D, double scale, int causal,
                 int nthreads)
{
    if (bad_args(q, k, v, enc, B, H, N, D) || !o || !lse) return -1;
    set_threads(nthreads);
    long rows = B * H * N;
    int failed = 0;
#pragma omp parallel
    {
        double* s = (double*)malloc(sizeof(double) * (size_t)N);
        if (!s) {
#pragma omp atomic write
            failed = 1;
        }
#pragma omp for schedule(dynamic, 16)
        for (long r = 0; r < rows; ++r) {
            if (!s) continue;
            long bh = r / N, i = r % N;
            size_t head_base = (size_t)bh * (size_t)N * (size_t)D;
            naive_row(q, k, v, enc, N, D, scale, causal, head_base, head_base, i, s,
                      o + (size_t)r * (size_t)D, lse + r);
        }
        free(s);
    }
    return failed ? -2 : 0;
}

int fa_ref_naive_rows(const void* q, const void* k, const void* v, int enc,
                      long B, long H, long N, long D, double scale, int causal,
                      const long* bh_idx, const long* row_idx, long nrows,
                      double* o_rows, double* lse_rows, int nthreads)
{
    if (bad_args(q, k, v, enc, B, H, N, D) || !bh_idx || !row_idx || !o_rows || !lse_rows)
        return -1;
    for (long r = 0; r < nrows; ++r)
        if (bh_idx[r] < 0 || bh_idx[r] >= B * H || row_idx[r] < 0 || row_idx[r] >= N) return -1;
    set_threads(nthreads);
    int failed = 0;
#pragma omp parallel
    {
        double* s = (double*)malloc(sizeof(double) * (size_t)N);
        if (!s) {
#pragma omp atomic write
            failed = 1;
        }
#pragma omp for schedule(dynamic, 1)
        for (long r = 0; r < nrows; ++r) {
            if (!s) continue;
            size_t head_base = (size_t)bh_idx[r] * (size_t)N * (size_t)D;
            naive_row(q, k, v, enc, N, D, scale, causal, head_base, head_base, row_idx[r], s,
                      o_rows + (size_t)r * (size_t)D, lse_rows + r);
        }
        free(s);
    }
    return failed ? -2 : 0;
}

/* ---- blocked online softmax --------------------------------------------- */

/* One (Q block i0, K/V block j0) update of the running state of one head:
 *   S      = scale * Q_i K_j^T, with masked entries set to -inf
 *   m_new  = max(m_old, rowmax S)
 *   P      = exp(S - m_new)
 *   corr   = 0 if m_old = -inf, else exp(m_old - m_new)
 *   l      = l * corr + rowsum P
 *   O      = O * corr + P V_j
 *   m      = m_new                                                       */
static void block_update(const void* q, const void* k, const void* v, int enc,
                         long N, long D, double scale, int causal, int rescale,
                         size_t head_base, long i0, long i1, long j0, long j1,
                         double* m, double* l, double* O, double* s,
                         long trace_row, double* trace, long trace_cap, long* trace_len)
{
    long bc = j1 - j0;
    for (long i = i0; i < i1; ++i) {
        size_t qrow = head_base + (size_t)i * (size_t)D;
        double m_blk = -INFINITY;
        for (long j = j0; j < j1; ++j) {
            double sij;
            if (causal && j > i) {
                sij = -INFINITY;
            } else {
                size_t krow = head_base + (size_t)j * (size_t)D;
                double dot = 0.0;
                for (long d = 0; d < D; ++d)
                    dot += load(q, enc, qrow + d) * load(k, enc, krow + d);
                sij = scale * dot;
            }
            s[j - j0] = sij;
            if (sij > m_blk) m_blk = sij;
        }
        double m_old = m[i];
        double m_new = m_old > m_blk ? m_old : m_blk;
        double corr;
        if (!rescale)
            corr = 1.0;
        else
            corr = isinf(m_old) && m_old < 0 ? 0.0 : exp(m_old - m_new);
        double l_blk = 0.0;
        double* o_row = O + (size_t)i * (size_t)D;
        for (long d = 0; d < D; ++d) o_row[d] *= corr;
        for (long c = 0; c < bc; ++c) {
            /* exp(-inf - m_new) is 0 for finite m_new; a row whose every score
             * so far is -inf keeps p = 0 instead of exp(-inf + inf). */
            double p = (isinf(s[c]) && s[c] < 0) ? 0.0 : exp(s[c] - m_new);
            if (p == 0.0) continue;
            size_t vrow = head_base + (size_t)(j0 + c) * (size_t)D;
            l_blk += p;
            for (long d = 0; d < D; ++d) o_row[d] += p * load(v, enc, vrow + d);
        }
        l[i] = l[i] * corr + l_blk;
        m[i] = m_new;
        if (trace && i == trace_row && *trace_len < trace_cap) {
            double* t = trace + 4 * (*trace_len);
            t[0] = (double)j0;
            t[1] = m_new;
            t[2] = l[i];
            t[3] = corr;
            ++*trace_len;
        }
    }
}

int fa_ref_blocked(const void* q, const void* k, const void* v, int enc,
                   double* o, double* lse,
                   long B, long H, long N, long D, double scale, int causal,
                   long Br, long Bc, int kv_outer, int rescale,
                   long trace_row, double* trace, long trace_cap, long* trace_len,
                   long* visited, int nthreads)
{
    if (bad_args(q, k, v, enc, B, H, N, D) || !o || !lse || Br < 1 || Bc < 1) return -1;
    if (trace && (!trace_len || trace_cap < 0)) return -1;
    if (trace_len) *trace_len = 0;
    set_threads(nthreads);
    long BH = B * H;
    long pairs_head0 = 0;
    int failed = 0;
#pragma omp parallel for schedule(dynamic, 1)
    for (long bh = 0; bh < BH; ++bh) {
        double* m = (double*)malloc(sizeof(double) * (size_t)N);
        double* l = (double*)malloc(sizeof(double) * (size_t)N);
        double* O = (double*)calloc((size_t)N * (size_t)D, sizeof(double));
        double* s = (double*)malloc(sizeof(double) * (size_t)Bc);
        if (!m || !l || !O || !s) {
#pragma omp atomic write
            failed = 1;
            free(m); free(l); free(O); free(s);
            continue;
        }
        for (long i = 0; i < N; ++i) { m[i] = -INFINITY; l[i] = 0.0; }
        size_t head_base = (size_t)bh * (size_t)N * (size_t)D;
        double* tr = (bh == 0) ? trace : NULL;
        long pairs = 0;
        long outer_n = kv_outer ? Bc : Br;
        long inner_n = kv_outer ? Br : Bc;
        for (long a0 = 0; a0 < N; a0 += outer_n) {
            for (long b0 = 0; b0 < N; b0 += inner_n) {
                long i0 = kv_outer ? b0 : a0;
                long j0 = kv_outer ? a0 : b0;
                long i1 = i0 + Br < N ? i0 + Br : N;
                long j1 = j0 + Bc < N ? j0 + Bc : N;
                /* every query of the block precedes every key of the block */
                if (causal && i1 - 1 < j0) continue;
                ++pairs;
                block_update(q, k, v, enc, N, D, scale, causal, rescale, head_base,
                             i0, i1, j0, j1, m, l, O, s, trace_row, tr, trace_cap,
                             trace_len);
            }
        }
        for (long i = 0; i < N; ++i) {
            double* dst = o + ((size_t)bh * (size_t)N + (size_t)i) * (size_t)D;
            const double* src = O + (size_t)i * (size_t)D;
            if (l[i] > 0.0) {
                for (long d = 0; d < D; ++d) dst[d] = src[d] / l[i];
                lse[(size_t)bh * (size_t)N + (size_t)i] = m[i] + log(l[i]);
            } else {
                for (long d = 0; d < D; ++d) dst[d] = 0.0;
                lse[(size_t)bh * (size_t)N + (size_t)i] = -INFINITY;
            }
        }
        if (bh == 0) pairs_head0 = pairs;
        free(m); free(l); free(O); free(s);
    }
    if (visited) *visited = pairs_head0;
    return failed ? -2 : 0;
}

/* ---- split along the keys, then merge ----------------------------------- */

int fa_ref_split_merge(const void* q, const void* k, const void* v, int enc,
                       double* o, double* lse,
                       long B, long H, long N, long D, double scale, int causal,
                       long chunk, double* part_m, double* part_l, long part_cap,
                       int nthreads)
{
    if (bad_args(q, k, v, enc, B, H, N, D) || !o || !lse || chunk < 1) return -1;
    set_threads(nthreads);
    long rows = B * H * N;
    long nchunks = (N + chunk - 1) / chunk;
    int failed = 0;
#pragma omp parallel
    {
        double* pm = (double*)malloc(sizeof(double) * (size_t)nchunks);
        double* pl = (double*)malloc(sizeof(double) * (size_t)nchunks);
        double* po = (double*)malloc(sizeof(double) * (size_t)nchunks * (size_t)D);
        if (!pm || !pl || !po) {
#pragma omp atomic write
            failed = 1;
        }
#pragma omp for schedule(dynamic, 16)
        for (long r = 0; r < rows; ++r) {
            if (!pm || !pl || !po) continue;
            long bh = r / N, i = r % N;
            size_t head_base = (size_t)bh * (size_t)N * (size_t)D;
            size_t qrow = head_base + (size_t)i * (size_t)D;
            long nvis = causal ? (i + 1 < N ? i + 1 : N) : N;
            /* the partial of each chunk, by the definition over its keys */
            for (long c = 0; c < nchunks; ++c) {
                long j0 = c * chunk, j1 = j0 + chunk < nvis ? j0 + chunk : nvis;
                double* oc = po + (size_t)c * (size_t)D;
                for (long d = 0; d < D; ++d) oc[d] = 0.0;
                pm[c] = -INFINITY;
                pl[c] = 0.0;
                for (long j = j0; j < j1; ++j) {
                    size_t krow = head_base + (size_t)j * (size_t)D;
                    double dot = 0.0;
                    for (long d = 0; d < D; ++d) dot += load(q, enc, qrow + d) * load(k, enc, krow + d);
                    if (scale * dot > pm[c]) pm[c] = scale * dot;
                }
                for (long j = j0; j < j1; ++j) {
                    size_t krow = head_base + (size_t)j * (size_t)D;
                    size_t vrow = head_base + (size_t)j * (size_t)D;
                    double dot = 0.0;
                    for (long d = 0; d < D; ++d) dot += load(q, enc, qrow + d) * load(k, enc, krow + d);
                    double p = exp(scale * dot - pm[c]);
                    pl[c] += p;
                    for (long d = 0; d < D; ++d) oc[d] += p * load(v, enc, vrow + d);
                }
            }
            if (r == 0 && part_m && part_l) {
                for (long c = 0; c < nchunks && c < part_cap; ++c) {
                    part_m[c] = pm[c];
                    part_l[c] = pl[c];
                }
            }
            /* the merge */
            double m = -INFINITY;
            for (long c = 0; c < nchunks; ++c)
                if (pl[c] > 0.0 && pm[c] > m) m = pm[c];
            double l = 0.0;
            double* orow = o + (size_t)r * (size_t)D;
            for (long d = 0; d < D; ++d) orow[d] = 0.0;
            for (long c = 0; c < nchunks; ++c) {
                if (!(pl[c] > 0.0)) continue;
                double w = exp(pm[c] - m);
                l += w * pl[c];
                for (long d = 0; d < D; ++d) orow[d] += w * po[(size_t)c * (size_t)D + d];
            }
            if (l > 0.0) {
                for (long d = 0; d < D; ++d) orow[d] /= l;
                lse[r] = m + log(l);
            } else {
                lse[r] = -INFINITY;
            }
        }
        free(pm); free(pl); free(po);
    }
    return failed ? -2 : 0;
}

/* ---- grouped key/value heads ------------------------------------------- */

int fa_ref_naive_gqa(const void* q, const void* k, const void* v, int enc,
                     double* o, double* lse,
                     long B, long H, long H_kv, long N, long D, double scale, int causal,
                     int nthreads)
{
    if (bad_args(q, k, v, enc, B, H, N, D) || !o || !lse) return -1;
    if (H_kv < 1 || H % H_kv != 0) return -1;
    set_threads(nthreads);
    long rows = B * H * N;
    long group = H / H_kv;
    int failed = 0;
#pragma omp parallel
    {
        double* s = (double*)malloc(sizeof(double) * (size_t)N);
        if (!s) {
#pragma omp atomic write
            failed = 1;
        }
#pragma omp for schedule(dynamic, 16)
        for (long r = 0; r < rows; ++r) {
            if (!s) continue;
            long bh = r / N, i = r % N;
            long b = bh / H, h = bh % H;
            size_t q_base = (size_t)bh * (size_t)N * (size_t)D;
            size_t kv_base = ((size_t)b * (size_t)H_kv + (size_t)(h / group)) * (size_t)N * (size_t)D;
            naive_row(q, k, v, enc, N, D, scale, causal, q_base, kv_base, i, s,
                      o + (size_t)r * (size_t)D, lse + r);
        }
        free(s);
    }
    return failed ? -2 : 0;
}

/* ---- backward pass ------------------------------------------------------ */

/* Row i of a head ("Why FlashAttention does not need to store the attention
 * matrix", section 3.3; "CUDA FlashAttention: from online softmax to the
 * long-sequence IO limit", section 4.3.1): the scores s_ij, the row's
 * log-sum-exp, P_ij = exp(s_ij - LSE_i), dP_ij = dO_i . v_j, the softmax
 * correction term Delta_i = rowsum(dP_i (x) P_i), and, if dq_row is given,
 * dQ_i = scale * sum_j P_ij (dP_ij - Delta_i) k_j.  s and dp are scratch of
 * length N.  A row without visible keys gives LSE = -inf, Delta = 0, dQ = 0. */
static void bwd_row(const void* q, const void* k, const void* v, const void* dout, int enc,
                    long N, long D, double scale, int causal, size_t q_base, size_t kv_base,
                    long i, double* s, double* dp, double* lse_out, double* delta_out, double* dq_row)
{
    long nvis = causal ? (i + 1 < N ? i + 1 : N) : N;
    size_t qrow = q_base + (size_t)i * (size_t)D;
    if (dq_row)
        for (long d = 0; d < D; ++d) dq_row[d] = 0.0;
    if (nvis <= 0) {
        *lse_out = -INFINITY;
        *delta_out = 0.0;
        return;
    }
    double m = -INFINITY;
    for (long j = 0; j < nvis; ++j) {
        size_t kvrow = kv_base + (size_t)j * (size_t)D;
        double dot = 0.0, dpo = 0.0;
        for (long d = 0; d < D; ++d) {
            dot += load(q, enc, qrow + d) * load(k, enc, kvrow + d);
            dpo += load(dout, enc, qrow + d) * load(v, enc, kvrow + d);
        }
        s[j] = scale * dot;
        dp[j] = dpo;
        if (s[j] > m) m = s[j];
    }
    double l = 0.0;
    for (long j = 0; j < nvis; ++j) l += exp(s[j] - m);
    double lse = m + log(l);
    double delta = 0.0;
    for (long j = 0; j < nvis; ++j) delta += exp(s[j] - lse) * dp[j];
    if (dq_row) {
        for (long j = 0; j < nvis; ++j) {
            double ds = exp(s[j] - lse) * (dp[j] - delta);
            size_t kvrow = kv_base + (size_t)j * (size_t)D;
            for (long d = 0; d < D; ++d) dq_row[d] += scale * ds * load(k, enc, kvrow + d);
        }
    }
    *lse_out = lse;
    *delta_out = delta;
}

/* Key j of a head, given LSE_i and Delta_i of every row: over the rows that
 * see key j, dV_j = sum_i P_ij dO_i and dK_j = scale * sum_i dS_ij q_i with
 * dS_ij = P_ij (dP_ij - Delta_i) (same sections). */
static void bwd_col(const void* q, const void* k, const void* v, const void* dout, int enc,
                    long N, long D, double scale, int causal, size_t q_base, size_t kv_base,
                    long j, const double* lse, const double* delta, double* dk_row, double* dv_row)
{
    size_t kvrow = kv_base + (size_t)j * (size_t)D;
    for (long d = 0; d < D; ++d) dk_row[d] = dv_row[d] = 0.0;
    for (long i = causal ? j : 0; i < N; ++i) {
        if (lse[i] == -INFINITY) continue;
        size_t qrow = q_base + (size_t)i * (size_t)D;
        double dot = 0.0, dpo = 0.0;
        for (long d = 0; d < D; ++d) {
            dot += load(q, enc, qrow + d) * load(k, enc, kvrow + d);
            dpo += load(dout, enc, qrow + d) * load(v, enc, kvrow + d);
        }
        double p = exp(scale * dot - lse[i]);
        double ds = p * (dpo - delta[i]);
        for (long d = 0; d < D; ++d) {
            dv_row[d] += p * load(dout, enc, qrow + d);
            dk_row[d] += scale * ds * load(q, enc, qrow + d);
        }
    }
}

/* LSE and Delta of every row of head bh (OpenMP over rows). */
static int bwd_head_stats(const void* q, const void* k, const void* v, const void* dout, int enc,
                          long N, long D, double scale, int causal, size_t base, double* lse, double* delta)
{
    int err = 0;
#pragma omp parallel
    {
        double* s = (double*)malloc(sizeof(double) * (size_t)N);
        double* dp = (double*)malloc(sizeof(double) * (size_t)N);
        if (!s || !dp) {
#pragma omp atomic write
            err = 1;
        } else {
#pragma omp for schedule(dynamic, 16)
            for (long i = 0; i < N; ++i)
                bwd_row(q, k, v, dout, enc, N, D, scale, causal, base, base, i, s, dp, &lse[i], &delta[i], NULL);
        }
        free(s);
        free(dp);
    }
    return err;
}

int fa_ref_backward(const void* q, const void* k, const void* v, const void* dout, int enc,
                    double* dq, double* dk, double* dv, double* delta_out,
                    long B, long H, long N, long D, double scale, int causal, int nthreads)
{
    if (bad_args(q, k, v, enc, B, H, N, D) || !dout || !dq || !dk || !dv) return -1;
    set_threads(nthreads);
    double* lse = (double*)malloc(sizeof(double) * (size_t)N);
    double* dlt = (double*)malloc(sizeof(double) * (size_t)N);
    if (!lse || !dlt) {
        free(lse);
        free(dlt);
        return -2;
    }
    int err = 0;
    for (long bh = 0; bh < B * H && !err; ++bh) {
        size_t base = (size_t)bh * (size_t)N * (size_t)D;
#pragma omp parallel
        {
            double* s = (double*)malloc(sizeof(double) * (size_t)N);
            double* dp = (double*)malloc(sizeof(double) * (size_t)N);
            if (!s || !dp) {
#pragma omp atomic write
                err = 1;
            } else {
#pragma omp for schedule(dynamic, 16)
                for (long i = 0; i < N; ++i)
                    bwd_row(q, k, v, dout, enc, N, D, scale, causal, base, base, i, s, dp, &lse[i], &dlt[i],
                            dq + base + (size_t)i * (size_t)D);
            }
            free(s);
            free(dp);
        }
        if (err) break;
#pragma omp parallel for schedule(dynamic, 16)
        for (long j = 0; j < N; ++j)
            bwd_col(q, k, v, dout, enc, N, D, scale, causal, base, base, j, lse, dlt,
                    dk + base + (size_t)j * (size_t)D, dv + base + (size_t)j * (size_t)D);
        if (delta_out)
            for (long i = 0; i < N; ++i) delta_out[(size_t)bh * (size_t)N + (size_t)i] = dlt[i];
    }
    free(lse);
    free(dlt);
    return err ? -2 : 0;
}

int fa_ref_backward_sample(const void* q, const void* k, const void* v, const void* dout, int enc,
                           long B, long H, long N, long D, double scale, int causal,
                           const long* dq_bh, const long* dq_rows, long n_dq, double* dq_out,
                           const long* kv_bh, const long* kv_keys, long n_kv, double* dk_out, double* dv_out,
                           int nthreads)
{
    if (bad_args(q, k, v, enc, B, H, N, D) || !dout) return -1;
    if ((n_dq > 0 && (!dq_bh || !dq_rows || !dq_out)) || (n_kv > 0 && (!kv_bh || !kv_keys || !dk_out || !dv_out)))
        return -1;
    for (long r = 0; r < n_dq; ++r)
        if (dq_bh[r] < 0 || dq_bh[r] >= B * H || dq_rows[r] < 0 || dq_rows[r] >= N) return -1;
    for (long r = 0; r < n_kv; ++r)
        if (kv_bh[r] < 0 || kv_bh[r] >= B * H || kv_keys[r] < 0 || kv_keys[r] >= N) return -1;
    set_threads(nthreads);
    int err = 0;
    /* dQ rows: each is local to its row */
#pragma omp parallel
    {
        double* s = (double*)malloc(sizeof(double) * (size_t)N);
        double* dp = (double*)malloc(sizeof(double) * (size_t)N);
        if (!s || !dp) {
#pragma omp atomic write
            err = 1;
        } else {
#pragma omp for schedule(dynamic, 1)
            for (long r = 0; r < n_dq; ++r) {
                size_t base = (size_t)dq_bh[r] * (size_t)N * (size_t)D;
                double lse_r, dlt_r;
                bwd_row(q, k, v, dout, enc, N, D, scale, causal, base, base, dq_rows[r], s, dp, &lse_r, &dlt_r,
                        dq_out + (size_t)r * (size_t)D);
            }
        }
        free(s);
        free(dp);
    }
    if (err) return -2;
    /* dK / dV keys: the row statistics of each sampled head, then the columns */
    if (n_kv > 0) {
        double* lse = (double*)malloc(sizeof(double) * (size_t)N);
        double* dlt = (double*)malloc(sizeof(double) * (size_t)N);
        if (!lse || !dlt) {
            free(lse);
            free(dlt);
            return -2;
        }
        for (long bh = 0; bh < B * H && !err; ++bh) {
            int used = 0;
            for (long r = 0; r < n_kv && !used; ++r) used = kv_bh[r] == bh;
            if (!used) continue;
            size_t base = (size_t)bh * (size_t)N * (size_t)D;
            err = bwd_head_stats(q, k, v, dout, enc, N, D, scale, causal, base, lse, dlt);
            if (err) break;
#pragma omp parallel for schedule(dynamic, 1)
            for (long r = 0; r < n_kv; ++r)
                if (kv_bh[r] == bh)
                    bwd_col(q, k, v, dout, enc, N, D, scale, causal, base, base, kv_keys[r], lse, dlt,
                            dk_out + (size_t)r * (size_t)D, dv_out + (size_t)r * (size_t)D);
        }
        free(lse);
        free(dlt);
    }
    return err ? -2 : 0;
}

/* ---- FP8 (E4M3) inputs with per-block scales ---------------------------- */

/* OCP 8-bit E4M3 ("FN": no infinities): 1 sign bit, 4 exponent bits (bias 7),
 * 3 fraction bits; exponent 0 is subnormal (f * 2^-9); S.1111.111 is NaN. */
double fa_ref_decode_e4m3(uint8_t x)
{
    int sign = (x >> 7) & 1;
    int e = (x >> 3) & 0xf;
    int f = x & 7;
    double mag;
    if (e == 15 && f == 7)
        mag = NAN;
    else if (e == 0)
        mag = ldexp((double)f, -9);
    else
        mag = ldexp((double)(8 + f), e - 10);     /* (1.f) * 2^(e-7) */
    return sign ? -mag : mag;
}

int fa_ref_dequant_e4m3(const uint8_t* x, const float* block_scale, long BH, long N, long D, long block_rows,
                        double* out)
{
    if (!x || !block_scale || !out || BH < 1 || N < 1 || D < 1 || block_rows < 1) return -1;
    long nb = (N + block_rows - 1) / block_rows;
    for (long bh = 0; bh < BH; ++bh)
        for (long n = 0; n < N; ++n) {
            double s = (double)block_scale[bh * nb + n / block_rows];
            size_t row = ((size_t)bh * (size_t)N + (size_t)n) * (size_t)D;
            for (long d = 0; d < D; ++d) out[row + d] = fa_ref_decode_e4m3(x[row + d]) * s;
        }
    return 0;
}

/* ---- queries against a longer key/value sequence ------------------------- */

int fa_ref_naive_kv(const void* q, const void* k, const void* v, int enc, double* o, double* lse, long B, long H,
                    long H_kv, long Nq, long Nk, long D, double scale, int causal, int nthreads)
{
    if (bad_args(q, k, v, enc, B, H, Nq, D) || !o || !lse || Nk < 1 || H_kv < 1 || H % H_kv != 0) return -1;
    if (causal && Nq > Nk) return -1;
    set_threads(nthreads);
    const long group = H / H_kv;
    int err = 0;
#pragma omp parallel
    {
        double* s = (double*)malloc(sizeof(double) * (size_t)Nk);
        if (!s) {
#pragma omp atomic write
            err = 1;
        } else {
#pragma omp for schedule(dynamic, 16)
            for (long r = 0; r < B * H * Nq; ++r) {
                long bh = r / Nq, i = r - bh * Nq;
                long b = bh / H, h = bh - b * H;
                size_t q_base = (size_t)bh * (size_t)Nq * (size_t)D;
                size_t kv_base = ((size_t)b * (size_t)H_kv + (size_t)(h / group)) * (size_t)Nk * (size_t)D;
                /* query i sits at position i + Nk - Nq of the key sequence */
                long nvis = causal ? i + (Nk - Nq) + 1 : Nk;
                double* orow = o + (size_t)r * (size_t)D;
                size_t qrow = q_base + (size_t)i * (size_t)D;
                double m = -INFINITY;
                for (long j = 0; j < nvis; ++j) {
                    size_t krow = kv_base + (size_t)j * (size_t)D;
                    double dot = 0.0;
                    for (long d = 0; d < D; ++d) dot += load(q, enc, qrow + d) * load(k, enc, krow + d);
                    s[j] = scale * dot;
                    if (s[j] > m) m = s[j];
                }
                for (long d = 0; d < D; ++d) orow[d] = 0.0;
                double l = 0.0;
                for (long j = 0; j < nvis; ++j) {
                    double p = exp(s[j] - m);
                    size_t vrow = kv_base + (size_t)j * (size_t)D;
                    l += p;
                    for (long d = 0; d < D; ++d) orow[d] += p * load(v, enc, vrow + d);
                }
                for (long d = 0; d < D; ++d) orow[d] /= l;
                lse[r] = m + log(l);
            }
        }
        free(s);
    }
    return err ? -2 : 0;
}
