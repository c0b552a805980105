/*
 * Exact-attention oracle: plain, slow, fp64, single source of truth for the
 * parity tests.  TEST INFRASTRUCTURE ONLY: nothing in the product path links,
 * loads or calls this file; only tests/, the smoke check and the bench's CPU
 * baseline leg do.  It shares no code with the CUDA library.
 *
 * What it computes, and where each step is stated:
 *   S = scale * Q K^T                 "TileLang tutorial, ch.15 Operators:
 *                                       Attention", section 1.1; "llm-course
 *                                       ch.19 Flash Attention", section 19.1
 *   P = softmax(S) row by row, with the row maximum subtracted first
 *                                      (safe softmax, ch.15 sections 2.1-2.2)
 *   O = P V, LSE_i = m_i + ln(sum_j exp(S_ij - m_i))   (natural log)
 *
 * The two-pass functions materialise one full row of S and P at a time (the
 * "naive" version of ch.15 section 3.1), so a reader can check them against
 * the formulas above by eye.  The blockwise function follows the online
 * softmax recurrence of ch.15 section 2.3 (running max m, rescale factor
 * c = exp(m_old - m_new), running sum l, unnormalised O, one final O / l),
 * with the check_inf guard of ch.15 section 5.1(1); it exists only so the
 * tests can pin the recurrence against the two-pass definition.
 *
 * Masks (ch.15 sections 3.4 and 5.2; varlen right alignment, section 5.3):
 *   off = Skv - Sq (bottom-right aligned causal diagonal)
 *   key j is visible to query i iff
 *       j < Skv, and, when causal,   j <= i + off, and, when window W > 0,
 *       (j > i + off - W  or  j < n_sink).
 *   A row that sees no key returns O = 0 and LSE = -inf (ch.15 section 5.1(2)).
 *
 * Logit sink (optional, one value per query head; ch.15 section 4.6, the
 * "attention sink" row of the variant table: the sink only adds one term to
 * the softmax denominator).  Read here as a logit sigma_h in the units of S
 * (natural log, after the scale) that joins the row's softmax as one more
 * column with no value row:
 *       m   = max(sigma_h, max_j S_ij)
 *       O_i = sum_j exp(S_ij - m) V_j / (exp(sigma_h - m) + sum_j exp(S_ij - m))
 *       LSE = m + ln(exp(sigma_h - m) + sum_j exp(S_ij - m))
 *   sigma_h = -inf is no sink.  A row that sees no key but has a finite sink
 *   returns O = 0 and LSE = sigma_h.
 *
 * Layouts (row-major, contiguous):
 *   dense : q,o [B,Sq,Hq,d]   k,v [B,Skv,Hkv,d]   lse [B,Hq,Sq]
 *   varlen: q,o [Tq,Hq,d]     k,v [Tk,Hkv,d]      lse [Hq,Tq]
 *   decode: q,o [B,Hq,d]      k,v [B,Lmax,Hkv,d]  lse [B,Hq]
 * GQA: query head h reads key/value head h / (Hq / Hkv) (ch.15 section 4.8(1)).
 */
#include <math.h>
#include <stddef.h>
#include <stdlib.h>
#include <string.h>

#define ORACLE_API __attribute__((visibility("default")))

static int visible(long i, long j, long Sq, long Skv, int causal, int window, int n_sink)
{
    long off = Skv - Sq;
    if (j < 0 || j >= Skv) return 0;
    if (!causal) return 1;
    if (j > i + off) return 0;
    if (window > 0) return (j > i + off - window) || (j < n_sink);
    return 1;
}

/* One query row against one key/value head, two-pass definition.
 * qrow: d values; k, v: rows of stride kv_stride (elements), Skv of them.
 * sink: the row's sink logit, -INFINITY for none.
 * srow: scratch of Skv doubles (holds S, then P). */
static void row_two_pass(const double *qrow, const double *k, const double *v, long kv_stride,
                         long i, long Sq, long Skv, int d, double scale, int causal, int window,
                         int n_sink, double sink, double *srow, double *orow, double *lse_out)
{
    double m = sink; /* the sink's column takes part in the row maximum */
    for (long j = 0; j < Skv; ++j) {
        if (!visible(i, j, Sq, Skv, causal, window, n_sink)) {
            srow[j] = -INFINITY;
            continue;
        }
        const double *kj = k + j * kv_stride;
        double dot = 0.0;
        for (int t = 0; t < d; ++t) dot += qrow[t] * kj[t];
        srow[j] = scale * dot;
        if (srow[j] > m) m = srow[j];
    }
    if (m == -INFINITY) { /* no visible key and no sink */
        for (int t = 0; t < d; ++t) orow[t] = 0.0;
        *lse_out = -INFINITY;
        return;
    }
    double sum = (sink == -INFINITY) ? 0.0 : exp(sink - m);
    for (long j = 0; j < Skv; ++j) {
        double p = (srow[j] == -INFINITY) ? 0.0 : exp(srow[j] - m);
        srow[j] = p;
        sum += p;
    }
    for (int t = 0; t < d; ++t) orow[t] = 0.0;
    for (long j = 0; j < Skv; ++j) {
        double pj = srow[j] / sum;
        if (pj == 0.0) continue;
        const double *vj = v + j * kv_stride;
        for (int t = 0; t < d; ++t) orow[t] += pj * vj[t];
    }
    *lse_out = m + log(sum);
}

/*
 * Dense attention forward, two-pass definition.
 * rows / n_rows: optional subset of query rows (same subset for every batch
 * and head); rows == NULL means every row 0..Sq-1 and n_rows must equal Sq.
 * Outputs are compact over the subset: o [B, n_rows, Hq, d], lse [B, Hq, n_rows].
 * sink: NULL, or the logit sink of every query head [Hq].
 */
ORACLE_API int oracle_attn_fwd(const double *q, const double *k, const double *v, double *o,
                               double *lse, int B, int Hq, int Hkv, int Sq, int Skv, int d,
                               double scale, int causal, int window, int n_sink,
                               const int *rows, int n_rows, const double *sink)
{
    if (Hkv <= 0 || Hq % Hkv != 0 || d <= 0) return 1;
    if (!rows && n_rows != Sq) return 1;
    const int groups = Hq / Hkv;
    const long total = (long)B * Hq * n_rows;
    int bad = 0;
#pragma omp parallel
    {
        double *srow = (double *)malloc(sizeof(double) * (Skv > 0 ? Skv : 1));
        if (!srow) {
#pragma omp atomic write
            bad = 1;
        } else {
#pragma omp for schedule(dynamic, 16)
            for (long w = 0; w < total; ++w) {
                long r = w % n_rows;
                long h = (w / n_rows) % Hq;
                long b = w / ((long)n_rows * Hq);
                long i = rows ? rows[r] : r;
                long hk = h / groups;
                const double *qrow = q + (((b * Sq + i) * Hq) + h) * d;
                const double *kb = k + ((b * (long)Skv) * Hkv + hk) * d;
                const double *vb = v + ((b * (long)Skv) * Hkv + hk) * d;
                double *orow = o + (((b * n_rows + r) * Hq) + h) * d;
                double *lrow = lse + ((b * Hq + h) * (long)n_rows + r);
                row_two_pass(qrow, kb, vb, (long)Hkv * d, i, Sq, Skv, d, scale, causal, window,
                             n_sink, sink ? sink[h] : -INFINITY, srow, orow, lrow);
            }
            free(srow);
        }
    }
    return bad ? 2 : 0;
}

/*
 * Variable-length (packed) attention forward, two-pass definition.
 * cu_q / cu_k: [nseq + 1] prefix sums of the query / key lengths
 * (ch.15 section 5.3).  Causal alignment per sequence is bottom-right
 * (off = Lk - Lq).  o [Tq,Hq,d], lse [Hq,Tq], Tq = cu_q[nseq].
 * sink: NULL, or the logit sink of every query head [Hq].
 */
ORACLE_API int oracle_attn_fwd_varlen(const double *q, const double *k, const double *v,
                                      double *o, double *lse, const int *cu_q, const int *cu_k,
                                      int nseq, int Hq, int Hkv, int d, double scale, int causal,
                                      int window, int n_sink, const double *sink)
{
    if (Hkv <= 0 || Hq % Hkv != 0 || d <= 0) return 1;
    const int groups = Hq / Hkv;
    const long Tq = cu_q[nseq];
    long maxk = 1;
    for (int s = 0; s < nseq; ++s)
        if (cu_k[s + 1] - cu_k[s] > maxk) maxk = cu_k[s + 1] - cu_k[s];
    const long total = Tq * Hq;
    int bad = 0;
#pragma omp parallel
    {
        double *srow = (double *)malloc(sizeof(double) * maxk);
        if (!srow) {
#pragma omp atomic write
            bad = 1;
        } else {
#pragma omp for schedule(dynamic, 16)
            for (long w = 0; w < total; ++w) {
                long t = w / Hq, h = w % Hq, hk = h / groups;
                int s = 0;
                while (cu_q[s + 1] <= t) ++s; /* sequence holding token t */
                long i = t - cu_q[s];
                long Lq = cu_q[s + 1] - cu_q[s], Lk = cu_k[s + 1] - cu_k[s];
                const double *qrow = q + (t * Hq + h) * d;
                const double *kb = k + ((long)cu_k[s] * Hkv + hk) * d;
                const double *vb = v + ((long)cu_k[s] * Hkv + hk) * d;
                row_two_pass(qrow, kb, vb, (long)Hkv * d, i, Lq, Lk, d, scale, causal, window,
                             n_sink, sink ? sink[h] : -INFINITY, srow, o + (t * Hq + h) * d,
                             lse + h * Tq + t);
            }
            free(srow);
        }
    }
    return bad ? 2 : 0;
}

/*
 * Single-token decode against contiguous per-request caches: query b sees
 * the first seqlens[b] keys of k[b] (the causal diagonal of a one-row query
 * aligned bottom-right, ch.15 sections 5.2-5.3).  k, v [B, Lmax, Hkv, d].
 * sink: NULL, or the logit sink of every query head [Hq].
 */
ORACLE_API int oracle_attn_decode(const double *q, const double *k, const double *v,
                                  const int *seqlens, double *o, double *lse, int B, int Hq,
                                  int Hkv, int d, int Lmax, double scale, const double *sink)
{
    if (Hkv <= 0 || Hq % Hkv != 0 || d <= 0) return 1;
    const int groups = Hq / Hkv;
    int bad = 0;
#pragma omp parallel
    {
        double *srow = (double *)malloc(sizeof(double) * (Lmax > 0 ? Lmax : 1));
        if (!srow) {
#pragma omp atomic write
            bad = 1;
        } else {
#pragma omp for schedule(dynamic, 4)
            for (long w = 0; w < (long)B * Hq; ++w) {
                long b = w / Hq, h = w % Hq, hk = h / groups;
                long L = seqlens[b];
                const double *kb = k + ((b * (long)Lmax) * Hkv + hk) * d;
                const double *vb = v + ((b * (long)Lmax) * Hkv + hk) * d;
                row_two_pass(q + w * d, kb, vb, (long)Hkv * d, 0, 1, L, d, scale, 0, 0, 0,
                             sink ? sink[h] : -INFINITY, srow, o + w * d, lse + w);
            }
            free(srow);
        }
    }
    return bad ? 2 : 0;
}

/*
 * Blockwise online-softmax forward (ch.15 section 2.3; FA-2 order of
 * "TileLang in practice: FlashAttention forward kernel", section 2.4): keys
 * are visited in blocks of `block`; per query row the state (m, l, O) is
 * updated as
 *     m_new = max(m, rowmax(S_blk))
 *     c     = exp(m - m_new)        with m_new = -inf treated as 0 (check_inf)
 *     l     = c * l + sum exp(S_blk - m_new)
 *     O     = c * O + exp(S_blk - m_new) V_blk
 * and O / l is returned at the end (O = 0, LSE = -inf when l == 0).
 * trace (nullable): after each block, the (m, l, O[0..d)) state of query row 0
 * of batch 0, head 0 is appended: (2 + d) doubles per block.
 * sink (nullable, [Hq]): the logit sink enters only after the last block, as
 * one more term of the denominator taken against m* = max(sigma, m) (the
 * epilogue form of ch.15 section 4.6; m* rather than m keeps exp(sigma - m*)
 * finite when the sink exceeds every score):
 *     l* = l exp(m - m*) + exp(sigma - m*),   O = acc exp(m - m*) / l*,
 *     LSE = m* + ln(l*).
 */
ORACLE_API int oracle_attn_fwd_blockwise(const double *q, const double *k, const double *v,
                                         double *o, double *lse, int B, int Hq, int Hkv, int Sq,
                                         int Skv, int d, double scale, int causal, int window,
                                         int n_sink, int block, double *trace, const double *sink)
{
    if (Hkv <= 0 || Hq % Hkv != 0 || d <= 0 || block <= 0) return 1;
    const int groups = Hq / Hkv;
    const long total = (long)B * Hq * Sq;
    int bad = 0;
#pragma omp parallel
    {
        double *sblk = (double *)malloc(sizeof(double) * block);
        double *acc = (double *)malloc(sizeof(double) * d);
        if (!sblk || !acc) {
#pragma omp atomic write
            bad = 1;
        } else {
#pragma omp for schedule(dynamic, 16)
            for (long w = 0; w < total; ++w) {
                long i = w % Sq, h = (w / Sq) % Hq, b = w / ((long)Sq * Hq), hk = h / groups;
                const double *qrow = q + (((b * Sq + i) * Hq) + h) * d;
                const double *kb = k + ((b * (long)Skv) * Hkv + hk) * d;
                const double *vb = v + ((b * (long)Skv) * Hkv + hk) * d;
                const long kvs = (long)Hkv * d;
                double m = -INFINITY, l = 0.0;
                for (int t = 0; t < d; ++t) acc[t] = 0.0;
                long nblk = 0;
                for (long j0 = 0; j0 < Skv; j0 += block, ++nblk) {
                    long j1 = j0 + block < Skv ? j0 + block : Skv;
                    double mblk = -INFINITY;
                    for (long j = j0; j < j1; ++j) {
                        double s = -INFINITY;
                        if (visible(i, j, Sq, Skv, causal, window, n_sink)) {
                            double dot = 0.0;
                            for (int t = 0; t < d; ++t) dot += qrow[t] * kb[j * kvs + t];
                            s = scale * dot;
                        }
                        sblk[j - j0] = s;
                        if (s > mblk) mblk = s;
                    }
                    double m_new = m > mblk ? m : mblk;
                    double m_use = (m_new == -INFINITY) ? 0.0 : m_new; /* check_inf */
                    double c = exp(m - m_use);
                    double lblk = 0.0;
                    for (int t = 0; t < d; ++t) acc[t] *= c;
                    for (long j = j0; j < j1; ++j) {
                        double p = exp(sblk[j - j0] - m_use);
                        lblk += p;
                        if (p != 0.0)
                            for (int t = 0; t < d; ++t) acc[t] += p * vb[j * kvs + t];
                    }
                    l = c * l + lblk;
                    m = m_new;
                    if (trace && w == 0) {
                        double *tr = trace + nblk * (2 + d);
                        tr[0] = m;
                        tr[1] = l;
                        for (int t = 0; t < d; ++t) tr[2 + t] = acc[t];
                    }
                }
                double *orow = o + (((b * Sq + i) * Hq) + h) * d;
                const double sg = sink ? sink[h] : -INFINITY;
                if (sg != -INFINITY) {
                    double ms = (m > sg) ? m : sg;
                    double e1 = (l == 0.0) ? 0.0 : exp(m - ms);
                    double ls = l * e1 + exp(sg - ms);
                    for (int t = 0; t < d; ++t) orow[t] = acc[t] * e1 / ls;
                    lse[(b * Hq + h) * (long)Sq + i] = ms + log(ls);
                } else if (l == 0.0) {
                    for (int t = 0; t < d; ++t) orow[t] = 0.0;
                    lse[(b * Hq + h) * (long)Sq + i] = -INFINITY;
                } else {
                    for (int t = 0; t < d; ++t) orow[t] = acc[t] / l;
                    lse[(b * Hq + h) * (long)Sq + i] = m + log(l);
                }
            }
        }
        free(sblk);
        free(acc);
    }
    return bad ? 2 : 0;
}

/*
 * Split-KV decode partials (ch.15 sections 4.6, 4.8(3) and 5.4).  The keys
 * of request b are cut at page granularity: with np = ceil(L_b / page) pages
 * and pps = ceil(np / num_splits), split s covers pages
 * [s*pps, min((s+1)*pps, np)), its tokens capped at L_b.  Each split returns
 * its own normalised output O_s and log-sum-exp lse_s (natural log); an empty
 * split returns O_s = 0, lse_s = -inf.
 * o_part [B, Hq, num_splits, d], lse_part [B, Hq, num_splits].
 */
ORACLE_API int oracle_decode_split(const double *q, const double *k, const double *v,
                                   const int *seqlens, double *o_part, double *lse_part, int B,
                                   int Hq, int Hkv, int d, int Lmax, double scale, int num_splits,
                                   int page)
{
    if (Hkv <= 0 || Hq % Hkv != 0 || d <= 0 || num_splits <= 0 || page <= 0) return 1;
    const int groups = Hq / Hkv;
    int bad = 0;
#pragma omp parallel
    {
        double *srow = (double *)malloc(sizeof(double) * (Lmax > 0 ? Lmax : 1));
        if (!srow) {
#pragma omp atomic write
            bad = 1;
        } else {
#pragma omp for schedule(dynamic, 4)
            for (long w = 0; w < (long)B * Hq * num_splits; ++w) {
                long s = w % num_splits, h = (w / num_splits) % Hq, b = w / ((long)num_splits * Hq);
                long hk = h / groups, L = seqlens[b];
                long np = (L + page - 1) / page, pps = (np + num_splits - 1) / num_splits;
                long t0 = s * pps * page, t1 = (s + 1) * pps * page;
                if (t1 > L) t1 = L;
                if (t0 > L) t0 = L;
                const double *kb = k + ((b * (long)Lmax + t0) * Hkv + hk) * d;
                const double *vb = v + ((b * (long)Lmax + t0) * Hkv + hk) * d;
                /* the split's keys form their own row: no mask inside it */
                row_two_pass(q + (b * Hq + h) * d, kb, vb, (long)Hkv * d, 0, 1, t1 - t0, d,
                             scale, 0, 0, 0, -INFINITY, srow, o_part + w * d, lse_part + w);
            }
            free(srow);
        }
    }
    return bad ? 2 : 0;
}

/*
 * Log-sum-exp merge of split partials (ch.15 section 5.4): with
 * M = max_s lse_s and w_s = exp(lse_s - M),
 *     O   = sum_s w_s O_s / sum_s w_s,     LSE = M + ln(sum_s w_s),
 * summed in ascending split order.  All splits empty: O = 0, LSE = -inf.
 * sink (nullable, one logit per row): the sink joins the merge as one more
 * term of the denominator with no output, M = max(sigma, max_s lse_s),
 *     O = sum_s w_s O_s / (exp(sigma - M) + sum_s w_s),
 *     LSE = M + ln(exp(sigma - M) + sum_s w_s).
 */
ORACLE_API int oracle_combine(const double *o_part, const double *lse_part, double *o,
                              double *lse, long rows, int num_splits, int d, const double *sink)
{
    if (num_splits <= 0 || d <= 0) return 1;
#pragma omp parallel for schedule(static)
    for (long r = 0; r < rows; ++r) {
        const double *ls = lse_part + r * num_splits;
        const double *os = o_part + r * num_splits * (long)d;
        const double sg = sink ? sink[r] : -INFINITY;
        double M = sg;
        for (int s = 0; s < num_splits; ++s)
            if (ls[s] > M) M = ls[s];
        double *orow = o + r * d;
        for (int t = 0; t < d; ++t) orow[t] = 0.0;
        if (M == -INFINITY) {
            lse[r] = -INFINITY;
            continue;
        }
        double wsum = (sg == -INFINITY) ? 0.0 : exp(sg - M);
        for (int s = 0; s < num_splits; ++s) {
            double wt = exp(ls[s] - M);
            wsum += wt;
            if (wt != 0.0)
                for (int t = 0; t < d; ++t) orow[t] += wt * os[s * (long)d + t];
        }
        for (int t = 0; t < d; ++t) orow[t] /= wsum;
        lse[r] = M + log(wsum);
    }
    return 0;
}

/*
 * Backward pass of the dense forward (two-pass definition, per query row).
 * The pages state no formulas for it ("TileLang tutorial, ch.15", section
 * 5.4 only reports how much a low-precision, atomically accumulated dQ
 * loses); these are the chain rule through O = P V and the row softmax.
 * With P_i the row's probabilities and dO the gradient of O,
 *     dV_j += P_ij dO_i,          dP_ij = dO_i . V_j,
 *     D_i   = sum_j P_ij dP_ij,   dS_ij = P_ij (dP_ij - D_i),
 *     dQ_i  = scale sum_j dS_ij K_j,   dK_j += scale dS_ij Q_i.
 * Rows that see no key contribute nothing (their dQ is 0).  dK and dV of a
 * key/value head sum over the Hq/Hkv query heads that read it, in ascending
 * head, then row order.  dq [B,Sq,Hq,d], dk/dv [B,Skv,Hkv,d].
 * sink: NULL, or the logit sink of every query head [Hq]: one more softmax
 * column with no value row (the forward's reading), so P_ij is normalised
 * over the keys and the sink; its own gradient is
 *     dsink_h = sum over rows i of head h of  -P_i,sink D_i
 * (dS of the sink column, whose dP is 0), summed over the batch in ascending
 * order into dsink [Hq].
 */
ORACLE_API int oracle_attn_bwd(const double *q, const double *k, const double *v,
                               const double *dout, double *dq, double *dk, double *dv, int B,
                               int Hq, int Hkv, int Sq, int Skv, int d, double scale, int causal,
                               int window, int n_sink, const double *sink, double *dsink)
{
    if (Hkv <= 0 || Hq % Hkv != 0 || d <= 0) return 1;
    if (sink && !dsink) return 1;
    const int groups = Hq / Hkv;
    int bad = 0;
    /* per (batch, head) sink gradients, summed in ascending batch order below */
    double *dsink_part = sink ? (double *)calloc((size_t)(B > 0 ? B : 1) * Hq, sizeof(double))
                              : NULL;
    if (sink && !dsink_part) return 2;
#pragma omp parallel
    {
        double *p = (double *)malloc(sizeof(double) * (Skv > 0 ? Skv : 1));
        double *dp = (double *)malloc(sizeof(double) * (Skv > 0 ? Skv : 1));
        if (!p || !dp) {
#pragma omp atomic write
            bad = 1;
        } else {
#pragma omp for schedule(dynamic, 1)
            for (long w = 0; w < (long)B * Hkv; ++w) {
                long b = w / Hkv, hk = w % Hkv;
                const long kvs = (long)Hkv * d;
                const double *kb = k + ((b * (long)Skv) * Hkv + hk) * d;
                const double *vb = v + ((b * (long)Skv) * Hkv + hk) * d;
                double *dkb = dk + ((b * (long)Skv) * Hkv + hk) * d;
                double *dvb = dv + ((b * (long)Skv) * Hkv + hk) * d;
                for (long j = 0; j < Skv; ++j)
                    for (int t = 0; t < d; ++t) dkb[j * kvs + t] = dvb[j * kvs + t] = 0.0;
                for (long h = hk * groups; h < (hk + 1) * groups; ++h) {
                    for (long i = 0; i < Sq; ++i) {
                        const double *qi = q + (((b * Sq + i) * Hq) + h) * d;
                        const double *gi = dout + (((b * Sq + i) * Hq) + h) * d;
                        double *dqi = dq + (((b * Sq + i) * Hq) + h) * d;
                        for (int t = 0; t < d; ++t) dqi[t] = 0.0;
                        const double sg = sink ? sink[h] : -INFINITY;
                        double m = sg; /* the sink's column takes part in the row maximum */
                        for (long j = 0; j < Skv; ++j) {
                            if (!visible(i, j, Sq, Skv, causal, window, n_sink)) {
                                p[j] = -INFINITY;
                                continue;
                            }
                            double dot = 0.0;
                            for (int t = 0; t < d; ++t) dot += qi[t] * kb[j * kvs + t];
                            p[j] = scale * dot;
                            if (p[j] > m) m = p[j];
                        }
                        if (m == -INFINITY) continue; /* no visible key and no sink */
                        double sum = (sg == -INFINITY) ? 0.0 : exp(sg - m);
                        for (long j = 0; j < Skv; ++j) {
                            p[j] = (p[j] == -INFINITY) ? 0.0 : exp(p[j] - m);
                            sum += p[j];
                        }
                        double D = 0.0;
                        for (long j = 0; j < Skv; ++j) {
                            p[j] /= sum;
                            double g = 0.0;
                            for (int t = 0; t < d; ++t) g += gi[t] * vb[j * kvs + t];
                            dp[j] = g;
                            D += p[j] * g;
                        }
                        for (long j = 0; j < Skv; ++j) {
                            if (p[j] == 0.0) continue;
                            const double ds = p[j] * (dp[j] - D);
                            for (int t = 0; t < d; ++t) {
                                dvb[j * kvs + t] += p[j] * gi[t];
                                dqi[t] += scale * ds * kb[j * kvs + t];
                                dkb[j * kvs + t] += scale * ds * qi[t];
                            }
                        }
                        if (sg != -INFINITY) dsink_part[b * Hq + h] -= exp(sg - m) / sum * D;
                    }
                }
            }
        }
        free(p);
        free(dp);
    }
    if (sink) {
        for (int h = 0; h < Hq; ++h) {
            double acc = 0.0;
            for (int b = 0; b < B; ++b) acc += dsink_part[(long)b * Hq + h];
            dsink[h] = acc;
        }
        free(dsink_part);
    }
    return bad ? 2 : 0;
}

ORACLE_API int oracle_num_threads(void)
{
    int n = 1;
#pragma omp parallel
    {
#pragma omp single
        {
#ifdef _OPENMP
            extern int omp_get_num_threads(void);
            n = omp_get_num_threads();
#endif
        }
    }
    return n;
}

/* Sets the number of OpenMP threads later calls use (n >= 1); returns the
 * previous count.  Timing plumbing only: results do not depend on it. */
ORACLE_API int oracle_set_num_threads(int n)
{
    int prev = oracle_num_threads();
#ifdef _OPENMP
    extern void omp_set_num_threads(int);
    if (n >= 1) omp_set_num_threads(n);
#else
    (void)n;
#endif
    return prev;
}
