/*
 * attn_oracle.c -- plain fp64 CPU oracle for exact attention forward.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path links, loads or
 * calls this file: only the test suite, the package's smoke check and the
 * benchmark's CPU-baseline leg use it.  It shares no code, header, table or
 * constant with the CUDA library.
 *
 * What it computes (the plain definition, no blocking, no fusion):
 *
 *   s_ij = scale * sum_t q_it k_jt                      (fp64, inputs widened exactly)
 *   allowed(i, j) = !causal || j <= i + (Nk - Nq)        (bottom-right causal alignment)
 *   m_i  = max_{j allowed} s_ij
 *   p_ij = exp(s_ij - m_i) if allowed else 0
 *   l_i  = sum_j p_ij
 *   O_i  = sum_j p_ij v_j / l_i
 *   LSE_i = m_i + ln l_i        (natural log of the scaled scores)
 *
 * Sources:
 *  - "Lecture 25: why attention needs no intermediate matrix",
 *    §1.1 (standard attention O = softmax(QK^T/sqrt(d)) V) and §2.1 (safe
 *    softmax: subtract the row max, exponentiate, sum, divide).
 *  - "6.2 FlashAttention V2 explained", §5.1 (causal mask: -inf
 *    added before the softmax so row i sees only j <= i) and §6 (the forward
 *    algorithm and its L = m + log(l) output).
 *  - "02 · FA2: parallelism and work partitioning", §4 (the causal
 *    KV-block bound carries the offset seqlen_k - seqlen_q, i.e. the
 *    diagonal is aligned to the bottom-right corner when Nq != Nk).
 *  - Fully masked rows (possible only when causal and Nq > Nk) give O = 0 and
 *    LSE = -inf: the official FA2 epilogue quoted in "Flash Attention (4) v2.1
 *    forward", §3.5, guards l == 0 by using 1 instead of 1/l, which
 *    leaves the zero accumulator as the output.
 *
 * The backward (oracle_attn_bwd, at the end of this file) is the chain rule of
 * this definition.
 *
 * Two further modes exist only to check invariants of the method:
 *  - oracle_attn_tiled: the online-softmax loop of "6.2 FlashAttention V2
 *    explained" §6 in fp64, over KV tiles of a caller-chosen width (with the
 *    rule of "Flash Attention (4)" §2.5 that a running
 *    max of -inf is replaced by 0 before it is subtracted);
 *  - oracle_attn_split_partials + oracle_combine: the split-KV partial
 *    (O_s, LSE_s) per contiguous key range and their LSE-weighted merge
 *    ("02 · FA2" §2, "decode / split-KV").
 *
 * Every row is independent; rows may run on several OpenMP threads, which
 * changes no arithmetic inside a row.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

static int g_threads = 1;

int oracle_set_threads(int n) {
#ifdef _OPENMP
    g_threads = n > 0 ? n : 1;
    return g_threads;
#else
    (void)n;
    g_threads = 1;
    return 1;
#endif
}

int oracle_has_openmp(void) {
#ifdef _OPENMP
    return 1;
#else
    return 0;
#endif
}

/* Number of keys row i may see: keys 0 .. limit-1 (the causal mask is a prefix). */
static long allowed_limit(long i, long Nq, long Nk, int causal) {
    if (!causal) return Nk;
    long lim = i + (Nk - Nq) + 1;
    if (lim < 0) lim = 0;
    if (lim > Nk) lim = Nk;
    return lim;
}

/*
 * One row of the definition, with the S row and the P row held in full.
 * keys [j0, j1) are the candidate keys; within them the causal limit applies.
 * Writes o[0..d) and *lse.  Returns the row sum l (0 for an empty row).
 */
static double attn_row_range(const double *qi, const double *k, const double *v,
                             long i, long Nq, long Nk, int d, int causal, double scale,
                             long j0, long j1, double *s, double *p,
                             double *o, double *lse) {
    long lim = allowed_limit(i, Nq, Nk, causal);
    for (int t = 0; t < d; ++t) o[t] = 0.0;

    /* S row: s_j = scale * q_i . k_j, -inf where masked */
    for (long j = j0; j < j1; ++j) {
        if (j < lim) {
            double acc = 0.0;
            const double *kj = k + (size_t)j * d;
            for (int t = 0; t < d; ++t) acc += qi[t] * kj[t];
            s[j - j0] = scale * acc;
        } else {
            s[j - j0] = -INFINITY;
        }
    }
    /* m = row max over allowed entries */
    double m = -INFINITY;
    for (long j = j0; j < j1; ++j)
        if (s[j - j0] > m) m = s[j - j0];
    if (m == -INFINITY) { /* no allowed key in range */
        *lse = -INFINITY;
        return 0.0;
    }
    /* P row and its sum */
    double l = 0.0;
    for (long j = j0; j < j1; ++j) {
        double sj = s[j - j0];
        p[j - j0] = (sj == -INFINITY) ? 0.0 : exp(sj - m);
        l += p[j - j0];
    }
    /* O = P V / l */
    for (long j = j0; j < j1; ++j) {
        double pj = p[j - j0];
        if (pj == 0.0) continue;
        const double *vj = v + (size_t)j * d;
        for (int t = 0; t < d; ++t) o[t] += pj * vj[t];
    }
    for (int t = 0; t < d; ++t) o[t] /= l;
    *lse = m + log(l);
    return l;
}

/*
 * Full attention for BH independent heads.
 * q: [BH][Nq][d], k, v: [BH][Nk][d], o: [BH][Nq][d], lse: [BH][Nq]; all fp64, contiguous.
 */
int oracle_attn_full(const double *q, const double *k, const double *v,
                     int BH, int Nq, int Nk, int d, int causal, double scale,
                     double *o, double *lse) {
    if (BH < 0 || Nq < 0 || Nk < 0 || d <= 0) return -1;
    long total = (long)BH * Nq;
#pragma omp parallel num_threads(g_threads)
    {
        double *s = (double *)malloc(sizeof(double) * (size_t)(Nk > 0 ? Nk : 1));
        double *p = (double *)malloc(sizeof(double) * (size_t)(Nk > 0 ? Nk : 1));
#pragma omp for schedule(dynamic, 16)
        for (long r = 0; r < total; ++r) {
            long bh = r / Nq, i = r % Nq;
            const double *kb = k + (size_t)bh * Nk * d;
            const double *vb = v + (size_t)bh * Nk * d;
            attn_row_range(q + (size_t)r * d, kb, vb, i, Nq, Nk, d, causal, scale, 0, Nk,
                           s, p, o + (size_t)r * d, lse + r);
        }
        free(s);
        free(p);
    }
    return 0;
}

/*
 * Selected rows only.  Row n has query q_rows[n], index row_index[n] in [0, Nq)
 * and reads keys/values from slot kv_slot[n] of k, v: [nslots][Nk][d].
 */
int oracle_attn_rows(const double *q_rows, const int64_t *row_index, const int64_t *kv_slot,
                     const double *k, const double *v, int n, int Nq, int Nk, int d,
                     int causal, double scale, double *o, double *lse) {
    if (n < 0 || Nq <= 0 || Nk < 0 || d <= 0) return -1;
#pragma omp parallel num_threads(g_threads)
    {
        double *s = (double *)malloc(sizeof(double) * (size_t)(Nk > 0 ? Nk : 1));
        double *p = (double *)malloc(sizeof(double) * (size_t)(Nk > 0 ? Nk : 1));
#pragma omp for schedule(dynamic, 1)
        for (long r = 0; r < n; ++r) {
            const double *kb = k + (size_t)kv_slot[r] * Nk * d;
            const double *vb = v + (size_t)kv_slot[r] * Nk * d;
            attn_row_range(q_rows + (size_t)r * d, kb, vb, (long)row_index[r], Nq, Nk, d,
                           causal, scale, 0, Nk, s, p, o + (size_t)r * d, lse + r);
        }
        free(s);
        free(p);
    }
    return 0;
}

/*
 * The forward loop of "6.2 FlashAttention V2 explained" §6 in fp64: rows in
 * blocks of Br, keys in tiles of Bc,
 * running (m, l, O~) per row, deferred 1/l, L = m + ln l.  The causal KV bound
 * is the block's last allowed key (with the Nk - Nq offset).  Exists to show
 * that the tiled online softmax equals the full softmax.
 */
int oracle_attn_tiled(const double *q, const double *k, const double *v,
                      int BH, int Nq, int Nk, int d, int causal, double scale,
                      int Br, int Bc, double *o, double *lse) {
    if (Br <= 0 || Bc <= 0 || d <= 0) return -1;
    long nblk = (Nq + Br - 1) / Br;
    long total = (long)BH * nblk;
#pragma omp parallel num_threads(g_threads)
    {
        double *acc = (double *)malloc(sizeof(double) * (size_t)d);
        double *srow = (double *)malloc(sizeof(double) * (size_t)Bc);
#pragma omp for schedule(dynamic, 1)
        for (long w = 0; w < total; ++w) {
            long bh = w / nblk, blk = w % nblk;
            long i0 = blk * Br, i1 = i0 + Br < Nq ? i0 + Br : Nq;
            long kv_end = Nk;
            if (causal) {
                kv_end = i1 + (Nk - Nq); /* last row of the block sees keys < i1 + Nk - Nq */
                if (kv_end > Nk) kv_end = Nk;
                if (kv_end < 0) kv_end = 0;
            }
            const double *kb = k + (size_t)bh * Nk * d;
            const double *vb = v + (size_t)bh * Nk * d;
            for (long i = i0; i < i1; ++i) {
                const double *qi = q + ((size_t)bh * Nq + i) * d;
                long lim = allowed_limit(i, Nq, Nk, causal);
                double m = -INFINITY, l = 0.0;
                for (int t = 0; t < d; ++t) acc[t] = 0.0;
                for (long j0 = 0; j0 < kv_end; j0 += Bc) {
                    long j1 = j0 + Bc < kv_end ? j0 + Bc : kv_end;
                    double mt = -INFINITY;
                    for (long j = j0; j < j1; ++j) {
                        double sj = -INFINITY;
                        if (j < lim) {
                            double a = 0.0;
                            for (int t = 0; t < d; ++t) a += qi[t] * kb[(size_t)j * d + t];
                            sj = scale * a;
                        }
                        srow[j - j0] = sj;
                        if (sj > mt) mt = sj;
                    }
                    double m_new = m > mt ? m : mt;
                    double m_sub = (m_new == -INFINITY) ? 0.0 : m_new; /* -inf guard */
                    double alpha = exp(m - m_sub);                      /* exp(-inf) = 0 */
                    double lt = 0.0;
                    for (int t = 0; t < d; ++t) acc[t] *= alpha;
                    for (long j = j0; j < j1; ++j) {
                        double pj = exp(srow[j - j0] - m_sub);
                        lt += pj;
                        if (pj != 0.0)
                            for (int t = 0; t < d; ++t) acc[t] += pj * vb[(size_t)j * d + t];
                    }
                    l = l * alpha + lt;
                    m = m_new;
                }
                double *oi = o + ((size_t)bh * Nq + i) * d;
                if (l == 0.0) {
                    for (int t = 0; t < d; ++t) oi[t] = 0.0;
                    lse[bh * Nq + i] = -INFINITY;
                } else {
                    for (int t = 0; t < d; ++t) oi[t] = acc[t] / l;
                    lse[bh * Nq + i] = m + log(l);
                }
            }
        }
        free(acc);
        free(srow);
    }
    return 0;
}

/*
 * Split-KV partials: split s covers keys [s*split_len, min((s+1)*split_len, Nk)).
 * For each split and row: the definition restricted to that key range, giving a
 * normalised O_s and LSE_s (O_s = 0, LSE_s = -inf when the range has no allowed key).
 * o_part: [S][BH][Nq][d], lse_part: [S][BH][Nq].
 */
int oracle_attn_split_partials(const double *q, const double *k, const double *v,
                               int BH, int Nq, int Nk, int d, int causal, double scale,
                               int num_splits, long split_len,
                               double *o_part, double *lse_part) {
    if (num_splits <= 0 || split_len <= 0 || d <= 0) return -1;
    long rows = (long)BH * Nq;
    long total = rows * num_splits;
#pragma omp parallel num_threads(g_threads)
    {
        double *s = (double *)malloc(sizeof(double) * (size_t)(split_len));
        double *p = (double *)malloc(sizeof(double) * (size_t)(split_len));
#pragma omp for schedule(dynamic, 16)
        for (long w = 0; w < total; ++w) {
            long sp = w / rows, r = w % rows;
            long bh = r / Nq, i = r % Nq;
            long j0 = sp * split_len, j1 = j0 + split_len;
            if (j0 > Nk) j0 = Nk;
            if (j1 > Nk) j1 = Nk;
            attn_row_range(q + (size_t)r * d, k + (size_t)bh * Nk * d, v + (size_t)bh * Nk * d,
                           i, Nq, Nk, d, causal, scale, j0, j1, s, p,
                           o_part + (size_t)w * d, lse_part + w);
        }
        free(s);
        free(p);
    }
    return 0;
}

/*
 * LSE-weighted merge of S partials per row:
 *   M = max_s LSE_s;  w_s = exp(LSE_s - M);  LSE = M + ln sum_s w_s;
 *   O = sum_s w_s O_s / sum_s w_s.       A row whose partials are all empty
 * (every LSE_s = -inf) gives O = 0, LSE = -inf.
 * o_part: [S][rows][d], lse_part: [S][rows]; o: [rows][d], lse: [rows].
 */
int oracle_combine(const double *o_part, const double *lse_part, int num_splits, long rows,
                   int d, double *o, double *lse) {
    if (num_splits <= 0 || d <= 0) return -1;
    for (long r = 0; r < rows; ++r) {
        double M = -INFINITY;
        for (int s = 0; s < num_splits; ++s) {
            double ls = lse_part[(size_t)s * rows + r];
            if (ls > M) M = ls;
        }
        double *orow = o + (size_t)r * d;
        for (int t = 0; t < d; ++t) orow[t] = 0.0;
        if (M == -INFINITY) {
            lse[r] = -INFINITY;
            continue;
        }
        double wsum = 0.0;
        for (int s = 0; s < num_splits; ++s) {
            double ls = lse_part[(size_t)s * rows + r];
            double w = (ls == -INFINITY) ? 0.0 : exp(ls - M);
            wsum += w;
            if (w != 0.0) {
                const double *op = o_part + ((size_t)s * rows + r) * d;
                for (int t = 0; t < d; ++t) orow[t] += w * op[t];
            }
        }
        for (int t = 0; t < d; ++t) orow[t] /= wsum;
        lse[r] = M + log(wsum);
    }
    return 0;
}

/*
 * Backward of the definition: the gradients of O = softmax(scale * Q K^T + mask) V
 * with respect to Q, K and V, given dO (the gradient of a loss with respect to O).
 *
 *   P     = softmax(scale * Q K^T + mask)        (the forward's row-normalised weights)
 *   dV    = P^T dO
 *   dP    = dO V^T
 *   dS    = P o (dP - rowsum(dP o P))            (o: elementwise product)
 *   dQ    = scale * dS K,     dK = scale * dS^T Q
 *
 * ("Lecture 25" §3.3, the backward's chain-rule formulas, with P recomputed from
 * the scores rather than stored; the factor `scale` is the chain rule through
 * S = scale * Q K^T, which the page's formulas leave out because they write S
 * with the scale folded in.)  A row that sees no key has P = 0 and contributes
 * nothing.  Heads are independent and may run on several OpenMP threads; within
 * a head the rows are taken in order, so dK and dV are plain sums.
 * q, dout, dq: [BH][Nq][d]; k, v, dk, dv: [BH][Nk][d]; fp64, contiguous.
 */
int oracle_attn_bwd(const double *q, const double *k, const double *v, const double *dout,
                    int BH, int Nq, int Nk, int d, int causal, double scale,
                    double *dq, double *dk, double *dv) {
    if (BH < 0 || Nq < 0 || Nk < 0 || d <= 0) return -1;
    int bad = 0;
#ifdef _OPENMP
#pragma omp parallel for schedule(dynamic, 1) num_threads(g_threads) reduction(| : bad)
#endif
    for (int h = 0; h < BH; ++h) {
        const double *qh = q + (size_t)h * Nq * d, *kh = k + (size_t)h * Nk * d, *vh = v + (size_t)h * Nk * d;
        const double *doh = dout + (size_t)h * Nq * d;
        double *dqh = dq + (size_t)h * Nq * d, *dkh = dk + (size_t)h * Nk * d, *dvh = dv + (size_t)h * Nk * d;
        memset(dqh, 0, sizeof(double) * (size_t)Nq * d);
        memset(dkh, 0, sizeof(double) * (size_t)Nk * d);
        memset(dvh, 0, sizeof(double) * (size_t)Nk * d);
        double *s = (double *)malloc(sizeof(double) * (size_t)(Nk > 0 ? Nk : 1) * 3 + sizeof(double) * d);
        if (s == NULL) { bad = 1; continue; }
        double *p = s + (Nk > 0 ? Nk : 1), *dp = p + (Nk > 0 ? Nk : 1), *orow = dp + (Nk > 0 ? Nk : 1);
        for (long i = 0; i < Nq; ++i) {
            const double *qi = qh + (size_t)i * d, *doi = doh + (size_t)i * d;
            double lse;
            const double l = attn_row_range(qi, kh, vh, i, Nq, Nk, d, causal, scale, 0, Nk, s, p, orow, &lse);
            if (l == 0.0) continue; /* no visible key: P = 0 */
            /* P row normalised; dP = dO_i . v_j; D = rowsum(dP o P) */
            double D = 0.0;
            for (long j = 0; j < Nk; ++j) {
                p[j] /= l;
                double acc = 0.0;
                if (p[j] != 0.0) {
                    const double *vj = vh + (size_t)j * d;
                    for (int t = 0; t < d; ++t) acc += doi[t] * vj[t];
                }
                dp[j] = acc;
                D += p[j] * acc;
            }
            double *dqi = dqh + (size_t)i * d;
            for (long j = 0; j < Nk; ++j) {
                if (p[j] == 0.0) continue;
                const double ds = p[j] * (dp[j] - D);
                const double *kj = kh + (size_t)j * d;
                double *dkj = dkh + (size_t)j * d, *dvj = dvh + (size_t)j * d;
                for (int t = 0; t < d; ++t) {
                    dvj[t] += p[j] * doi[t];
                    dqi[t] += scale * ds * kj[t];
                    dkj[t] += scale * ds * qi[t];
                }
            }
        }
        free(s);
    }
    return bad ? -2 : 0;
}
