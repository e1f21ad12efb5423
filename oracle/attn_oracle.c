/*
 * fp64 CPU oracle for multi-head scaled dot-product attention.
 *
 * TEST INFRASTRUCTURE. Only the tests, the smoke check and the CPU-baseline
 * leg of the benchmark may build, load or call this file. The CUDA library
 * never links it, and it includes nothing from the CUDA path.
 *
 * What it computes is the plain definition, with no tiling, no online
 * softmax and no reordering beyond what the definition states:
 *
 *   "Attention Is All You Need", §3.2.1 eq. (1):
 *       Attention(Q, K, V) = softmax(Q K^T / sqrt(d_k)) V
 *   Figure 2 (left): MatMul -> Scale -> Mask (opt.) -> SoftMax -> MatMul.
 *   §3.2.3: in decoder self-attention every illegal connection (key j after
 *   query i) is set to -inf in the softmax input; position i itself stays
 *   visible. Masked weights are therefore exactly zero.
 *   §3.2.2: the h heads are independent problems run in parallel.
 *
 * The softmax subtracts the row maximum before exponentiating. That is a
 * numerical device only (exp(s - M) / sum exp(s - M) equals
 * exp(s) / sum exp(s) exactly in real arithmetic); the pages' numpy sketch of
 * eq. (1) does the same.
 *
 * The backward pass is the analytic derivative of the above for an upstream
 * gradient dO (the pages train the model, §5, but never write the derivative):
 *   D_i   = sum_c dO_ic O_ic
 *   dP_ij = sum_c dO_ic v_jc
 *   dS_ij = P_ij (dP_ij - D_i)
 *   dQ_i  = scale sum_j dS_ij k_j
 *   dK_j  = scale sum_i dS_ij q_i
 *   dV_j  = sum_i P_ij dO_i
 *
 * Readings where the pages are silent (each listed in the design notes):
 *   - scale is an explicit argument; callers pass 1/sqrt(d_k) for eq. (1).
 *   - causal masking is top-left aligned: key j is visible to query i iff
 *     j <= i, for any n and m.
 *   - lse_i = M_i + ln(l_i) = ln sum_j exp(s_ij), in natural-log units of the
 *     scaled score.
 *   - key padding (variable-length batches; the <pad> positions of Figure 3):
 *     sequence b has kv_len[b] real keys, the first ones; the others are
 *     masked like illegal connections (weight exactly 0, no gradient). A row
 *     that sees no key at all (kv_len[b] = 0) has O = 0, lse = -inf and zero
 *     gradients (the empty sum).
 *   - restricted self-attention (§4, Table 1: a neighbourhood of size r
 *     around the output position): key j is visible to query i only if
 *     i - wl <= j <= i + wr; wl = wr = (r - 1) / 2 for an odd r centred on i.
 *     A negative wl or wr leaves that side open. The window combines with the
 *     causal mask and with key padding (all conditions must hold); a row left
 *     with no visible key is the empty sum, as above.
 *
 * Layout: every tensor is a contiguous row-major [B, h, S, d] array of
 * doubles (lse is [B, h, n]). Built with -O2 -ffp-contract=off and without
 * -ffast-math so the C library's fp64 exp/log and IEEE rounding are used.
 */
#include <math.h>
#include <stddef.h>
#include <stdlib.h>
#include <string.h>

#ifdef _OPENMP
#include <omp.h>
#endif

#define ORACLE_OK 0
#define ORACLE_ERR_ARG 1
#define ORACLE_ERR_NOMEM 2

/* Number of keys visible to query i: all m, or j <= i when causal (§3.2.3). */
static long visible_keys(long i, long m, int causal) {
    if (!causal) return m;
    return (i + 1 < m) ? (i + 1) : m;
}

/* Keys visible to query i when only the first mb keys are real (key
 * padding, mb <= m): the causal limit, cut at mb. */
static long visible_padded(long i, long m, int causal, long mb) {
    const long v = visible_keys(i, m, causal);
    return v < mb ? v : mb;
}

/* The keys [lo, hi) visible to query i: the causal and padding limit above,
 * narrowed to the window i - wl <= j <= i + wr (a negative side is open).
 * hi <= lo means no key is visible. */
static void key_range(long i, long m, int causal, long mb, long wl, long wr,
                      long *lo, long *hi) {
    long h = visible_padded(i, m, causal, mb);
    if (wr >= 0 && i + wr + 1 < h) h = i + wr + 1;
    *lo = (wl >= 0 && i - wl > 0) ? i - wl : 0;
    *hi = h;
}

/* Real keys of head bh: kv_len[b] for its sequence b = bh / h, clamped to
 * [0, m]; all m without a length array. */
static long head_keys(const long *kv_len, long bh, long h, long m) {
    if (!kv_len) return m;
    const long mb = kv_len[bh / h];
    return mb < 0 ? 0 : (mb > m ? m : mb);
}

/* Step MatMul + Scale + Mask of Figure 2 for one query row:
 * s_j = scale * sum_c q_c k_jc for visible j, and -inf for masked j. */
static void score_row(const double *qi, const double *K, long m, long dk,
                      double scale, long lo, long hi, double *s) {
    for (long j = 0; j < m; ++j) {
        if (j < lo || j >= hi) {
            s[j] = -INFINITY;
            continue;
        }
        const double *kj = K + j * dk;
        double dot = 0.0;
        for (long c = 0; c < dk; ++c) dot += qi[c] * kj[c];
        s[j] = scale * dot;
    }
}

/* Step SoftMax of Figure 2, in place: s_j -> P_j = exp(s_j - M) / l with
 * M = max_j s_j and l = sum_j exp(s_j - M). Returns lse = M + ln l.
 * Masked entries hold -inf and come out as exactly 0. */
static double softmax_row(double *s, long m) {
    double M = -INFINITY;
    for (long j = 0; j < m; ++j)
        if (s[j] > M) M = s[j];
    if (M == -INFINITY) { /* no visible key: the empty sum */
        for (long j = 0; j < m; ++j) s[j] = 0.0;
        return -INFINITY;
    }
    double l = 0.0;
    for (long j = 0; j < m; ++j) {
        s[j] = exp(s[j] - M);
        l += s[j];
    }
    for (long j = 0; j < m; ++j) s[j] = s[j] / l;
    return M + log(l);
}

/* Second MatMul of Figure 2: O_i = sum_j P_j v_j. */
static void weighted_sum(const double *P, const double *V, long m, long dv,
                         double *oi) {
    for (long c = 0; c < dv; ++c) oi[c] = 0.0;
    for (long j = 0; j < m; ++j) {
        if (P[j] == 0.0) continue; /* masked or underflowed: contributes 0 */
        const double *vj = V + j * dv;
        for (long c = 0; c < dv; ++c) oi[c] += P[j] * vj[c];
    }
}

static int check_dims(long B, long h, long n, long m, long dk, long dv) {
    if (B < 0 || h < 0 || n < 0 || m < 1 || dk < 1 || dv < 1) return ORACLE_ERR_ARG;
    return ORACLE_OK;
}

/*
 * Scaled scores and attention weights of ONE head (Q: n x dk, K: m x dk).
 * s_out and p_out are n x m (either may be NULL). Masked scores are -inf.
 * Intended for small cases (inspection of the weight matrix, §3.2.1).
 */
int oracle_attn_weights(const double *Q, const double *K, long n, long m,
                        long dk, int causal, double scale, double *s_out,
                        double *p_out) {
    if (check_dims(1, 1, n, m, dk, 1) != ORACLE_OK) return ORACLE_ERR_ARG;
    double *row = (double *)malloc(sizeof(double) * (size_t)m);
    if (!row) return ORACLE_ERR_NOMEM;
    for (long i = 0; i < n; ++i) {
        score_row(Q + i * dk, K, m, dk, scale, 0, visible_keys(i, m, causal), row);
        if (s_out) memcpy(s_out + i * m, row, sizeof(double) * (size_t)m);
        softmax_row(row, m);
        if (p_out) memcpy(p_out + i * m, row, sizeof(double) * (size_t)m);
    }
    free(row);
    return ORACLE_OK;
}

/*
 * Forward pass, eq. (1) per (b, h) head.
 * q: [B,h,n,dk], k: [B,h,m,dk], v: [B,h,m,dv] -> o: [B,h,n,dv], lse: [B,h,n]
 * (lse may be NULL). rows/nrows: optional list of query indices to compute
 * (NULL = all n rows); rows not listed are left untouched in o and lse.
 */
int oracle_attn_fwd(const double *q, const double *k, const double *v,
                    double *o, double *lse, long B, long h, long n, long m,
                    long dk, long dv, int causal, double scale,
                    const long *rows, long nrows, const long *kv_len, long wl, long wr) {
    if (check_dims(B, h, n, m, dk, dv) != ORACLE_OK) return ORACLE_ERR_ARG;
    const long heads = B * h;
    const long R = rows ? nrows : n;
    if (rows)
        for (long r = 0; r < nrows; ++r)
            if (rows[r] < 0 || rows[r] >= n) return ORACLE_ERR_ARG;
    int status = ORACLE_OK;
#pragma omp parallel
    {
        double *row = (double *)malloc(sizeof(double) * (size_t)m);
        if (!row) {
#pragma omp atomic write
            status = ORACLE_ERR_NOMEM;
        }
#pragma omp for collapse(2) schedule(dynamic, 4)
        for (long bh = 0; bh < heads; ++bh) {
            for (long r = 0; r < R; ++r) {
                if (!row) continue;
                const long i = rows ? rows[r] : r;
                const double *Q = q + bh * n * dk;
                const double *K = k + bh * m * dk;
                const double *V = v + bh * m * dv;
                long lo, hi;
                key_range(i, m, causal, head_keys(kv_len, bh, h, m), wl, wr, &lo, &hi);
                score_row(Q + i * dk, K, m, dk, scale, lo, hi, row);
                const double l = softmax_row(row, m);
                weighted_sum(row, V, m, dv, o + (bh * n + i) * dv);
                if (lse) lse[bh * n + i] = l;
            }
        }
        free(row);
    }
    return status;
}

/*
 * Backward, one query row i of one head: the forward row (P_i., O_i,
 * lse_i), D_i = dO_i . O_i and, if dqi != NULL,
 * dQ_i = scale sum_j P_ij (dO_i . v_j - D_i) k_j.
 * row (m doubles) and oi (dv doubles) are scratch.
 */
static void bwd_query_row(const double *Q, const double *K, const double *V,
                          const double *dOi, long i, long m, long mb, long wl, long wr,
                          long dk, long dv, int causal, double scale, double *row,
                          double *oi, double *lse_i, double *D_i, double *dqi) {
    long lo, hi;
    key_range(i, m, causal, mb, wl, wr, &lo, &hi);
    score_row(Q + i * dk, K, m, dk, scale, lo, hi, row);
    const double l = softmax_row(row, m);
    weighted_sum(row, V, m, dv, oi);
    double Di = 0.0;
    for (long c = 0; c < dv; ++c) Di += dOi[c] * oi[c];
    *lse_i = l;
    *D_i = Di;
    if (dqi) {
        for (long c = 0; c < dk; ++c) dqi[c] = 0.0;
        for (long j = 0; j < m; ++j) {
            if (row[j] == 0.0) continue; /* P_ij = 0 => dS_ij = 0 */
            const double *vj = V + j * dv;
            double dP = 0.0;
            for (long c = 0; c < dv; ++c) dP += dOi[c] * vj[c];
            const double dS = row[j] * (dP - Di);
            const double *kj = K + j * dk;
            for (long c = 0; c < dk; ++c) dqi[c] += dS * kj[c];
        }
        for (long c = 0; c < dk; ++c) dqi[c] *= scale;
    }
}

/*
 * Backward, one key row j of one head, given lse_i and D_i of every query:
 * dK_j = scale sum_i dS_ij q_i and dV_j = sum_i P_ij dO_i with
 * P_ij = exp(s_ij - lse_i) (the softmax written through its normaliser).
 * Either output may be NULL.
 */
static void bwd_key_row(const double *Q, const double *kj, const double *vj,
                        const double *dO, const double *lse, const double *D,
                        long j, long n, long m, long mb, long wl, long wr, long dk, long dv,
                        int causal, double scale, double *dkj, double *dvj) {
    if (dkj) for (long c = 0; c < dk; ++c) dkj[c] = 0.0;
    if (dvj) for (long c = 0; c < dv; ++c) dvj[c] = 0.0;
    for (long i = 0; i < n; ++i) {
        long lo, hi;
        key_range(i, m, causal, mb, wl, wr, &lo, &hi);
        if (j < lo || j >= hi) continue; /* masked: P_ij = 0 */
        const double *qi = Q + i * dk;
        const double *dOi = dO + i * dv;
        double dot = 0.0;
        for (long c = 0; c < dk; ++c) dot += qi[c] * kj[c];
        const double P = exp(scale * dot - lse[i]);
        if (dvj)
            for (long c = 0; c < dv; ++c) dvj[c] += P * dOi[c];
        if (dkj) {
            double dP = 0.0;
            for (long c = 0; c < dv; ++c) dP += dOi[c] * vj[c];
            const double dS = P * (dP - D[i]);
            for (long c = 0; c < dk; ++c) dkj[c] += dS * qi[c];
        }
    }
    if (dkj) for (long c = 0; c < dk; ++c) dkj[c] *= scale;
}

/*
 * Backward pass: gradients of L = sum(dO * O) with respect to q, k and v,
 * for O from oracle_attn_fwd on the same inputs.
 * dq: [B,h,n,dk], dk_out: [B,h,m,dk], dv_out: [B,h,m,dv]; each may be NULL
 * to skip it. o_out / lse_out (optional) receive the forward results the
 * backward used.
 *
 * Pass 1 (per query row i): P_i., O_i, lse_i, D_i and dQ_i.
 * Pass 2 (per key row j): dK_j and dV_j.
 */
int oracle_attn_bwd(const double *q, const double *k, const double *v,
                    const double *dO, double *dq, double *dk_out,
                    double *dv_out, double *o_out, double *lse_out, long B,
                    long h, long n, long m, long dk, long dv, int causal,
                    double scale, const long *kv_len, long wl, long wr) {
    if (check_dims(B, h, n, m, dk, dv) != ORACLE_OK) return ORACLE_ERR_ARG;
    const long heads = B * h;
    double *lse = (double *)malloc(sizeof(double) * (size_t)(heads * n + 1));
    double *D = (double *)malloc(sizeof(double) * (size_t)(heads * n + 1));
    if (!lse || !D) {
        free(lse);
        free(D);
        return ORACLE_ERR_NOMEM;
    }
    int status = ORACLE_OK;
#pragma omp parallel
    {
        double *row = (double *)malloc(sizeof(double) * (size_t)m);
        double *oi = (double *)malloc(sizeof(double) * (size_t)dv);
        if (!row || !oi) {
#pragma omp atomic write
            status = ORACLE_ERR_NOMEM;
        }
#pragma omp for collapse(2) schedule(dynamic, 4)
        for (long bh = 0; bh < heads; ++bh) {
            for (long i = 0; i < n; ++i) {
                if (!row || !oi) continue;
                bwd_query_row(q + bh * n * dk, k + bh * m * dk, v + bh * m * dv,
                              dO + (bh * n + i) * dv, i, m, head_keys(kv_len, bh, h, m), wl, wr,
                              dk, dv, causal, scale,
                              row, oi, &lse[bh * n + i], &D[bh * n + i],
                              dq ? dq + (bh * n + i) * dk : NULL);
                if (o_out) memcpy(o_out + (bh * n + i) * dv, oi, sizeof(double) * (size_t)dv);
                if (lse_out) lse_out[bh * n + i] = lse[bh * n + i];
            }
        }
        /* implicit barrier: lse and D are complete */
        if (dk_out || dv_out) {
#pragma omp for collapse(2) schedule(dynamic, 4)
            for (long bh = 0; bh < heads; ++bh) {
                for (long j = 0; j < m; ++j) {
                    bwd_key_row(q + bh * n * dk, k + (bh * m + j) * dk, v + (bh * m + j) * dv,
                                dO + bh * n * dv, lse + bh * n, D + bh * n, j, n, m,
                                head_keys(kv_len, bh, h, m), wl, wr, dk, dv,
                                causal, scale, dk_out ? dk_out + (bh * m + j) * dk : NULL,
                                dv_out ? dv_out + (bh * m + j) * dv : NULL);
                }
            }
        }
        free(row);
        free(oi);
    }
    free(lse);
    free(D);
    return status;
}

/*
 * Sampled backward of ONE head (q: n x dk, k: m x dk, v: m x dv, dO: n x dv):
 * dQ for the listed query rows (dq_out: nq x dk) and dK, dV for the listed
 * key rows (dk_out: nk x dk, dv_out: nk x dv). Same arithmetic as
 * oracle_attn_bwd row by row; key rows need lse and D of all n queries, so
 * they cost a full forward of the head.
 */
int oracle_attn_bwd_rows(const double *q, const double *k, const double *v,
                         const double *dO, long n, long m, long dk, long dv,
                         int causal, double scale, const long *qrows, long nq,
                         double *dq_out, const long *krows, long nk,
                         double *dk_out, double *dv_out, long kv_len, long wl, long wr) {
    if (check_dims(1, 1, n, m, dk, dv) != ORACLE_OK || nq < 0 || nk < 0) return ORACLE_ERR_ARG;
    for (long r = 0; r < nq; ++r)
        if (qrows[r] < 0 || qrows[r] >= n) return ORACLE_ERR_ARG;
    for (long r = 0; r < nk; ++r)
        if (krows[r] < 0 || krows[r] >= m) return ORACLE_ERR_ARG;
    const long nall = nk > 0 ? n : 0;
    const long mb = kv_len < 0 ? m : (kv_len > m ? m : kv_len); /* < 0: no key padding */
    double *lse = (double *)malloc(sizeof(double) * (size_t)(nall + 1));
    double *D = (double *)malloc(sizeof(double) * (size_t)(nall + 1));
    if (!lse || !D) {
        free(lse);
        free(D);
        return ORACLE_ERR_NOMEM;
    }
    int status = ORACLE_OK;
#pragma omp parallel
    {
        double *row = (double *)malloc(sizeof(double) * (size_t)m);
        double *oi = (double *)malloc(sizeof(double) * (size_t)dv);
        if (!row || !oi) {
#pragma omp atomic write
            status = ORACLE_ERR_NOMEM;
        }
#pragma omp for schedule(dynamic, 4)
        for (long r = 0; r < nq; ++r) {
            if (!row || !oi) continue;
            double l, Di;
            const long i = qrows[r];
            bwd_query_row(q, k, v, dO + i * dv, i, m, mb, wl, wr, dk, dv, causal, scale, row, oi,
                          &l, &Di, dq_out + r * dk);
        }
#pragma omp for schedule(dynamic, 16)
        for (long i = 0; i < nall; ++i) {
            if (!row || !oi) continue;
            bwd_query_row(q, k, v, dO + i * dv, i, m, mb, wl, wr, dk, dv, causal, scale, row, oi,
                          &lse[i], &D[i], NULL);
        }
#pragma omp for schedule(dynamic, 1)
        for (long r = 0; r < nk; ++r) {
            const long j = krows[r];
            bwd_key_row(q, k + j * dk, v + j * dv, dO, lse, D, j, n, m, mb, wl, wr, dk, dv, causal,
                        scale, dk_out + r * dk, dv_out + r * dv);
        }
        free(row);
        free(oi);
    }
    free(lse);
    free(D);
    return status;
}

/* Threads the oracle will use (OpenMP team size), for reporting. */
int oracle_num_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
