/*
 * ra_oracle.c -- plain, slow, fp64 CPU oracle for packed causal varlen
 * ring attention.  TEST INFRASTRUCTURE ONLY: it is called by the tests, by
 * the smoke check and by the benchmark's CPU-baseline leg, never by the
 * product path.  It shares no code, header or constant with the CUDA
 * library; every function restates its definition directly.
 *
 * What the pages fix, and where (page title, then the part of the page):
 *  - packed sequences must not attend across documents: "Attention Mask for
 *    Packed Sequences (via Attention Bias)" (EasyDeL #129), opening request;
 *    the mask is written out explicitly as a per-pair predicate here;
 *  - the causal mask inside each document: maxtext PR #1133, description
 *    (the TE all-gather CP path supports only the causal mask type);
 *  - softmax scale 1/sqrt(head_dim): maxtext PR #1133, cudnn_flash_attention
 *    diff (scale_factor);
 *  - the zigzag split into 2*CP chunks, rank r holding chunks r and
 *    2*CP-1-r: ring-attention-pytorch #20 (`extract_local`) and maxtext
 *    PR #1133 review comment on reordering;
 *  - a ring attention step computes attention of the local queries against
 *    one KV shard and the partial results are merged: "Question about varlen
 *    ring attention" (MiniMax-01 #6) and FlagScale PR #910 (RingAttention
 *    with forward_impl / backward_impl).
 * The pages print no formula.  The attention, log-sum-exp, merge and
 * gradient below are the textbook definitions (plainest reading).
 *
 * Parity pins for every function live in tests/test_oracle_*.py.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

int orc_set_threads(int n) {
#ifdef _OPENMP
    if (n > 0) omp_set_num_threads(n);
    return omp_get_max_threads();
#else
    (void)n;
    return 1;
#endif
}

/* ------------------------------------------------------------------------
 * Attention of a set of queries against a set of keys, restricted to the
 * allowed pairs
 *      A(i) = { j : seg_k[j] == seg_q[i]  and  (causal == 0  or  k_pos[j] <= q_pos[i])
 *                   and  (window < 0  or  k_pos[j] >= q_pos[i] - window) }.
 * The window is the sliding-window mask named by the window_size argument of
 * the cuDNN flash-attention call ("Add Context Parallelism support to cudnn
 * Flash Attention #1133", maxtext, diff of cudnn_flash_attention), read as a
 * key reaching back at most `window` positions from its query.
 * With seg = document id and pos = packed index this is the full
 * block-diagonal causal attention; with a subset of keys it is one ring
 * step's partial result.
 *
 * Interval masks (the dynamic, per-token attention masks of "[Train]
 * Support custom attention with context parallel", FlagScale PR #910,
 * description: flex attention with context parallelism): with q_lo and
 * q_hi given (NULL = none), the allowed set is further restricted to
 *      q_lo[i] <= k_pos[j] <= q_hi[i],
 * the bounds being positions, like k_pos.  Causal, sliding-window,
 * chunked-local, prefix-LM and bidirectional document masks are all such
 * intervals.
 *
 *   s_ij  = scale * sum_c q[i,h,c] * k[j,g,c],      g = h / (Hq/Hkv)
 *   lse_i = m + log( sum_{j in A(i)} exp(s_ij - m) ),  m = max_{j in A(i)} s_ij
 *   o_i   = sum_{j in A(i)} exp(s_ij - lse_i) * v[j,g,:]
 *   A(i) empty:  o_i = 0,  lse_i = -inf.
 *
 * rows: the query indices to evaluate (NULL = all Tq rows in order).
 * out [nrows, Hq, d], lse [nrows, Hq] (natural log).
 * ------------------------------------------------------------------------ */
static int pair_allowed(int32_t sq, int32_t sk, int64_t qp, int64_t kp, int causal, int64_t window,
                        const int64_t *q_lo, const int64_t *q_hi, int64_t i)
{
    if (sk != sq) return 0;
    if (causal && kp > qp) return 0;
    if (window >= 0 && kp < qp - window) return 0;
    if (q_lo && kp < q_lo[i]) return 0;
    if (q_hi && kp > q_hi[i]) return 0;
    return 1;
}

int orc_partial_fwd(const double *q, const double *k, const double *v,
                    int64_t Tq, int64_t Tk, int Hq, int Hkv, int d,
                    const int32_t *seg_q, const int32_t *seg_k,
                    const int64_t *q_pos, const int64_t *k_pos,
                    int causal, int64_t window, double scale,
                    const int64_t *q_lo, const int64_t *q_hi,
                    const int64_t *rows, int64_t nrows,
                    double *out, double *lse)
{
    if (Hkv <= 0 || Hq % Hkv != 0 || d <= 0) return 1;
    const int G = Hq / Hkv;
    if (rows == NULL) nrows = Tq;
    int64_t total = nrows * (int64_t)Hq;
#pragma omp parallel
    {
        double *s = (double *)malloc(sizeof(double) * (size_t)(Tk > 0 ? Tk : 1));
        unsigned char *ok = (unsigned char *)malloc((size_t)(Tk > 0 ? Tk : 1));
#pragma omp for schedule(dynamic, 8)
        for (int64_t w = 0; w < total; ++w) {
            int64_t ri = w / Hq;
            int h = (int)(w % Hq);
            int64_t i = rows ? rows[ri] : ri;
            int g = h / G;
            const double *qi = q + (i * Hq + h) * (int64_t)d;
            double m = -INFINITY;
            int any = 0;
            for (int64_t j = 0; j < Tk; ++j) {
                int allowed = pair_allowed(seg_q[i], seg_k[j], q_pos[i], k_pos[j], causal, window, q_lo, q_hi, i);
                ok[j] = (unsigned char)allowed;
                if (!allowed) continue;
                const double *kj = k + (j * Hkv + g) * (int64_t)d;
                double acc = 0.0;
                for (int c = 0; c < d; ++c) acc += qi[c] * kj[c];
                s[j] = scale * acc;
                if (s[j] > m) m = s[j];
                any = 1;
            }
            double *oi = out + (ri * Hq + h) * (int64_t)d;
            for (int c = 0; c < d; ++c) oi[c] = 0.0;
            if (!any) {
                lse[ri * Hq + h] = -INFINITY;
                continue;
            }
            double sum = 0.0;
            for (int64_t j = 0; j < Tk; ++j)
                if (ok[j]) sum += exp(s[j] - m);
            double l = m + log(sum);
            lse[ri * Hq + h] = l;
            for (int64_t j = 0; j < Tk; ++j) {
                if (!ok[j]) continue;
                double p = exp(s[j] - l);
                const double *vj = v + (j * Hkv + g) * (int64_t)d;
                for (int c = 0; c < d; ++c) oi[c] += p * vj[c];
            }
        }
        free(s);
        free(ok);
    }
    return 0;
}

/* ------------------------------------------------------------------------
 * Merge of n partial results of the same queries over disjoint key sets:
 *   M     = max_p lse_p
 *   lse   = M + log( sum_p exp(lse_p - M) )
 *   o     = sum_p exp(lse_p - lse) * o_p
 * all lse_p = -inf  ->  o = 0, lse = -inf.
 * outs[p] [rows, H, d], lses[p] [rows, H].
 * ------------------------------------------------------------------------ */
int orc_lse_merge(int n, const double *const *outs, const double *const *lses,
                  int64_t rows, int H, int d, double *out, double *lse)
{
    int64_t total = rows * (int64_t)H;
#pragma omp parallel for schedule(static)
    for (int64_t w = 0; w < total; ++w) {
        double M = -INFINITY;
        for (int p = 0; p < n; ++p)
            if (lses[p][w] > M) M = lses[p][w];
        double *o = out + w * (int64_t)d;
        for (int c = 0; c < d; ++c) o[c] = 0.0;
        if (M == -INFINITY) {
            lse[w] = -INFINITY;
            continue;
        }
        double sum = 0.0;
        for (int p = 0; p < n; ++p) sum += exp(lses[p][w] - M);
        double l = M + log(sum);
        lse[w] = l;
        for (int p = 0; p < n; ++p) {
            double wt = exp(lses[p][w] - l);
            const double *op = outs[p] + w * (int64_t)d;
            for (int c = 0; c < d; ++c) o[c] += wt * op[c];
        }
    }
    return 0;
}

/* ------------------------------------------------------------------------
 * Gradient of the attention above (one KV set, all rows), textbook form:
 *   P_ij  = exp(s_ij - lse_i)                (j in A(i))
 *   D_i   = sum_c dO[i,c] * O[i,c]
 *   dP_ij = sum_c dO[i,c] * v[j,c]
 *   dS_ij = P_ij * (dP_ij - D_i)
 *   dQ_i  = scale * sum_j dS_ij k_j
 *   dK_j  = scale * sum_{h in group(g)} sum_i dS_ij q_i
 *   dV_j  =         sum_{h in group(g)} sum_i P_ij dO_i
 * o, lse are the forward results for the same inputs.  The allowed set is
 * that of orc_partial_fwd (with the same optional q_lo / q_hi bounds).
 * dq_rows / dk_rows: which rows of dQ / dK,dV to evaluate (NULL = all);
 * dq [ndq, Hq, d], dk/dv [ndk, Hkv, d].
 * ------------------------------------------------------------------------ */
static double dot(const double *a, const double *b, int d)
{
    double acc = 0.0;
    for (int c = 0; c < d; ++c) acc += a[c] * b[c];
    return acc;
}

int orc_attn_bwd(const double *q, const double *k, const double *v,
                 const double *o, const double *lse, const double *dout,
                 int64_t T, int Hq, int Hkv, int d,
                 const int32_t *seg, const int64_t *pos, int causal, int64_t window, double scale,
                 const int64_t *q_lo, const int64_t *q_hi,
                 const int64_t *dq_rows, int64_t ndq,
                 const int64_t *dk_rows, int64_t ndk,
                 double *dq, double *dk, double *dv)
{
    if (Hkv <= 0 || Hq % Hkv != 0) return 1;
    const int G = Hq / Hkv;
    if (dq_rows == NULL) ndq = T;
    if (dk_rows == NULL) ndk = T;
    /* D_i for every (i, h) */
    double *D = (double *)malloc(sizeof(double) * (size_t)(T * Hq > 0 ? T * Hq : 1));
#pragma omp parallel for schedule(static)
    for (int64_t w = 0; w < T * (int64_t)Hq; ++w)
        D[w] = dot(dout + w * d, o + w * d, d);

    /* dQ: query-major */
#pragma omp parallel for schedule(dynamic, 4)
    for (int64_t w = 0; w < ndq * (int64_t)Hq; ++w) {
        int64_t ri = w / Hq;
        int h = (int)(w % Hq);
        int64_t i = dq_rows ? dq_rows[ri] : ri;
        int g = h / G;
        const double *qi = q + (i * Hq + h) * (int64_t)d;
        const double *doi = dout + (i * Hq + h) * (int64_t)d;
        double *dqi = dq + (ri * Hq + h) * (int64_t)d;
        for (int c = 0; c < d; ++c) dqi[c] = 0.0;
        double li = lse[i * Hq + h];
        for (int64_t j = 0; j < T; ++j) {
            if (!pair_allowed(seg[i], seg[j], pos[i], pos[j], causal, window, q_lo, q_hi, i)) continue;
            const double *kj = k + (j * Hkv + g) * (int64_t)d;
            const double *vj = v + (j * Hkv + g) * (int64_t)d;
            double p = exp(scale * dot(qi, kj, d) - li);
            double ds = p * (dot(doi, vj, d) - D[i * Hq + h]);
            for (int c = 0; c < d; ++c) dqi[c] += scale * ds * kj[c];
        }
    }

    /* dK, dV: key-major */
#pragma omp parallel for schedule(dynamic, 4)
    for (int64_t w = 0; w < ndk * (int64_t)Hkv; ++w) {
        int64_t rj = w / Hkv;
        int g = (int)(w % Hkv);
        int64_t j = dk_rows ? dk_rows[rj] : rj;
        const double *kj = k + (j * Hkv + g) * (int64_t)d;
        const double *vj = v + (j * Hkv + g) * (int64_t)d;
        double *dkj = dk + (rj * Hkv + g) * (int64_t)d;
        double *dvj = dv + (rj * Hkv + g) * (int64_t)d;
        for (int c = 0; c < d; ++c) { dkj[c] = 0.0; dvj[c] = 0.0; }
        for (int h = g * G; h < (g + 1) * G; ++h) {
            for (int64_t i = 0; i < T; ++i) {
                if (!pair_allowed(seg[i], seg[j], pos[i], pos[j], causal, window, q_lo, q_hi, i)) continue;
                const double *qi = q + (i * Hq + h) * (int64_t)d;
                const double *doi = dout + (i * Hq + h) * (int64_t)d;
                double p = exp(scale * dot(qi, kj, d) - lse[i * Hq + h]);
                double ds = p * (dot(doi, vj, d) - D[i * Hq + h]);
                for (int c = 0; c < d; ++c) {
                    dvj[c] += p * doi[c];
                    dkj[c] += scale * ds * qi[c];
                }
            }
        }
    }
    free(D);
    return 0;
}

/* ------------------------------------------------------------------------
 * Zigzag ownership.  A stream of L tokens is cut into n = 2*cp chunks with
 * boundaries bound(c) = floor(c*L/n); chunk c belongs to rank c when c < cp
 * and to rank n-1-c otherwise (rank r holds chunks r and 2cp-1-r).
 * mode 0 (global): the stream is the whole packed batch of T tokens.
 * mode 1 (per document): every document is its own stream.
 * owner[i] = rank of packed token i.
 * ------------------------------------------------------------------------ */
static int64_t chunk_bound(int64_t c, int64_t L, int64_t n) { return (c * L) / n; }

static int owner_in_stream(int64_t x, int64_t L, int cp)
{
    int64_t n = 2 * (int64_t)cp;
    for (int64_t c = 0; c < n; ++c) {
        if (chunk_bound(c, L, n) <= x && x < chunk_bound(c + 1, L, n))
            return (int)(c < cp ? c : n - 1 - c);
    }
    return -1;
}

int orc_zigzag_owner(const int32_t *cu, int B, int cp, int mode, int32_t *owner)
{
    if (cp < 1 || B < 0) return 1;
    int64_t T = cu[B];
    for (int b = 0; b < B; ++b) {
        for (int64_t i = cu[b]; i < cu[b + 1]; ++i) {
            int r = mode == 0 ? owner_in_stream(i, T, cp)
                              : owner_in_stream(i - cu[b], (int64_t)cu[b + 1] - cu[b], cp);
            if (r < 0) return 2;
            owner[i] = r;
        }
    }
    return 0;
}

/* perm [T]: rank 0's tokens in increasing packed index, then rank 1's, ...
 * off [cp+1]: start of each rank in perm.
 * cu_local [cp*(B+1)]: for rank r, cumulative count of its tokens per document. */
int orc_zigzag_plan(const int32_t *cu, int B, int cp, int mode,
                    int32_t *perm, int32_t *off, int32_t *cu_local)
{
    int64_t T = cu[B];
    int32_t *owner = (int32_t *)malloc(sizeof(int32_t) * (size_t)(T > 0 ? T : 1));
    int rc = orc_zigzag_owner(cu, B, cp, mode, owner);
    if (rc) { free(owner); return rc; }
    int64_t p = 0;
    for (int r = 0; r < cp; ++r) {
        off[r] = (int32_t)p;
        int32_t *cl = cu_local + (int64_t)r * (B + 1);
        cl[0] = 0;
        for (int b = 0; b < B; ++b) {
            int32_t cnt = 0;
            for (int64_t i = cu[b]; i < cu[b + 1]; ++i)
                if (owner[i] == r) { perm[p++] = (int32_t)i; ++cnt; }
            cl[b + 1] = cl[b] + cnt;
        }
    }
    off[cp] = (int32_t)p;
    free(owner);
    return 0;
}

/* Allowed (query, key) pairs per rank: a rank computes its own queries
 * against every key of the same document (the union of all ring steps). */
int orc_rank_pairs(const int32_t *cu, int B, int cp, int mode, int causal, int64_t window, int64_t *counts)
{
    int64_t T = cu[B];
    int32_t *owner = (int32_t *)malloc(sizeof(int32_t) * (size_t)(T > 0 ? T : 1));
    int rc = orc_zigzag_owner(cu, B, cp, mode, owner);
    if (rc) { free(owner); return rc; }
    for (int r = 0; r < cp; ++r) counts[r] = 0;
    for (int b = 0; b < B; ++b)
        for (int64_t i = cu[b]; i < cu[b + 1]; ++i) {
            /* keys of the document in [lo, hi] */
            int64_t lo = cu[b], hi = causal ? i : (int64_t)cu[b + 1] - 1;
            if (window >= 0 && i - window > lo) lo = i - window;
            if (hi >= lo) counts[owner[i]] += hi - lo + 1;
        }
    free(owner);
    return 0;
}
