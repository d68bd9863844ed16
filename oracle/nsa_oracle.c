/*
 * nsa_oracle.c -- plain fp64 CPU oracle for Native-Sparse-Attention block
 * selection (forward and analytic backward) under grouped-query attention.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may call this file:
 * only the tests, the smoke check and the benchmark's CPU-baseline leg load
 * it.  It shares no code with the CUDA library.
 *
 * What it computes (the gradcheck-gate page, "test_kernel_backward.py":
 * run_one builds q,k,v [B,H,T,D], idx = make_block_idx(B,Hkv,T,bs,S) and
 * compares dQ/dK/dV of selection attention against autograd through the
 * plain torch forward; the definitions below are that forward and its exact
 * derivative, written out per output element):
 *
 *   G = Hq / Hkv, query head h reads kv head g = h / G.
 *   sel(t)  = { idx[b,g,t,s] : 0 <= s < S, idx != -1 }
 *   key k is attended by row (b,h,t) iff k <= t and k / bs is in sel(t)
 *   (and, with a sliding window W >= 1, t - k < W)
 *   s_tk    = scale * <q_t, k_k>
 *   LSE_t   = log sum_k exp(s_tk)        (max-shifted; -inf for an empty row)
 *   P_tk    = exp(s_tk - LSE_t)
 *   O_t     = sum_k P_tk v_k             (0 for an empty row)
 *   D_t     = <dO_t, O_t>
 *   dP_tk   = <dO_t, v_k>
 *   dS_tk   = P_tk (dP_tk - D_t)
 *   dQ_t    = scale * sum_k dS_tk k_k
 *   dK_k    = scale * sum_{h in group, t} dS_tk q_t
 *   dV_k    = sum_{h in group, t} P_tk dO_t
 *
 * The window is the sliding-window option of the cuDNN-frontend page's
 * dense causal backward (SWA); W = 0 means no window.  The *_w entry points
 * take it; the others use W = 0.
 *
 * Attention sinks (the *_s entry points; the same page's backward chain ends
 * in a dSink kernel but does not define the sink, so this is the plainest
 * reading): one logit sigma_h per query head joins every row's softmax
 * denominator and carries no value,
 *   LSE_t   = log( sum_k exp(s_tk) + exp(sigma_h) )   (= sigma_h for an empty row)
 *   P_tk, O_t, dS_tk, dQ, dK, dV as above with this LSE
 *   dsigma_h = - sum_{b,t} exp(sigma_h - LSE_t) D_t
 * (the sink's probability exp(sigma_h - LSE_t) times dP = 0 minus D_t).
 *
 * Readings of points the pages leave open: scale is passed in (callers use
 * 1/sqrt(D)); keys after t inside the own block are masked (causal); -1
 * slots are ignored wherever they sit; an index is invalid if it is < -1,
 * lies in the future (> t / bs), or repeats within a row.
 *
 * Layouts.  Fixed length ("BHTD"): q,o,dO,dq [B,Hq,T,D]; k,v,dk,dv
 * [B,Hkv,T,D]; idx [B,Hkv,T,S]; lse [B,Hq,T].  Packed variable length
 * ("THD", cu_seqlens != NULL, B = number of sequences): q [total,Hq,D],
 * k [total,Hkv,D], idx [total,Hkv,S] holding sequence-local block ids,
 * lse [total,Hq]; causality and block numbering are local to a sequence.
 *
 * Build: cc -O2 -fopenmp -fPIC -shared nsa_oracle.c -o liboracle.so -lm
 */
#include <math.h>
#include <omp.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

typedef struct {
    int64_t B, Hq, Hkv, T, D, bs, S;
    double scale;
    const int32_t *cu;    /* NULL: fixed length */
    int64_t window;       /* 0: none; else keys k with t - k < window only */
    const double *sinks;  /* NULL: none; else one logit per query head */
} prob_t;

static prob_t mk(int64_t B, int64_t Hq, int64_t Hkv, int64_t T, int64_t D,
                 int64_t bs, int64_t S, double scale, const int32_t *cu)
{
    prob_t p = {B, Hq, Hkv, T, D, bs, S, scale, cu, 0, NULL};
    return p;
}

/* 1 if the window lets row t see key kk (kk <= t is checked elsewhere) */
static int in_window(const prob_t *p, int64_t t, int64_t kk) { return p->window <= 0 || t - kk < p->window; }

static int64_t seq_len(const prob_t *p, int64_t b)
{
    return p->cu ? (int64_t)p->cu[b + 1] - p->cu[b] : p->T;
}

/* element offset of the D-vector of (b, head, t) in a tensor with H heads */
static int64_t row_off(const prob_t *p, int64_t H, int64_t b, int64_t h, int64_t t)
{
    if (p->cu)
        return (((int64_t)p->cu[b] + t) * H + h) * p->D;
    return ((b * H + h) * p->T + t) * p->D;
}

/* offset of a per-row scalar (lse, row sums) */
static int64_t stat_off(const prob_t *p, int64_t H, int64_t b, int64_t h, int64_t t)
{
    if (p->cu)
        return ((int64_t)p->cu[b] + t) * H + h;
    return (b * H + h) * p->T + t;
}

static const int32_t *idx_row(const prob_t *p, const int32_t *idx, int64_t b, int64_t g, int64_t t)
{
    if (p->cu)
        return idx + (((int64_t)p->cu[b] + t) * p->Hkv + g) * p->S;
    return idx + ((b * p->Hkv + g) * p->T + t) * p->S;
}

static double dot(const double *a, const double *b, int64_t n)
{
    double s = 0.0;
    for (int64_t i = 0; i < n; ++i)
        s += a[i] * b[i];
    return s;
}

/* 1 if block j is one of the row's selected blocks */
static int selects(const prob_t *p, const int32_t *row, int64_t j)
{
    for (int64_t s = 0; s < p->S; ++s)
        if (row[s] == j)
            return 1;
    return 0;
}

/*
 * Index validation.  Returns 0 when every entry is -1 or a distinct block id
 * in [0, t / bs]; 3 otherwise (the library's "bad index" status).
 */
int oracle_validate_index(int64_t B, int64_t Hkv, int64_t T, int64_t bs, int64_t S,
                          const int32_t *cu, const int32_t *idx)
{
    prob_t p = mk(B, Hkv, Hkv, T, 1, bs, S, 1.0, cu);
    for (int64_t b = 0; b < B; ++b)
        for (int64_t g = 0; g < Hkv; ++g)
            for (int64_t t = 0; t < seq_len(&p, b); ++t) {
                const int32_t *row = idx_row(&p, idx, b, g, t);
                for (int64_t s = 0; s < S; ++s) {
                    int64_t j = row[s];
                    if (j == -1)
                        continue;
                    if (j < -1 || j > t / bs)
                        return 3;
                    for (int64_t s2 = 0; s2 < s; ++s2)
                        if (row[s2] == j)
                            return 3;
                }
            }
    return 0;
}

/*
 * Scores of one row over its attended keys.  Fills keys[] (sequence-local key
 * positions) and sc[] (scale * q.k); returns the number of attended keys.
 * Keys come block by block in slot order; the set is what matters.
 */
static int64_t row_scores(const prob_t *p, const double *q, const double *k, const int32_t *idx,
                          int64_t b, int64_t h, int64_t t, int64_t *keys, double *sc)
{
    const int64_t G = p->Hq / p->Hkv, g = h / G;
    const int32_t *row = idx_row(p, idx, b, g, t);
    const double *qt = q + row_off(p, p->Hq, b, h, t);
    int64_t n = 0;
    for (int64_t s = 0; s < p->S; ++s) {
        int64_t j = row[s];
        if (j < 0)
            continue;
        for (int64_t kk = j * p->bs; kk < (j + 1) * p->bs && kk <= t; ++kk) {
            if (!in_window(p, t, kk))
                continue;
            keys[n] = kk;
            sc[n] = p->scale * dot(qt, k + row_off(p, p->Hkv, b, g, kk), p->D);
            ++n;
        }
    }
    return n;
}

/* log-sum-exp of sc[0..n) and, with sinks, head h's sink logit, with the
 * max shift; -inf when there is nothing to sum */
static double lse_of(const prob_t *p, int64_t h, const double *sc, int64_t n)
{
    const int has = p->sinks != NULL;
    if (n == 0 && !has)
        return -INFINITY;
    double m = has ? p->sinks[h] : sc[0];
    for (int64_t i = 0; i < n; ++i)
        if (sc[i] > m)
            m = sc[i];
    double l = has ? exp(p->sinks[h] - m) : 0.0;
    for (int64_t i = 0; i < n; ++i)
        l += exp(sc[i] - m);
    return m + log(l);
}

/* forward of one row: writes o (D values) and returns LSE */
static double row_forward(const prob_t *p, const double *q, const double *k, const double *v,
                          const int32_t *idx, int64_t b, int64_t h, int64_t t, double *o,
                          int64_t *keys, double *sc)
{
    const int64_t G = p->Hq / p->Hkv, g = h / G;
    int64_t n = row_scores(p, q, k, idx, b, h, t, keys, sc);
    double lse = lse_of(p, h, sc, n);
    for (int64_t d = 0; d < p->D; ++d)
        o[d] = 0.0;
    for (int64_t i = 0; i < n; ++i) {
        double pk = exp(sc[i] - lse);
        const double *vk = v + row_off(p, p->Hkv, b, g, keys[i]);
        for (int64_t d = 0; d < p->D; ++d)
            o[d] += pk * vk[d];
    }
    return lse;
}

static int64_t max_keys(const prob_t *p) { return p->S * p->bs + 1; }

static int64_t n_rows_total(const prob_t *p)
{
    int64_t n = 0;
    for (int64_t b = 0; b < p->B; ++b)
        n += seq_len(p, b);
    return n;
}

/* Forward: o (layout of q) and lse; sinks NULL or one logit per query head. */
void oracle_sel_fwd_s(int64_t B, int64_t Hq, int64_t Hkv, int64_t T, int64_t D, int64_t bs,
                      int64_t S, double scale, const int32_t *cu, const double *q,
                      const double *k, const double *v, const int32_t *idx, double *o,
                      double *lse, int64_t window, const double *sinks)
{
    prob_t p = mk(B, Hq, Hkv, T, D, bs, S, scale, cu);
    p.window = window;
    p.sinks = sinks;
#pragma omp parallel
    {
        int64_t *keys = (int64_t *)malloc(sizeof(int64_t) * max_keys(&p));
        double *sc = (double *)malloc(sizeof(double) * max_keys(&p));
#pragma omp for collapse(2) schedule(dynamic)
        for (int64_t b = 0; b < B; ++b)
            for (int64_t h = 0; h < Hq; ++h)
                for (int64_t t = 0; t < seq_len(&p, b); ++t)
                    lse[stat_off(&p, Hq, b, h, t)] =
                        row_forward(&p, q, k, v, idx, b, h, t, o + row_off(&p, Hq, b, h, t),
                                    keys, sc);
        free(keys);
        free(sc);
    }
}

void oracle_sel_fwd_w(int64_t B, int64_t Hq, int64_t Hkv, int64_t T, int64_t D, int64_t bs,
                      int64_t S, double scale, const int32_t *cu, const double *q,
                      const double *k, const double *v, const int32_t *idx, double *o,
                      double *lse, int64_t window)
{
    oracle_sel_fwd_s(B, Hq, Hkv, T, D, bs, S, scale, cu, q, k, v, idx, o, lse, window, NULL);
}

/*
 * Backward.  Recomputes the forward in fp64 (O, LSE), then
 *   pass 1, one query row at a time: D_t, dQ_t and (optionally) sum_k dS_tk;
 *   pass 2, one key at a time: dK_k and dV_k as sums over every row (h, t) of
 *           the group that attends k.
 * o_out / lse_out / dsum_out may be NULL.
 */
void oracle_sel_bwd_s(int64_t B, int64_t Hq, int64_t Hkv, int64_t T, int64_t D, int64_t bs,
                      int64_t S, double scale, const int32_t *cu, const double *q,
                      const double *k, const double *v, const int32_t *idx, const double *dO,
                      double *dq, double *dk, double *dv, double *o_out, double *lse_out,
                      double *dsum_out, int64_t window, const double *sinks, double *dsinks_out)
{
    prob_t p = mk(B, Hq, Hkv, T, D, bs, S, scale, cu);
    p.window = window;
    p.sinks = sinks;
    const int64_t G = Hq / Hkv;
    const int64_t nrow = n_rows_total(&p) * Hq;
    double *O = o_out ? o_out : (double *)malloc(sizeof(double) * nrow * D);
    double *L = lse_out ? lse_out : (double *)malloc(sizeof(double) * nrow);
    double *Dt = (double *)malloc(sizeof(double) * nrow);

    /* pass 1: per query row */
#pragma omp parallel
    {
        int64_t *keys = (int64_t *)malloc(sizeof(int64_t) * max_keys(&p));
        double *sc = (double *)malloc(sizeof(double) * max_keys(&p));
#pragma omp for collapse(2) schedule(dynamic)
        for (int64_t b = 0; b < B; ++b)
            for (int64_t h = 0; h < Hq; ++h)
                for (int64_t t = 0; t < seq_len(&p, b); ++t) {
                    const int64_t ro = row_off(&p, Hq, b, h, t), so = stat_off(&p, Hq, b, h, t);
                    const int64_t g = h / G;
                    double lse = row_forward(&p, q, k, v, idx, b, h, t, O + ro, keys, sc);
                    L[so] = lse;
                    const double *dOt = dO + ro;
                    double Dv = dot(dOt, O + ro, D);
                    Dt[so] = Dv;
                    int64_t n = row_scores(&p, q, k, idx, b, h, t, keys, sc);
                    double *dqt = dq + ro;
                    for (int64_t d = 0; d < D; ++d)
                        dqt[d] = 0.0;
                    double dsum = 0.0;
                    for (int64_t i = 0; i < n; ++i) {
                        const double *kk = k + row_off(&p, Hkv, b, g, keys[i]);
                        const double *vk = v + row_off(&p, Hkv, b, g, keys[i]);
                        double P = exp(sc[i] - lse);
                        double dP = dot(dOt, vk, D);
                        double dS = P * (dP - Dv);
                        dsum += dS;
                        for (int64_t d = 0; d < D; ++d)
                            dqt[d] += scale * dS * kk[d];
                    }
                    if (dsum_out)
                        dsum_out[so] = dsum;
                }
        free(keys);
        free(sc);
    }

    /* the sinks' gradient: each row's term, then a sum per head in (b, t) order */
    if (sinks && dsinks_out)
        for (int64_t h = 0; h < Hq; ++h) {
            double acc = 0.0;
            for (int64_t b = 0; b < B; ++b)
                for (int64_t t = 0; t < seq_len(&p, b); ++t) {
                    const int64_t so = stat_off(&p, Hq, b, h, t);
                    acc -= exp(sinks[h] - L[so]) * Dt[so];
                }
            dsinks_out[h] = acc;
        }

    /* pass 2: per key, sum over every row of the group that attends it */
#pragma omp parallel for collapse(2) schedule(dynamic)
    for (int64_t b = 0; b < B; ++b)
        for (int64_t g = 0; g < Hkv; ++g)
            for (int64_t kk = 0; kk < seq_len(&p, b); ++kk) {
                const int64_t ko = row_off(&p, Hkv, b, g, kk);
                const double *kv = k + ko, *vv = v + ko;
                double *dkk = dk + ko, *dvk = dv + ko;
                for (int64_t d = 0; d < D; ++d) {
                    dkk[d] = 0.0;
                    dvk[d] = 0.0;
                }
                const int64_t j = kk / bs;
                for (int64_t t = kk; t < seq_len(&p, b) && in_window(&p, t, kk); ++t) {
                    if (!selects(&p, idx_row(&p, idx, b, g, t), j))
                        continue;
                    for (int64_t h = g * G; h < (g + 1) * G; ++h) {
                        const int64_t ro = row_off(&p, Hq, b, h, t), so = stat_off(&p, Hq, b, h, t);
                        const double *qt = q + ro, *dOt = dO + ro;
                        double s = scale * dot(qt, kv, D);
                        double P = exp(s - L[so]);
                        double dP = dot(dOt, vv, D);
                        double dS = P * (dP - Dt[so]);
                        for (int64_t d = 0; d < D; ++d) {
                            dkk[d] += scale * dS * qt[d];
                            dvk[d] += P * dOt[d];
                        }
                    }
                }
            }

    if (!o_out)
        free(O);
    if (!lse_out)
        free(L);
    free(Dt);
}

void oracle_sel_bwd_w(int64_t B, int64_t Hq, int64_t Hkv, int64_t T, int64_t D, int64_t bs,
                      int64_t S, double scale, const int32_t *cu, const double *q,
                      const double *k, const double *v, const int32_t *idx, const double *dO,
                      double *dq, double *dk, double *dv, double *o_out, double *lse_out,
                      double *dsum_out, int64_t window)
{
    oracle_sel_bwd_s(B, Hq, Hkv, T, D, bs, S, scale, cu, q, k, v, idx, dO, dq, dk, dv, o_out, lse_out,
                     dsum_out, window, NULL, NULL);
}

/*
 * Inverse index (block -> selecting tokens), by brute force.
 * offsets has B*Hkv*nbmax + 1 entries, nbmax = ceil(max sequence length / bs);
 * entry (b,g,j) lists, in ascending order, every sequence-local token t whose
 * row selects block j.  Blocks past a sequence's end have empty lists.
 * rows must hold offsets[B*Hkv*nbmax] entries (at most total_tokens*Hkv*S).
 */
void oracle_inverse_index(int64_t B, int64_t Hkv, int64_t T, int64_t bs, int64_t S,
                          const int32_t *cu, const int32_t *idx, int64_t nbmax,
                          int32_t *offsets, int32_t *rows)
{
    prob_t p = mk(B, Hkv, Hkv, T, 1, bs, S, 1.0, cu);
    int64_t n = 0;
    for (int64_t b = 0; b < B; ++b)
        for (int64_t g = 0; g < Hkv; ++g)
            for (int64_t j = 0; j < nbmax; ++j) {
                offsets[(b * Hkv + g) * nbmax + j] = (int32_t)n;
                for (int64_t t = 0; t < seq_len(&p, b); ++t)
                    if (selects(&p, idx_row(&p, idx, b, g, t), j))
                        rows[n++] = (int32_t)t;
            }
    offsets[B * Hkv * nbmax] = (int32_t)n;
}

/* D_t = <dO_t, O_t> for every row (layout of lse) */
void oracle_do_dot(int64_t B, int64_t Hq, int64_t T, int64_t D, const int32_t *cu,
                   const double *o, const double *dO, double *out)
{
    prob_t p = mk(B, Hq, Hq, T, D, 1, 1, 1.0, cu);
    for (int64_t b = 0; b < B; ++b)
        for (int64_t h = 0; h < Hq; ++h)
            for (int64_t t = 0; t < seq_len(&p, b); ++t) {
                int64_t ro = row_off(&p, Hq, b, h, t);
                out[stat_off(&p, Hq, b, h, t)] = dot(dO + ro, o + ro, D);
            }
}

/* Number of (query row, attended key) pairs summed over query heads. */
int64_t oracle_count_pairs_w(int64_t B, int64_t Hq, int64_t Hkv, int64_t T, int64_t bs, int64_t S,
                             const int32_t *cu, const int32_t *idx, int64_t window)
{
    prob_t p = mk(B, Hq, Hkv, T, 1, bs, S, 1.0, cu);
    p.window = window;
    const int64_t G = Hq / Hkv;
    int64_t n = 0;
    for (int64_t b = 0; b < B; ++b)
        for (int64_t g = 0; g < Hkv; ++g)
            for (int64_t t = 0; t < seq_len(&p, b); ++t) {
                const int32_t *row = idx_row(&p, idx, b, g, t);
                for (int64_t s = 0; s < S; ++s) {
                    int64_t j = row[s];
                    if (j < 0)
                        continue;
                    int64_t hi = (j + 1) * bs - 1, lo = j * bs;
                    if (hi > t)
                        hi = t;
                    if (window > 0 && lo < t - window + 1)
                        lo = t - window + 1;
                    if (hi >= lo)
                        n += G * (hi - lo + 1);
                }
            }
    return n;
}

/*
 * Sampled outputs, for problems too large to run whole: the same definitions
 * evaluated only at the requested rows / keys.
 *
 * oracle_sel_rows: for each (b, h, t) in the list, O_t, LSE_t and dQ_t.
 */
void oracle_sel_rows_w(int64_t B, int64_t Hq, int64_t Hkv, int64_t T, int64_t D, int64_t bs,
                       int64_t S, double scale, const int32_t *cu, const double *q,
                       const double *k, const double *v, const int32_t *idx, const double *dO,
                       int64_t n, const int64_t *rb, const int64_t *rh, const int64_t *rt,
                       double *o_out, double *lse_out, double *dq_out, int64_t window)
{
    prob_t p = mk(B, Hq, Hkv, T, D, bs, S, scale, cu);
    p.window = window;
    const int64_t G = Hq / Hkv;
#pragma omp parallel
    {
        int64_t *keys = (int64_t *)malloc(sizeof(int64_t) * max_keys(&p));
        double *sc = (double *)malloc(sizeof(double) * max_keys(&p));
#pragma omp for schedule(dynamic)
        for (int64_t i = 0; i < n; ++i) {
            const int64_t b = rb[i], h = rh[i], t = rt[i], g = h / G;
            double *o = o_out + i * D, *dqt = dq_out + i * D;
            const double *dOt = dO + row_off(&p, Hq, b, h, t);
            double lse = row_forward(&p, q, k, v, idx, b, h, t, o, keys, sc);
            lse_out[i] = lse;
            double Dv = dot(dOt, o, D);
            int64_t m = row_scores(&p, q, k, idx, b, h, t, keys, sc);
            for (int64_t d = 0; d < D; ++d)
                dqt[d] = 0.0;
            for (int64_t c = 0; c < m; ++c) {
                const int64_t ko = row_off(&p, Hkv, b, g, keys[c]);
                double P = exp(sc[c] - lse);
                double dS = P * (dot(dOt, v + ko, D) - Dv);
                for (int64_t d = 0; d < D; ++d)
                    dqt[d] += scale * dS * k[ko + d];
            }
        }
        free(keys);
        free(sc);
    }
}

/*
 * oracle_sel_keys: for each (b, g, key) in the list, dK and dV of that key;
 * LSE_t and D_t of every attending row are recomputed from scratch.
 */
void oracle_sel_keys_w(int64_t B, int64_t Hq, int64_t Hkv, int64_t T, int64_t D, int64_t bs,
                       int64_t S, double scale, const int32_t *cu, const double *q,
                       const double *k, const double *v, const int32_t *idx, const double *dO,
                       int64_t n, const int64_t *kb, const int64_t *kg, const int64_t *kk_,
                       double *dk_out, double *dv_out, int64_t window)
{
    prob_t p = mk(B, Hq, Hkv, T, D, bs, S, scale, cu);
    p.window = window;
    const int64_t G = Hq / Hkv;
#pragma omp parallel
    {
        int64_t *keys = (int64_t *)malloc(sizeof(int64_t) * max_keys(&p));
        double *sc = (double *)malloc(sizeof(double) * max_keys(&p));
        double *o = (double *)malloc(sizeof(double) * D);
#pragma omp for schedule(dynamic)
        for (int64_t i = 0; i < n; ++i) {
            const int64_t b = kb[i], g = kg[i], kk = kk_[i], j = kk / bs;
            const int64_t ko = row_off(&p, Hkv, b, g, kk);
            double *dkk = dk_out + i * D, *dvk = dv_out + i * D;
            for (int64_t d = 0; d < D; ++d) {
                dkk[d] = 0.0;
                dvk[d] = 0.0;
            }
            for (int64_t t = kk; t < seq_len(&p, b) && in_window(&p, t, kk); ++t) {
                if (!selects(&p, idx_row(&p, idx, b, g, t), j))
                    continue;
                for (int64_t h = g * G; h < (g + 1) * G; ++h) {
                    const int64_t ro = row_off(&p, Hq, b, h, t);
                    const double *qt = q + ro, *dOt = dO + ro;
                    double lse = row_forward(&p, q, k, v, idx, b, h, t, o, keys, sc);
                    double Dv = dot(dOt, o, D);
                    double P = exp(scale * dot(qt, k + ko, D) - lse);
                    double dS = P * (dot(dOt, v + ko, D) - Dv);
                    for (int64_t d = 0; d < D; ++d) {
                        dkk[d] += scale * dS * qt[d];
                        dvk[d] += P * dOt[d];
                    }
                }
            }
        }
        free(keys);
        free(sc);
        free(o);
    }
}

/*
 * oracle_sel_blocks: for each (b, g, j) in the list, dK and dV of every key
 * of block j (bs keys x D each, keys past the sequence's end left 0), by the
 * same definitions as oracle_sel_keys.  Each attending row -- a token t of
 * the block's sequence whose row selects j, with every query head of group
 * g -- has its forward (LSE_t, O_t) recomputed once for the whole block
 * instead of once per key, which is what makes whole heavily selected
 * blocks of the long workloads affordable.
 */
void oracle_sel_blocks_w(int64_t B, int64_t Hq, int64_t Hkv, int64_t T, int64_t D, int64_t bs,
                         int64_t S, double scale, const int32_t *cu, const double *q,
                         const double *k, const double *v, const int32_t *idx, const double *dO,
                         int64_t n, const int64_t *jb, const int64_t *jg, const int64_t *jj,
                         double *dk_out, double *dv_out, int64_t window)
{
    prob_t p = mk(B, Hq, Hkv, T, D, bs, S, scale, cu);
    p.window = window;
    const int64_t G = Hq / Hkv;
    for (int64_t i = 0; i < n; ++i) {
        const int64_t b = jb[i], g = jg[i], j = jj[i], L = seq_len(&p, b);
        const int64_t k0 = j * bs, nk = (k0 + bs <= L ? bs : L - k0);
        double *dkb = dk_out + i * bs * D, *dvb = dv_out + i * bs * D;
        memset(dkb, 0, sizeof(double) * bs * D);
        memset(dvb, 0, sizeof(double) * bs * D);
        if (nk <= 0)
            continue;
        /* the attending rows' contributions, summed per thread, then added in
           thread order */
#pragma omp parallel
        {
            int64_t *keys = (int64_t *)malloc(sizeof(int64_t) * max_keys(&p));
            double *sc = (double *)malloc(sizeof(double) * max_keys(&p));
            double *o = (double *)malloc(sizeof(double) * D);
            double *acc_k = (double *)calloc((size_t)(bs * D), sizeof(double));
            double *acc_v = (double *)calloc((size_t)(bs * D), sizeof(double));
#pragma omp for schedule(dynamic, 4)
            for (int64_t t = k0; t < L; ++t) {
                if (!selects(&p, idx_row(&p, idx, b, g, t), j))
                    continue;
                for (int64_t h = g * G; h < (g + 1) * G; ++h) {
                    const int64_t ro = row_off(&p, Hq, b, h, t);
                    const double *qt = q + ro, *dOt = dO + ro;
                    double lse = row_forward(&p, q, k, v, idx, b, h, t, o, keys, sc);
                    double Dv = dot(dOt, o, D);
                    for (int64_t c = 0; c < nk; ++c) {
                        const int64_t kk = k0 + c;
                        if (kk > t || !in_window(&p, t, kk))
                            continue;
                        const int64_t ko = row_off(&p, Hkv, b, g, kk);
                        double P = exp(scale * dot(qt, k + ko, D) - lse);
                        double dS = P * (dot(dOt, v + ko, D) - Dv);
                        for (int64_t d = 0; d < D; ++d) {
                            acc_k[c * D + d] += scale * dS * qt[d];
                            acc_v[c * D + d] += P * dOt[d];
                        }
                    }
                }
            }
#pragma omp for ordered schedule(static, 1)
            for (int th = 0; th < omp_get_num_threads(); ++th) {
#pragma omp ordered
                for (int64_t x = 0; x < bs * D; ++x) {
                    dkb[x] += acc_k[x];
                    dvb[x] += acc_v[x];
                }
            }
            free(keys);
            free(sc);
            free(o);
            free(acc_k);
            free(acc_v);
        }
    }
}

/*
 * Dense causal attention with separate query and key lengths (the
 * cuDNN-frontend page: the SDPA backward's THD path takes cum_seqlen_q and
 * cum_seqlen_k, and its causal mask comes in two alignments,
 * causal_bottom_right beside plain causal, each optionally with a sliding
 * window).  For sequence b with Lq query rows and Lk keys, row t sits at
 * key position
 *     c_t = t                 (top-left alignment)
 *     c_t = t + Lk - Lq       (bottom-right alignment)
 * and attends key k iff 0 <= k <= c_t, k < Lk and (window W > 0) c_t - k < W.
 * A row with no such key gets O = 0, LSE = -inf and no gradient.  Everything
 * else is the plain softmax attention of the header, per query head h with
 * kv head h / G.
 *
 * Layouts: fixed length (cu_q = cu_k = NULL): q, o, dO, dq [B,Hq,Tq,D],
 * k, v, dk, dv [B,Hkv,Tk,D], lse [B,Hq,Tq]; packed: q [cu_q[B],Hq,D],
 * k [cu_k[B],Hkv,D], lse [cu_q[B],Hq].
 */
typedef struct {
    int64_t B, Hq, Hkv, Tq, Tk, D, window, bottom_right;
    double scale;
    const int32_t *cu_q, *cu_k;
} cprob_t;

static int64_t c_lq(const cprob_t *p, int64_t b) { return p->cu_q ? (int64_t)p->cu_q[b + 1] - p->cu_q[b] : p->Tq; }
static int64_t c_lk(const cprob_t *p, int64_t b) { return p->cu_k ? (int64_t)p->cu_k[b + 1] - p->cu_k[b] : p->Tk; }

static int64_t c_qoff(const cprob_t *p, int64_t H, int64_t b, int64_t h, int64_t t)
{
    if (p->cu_q)
        return (((int64_t)p->cu_q[b] + t) * H + h) * p->D;
    return ((b * H + h) * p->Tq + t) * p->D;
}

static int64_t c_koff(const cprob_t *p, int64_t b, int64_t g, int64_t kk)
{
    if (p->cu_k)
        return (((int64_t)p->cu_k[b] + kk) * p->Hkv + g) * p->D;
    return ((b * p->Hkv + g) * p->Tk + kk) * p->D;
}

static int64_t c_soff(const cprob_t *p, int64_t b, int64_t h, int64_t t)
{
    if (p->cu_q)
        return ((int64_t)p->cu_q[b] + t) * p->Hq + h;
    return (b * p->Hq + h) * p->Tq + t;
}

/* 1 if row t of sequence b attends key kk */
static int c_attends(const cprob_t *p, int64_t b, int64_t t, int64_t kk)
{
    const int64_t Lk = c_lk(p, b);
    const int64_t c = p->bottom_right ? t + Lk - c_lq(p, b) : t;
    return kk >= 0 && kk < Lk && kk <= c && (p->window <= 0 || c - kk < p->window);
}

/* forward of one row: o (D values) and the returned LSE */
static double c_row_forward(const cprob_t *p, const double *q, const double *k, const double *v, int64_t b,
                            int64_t h, int64_t t, double *o, double *sc)
{
    const int64_t g = h / (p->Hq / p->Hkv), Lk = c_lk(p, b);
    const double *qt = q + c_qoff(p, p->Hq, b, h, t);
    double m = -INFINITY;
    for (int64_t kk = 0; kk < Lk; ++kk) {
        sc[kk] = c_attends(p, b, t, kk) ? p->scale * dot(qt, k + c_koff(p, b, g, kk), p->D) : -INFINITY;
        if (sc[kk] > m)
            m = sc[kk];
    }
    for (int64_t d = 0; d < p->D; ++d)
        o[d] = 0.0;
    if (m == -INFINITY)
        return -INFINITY;
    double l = 0.0;
    for (int64_t kk = 0; kk < Lk; ++kk)
        if (sc[kk] != -INFINITY)
            l += exp(sc[kk] - m);
    const double lse = m + log(l);
    for (int64_t kk = 0; kk < Lk; ++kk)
        if (sc[kk] != -INFINITY) {
            const double pk = exp(sc[kk] - lse);
            const double *vk = v + c_koff(p, b, g, kk);
            for (int64_t d = 0; d < p->D; ++d)
                o[d] += pk * vk[d];
        }
    return lse;
}

static int64_t c_maxlen(const int32_t *cu, int64_t B, int64_t T)
{
    if (!cu)
        return T;
    int64_t m = 0;
    for (int64_t b = 0; b < B; ++b)
        if (cu[b + 1] - cu[b] > m)
            m = cu[b + 1] - cu[b];
    return m;
}

/*
 * Forward and backward together: o, lse, dq, dk, dv (dO may be NULL for the
 * forward only; then dq, dk, dv are not touched).  Pass 1 per query row
 * (LSE, O, D_t, dQ), pass 2 per key (dK, dV over every attending row of the
 * key's group).
 */
void oracle_causal(int64_t B, int64_t Hq, int64_t Hkv, int64_t Tq, int64_t Tk, int64_t D, double scale,
                   const int32_t *cu_q, const int32_t *cu_k, int64_t window, int64_t bottom_right, const double *q,
                   const double *k, const double *v, const double *dO, double *o, double *lse, double *dq, double *dk,
                   double *dv)
{
    cprob_t p = {B, Hq, Hkv, Tq, Tk, D, window, bottom_right, scale, cu_q, cu_k};
    const int64_t G = Hq / Hkv, mk_ = c_maxlen(cu_k, B, Tk) + 1;
    int64_t nq = 0;
    for (int64_t b = 0; b < B; ++b)
        nq += c_lq(&p, b);
    double *Dt = (double *)calloc((size_t)(nq * Hq + 1), sizeof(double));
#pragma omp parallel
    {
        double *sc = (double *)malloc(sizeof(double) * mk_);
#pragma omp for collapse(2) schedule(dynamic)
        for (int64_t b = 0; b < B; ++b)
            for (int64_t h = 0; h < Hq; ++h)
                for (int64_t t = 0; t < c_lq(&p, b); ++t) {
                    const int64_t ro = c_qoff(&p, Hq, b, h, t), so = c_soff(&p, b, h, t), g = h / G;
                    const double L = c_row_forward(&p, q, k, v, b, h, t, o + ro, sc);
                    lse[so] = L;
                    if (!dO)
                        continue;
                    const double *dOt = dO + ro;
                    const double Dv = dot(dOt, o + ro, D);
                    Dt[so] = Dv;
                    double *dqt = dq + ro;
                    for (int64_t d = 0; d < D; ++d)
                        dqt[d] = 0.0;
                    for (int64_t kk = 0; kk < c_lk(&p, b); ++kk) {
                        if (sc[kk] == -INFINITY)
                            continue;
                        const int64_t ko = c_koff(&p, b, g, kk);
                        const double P = exp(sc[kk] - L);
                        const double dS = P * (dot(dOt, v + ko, D) - Dv);
                        for (int64_t d = 0; d < D; ++d)
                            dqt[d] += scale * dS * k[ko + d];
                    }
                }
        free(sc);
    }
    if (dO) {
#pragma omp parallel for collapse(2) schedule(dynamic)
        for (int64_t b = 0; b < B; ++b)
            for (int64_t g = 0; g < Hkv; ++g)
                for (int64_t kk = 0; kk < c_lk(&p, b); ++kk) {
                    const int64_t ko = c_koff(&p, b, g, kk);
                    double *dkk = dk + ko, *dvk = dv + ko;
                    for (int64_t d = 0; d < D; ++d) {
                        dkk[d] = 0.0;
                        dvk[d] = 0.0;
                    }
                    for (int64_t t = 0; t < c_lq(&p, b); ++t) {
                        if (!c_attends(&p, b, t, kk))
                            continue;
                        for (int64_t h = g * G; h < (g + 1) * G; ++h) {
                            const int64_t ro = c_qoff(&p, Hq, b, h, t), so = c_soff(&p, b, h, t);
                            const double *qt = q + ro, *dOt = dO + ro;
                            const double P = exp(scale * dot(qt, k + ko, D) - lse[so]);
                            const double dS = P * (dot(dOt, v + ko, D) - Dt[so]);
                            for (int64_t d = 0; d < D; ++d) {
                                dkk[d] += scale * dS * qt[d];
                                dvk[d] += P * dOt[d];
                            }
                        }
                    }
                }
    }
    free(Dt);
}

/* ------------------------------------------------------------ block selection
 *
 * The step that produces idx.  The pages take the index as given (the
 * gradcheck-gate page names "NSA selection" and builds idx with a helper it
 * does not print), so this is the plainest reading of NSA's selection step,
 * kept consistent with the index the pages' tests use (slot 0 is the row's
 * own block):
 *
 *   block j of a sequence is complete at row t  iff  (j + 1) * bs - 1 <= t
 *   kc_{g,j}      the compressed key of block j of kv head g -- an input,
 *                 since NSA learns its compression; the stand-in provided
 *                 is the mean of the block's bs keys (complete blocks only)
 *   p_{h,t,j}     = exp(scale <q_{h,t}, kc_{g,j}>) / sum_{j' complete at t} exp(scale <q_{h,t}, kc_{g,j'}>)
 *                   for j complete at t (h in group g)
 *   score_{g,t,j} = sum_{h in group g} p_{h,t,j}    (0 where j is not complete at t)
 *   idx_{g,t}     = [ t / bs,  then the S - 1 blocks j != t / bs complete at t
 *                     with the largest scores, in decreasing order of score
 *                     (equal scores: the smaller j first; a NaN score counts
 *                     as -infinity),  then -1 for the slots left ]
 *
 * Layouts: kc [B, Hkv, nb, D], nb = ceil(T / bs) (THD: of the longest
 * sequence), zero rows for blocks that are not complete; scores
 * [B, Hkv, T, nb] (THD: [total, Hkv, nb]).
 */

static int64_t n_complete(int64_t t, int64_t bs) { return (t + 1) / bs; }

static int64_t score_off(const prob_t *p, int64_t nb, int64_t b, int64_t g, int64_t t)
{
    if (p->cu)
        return (((int64_t)p->cu[b] + t) * p->Hkv + g) * nb;
    return ((b * p->Hkv + g) * p->T + t) * nb;
}

/* kc_{g,j} = (1 / bs) * sum of keys j*bs .. j*bs + bs - 1, for complete blocks */
void oracle_compress_mean(int64_t B, int64_t Hkv, int64_t T, int64_t D, int64_t bs, int64_t nb,
                          const int32_t *cu, const double *k, double *kc)
{
    prob_t p = mk(B, Hkv, Hkv, T, D, bs, 1, 1.0, cu);
    for (int64_t b = 0; b < B; ++b)
        for (int64_t g = 0; g < Hkv; ++g)
            for (int64_t j = 0; j < nb; ++j) {
                double *out = kc + ((b * Hkv + g) * nb + j) * D;
                for (int64_t d = 0; d < D; ++d)
                    out[d] = 0.0;
                if ((j + 1) * bs > seq_len(&p, b))
                    continue;  /* not complete in this sequence */
                for (int64_t kk = j * bs; kk < (j + 1) * bs; ++kk) {
                    const double *kr = k + row_off(&p, Hkv, b, g, kk);
                    for (int64_t d = 0; d < D; ++d)
                        out[d] += kr[d];
                }
                for (int64_t d = 0; d < D; ++d)
                    out[d] /= (double)bs;
            }
}

/* score_{g,t,j}: the compressed-attention probabilities of the group's heads, summed */
void oracle_block_scores(int64_t B, int64_t Hq, int64_t Hkv, int64_t T, int64_t D, int64_t bs, int64_t nb,
                         double scale, const int32_t *cu, const double *q, const double *kc, double *scores)
{
    prob_t p = mk(B, Hq, Hkv, T, D, bs, 1, scale, cu);
    const int64_t G = Hq / Hkv;
#pragma omp parallel for collapse(2) schedule(dynamic)
    for (int64_t b = 0; b < B; ++b)
        for (int64_t g = 0; g < Hkv; ++g) {
            double *s = (double *)malloc(sizeof(double) * (nb > 0 ? nb : 1));
            for (int64_t t = 0; t < seq_len(&p, b); ++t) {
                double *out = scores + score_off(&p, nb, b, g, t);
                for (int64_t j = 0; j < nb; ++j)
                    out[j] = 0.0;
                const int64_t nc = n_complete(t, bs);
                for (int64_t h = g * G; h < (g + 1) * G; ++h) {
                    const double *qt = q + row_off(&p, Hq, b, h, t);
                    double m = -INFINITY, sum = 0.0;
                    for (int64_t j = 0; j < nc; ++j) {
                        s[j] = scale * dot(qt, kc + ((b * Hkv + g) * nb + j) * D, D);
                        if (s[j] > m)
                            m = s[j];
                    }
                    for (int64_t j = 0; j < nc; ++j)
                        sum += exp(s[j] - m);
                    for (int64_t j = 0; j < nc; ++j)
                        out[j] += exp(s[j] - m) / sum;
                }
            }
            free(s);
        }
}

/* 1 if (x, i) comes before (y, j) in the selection order: larger score
 * first, then smaller block id; NaN as -infinity */
static int ranks_before(double x, int64_t i, double y, int64_t j)
{
    if (isnan(x))
        x = -INFINITY;
    if (isnan(y))
        y = -INFINITY;
    return x > y || (x == y && i < j);
}

/* idx rows from scores: the own block, then the S - 1 best complete blocks */
void oracle_select_topk(int64_t B, int64_t Hkv, int64_t T, int64_t bs, int64_t S, int64_t nb,
                        const int32_t *cu, const double *scores, int32_t *idx)
{
    prob_t p = mk(B, Hkv, Hkv, T, 1, bs, S, 1.0, cu);
    for (int64_t b = 0; b < B; ++b)
        for (int64_t g = 0; g < Hkv; ++g)
            for (int64_t t = 0; t < seq_len(&p, b); ++t) {
                const double *sc = scores + score_off(&p, nb, b, g, t);
                int32_t *row = (int32_t *)idx_row(&p, idx, b, g, t);
                const int64_t own = t / bs, nc = n_complete(t, bs);
                for (int64_t s = 0; s < S; ++s)
                    row[s] = -1;
                row[0] = (int32_t)own;
                for (int64_t s = 1; s < S; ++s) {
                    /* the best complete block not yet taken */
                    int64_t best = -1;
                    for (int64_t j = 0; j < nc; ++j) {
                        if (j == own)
                            continue;
                        int taken = 0;
                        for (int64_t u = 1; u < s; ++u)
                            taken |= row[u] == j;
                        if (taken)
                            continue;
                        if (best < 0 || ranks_before(sc[j], j, sc[best], best))
                            best = j;
                    }
                    if (best < 0)
                        break;
                    row[s] = (int32_t)best;
                }
            }
}
