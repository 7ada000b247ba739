/*
 * kda_oracle.c -- plain, slow, single-threaded CPU oracle for the speculative
 * verify walk through one Kimi-Delta-Attention (KDA) layer.
 *
 * TEST INFRASTRUCTURE ONLY.  The tests, the package smoke check and the CPU
 * baseline leg of the benchmark call it; the CUDA library never does.  It
 * shares no code, header, table or helper with the CUDA path.
 *
 * Precision: inputs and stored state are f32 (the pages keep the KDA state as
 * f32: one glm5_next KDA state is 64 heads x 128 x 128 f32, glm_spec.rs module
 * doc, ROLLBACK).  Every arithmetic step here runs in double and is rounded to
 * f32 only where a result is stored (state, conv ring, output rows).  bf16 raw
 * rows are widened exactly by a 16-bit left shift (dflash.rs, bf16_to_f32).
 *
 * What is computed, per (session, layer), for one head h and rows t = 0..T-1:
 *   short conv (width 4, depthwise, causal) over the raw q, k, v rows, with the
 *     3-slot ring of the previous raw inputs supplying x[t-3..t-1] for early rows,
 *     then SiLU:  y = a * sigmoid(a),  a = w0 x[t-3] + w1 x[t-2] + w2 x[t-1] + w3 x[t]
 *   L2 normalisation of q and k:  x_hat = y / sqrt(sum y^2 + 1e-6)
 *   gates:  g = -5 * sigmoid(raw_g) per key channel (gate_lower_bound -5.0 in the
 *     linear_attn_config of the mini fixture, glm5_spec_ppn_gate.rs);
 *     beta = sigmoid(raw_beta) per head
 *   gated delta rule on S [d_k = 128][d_v = 128]:
 *     S' = diag(exp g) S ;  u = S'^T k_hat ;  w = beta (v - u) ;
 *     S  = S' + k_hat w^T ;  o = S^T q_hat / sqrt(128)
 *   ring <- the last 3 of [ring, x_0 .. x_{T-1}]            (per stream)
 * The recurrence is sequential in t, one row at a time (glm_spec.rs module doc,
 * VERIFY-ROW BATCHING: the in-kernel T-loop is the chained t=1 program).
 *
 * Greedy accept (glm_spec.rs, glm5_spec_round step 4; dflash.rs,
 * dspark_accept_prefix): vam[r] = first index of the row maximum, j = the first
 * r < K with drafts[r] != vam[r] (else K), bonus = vam[j]; a NaN row yields a
 * sentinel that is refused loudly (the guard_vocab_token convention).
 *
 * Rollback (glm_spec.rs, glm5_verify_rollback and the KDA arm of
 * glm5_rollback_layer): keep must lie in 1..T; keep == T leaves the state as it
 * is; otherwise state and ring are rebuilt from the pre-round snapshot by running
 * rows 0..keep-1 again.
 *
 * Layouts of one (session, layer) unit, all row-major:
 *   raw rows q, k, v, g   [T][H][128]   (f32 or bf16 bits)
 *   raw beta              [T][H]
 *   conv_w                [H][3 stream: q,k,v][128][4 taps]  (tap 3 = current row)
 *   ring                  [H][3 stream][3 slot][128]         (slot 0 = oldest)
 *   state                 [H][128 d_k][128 d_v]
 *   out                   [T][H][128]
 */
#include "kda_oracle.h"

#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define D KDAO_D

/* bf16 -> f32: the 16 stored bits become the high half of an f32. */
static double widen(const void *base, int dtype, size_t idx)
{
    if (dtype == KDAO_BF16) {
        uint32_t bits = (uint32_t)((const uint16_t *)base)[idx] << 16;
        float f;
        memcpy(&f, &bits, sizeof f);
        return (double)f;
    }
    return (double)((const float *)base)[idx];
}

static double sigmoid(double z) { return 1.0 / (1.0 + exp(-z)); }

/* ---------------------------------------------------------------------------
 * Activations: conv + SiLU, L2 norm, gates, ring re-roll.
 * ------------------------------------------------------------------------- */
int kdao_prepare(int H, int T, int dtype,
                 const void *xq, const void *xk, const void *xv,
                 const void *xg, const void *xb,
                 const float *conv_w, const float *ring_in,
                 double *q_hat, double *k_hat, double *v_out,
                 double *g_out, double *beta_out, float *ring_out)
{
    if (H < 0 || T < 1 || (dtype != KDAO_F32 && dtype != KDAO_BF16))
        return KDAO_EINVAL;
    const void *raw[3] = {xq, xk, xv};
    /* hist[s][n][c]: n = 0..2 the ring slots (oldest first), n = 3 + t raw row t */
    double *hist = (double *)malloc(sizeof(double) * 3 * (size_t)(T + 3) * D);
    double *y = (double *)malloc(sizeof(double) * 3 * (size_t)T * D);
    if (!hist || !y) {
        free(hist);
        free(y);
        return KDAO_ENOMEM;
    }
    for (int h = 0; h < H; ++h) {
        for (int s = 0; s < 3; ++s) {
            for (int n = 0; n < 3; ++n)
                for (int c = 0; c < D; ++c)
                    hist[((size_t)s * (T + 3) + n) * D + c] =
                        ring_in[(((size_t)h * 3 + s) * 3 + n) * D + c];
            for (int t = 0; t < T; ++t)
                for (int c = 0; c < D; ++c)
                    hist[((size_t)s * (T + 3) + 3 + t) * D + c] =
                        widen(raw[s], dtype, ((size_t)t * H + h) * D + c);
        }
        /* depthwise causal conv, width 4, then SiLU */
        for (int s = 0; s < 3; ++s)
            for (int t = 0; t < T; ++t)
                for (int c = 0; c < D; ++c) {
                    const float *w = conv_w + (((size_t)h * 3 + s) * D + c) * 4;
                    const double *x = hist + ((size_t)s * (T + 3) + t) * D + c;
                    double a = (double)w[0] * x[0] + (double)w[1] * x[D] +
                               (double)w[2] * x[2 * D] + (double)w[3] * x[3 * D];
                    y[((size_t)s * T + t) * D + c] = a * sigmoid(a);
                }
        for (int t = 0; t < T; ++t) {
            size_t row = ((size_t)t * H + h) * D;
            /* L2 normalisation of q (s = 0) and k (s = 1) */
            for (int s = 0; s < 2; ++s) {
                const double *ys = y + ((size_t)s * T + t) * D;
                double ss = 0.0;
                for (int c = 0; c < D; ++c)
                    ss += ys[c] * ys[c];
                double r = 1.0 / sqrt(ss + KDAO_L2_EPS);
                double *dst = (s == 0) ? q_hat : k_hat;
                for (int c = 0; c < D; ++c)
                    dst[row + c] = ys[c] * r;
            }
            for (int c = 0; c < D; ++c)
                v_out[row + c] = y[((size_t)2 * T + t) * D + c];
            /* forget gate per key channel, write strength per head */
            for (int c = 0; c < D; ++c)
                g_out[row + c] = KDAO_GATE_LOWER_BOUND * sigmoid(widen(xg, dtype, row + c));
            beta_out[(size_t)t * H + h] = sigmoid(widen(xb, dtype, (size_t)t * H + h));
        }
        /* ring <- the last three raw inputs of each stream */
        if (ring_out)
            for (int s = 0; s < 3; ++s)
                for (int n = 0; n < 3; ++n)
                    for (int c = 0; c < D; ++c)
                        ring_out[(((size_t)h * 3 + s) * 3 + n) * D + c] =
                            (float)hist[((size_t)s * (T + 3) + T + n) * D + c];
    }
    free(hist);
    free(y);
    return KDAO_OK;
}

/* ---------------------------------------------------------------------------
 * The gated delta rule, row by row, on post-activation inputs.
 * S is [H][d_k][d_v] in double, updated in place; out [T][H][d_v] may be NULL.
 * ------------------------------------------------------------------------- */
int kdao_core(int H, int T, const double *q_hat, const double *k_hat,
              const double *v, const double *g, const double *beta,
              double *S, double *out)
{
    if (H < 0 || T < 0)
        return KDAO_EINVAL;
    const double scale = 1.0 / sqrt((double)D);
    double u[D], w[D];
    for (int t = 0; t < T; ++t) {
        for (int h = 0; h < H; ++h) {
            size_t row = ((size_t)t * H + h) * D;
            const double *q = q_hat + row, *k = k_hat + row, *vv = v + row, *gg = g + row;
            double b = beta[(size_t)t * H + h];
            double *Sh = S + (size_t)h * D * D;
            /* S' = diag(exp g) S : row i of S (key channel i) decays by exp(g_i) */
            for (int i = 0; i < D; ++i) {
                double d = exp(gg[i]);
                for (int j = 0; j < D; ++j)
                    Sh[i * D + j] *= d;
            }
            /* u = S'^T k */
            for (int j = 0; j < D; ++j) {
                double acc = 0.0;
                for (int i = 0; i < D; ++i)
                    acc += Sh[i * D + j] * k[i];
                u[j] = acc;
            }
            /* w = beta (v - u) */
            for (int j = 0; j < D; ++j)
                w[j] = b * (vv[j] - u[j]);
            /* S = S' + k w^T */
            for (int i = 0; i < D; ++i)
                for (int j = 0; j < D; ++j)
                    Sh[i * D + j] += k[i] * w[j];
            /* o = S^T q / sqrt(d_k) */
            if (out)
                for (int j = 0; j < D; ++j) {
                    double acc = 0.0;
                    for (int i = 0; i < D; ++i)
                        acc += Sh[i * D + j] * q[i];
                    out[row + j] = acc * scale;
                }
        }
    }
    return KDAO_OK;
}

/* ---------------------------------------------------------------------------
 * One verify launch for one (session, layer): T rows from state_in/ring_in.
 * state_out / ring_out receive the state after row T-1 (f32); out the T rows.
 * ------------------------------------------------------------------------- */
int kdao_verify(int H, int T, int dtype,
                const void *xq, const void *xk, const void *xv,
                const void *xg, const void *xb,
                const float *conv_w, const float *ring_in, const float *state_in,
                float *ring_out, float *state_out, float *out)
{
    if (H < 0 || T < 1 || T > KDAO_TMAX)
        return KDAO_EINVAL;
    size_t nrow = (size_t)T * H * D, nst = (size_t)H * D * D;
    double *q = (double *)malloc(sizeof(double) * nrow + 1);
    double *k = (double *)malloc(sizeof(double) * nrow + 1);
    double *v = (double *)malloc(sizeof(double) * nrow + 1);
    double *g = (double *)malloc(sizeof(double) * nrow + 1);
    double *b = (double *)malloc(sizeof(double) * (size_t)T * H + 1);
    double *S = (double *)malloc(sizeof(double) * nst + 1);
    double *o = (double *)malloc(sizeof(double) * nrow + 1);
    int rc = KDAO_ENOMEM;
    if (q && k && v && g && b && S && o) {
        rc = kdao_prepare(H, T, dtype, xq, xk, xv, xg, xb, conv_w, ring_in, q, k, v, g, b,
                          ring_out);
        if (rc == KDAO_OK) {
            for (size_t n = 0; n < nst; ++n)
                S[n] = (double)state_in[n];
            rc = kdao_core(H, T, q, k, v, g, b, S, o);
        }
        if (rc == KDAO_OK) {
            for (size_t n = 0; n < nst; ++n)
                state_out[n] = (float)S[n];
            if (out)
                for (size_t n = 0; n < nrow; ++n)
                    out[n] = (float)o[n];
        }
    }
    free(q);
    free(k);
    free(v);
    free(g);
    free(b);
    free(S);
    free(o);
    return rc;
}

/* ---------------------------------------------------------------------------
 * Accept-j rollback for one (session, layer).  T is the row count of the round
 * the snapshots belong to; the raw rows are that round's [T][H][128] rows.
 * ------------------------------------------------------------------------- */
int kdao_rollback(int H, int T, int keep, int dtype,
                  const void *xq, const void *xk, const void *xv,
                  const void *xg, const void *xb, const float *conv_w,
                  const float *ring_snap, const float *state_snap,
                  const float *ring_cur, const float *state_cur,
                  float *ring_out, float *state_out)
{
    if (keep < 1 || keep > T)
        return KDAO_EINVAL;
    if (keep == T) {
        /* the resident state is the state after the last kept row */
        memmove(state_out, state_cur, sizeof(float) * (size_t)H * D * D);
        memmove(ring_out, ring_cur, sizeof(float) * (size_t)H * 3 * 3 * D);
        return KDAO_OK;
    }
    return kdao_verify(H, keep, dtype, xq, xk, xv, xg, xb, conv_w, ring_snap, state_snap,
                       ring_out, state_out, NULL);
}

/* ---------------------------------------------------------------------------
 * Greedy accept for one session: logits [T][V], drafts [T-1].
 * ------------------------------------------------------------------------- */
int kdao_accept(int T, int V, int dtype, const void *logits, const int *drafts,
                int *vam, int *j_out, int *bonus_out)
{
    if (T < 1 || V < 1 || (dtype != KDAO_F32 && dtype != KDAO_BF16))
        return KDAO_EINVAL;
    for (int r = 0; r < T; ++r) {
        int best = 0, nan_row = 0;
        double bv = widen(logits, dtype, (size_t)r * V);
        for (int c = 0; c < V; ++c) {
            double x = widen(logits, dtype, (size_t)r * V + c);
            if (isnan(x))
                nan_row = 1;
            else if (isnan(bv) || x > bv) {
                bv = x;
                best = c;
            }
        }
        vam[r] = nan_row ? KDAO_SENTINEL : best;
    }
    int K = T - 1, j = 0;
    while (j < K && vam[j] != KDAO_SENTINEL && drafts[j] == vam[j])
        ++j;
    *j_out = j;
    *bonus_out = vam[j];
    return vam[j] == KDAO_SENTINEL ? KDAO_ENAN : KDAO_OK;
}

/* ---------------------------------------------------------------------------
 * Verify-window policies: how many drafted rows a session sends through verify.
 * They decide integers from f32 arithmetic, so they compute in f32 with the
 * operations the pages use (the host's expf, IEEE division), not in double.
 * ------------------------------------------------------------------------- */

/* glm_spec.rs, glm5_conf_keep and its conf_keep_tests: the p-min break of the
 * draft chain.  q[0..n-1] are the drafter's confidences of draft slots 0..n-1.
 * Slots are kept in order until the first slot whose confidence is strictly
 * below p_min; a miss at slot 0 only breaks the chain when pmin0 is set (slot 0
 * is otherwise judged on its own and does not latch).  Returns the kept count. */
int kdao_conf_keep(int n, const float *q, float p_min, int pmin0)
{
    int kept = 0;
    for (int j = 0; j < n; ++j) {
        if (q[j] < p_min && (j > 0 || pmin0))
            break;
        ++kept;
    }
    return kept;
}

static float sigmoid_f32(float r)
{
    return 1.0f / (1.0f + expf(-r));
}

static int clamp_vt(int kept, int vt_cap)
{
    int hi = vt_cap > 2 ? vt_cap : 2;
    int vt = 1 + kept;
    return vt < 2 ? 2 : (vt > hi ? hi : vt);
}

/* dflash.rs, dspark_confidence_vt: raws[k] is the pre-sigmoid accept score of
 * draft slot k+1; the survival S_k = prod_{j<=k} sigmoid(raws[j]) (accumulated in
 * f32 in slot order) keeps leading slots while S_k >= tau.  Returns the verify
 * row count 1 + kept, clamped to [2, max(vt_cap, 2)]. */
int kdao_confidence_vt(int n, const float *raws, float tau, int vt_cap)
{
    float surv = 1.0f;
    int kept = 0;
    for (int k = 0; k < n; ++k) {
        surv *= sigmoid_f32(raws[k]);
        if (surv < tau)
            break;
        ++kept;
    }
    return clamp_vt(kept, vt_cap);
}

/* dflash.rs, dspark_slot_confidence_vt: the same window with the per-slot
 * statistic: keep the longest prefix whose every slot has sigmoid(raw) >= tau. */
int kdao_slot_confidence_vt(int n, const float *raws, float tau, int vt_cap)
{
    int kept = 0;
    for (int k = 0; k < n; ++k) {
        if (sigmoid_f32(raws[k]) < tau)
            break;
        ++kept;
    }
    return clamp_vt(kept, vt_cap);
}

/* ---------------------------------------------------------------------------
 * Sampled acceptance (glm_spec.rs module doc, SAMPLED ACCEPTANCE, and
 * glm5_sampled_accept / glm5_sampled_bonus): the rejection-sampling walk over the
 * verify rows, with target p and draft q taken through the same filter.
 *
 * Filtered distribution of one logits row x[0..V-1] (filter_stats +
 * softmax_gather_filtered; their internals are not printed, so this is the plain
 * reading: each filter is a threshold on the one unfiltered distribution and a
 * token is kept when it passes all of them):
 *   z = x / temperature,  e_v = exp(z_v - max z)  (so max e = 1),  S = sum e
 *   top_k in 1..V-1: kept iff e_v >= the k-th largest e        (ties at it kept)
 *   top_p < 1:       with e sorted descending, n = the first count whose running
 *                    sum reaches top_p * S; kept iff e_v >= e_(n) (ties kept)
 *   min_p > 0:       kept iff e_v >= min_p  (p_v >= min_p * max p)
 *   p~_v = e_v / Z over the kept tokens, Z = sum of their e; 0 elsewhere.
 * ------------------------------------------------------------------------- */
static int cmp_desc(const void *a, const void *b)
{
    double x = *(const double *)a, y = *(const double *)b;
    return x < y ? 1 : (x > y ? -1 : 0);
}

int kdao_filtered(int V, int dtype, const void *row, double temperature, int top_k, double top_p,
                  double min_p, double *p)
{
    if (V < 1 || !(temperature > 0.0) || top_k < 0 || !(top_p > 0.0) || !(min_p >= 0.0) || min_p >= 1.0)
        return KDAO_EINVAL;
    double m = -INFINITY;
    for (int v = 0; v < V; ++v) {
        double z = widen(row, dtype, (size_t)v) / temperature;
        if (isnan(z))
            return KDAO_ENAN;
        p[v] = z;
        if (z > m)
            m = z;
    }
    if (isinf(m))  /* every logit -inf, or a +inf logit: no distribution */
        return KDAO_EINVAL;
    double S = 0.0;
    for (int v = 0; v < V; ++v) {
        p[v] = exp(p[v] - m);
        S += p[v];
    }
    double *sorted = malloc(sizeof(double) * (size_t)V);
    if (!sorted)
        return KDAO_ENOMEM;
    memcpy(sorted, p, sizeof(double) * (size_t)V);
    qsort(sorted, (size_t)V, sizeof(double), cmp_desc);
    double th = 0.0;
    if (top_k > 0 && top_k < V && sorted[top_k - 1] > th)
        th = sorted[top_k - 1];
    if (top_p < 1.0) {
        double run = 0.0;
        for (int i = 0; i < V; ++i) {
            run += sorted[i];
            if (run >= top_p * S) {
                if (sorted[i] > th)
                    th = sorted[i];
                break;
            }
        }
    }
    free(sorted);
    if (min_p > th)
        th = min_p;
    double Z = 0.0;
    for (int v = 0; v < V; ++v)
        if (p[v] >= th)
            Z += p[v];
    for (int v = 0; v < V; ++v)
        p[v] = p[v] >= th ? p[v] / Z : 0.0;
    return KDAO_OK;
}

/* One draw from weights w[0..V-1] (not all zero) with the uniform u in [0, 1):
 * the first index whose running sum, in index order, exceeds u * sum(w). */
static int draw_index(int V, const double *w, double u)
{
    double W = 0.0;
    for (int v = 0; v < V; ++v)
        W += w[v];
    double target = u * W, run = 0.0;
    int last = -1;
    for (int v = 0; v < V; ++v) {
        if (w[v] > 0.0)
            last = v;
        run += w[v];
        if (run > target)
            return v;
    }
    return last;  /* u * W rounded up to W: the last token with weight */
}

/* The sampled accept walk of one session.  logits [T][V] (target rows),
 * draft_logits [T-1][V] (the rows the drafts were drawn from), drafts [T-1];
 * u_accept[r] is the accept-test uniform of draft r, u_sample the uniform of the
 * final draw.  Draft r is accepted iff u_accept[r] * q~_r(x_r) < p~_r(x_r); the walk
 * stops at the first rejection j.  j < K: the token is drawn from the residual
 * max(0, p~_j - q~_j) (from p~_j when that residual is zero everywhere); j = K: the
 * bonus is drawn from p~_K, the last verify row. */
int kdao_sampled_accept(int T, int V, int dtype, const void *logits, const void *draft_logits,
                        const int *drafts, const double *u_accept, double u_sample, double temperature,
                        int top_k, double top_p, double min_p, int *j_out, int *token_out)
{
    if (T < 1 || V < 1)
        return KDAO_EINVAL;
    const int K = T - 1;
    size_t es = dtype == KDAO_BF16 ? 2 : 4;
    double *pr = malloc(sizeof(double) * (size_t)V), *qr = malloc(sizeof(double) * (size_t)V);
    if (!pr || !qr) {
        free(pr);
        free(qr);
        return KDAO_ENOMEM;
    }
    int rc = KDAO_OK, j = 0;
    for (; j < K; ++j) {
        if (drafts[j] < 0 || drafts[j] >= V) {
            rc = KDAO_EINVAL;
            goto done;
        }
        if ((rc = kdao_filtered(V, dtype, (const char *)logits + (size_t)j * V * es, temperature, top_k, top_p,
                                min_p, pr)))
            goto done;
        if ((rc = kdao_filtered(V, dtype, (const char *)draft_logits + (size_t)j * V * es, temperature, top_k,
                                top_p, min_p, qr)))
            goto done;
        /* the page compares its f32 gathers of p~ and q~ in double:
         * (u as f64) * (qj as f64) < pj as f64 */
        if (!(u_accept[j] * (double)(float)qr[drafts[j]] < (double)(float)pr[drafts[j]]))
            break;
    }
    if (j < K) {  /* pr, qr hold row j */
        int any = 0;
        for (int v = 0; v < V; ++v) {
            double r = pr[v] - qr[v];
            qr[v] = r > 0.0 ? r : 0.0;
            any |= qr[v] > 0.0;
        }
        *token_out = draw_index(V, any ? qr : pr, u_sample);
    } else {
        if ((rc = kdao_filtered(V, dtype, (const char *)logits + (size_t)K * V * es, temperature, top_k, top_p,
                                min_p, pr)))
            goto done;
        *token_out = draw_index(V, pr, u_sample);
    }
    *j_out = j;
done:
    free(pr);
    free(qr);
    return rc;
}

/* Philox4x32-10 (Salmon, Moraes, Dror and Shaw, "Parallel random numbers: as easy
 * as 1, 2, 3", SC'11): ten rounds on a 128-bit counter under a 64-bit key.  A round
 * multiplies counter words 0 and 2 by the two round multipliers (full 64-bit
 * products), and the new counter is (hi(M1 c2) ^ c1 ^ k0, lo(M1 c2),
 * hi(M0 c0) ^ c3 ^ k1, lo(M0 c0)); the key is bumped by the two Weyl constants
 * between rounds. */
void kdao_philox4x32_10(const unsigned int ctr[4], const unsigned int key[2], unsigned int out[4])
{
    const uint32_t M0 = 0xD2511F53u, M1 = 0xCD9E8D57u;
    const uint32_t W0 = 0x9E3779B9u, W1 = 0xBB67AE85u;
    uint32_t c0 = ctr[0], c1 = ctr[1], c2 = ctr[2], c3 = ctr[3];
    uint32_t k0 = key[0], k1 = key[1];
    for (int r = 0; r < 10; ++r) {
        if (r > 0) {
            k0 += W0;
            k1 += W1;
        }
        const uint64_t p0 = (uint64_t)M0 * c0, p1 = (uint64_t)M1 * c2;
        const uint32_t n0 = (uint32_t)(p1 >> 32) ^ c1 ^ k0;
        const uint32_t n1 = (uint32_t)p1;
        const uint32_t n2 = (uint32_t)(p0 >> 32) ^ c3 ^ k1;
        const uint32_t n3 = (uint32_t)p0;
        c0 = n0;
        c1 = n1;
        c2 = n2;
        c3 = n3;
    }
    out[0] = c0;
    out[1] = c1;
    out[2] = c2;
    out[3] = c3;
}

/* One uniform in [0, 1) of a session's stream: Philox4x32-10 under key (seed low,
 * seed high) at counter (counter, 0, 0, tag), the top 24 bits of output word 0 times
 * 2^-24 (exact in f32).  glm_spec.rs draws the accept-test uniforms on the host from
 * the session's uctr with stream tag 0xFFFF_FFFE (spec::host_u01), and the device
 * draws from its sctr; the word layout is this library's reading. */
float kdao_u01(unsigned long long seed, unsigned int counter, unsigned int tag)
{
    const unsigned int key[2] = {(unsigned int)seed, (unsigned int)(seed >> 32)};
    const unsigned int ctr[4] = {counter, 0u, 0u, tag};
    unsigned int o[4];
    kdao_philox4x32_10(ctr, key, o);
    return (float)((double)(o[0] >> 8) * (1.0 / 16777216.0));
}

/* The sampled accept walk with the session's counters (glm_spec.rs,
 * glm5_sampled_accept / glm5_sampled_bonus, and the Glm5SpecSession doc: the
 * counters live on the session and are never reset).  Accept test r draws
 * u01(seed, uctr, KDAO_TAG_ACCEPT) and advances uctr by one; the walk stops at the
 * first rejection, so a round runs j + 1 tests when it rejects draft j and K when it
 * accepts every draft.  The residual or bonus draw takes u01(seed, sctr,
 * KDAO_TAG_DRAW) and advances sctr by one. */
int kdao_sampled_accept_session(int T, int V, int dtype, const void *logits, const void *draft_logits,
                                const int *drafts, unsigned long long seed, unsigned int *uctr,
                                unsigned int *sctr, double temperature, int top_k, double top_p,
                                double min_p, int *j_out, int *token_out)
{
    if (T < 1 || T > KDAO_TMAX)
        return KDAO_EINVAL;
    const int K = T - 1;
    double u_accept[KDAO_TMAX];
    for (int r = 0; r < K; ++r)
        u_accept[r] = kdao_u01(seed, *uctr + (unsigned int)r, KDAO_TAG_ACCEPT);
    const double u_sample = kdao_u01(seed, *sctr, KDAO_TAG_DRAW);
    const int rc = kdao_sampled_accept(T, V, dtype, logits, draft_logits, drafts, u_accept, u_sample, temperature,
                                       top_k, top_p, min_p, j_out, token_out);
    if (rc)
        return rc;
    *uctr += (unsigned int)(*j_out < K ? *j_out + 1 : K);
    *sctr += 1u;
    return KDAO_OK;
}
