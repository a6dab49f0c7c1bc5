/*
 * Depthwise causal conv1d -- plain CPU oracle, fp64 arithmetic.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the slow, obviously-correct
 * restatement of the operation that the CUDA path is checked against.  Only the
 * tests, the smoke check and the benchmark's CPU-baseline leg may load it.  It
 * shares no code, header, table or helper with the CUDA library.
 *
 * What it computes (cuDNN frontend "Causal Conv1d" page: the list of tensors
 * -- weight[D, W], states [., D, W - 1] -- the paragraph on the optimized route
 * -- width four, SiLU, W-1 initial and final state, cu_seqlens packing -- and
 * the paragraph on causal_conv1d_update; tap order from the causal-padding
 * derivation on the POPCORNBENCH conv1d page, where tap k of a width-K filter
 * reads input position t + k - (K-1)).  For a width W in 2..4 and S = W - 1:
 *
 *   extended sequence   xe[j] = x[j]            for 0 <= j < len
 *                       xe[j] = init[j + S]     for -S <= j < 0 (0 if no init)
 *   pre-activation      pre[t] = bias + sum_{k=0..W-1} w[k] * xe[t - S + k]
 *   output              out[t] = silu(pre[t]) = pre[t] * s(pre[t]),  s(p) = 1/(1+exp(-p))
 *                       (or out = pre with the identity activation)
 *   final state         final[i] = xe[len - S + i], i = 0..S-1
 *
 * A "sequence" is one batch row of a dense call, or one cu_seqlens range of a
 * packed call (each with its own initial/final state, nothing crosses a
 * boundary).
 *
 * Per-token sequence ids (the cuDNN page's seq_idx[B, T] keyword, mutually
 * exclusive with cu_seqlens): tokens of a dense row that carry the same id
 * form one sequence, so tap k of token t reads xe[t - S + k] only when that
 * token carries the id of token t, and reads zero otherwise.  The pages fix
 * nothing more; initial and final states are not defined with seq_idx and are
 * rejected in combination with it.
 *
 * Backward (gradients of L with g = dL/dout and gf = dL/dfinal):
 *   gp[t]    = g[t] * silu'(pre[t]),   silu'(p) = s(p) * (1 + p * (1 - s(p)))
 *   dxe[j]   = sum_k w[k] * gp[j + S - k]   (only terms with 0 <= j+S-k < len)
 *              + gf[j - (len - S)]          (when j >= len - S)
 *   dx[t]    = dxe[t],   dinit[i] = dxe[i - S]
 *   dw[k]    = sum_seq sum_t gp[t] * xe[t - S + k],    db = sum_seq sum_t gp[t]
 *
 * Single-token update (causal_conv1d_update): xe = [s0 .. s(S-1), x],
 * out = act(bias + sum_k w[k] * xe[k]), new state = [s1 .. s(S-1), x].
 *
 * Every input and output here is a double.  The Python side decodes BF16
 * inputs exactly into doubles and rounds results once (nearest-even) to the
 * output type with oracle_bf16_encode_array below.  Products of a BF16 value
 * and a BF16/FP32 weight are exact in double, so pre[] is the exact value up to
 * the double rounding of a (W+1)-term sum.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define CONV_WMAX 4 /* widths 2..4 */

enum { ORC_OK = 0, ORC_BAD_CU_SEQLENS = 7, ORC_NO_MEMORY = 100, ORC_BAD_WIDTH = 101,
       ORC_BAD_SEQ_IDX = 102 };

/* ---- BF16 rounding ------------------------------------------------------ */

/* Round a double to the nearest BF16 value (ties to even), returned as bits.
 * BF16 keeps 8 significant bits; for |v| in [2^(e-1), 2^e) the spacing of
 * representable values is 2^(e-8).  Below the smallest normal (2^-126) the
 * spacing stays 2^-133.  Values that round to 2^128 or beyond overflow to inf. */
uint16_t oracle_bf16_encode(double v)
{
    if (isnan(v))
        return 0x7FC0;
    uint16_t sign = signbit(v) ? 0x8000 : 0;
    double a = fabs(v);
    if (a == 0.0)
        return sign;
    if (isinf(a))
        return (uint16_t)(sign | 0x7F80);
    int e;
    (void)frexp(a, &e);
    int qexp = (e < -125 ? -125 : e) - 8;
    double r = rint(ldexp(a, -qexp)); /* default rounding mode: nearest-even */
    double q = ldexp(r, qexp);
    if (q >= ldexp(1.0, 128))
        return (uint16_t)(sign | 0x7F80);
    float f = (float)q; /* exact: q is a BF16 value */
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    return (uint16_t)(sign | ((u >> 16) & 0x7FFF));
}

void oracle_bf16_encode_array(const double *v, int64_t n, uint16_t *out)
{
    for (int64_t i = 0; i < n; ++i)
        out[i] = oracle_bf16_encode(v[i]);
}

/* ---- activation --------------------------------------------------------- */

static double sigmoid(double p) { return 1.0 / (1.0 + exp(-p)); }

static double activate(double p, int act) { return act ? p * sigmoid(p) : p; }

static double activate_grad(double p, int act)
{
    if (!act)
        return 1.0;
    double s = sigmoid(p);
    return s * (1.0 + p * (1.0 - s));
}

/* ---- sequences ---------------------------------------------------------- */

/* cu_seqlens rules (cuDNN page, paragraph on packed metadata): first offset 0,
 * last offset equal to the runtime token total, strictly increasing offsets
 * (an empty sequence is malformed). */
int oracle_check_cu_seqlens(const int32_t *cu, int n_seq, int64_t total)
{
    if (n_seq < 1 || cu[0] != 0 || (int64_t)cu[n_seq] != total)
        return ORC_BAD_CU_SEQLENS;
    for (int n = 0; n < n_seq; ++n)
        if (cu[n + 1] <= cu[n])
            return ORC_BAD_CU_SEQLENS;
    return ORC_OK;
}

/* Sequence n: batch row, first token within the row, and length.  Dense: row
 * n, tokens 0..T-1.  Packed: row 0, tokens cu[n]..cu[n+1]-1. */
static void seq_range(int n, const int32_t *cu, int64_t T, int64_t *row, int64_t *start, int64_t *len)
{
    if (cu) {
        *row = 0;
        *start = cu[n];
        *len = (int64_t)cu[n + 1] - cu[n];
    } else {
        *row = n;
        *start = 0;
        *len = T;
    }
}

/* xe[j] of one (sequence, channel); x points at token 0 of the sequence,
 * init at its S state entries (or NULL). */
static double xe(const double *x, const double *init, int S, int64_t j)
{
    if (j >= 0)
        return x[j];
    return init ? init[j + S] : 0.0;
}

/* Whether input position j (of the same row) feeds token t: always without
 * per-token ids (positions before the row read the initial state or zero);
 * with ids, only positions carrying the id of token t. */
static int same_seq(const int32_t *ids, int64_t j, int64_t t)
{
    return !ids || j < 0 || ids[j] == ids[t];
}

static double pre_activation(const double *x, const double *init, const int32_t *ids,
                             const double *w, int W, double b, int64_t t)
{
    double p = b;
    for (int k = 0; k < W; ++k)
        if (same_seq(ids, t - (W - 1) + k, t))
            p += w[k] * xe(x, init, W - 1, t - (W - 1) + k);
    return p;
}

/* seq_idx excludes cu_seqlens and the states (see the header comment). */
static int seq_idx_ok(const int32_t *seq_idx, const int32_t *cu, const void *init, const void *fin)
{
    return !seq_idx || (!cu && !init && !fin);
}

/* ---- forward ------------------------------------------------------------ */

/*
 * x:     [B][D][T] (packed: B == 1 and T == token total)
 * w:     [D][W], 2 <= W <= 4;  bias: [D] or NULL
 * cu:    [n_seq + 1] or NULL (dense: n_seq is taken as B)
 * seq_idx: [B][T] per-token sequence ids or NULL (dense only, no states)
 * init:  [n_seq][D][W-1] or NULL
 * out, pre: [B][D][T] (pre may be NULL);  fin: [n_seq][D][W-1] or NULL
 */
int oracle_fwd(const double *x, int64_t B, int64_t D, int64_t T,
               const double *w, int W, const double *bias, const int32_t *cu, int n_seq,
               const int32_t *seq_idx, const double *init, int act, double *out, double *pre,
               double *fin)
{
    if (W < 2 || W > CONV_WMAX)
        return ORC_BAD_WIDTH;
    const int S = W - 1;
    if (!seq_idx_ok(seq_idx, cu, init, fin))
        return ORC_BAD_SEQ_IDX;
    if (cu && oracle_check_cu_seqlens(cu, n_seq, T))
        return ORC_BAD_CU_SEQLENS;
    if (!cu)
        n_seq = (int)B;
    for (int n = 0; n < n_seq; ++n) {
        int64_t row, start, len;
        seq_range(n, cu, T, &row, &start, &len);
        for (int64_t d = 0; d < D; ++d) {
            const double *wd = w + d * W;
            double b = bias ? bias[d] : 0.0;
            int64_t base = (row * D + d) * T + start;
            const double *xs = x + base;
            const double *is = init ? init + ((int64_t)n * D + d) * S : NULL;
            const int32_t *ids = seq_idx ? seq_idx + row * T + start : NULL;
            for (int64_t t = 0; t < len; ++t) {
                double p = pre_activation(xs, is, ids, wd, W, b, t);
                out[base + t] = activate(p, act);
                if (pre)
                    pre[base + t] = p;
            }
            if (fin) {
                double *fs = fin + ((int64_t)n * D + d) * S;
                for (int i = 0; i < S; ++i)
                    fs[i] = xe(xs, is, S, len - S + i);
            }
        }
    }
    return ORC_OK;
}

/* ---- backward ----------------------------------------------------------- */

/*
 * Inputs as oracle_fwd, plus g: [B][D][T] and gfin: [n_seq][D][W-1] or NULL.
 * Outputs (any may be NULL):
 *   dx [B][D][T];  dinit [n_seq][D][W-1]
 *   dw [D][W], dw_abs [D][W] = sum |gp * xe|;  db [D], db_abs [D] = sum |gp|
 * The sums run over sequences in ascending order, then tokens in ascending
 * order, in one double accumulator per (channel, tap).
 */
int oracle_bwd(const double *x, int64_t B, int64_t D, int64_t T,
               const double *w, int W, const double *bias, const int32_t *cu, int n_seq,
               const int32_t *seq_idx, const double *init, int act, const double *g,
               const double *gfin, double *dx, double *dinit, double *dw, double *dw_abs,
               double *db, double *db_abs)
{
    if (W < 2 || W > CONV_WMAX)
        return ORC_BAD_WIDTH;
    const int S = W - 1;
    if (!seq_idx_ok(seq_idx, cu, init, gfin))
        return ORC_BAD_SEQ_IDX;
    if (cu && oracle_check_cu_seqlens(cu, n_seq, T))
        return ORC_BAD_CU_SEQLENS;
    if (!cu)
        n_seq = (int)B;
    double *gp = (double *)malloc((size_t)(T > 0 ? T : 1) * sizeof(double));
    if (!gp)
        return ORC_NO_MEMORY;
    for (int64_t d = 0; d < D; ++d) {
        const double *wd = w + d * W;
        double b = bias ? bias[d] : 0.0;
        double sdw[CONV_WMAX] = {0, 0, 0, 0}, sdw_abs[CONV_WMAX] = {0, 0, 0, 0};
        double sdb = 0.0, sdb_abs = 0.0;
        for (int n = 0; n < n_seq; ++n) {
            int64_t row, start, len;
            seq_range(n, cu, T, &row, &start, &len);
            int64_t base = (row * D + d) * T + start;
            const double *xs = x + base;
            const double *gs = g + base;
            const double *is = init ? init + ((int64_t)n * D + d) * S : NULL;
            const double *gfs = gfin ? gfin + ((int64_t)n * D + d) * S : NULL;
            const int32_t *ids = seq_idx ? seq_idx + row * T + start : NULL;
            /* gradient at the pre-activation; weight and bias sums */
            for (int64_t t = 0; t < len; ++t) {
                gp[t] = gs[t] * activate_grad(pre_activation(xs, is, ids, wd, W, b, t), act);
                for (int k = 0; k < W; ++k) {
                    double term = gp[t] * xe(xs, is, S, t - (W - 1) + k);
                    if (!same_seq(ids, t - (W - 1) + k, t))
                        term = 0.0; /* tap reads another sequence: zero */
                    sdw[k] += term;
                    sdw_abs[k] += fabs(term);
                }
                sdb += gp[t];
                sdb_abs += fabs(gp[t]);
            }
            /* gradient at every entry of the extended sequence */
            for (int64_t j = -S; j < len; ++j) {
                double acc = 0.0;
                for (int k = 0; k < W; ++k) {
                    int64_t t = j + (W - 1) - k; /* the output that tap k reads xe[j] for */
                    if (t >= 0 && t < len && same_seq(ids, j, t))
                        acc += wd[k] * gp[t];
                }
                if (gfs && j >= len - S)
                    acc += gfs[j - (len - S)];
                if (j >= 0) {
                    if (dx)
                        dx[base + j] = acc;
                } else if (dinit) {
                    dinit[((int64_t)n * D + d) * S + (j + S)] = acc;
                }
            }
        }
        for (int k = 0; k < W; ++k) {
            if (dw)
                dw[d * W + k] = sdw[k];
            if (dw_abs)
                dw_abs[d * W + k] = sdw_abs[k];
        }
        if (db)
            db[d] = sdb;
        if (db_abs)
            db_abs[d] = sdb_abs;
    }
    free(gp);
    return ORC_OK;
}

/* ---- single-token update ------------------------------------------------ */

/*
 * x:     [B][D] (one token);  w [D][W], 2 <= W <= 4;  bias [D] or NULL
 * state: [B][D][W-1], read, then overwritten with [s1 .. s(W-2), x]
 * out:   [B][D]
 */
int oracle_update(const double *x, int64_t B, int64_t D, const double *w, int W,
                  const double *bias, int act, double *state, double *out)
{
    if (W < 2 || W > CONV_WMAX)
        return ORC_BAD_WIDTH;
    const int S = W - 1;
    for (int64_t bb = 0; bb < B; ++bb) {
        for (int64_t d = 0; d < D; ++d) {
            const double *wd = w + d * W;
            double *s = state + (bb * D + d) * S;
            double ext[CONV_WMAX];
            for (int i = 0; i < S; ++i)
                ext[i] = s[i];
            ext[S] = x[bb * D + d];
            double p = bias ? bias[d] : 0.0;
            for (int k = 0; k < W; ++k)
                p += wd[k] * ext[k];
            out[bb * D + d] = activate(p, act);
            for (int i = 0; i < S; ++i)
                s[i] = ext[i + 1];
        }
    }
    return ORC_OK;
}

/* ---- full-channel dilated causal conv1d ---------------------------------- */

/*
 * POPCORNBENCH conv1d page (the reasoning section and both listings): a Conv1d
 * over all input channels with dilation, made causal by left padding
 * P = (K-1)*dil; tap k reads input position t + k*dil - P, and positions before
 * 0 read zero:
 *
 *   out[b,oc,t] = bias[oc] + sum_{ic<Cin} sum_{k<K} w[oc,ic,k] * x[b,ic,t + k*dil - P]
 *
 * x [B][Cin][T], w [Cout][Cin][K], bias [Cout] or NULL, out [B][Cout][T];
 * abs_sum (or NULL) [B][Cout][T] receives |bias| + sum |w * x| over the same
 * terms (the scale of the rounding error of any summation order).  The sum runs
 * over ic, then k, in ascending order, in one double accumulator.
 */
int oracle_fullconv_fwd(const double *x, int64_t B, int64_t Cin, int64_t T, const double *w,
                        int64_t Cout, int K, int dil, const double *bias, double *out,
                        double *abs_sum)
{
    if (K < 1 || dil < 1)
        return ORC_BAD_WIDTH;
    const int64_t P = (int64_t)(K - 1) * dil;
    for (int64_t b = 0; b < B; ++b) {
        for (int64_t oc = 0; oc < Cout; ++oc) {
            for (int64_t t = 0; t < T; ++t) {
                double s = bias ? bias[oc] : 0.0;
                double a = bias ? fabs(bias[oc]) : 0.0;
                for (int64_t ic = 0; ic < Cin; ++ic) {
                    for (int k = 0; k < K; ++k) {
                        int64_t pos = t + (int64_t)k * dil - P;
                        if (pos < 0)
                            continue; /* the causal padding */
                        double term = w[(oc * Cin + ic) * K + k] * x[(b * Cin + ic) * T + pos];
                        s += term;
                        a += fabs(term);
                    }
                }
                out[(b * Cout + oc) * T + t] = s;
                if (abs_sum)
                    abs_sum[(b * Cout + oc) * T + t] = a;
            }
        }
    }
    return ORC_OK;
}
