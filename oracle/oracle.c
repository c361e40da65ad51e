/*
 * oracle.c -- plain, slow fp64 CPU reference of one Mixture-of-Experts layer,
 * forward and backward.
 *
 * TEST INFRASTRUCTURE ONLY. Only the tests, the smoke check and the
 * benchmark's CPU-baseline leg may load this file's library. The product
 * (the CUDA library and its Python binding) never calls it and shares no
 * code, header, table or helper with it.
 *
 * Source of the method: "Scalable Training of Mixture-of-Experts Models with
 * Megatron Core", §2 (Megatron-Core MoE Architecture): an MoE layer runs
 * Route (token hidden states -> expert logits -> probabilities -> top-k
 * experts; the router outputs routing weights and a token-expert
 * assignment), Dispatch (permute tokens by destination expert), Expert
 * Computation (each expert's FFN over its tokens; "SequentialMLP" runs one
 * expert at a time, which is how this file is organised) and Combine
 * (restore token order, add the shared expert's output). §5 (Selective
 * precision) keeps the router in FP32; here everything is fp64.
 *
 * Readings where the pages are silent (the layer's formulas are not printed):
 *   - score: softmax over all E logits, or the logistic sigmoid of each logit;
 *     the per-expert bias b is added to the logits before scoring and is used
 *     for both selection and gate values;
 *   - top-k: the k largest scores; slots ordered by score, descending; equal
 *     scores resolved towards the lower expert index;
 *   - gates: the selected scores divided by their sum (for softmax this equals
 *     the softmax over the selected logits);
 *   - expert FFN (SwiGLU): a = x Wg_e, u = x Wu_e, h = silu(a) * u,
 *     y_e = h Wd_e with silu(a) = a / (1 + exp(-a));
 *   - output: y_t = sum_j g_tj y_{e_tj}(x_t) + shared(x_t), the shared expert
 *     unweighted;
 *   - backward: the exact gradient of L = sum(dY * y) with the routing held
 *     fixed (top-k selection is piecewise constant); no gradient reaches b.
 *
 * Layouts (row-major): x T*H, Wr H*E, b E, Wg/Wu E*H*F, Wd E*F*H,
 * Wsg/Wsu H*Fs, Wsd Fs*H, topk and gates T*k, Yp and dXp R*H with R = T*k.
 *
 * Every function returns 0 on success and -1 on a bad argument.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define SCORE_SOFTMAX 0
#define SCORE_SIGMOID 1

static double silu(double a) { return a / (1.0 + exp(-a)); }
static double sigm(double a) { return 1.0 / (1.0 + exp(-a)); }
/* d silu / da = s(a) (1 + a (1 - s(a))) */
static double dsilu(double a) {
    double s = sigm(a);
    return s * (1.0 + a * (1.0 - s));
}

/* ------------------------------------------------------------------ Route */
/*
 * Route (§2, "Route"): logits z = x Wr + b, scores, top-k, gates.
 *
 * replay (optional, with replay_topk): for tokens with replay[t] != 0 the
 * selection and its slot order are taken from replay_topk instead of being
 * recomputed ("Router replay" in §10 records an assignment and enforces it).
 * Gates are still the oracle's own, from its own scores.
 *
 * gap_set[t]  = relative gap between the k-th and (k+1)-th largest score
 *               (+HUGE_VAL when k == E);
 * gap_order[t] = smallest relative gap between consecutive scores among the
 *               top k (+HUGE_VAL when k == 1).
 */
int oracle_route(int T, int H, int E, int k, int score_fn,
                 const double* x, const double* Wr, const double* b,
                 const int* replay_topk, const unsigned char* replay,
                 double* logits, double* scores, int* topk, double* gates,
                 double* gap_set, double* gap_order)
{
    if (T < 0 || H <= 0 || E <= 0 || E > 1024 || k <= 0 || k > E) return -1;
    if (score_fn != SCORE_SOFTMAX && score_fn != SCORE_SIGMOID) return -1;
#pragma omp parallel for schedule(static)
    for (int t = 0; t < T; ++t) {
        double* z = logits + (size_t)t * E;
        double* s = scores + (size_t)t * E;
        for (int e = 0; e < E; ++e) {
            double acc = 0.0;
            for (int h = 0; h < H; ++h) acc += x[(size_t)t * H + h] * Wr[(size_t)h * E + e];
            z[e] = acc + (b ? b[e] : 0.0);
        }
        if (score_fn == SCORE_SOFTMAX) {
            double zmax = z[0];
            for (int e = 1; e < E; ++e) if (z[e] > zmax) zmax = z[e];
            double den = 0.0;
            for (int e = 0; e < E; ++e) den += exp(z[e] - zmax);
            for (int e = 0; e < E; ++e) s[e] = exp(z[e] - zmax) / den;
        } else {
            for (int e = 0; e < E; ++e) s[e] = sigm(z[e]);
        }
        /* k+1 rounds of "largest remaining score, lower index on equality" */
        int order[1024];
        int nsel = (k < E) ? k + 1 : k;
        unsigned char taken[1024];
        memset(taken, 0, (size_t)E);
        for (int r = 0; r < nsel; ++r) {
            int best = -1;
            for (int e = 0; e < E; ++e)
                if (!taken[e] && (best < 0 || s[e] > s[best])) best = e;
            taken[best] = 1;
            order[r] = best;
        }
        double gs = HUGE_VAL, go = HUGE_VAL;
        if (k < E) gs = (s[order[k - 1]] - s[order[k]]) / fabs(s[order[k - 1]]);
        for (int r = 0; r + 1 < k; ++r) {
            double g = (s[order[r]] - s[order[r + 1]]) / fabs(s[order[r]]);
            if (g < go) go = g;
        }
        gap_set[t] = gs;
        gap_order[t] = go;
        int* sel = topk + (size_t)t * k;
        if (replay && replay[t]) {
            for (int j = 0; j < k; ++j) sel[j] = replay_topk[(size_t)t * k + j];
        } else {
            for (int j = 0; j < k; ++j) sel[j] = order[j];
        }
        double den = 0.0;
        for (int j = 0; j < k; ++j) den += s[sel[j]];
        for (int j = 0; j < k; ++j) gates[(size_t)t * k + j] = s[sel[j]] / den;
    }
    return 0;
}

/* --------------------------------------------------------------- Dispatch */
/*
 * Dispatch (§2, "Dispatch"): group the T*k (token, slot) pairs by expert.
 * counts[e] = number of tokens that chose e; offsets = exclusive prefix sum
 * (E+1 entries). Rows are ordered by expert, then by token. row_of[t*k+j] is
 * the row of pair (t, j); slot_of[row] = t*k + j is its inverse.
 */
int oracle_dispatch(int T, int E, int k, const int* topk,
                    int* counts, int* offsets, int* row_of, int* slot_of)
{
    if (T < 0 || E <= 0 || k <= 0) return -1;
    for (int e = 0; e < E; ++e) counts[e] = 0;
    for (int i = 0; i < T * k; ++i) {
        if (topk[i] < 0 || topk[i] >= E) return -1;
        counts[topk[i]] += 1;
    }
    offsets[0] = 0;
    for (int e = 0; e < E; ++e) offsets[e + 1] = offsets[e] + counts[e];
    int row = 0;
    for (int e = 0; e < E; ++e)
        for (int t = 0; t < T; ++t)
            for (int j = 0; j < k; ++j)
                if (topk[(size_t)t * k + j] == e) {
                    row_of[(size_t)t * k + j] = row;
                    slot_of[row] = t * k + j;
                    ++row;
                }
    return 0;
}

/* ------------------------------------------------------- one expert (SwiGLU) */
/* For M rows X (M*H): A = X Wg, U = X Wu (M*F), Hh = silu(A) * U, Y = Hh Wd. */
static void swiglu_forward(int M, int H, int F, const double* X,
                           const double* Wg, const double* Wu, const double* Wd,
                           double* A, double* U, double* Hh, double* Y)
{
#pragma omp parallel for schedule(static)
    for (int m = 0; m < M; ++m) {
        for (int f = 0; f < F; ++f) {
            double a = 0.0, u = 0.0;
            for (int h = 0; h < H; ++h) {
                a += X[(size_t)m * H + h] * Wg[(size_t)h * F + f];
                u += X[(size_t)m * H + h] * Wu[(size_t)h * F + f];
            }
            A[(size_t)m * F + f] = a;
            U[(size_t)m * F + f] = u;
            Hh[(size_t)m * F + f] = silu(a) * u;
        }
        for (int h = 0; h < H; ++h) {
            double acc = 0.0;
            for (int f = 0; f < F; ++f) acc += Hh[(size_t)m * F + f] * Wd[(size_t)f * H + h];
            Y[(size_t)m * H + h] = acc;
        }
    }
}

/*
 * Backward of one expert over M rows, given dY (M*H) for its output and the
 * forward intermediates: dH = dY Wd^T, dA = dH * U * silu'(A),
 * dU = dH * silu(A); dWd = Hh^T dY, dWg = X^T dA, dWu = X^T dU,
 * dX = dA Wg^T + dU Wu^T. Weight gradients are overwritten.
 */
static void swiglu_backward(int M, int H, int F, const double* X,
                            const double* Wg, const double* Wu, const double* Wd,
                            const double* A, const double* U, const double* Hh,
                            const double* dY, double* dX,
                            double* dWg, double* dWu, double* dWd)
{
    double* dA = (double*)malloc(sizeof(double) * (size_t)(M > 0 ? M : 1) * F);
    double* dU = (double*)malloc(sizeof(double) * (size_t)(M > 0 ? M : 1) * F);
#pragma omp parallel for schedule(static)
    for (int m = 0; m < M; ++m) {
        for (int f = 0; f < F; ++f) {
            double dh = 0.0;
            for (int h = 0; h < H; ++h) dh += dY[(size_t)m * H + h] * Wd[(size_t)f * H + h];
            double a = A[(size_t)m * F + f];
            dA[(size_t)m * F + f] = dh * U[(size_t)m * F + f] * dsilu(a);
            dU[(size_t)m * F + f] = dh * silu(a);
        }
        for (int h = 0; h < H; ++h) {
            double acc = 0.0;
            for (int f = 0; f < F; ++f)
                acc += dA[(size_t)m * F + f] * Wg[(size_t)h * F + f]
                     + dU[(size_t)m * F + f] * Wu[(size_t)h * F + f];
            dX[(size_t)m * H + h] = acc;
        }
    }
#pragma omp parallel for schedule(static)
    for (int f = 0; f < F; ++f)
        for (int h = 0; h < H; ++h) {
            double acc = 0.0;
            for (int m = 0; m < M; ++m) acc += Hh[(size_t)m * F + f] * dY[(size_t)m * H + h];
            dWd[(size_t)f * H + h] = acc;
        }
#pragma omp parallel for schedule(static)
    for (int h = 0; h < H; ++h)
        for (int f = 0; f < F; ++f) {
            double ag = 0.0, au = 0.0;
            for (int m = 0; m < M; ++m) {
                ag += X[(size_t)m * H + h] * dA[(size_t)m * F + f];
                au += X[(size_t)m * H + h] * dU[(size_t)m * F + f];
            }
            dWg[(size_t)h * F + f] = ag;
            dWu[(size_t)h * F + f] = au;
        }
    free(dA);
    free(dU);
}

/* ---------------------------------------------------------------- Forward */
/*
 * Forward of the layer with a given routing (topk, gates): Dispatch, then
 * Expert Computation one expert at a time, then Combine (§2).
 * Yp (optional, R*H) receives the unweighted expert outputs in dispatch
 * order; y (T*H) the layer output.
 */
/*
 * keep (optional, T*k): capacity-limited dropping ("Scalable Training of
 * Mixture-of-Experts Models with Megatron Core", §7 Load Balancing); a slot
 * with keep = 0 is dropped: its expert output does not enter y.
 */
int oracle_forward(int T, int H, int E, int k, int F, int Fs,
                   const double* x, const double* Wg, const double* Wu, const double* Wd,
                   const double* Wsg, const double* Wsu, const double* Wsd,
                   const int* topk, const double* gates, double* y, double* Yp_out,
                   const unsigned char* keep)
{
    if (T <= 0 || H <= 0 || E <= 0 || k <= 0 || k > E || F <= 0 || Fs < 0) return -1;
    const int R = T * k;
    int* counts = (int*)malloc(sizeof(int) * E);
    int* offsets = (int*)malloc(sizeof(int) * (E + 1));
    int* row_of = (int*)malloc(sizeof(int) * R);
    int* slot_of = (int*)malloc(sizeof(int) * R);
    if (oracle_dispatch(T, E, k, topk, counts, offsets, row_of, slot_of)) return -1;
    double* Xp = (double*)malloc(sizeof(double) * (size_t)R * H);
    double* Yp = (double*)malloc(sizeof(double) * (size_t)R * H);
    /* permute */
    for (int r = 0; r < R; ++r)
        memcpy(Xp + (size_t)r * H, x + (size_t)(slot_of[r] / k) * H, sizeof(double) * H);
    /* experts, one at a time */
    for (int e = 0; e < E; ++e) {
        int M = counts[e];
        if (M == 0) continue;
        double* A = (double*)malloc(sizeof(double) * (size_t)M * F);
        double* U = (double*)malloc(sizeof(double) * (size_t)M * F);
        double* Hh = (double*)malloc(sizeof(double) * (size_t)M * F);
        swiglu_forward(M, H, F, Xp + (size_t)offsets[e] * H,
                       Wg + (size_t)e * H * F, Wu + (size_t)e * H * F, Wd + (size_t)e * F * H,
                       A, U, Hh, Yp + (size_t)offsets[e] * H);
        free(A); free(U); free(Hh);
    }
    /* combine: restore token order, weight by gates, add the shared expert */
    for (int t = 0; t < T; ++t)
        for (int h = 0; h < H; ++h) {
            double acc = 0.0;
            for (int j = 0; j < k; ++j) {
                if (keep && !keep[(size_t)t * k + j]) continue;
                acc += gates[(size_t)t * k + j] * Yp[(size_t)row_of[(size_t)t * k + j] * H + h];
            }
            y[(size_t)t * H + h] = acc;
        }
    if (Fs > 0) {
        double* A = (double*)malloc(sizeof(double) * (size_t)T * Fs);
        double* U = (double*)malloc(sizeof(double) * (size_t)T * Fs);
        double* Hh = (double*)malloc(sizeof(double) * (size_t)T * Fs);
        double* Ys = (double*)malloc(sizeof(double) * (size_t)T * H);
        swiglu_forward(T, H, Fs, x, Wsg, Wsu, Wsd, A, U, Hh, Ys);
        for (size_t i = 0; i < (size_t)T * H; ++i) y[i] += Ys[i];
        free(A); free(U); free(Hh); free(Ys);
    }
    if (Yp_out) memcpy(Yp_out, Yp, sizeof(double) * (size_t)R * H);
    free(Xp); free(Yp); free(counts); free(offsets); free(row_of); free(slot_of);
    return 0;
}

/* ------------------------------------------------------- router backward */
/*
 * dz for one token from the gate gradients dg (k values): gates
 * g_j = s_j / sum_i s_i over the selected set S.
 *   softmax: g is the softmax over the selected logits, so
 *            dz_j = g_j (dg_j - sum_i g_i dg_i);
 *   sigmoid: dL/ds_j = (dg_j - sum_i g_i dg_i) / sum_i s_i and
 *            ds_j/dz_j = s_j (1 - s_j).
 * Experts outside S get dz = 0 (the gates do not depend on their logits).
 */
static void router_dz(int k, int score_fn, const int* sel, const double* g, const double* s_all,
                      const double* dg, double* dz)
{
    double gd = 0.0;
    for (int j = 0; j < k; ++j) gd += g[j] * dg[j];
    if (score_fn == SCORE_SOFTMAX) {
        for (int j = 0; j < k; ++j) dz[j] = g[j] * (dg[j] - gd);
    } else {
        double ssum = 0.0;
        for (int j = 0; j < k; ++j) ssum += s_all[sel[j]];
        for (int j = 0; j < k; ++j) {
            double s = s_all[sel[j]];
            dz[j] = s * (1.0 - s) * (dg[j] - gd) / ssum;
        }
    }
}

/* --------------------------------------------------------------- Backward */
/*
 * Backward of the layer for L = sum(dY * y), routing fixed. scores is the
 * T*E output of oracle_route (softmax probabilities or sigmoids).
 * Outputs (overwritten): dX T*H, dWr H*E, dWg/dWu E*H*F, dWd E*F*H,
 * dWsg/dWsu H*Fs, dWsd Fs*H (when Fs > 0), dg T*k (optional).
 * Experts that received no token get zero weight gradients.
 */
int oracle_backward(int T, int H, int E, int k, int F, int Fs, int score_fn,
                    const double* x, const double* Wr,
                    const double* Wg, const double* Wu, const double* Wd,
                    const double* Wsg, const double* Wsu, const double* Wsd,
                    const int* topk, const double* gates, const double* scores,
                    const double* dY,
                    double* dX, double* dWr, double* dWg, double* dWu, double* dWd,
                    double* dWsg, double* dWsu, double* dWsd, double* dg_out,
                    const unsigned char* keep)
{
    if (T <= 0 || H <= 0 || E <= 0 || k <= 0 || k > E || k > 1024 || F <= 0 || Fs < 0) return -1;
    const int R = T * k;
    int* counts = (int*)malloc(sizeof(int) * E);
    int* offsets = (int*)malloc(sizeof(int) * (E + 1));
    int* row_of = (int*)malloc(sizeof(int) * R);
    int* slot_of = (int*)malloc(sizeof(int) * R);
    if (oracle_dispatch(T, E, k, topk, counts, offsets, row_of, slot_of)) return -1;
    double* Xp = (double*)malloc(sizeof(double) * (size_t)R * H);
    double* Yp = (double*)malloc(sizeof(double) * (size_t)R * H);
    double* dYp = (double*)malloc(sizeof(double) * (size_t)R * H);
    double* dXp = (double*)malloc(sizeof(double) * (size_t)R * H);
    double* dg = (double*)malloc(sizeof(double) * (size_t)R);
    for (int r = 0; r < R; ++r)
        memcpy(Xp + (size_t)r * H, x + (size_t)(slot_of[r] / k) * H, sizeof(double) * H);

    /* recompute the forward per expert, then its backward */
    for (int e = 0; e < E; ++e) {
        int M = counts[e];
        double* dWg_e = dWg + (size_t)e * H * F;
        double* dWu_e = dWu + (size_t)e * H * F;
        double* dWd_e = dWd + (size_t)e * F * H;
        if (M == 0) {
            memset(dWg_e, 0, sizeof(double) * (size_t)H * F);
            memset(dWu_e, 0, sizeof(double) * (size_t)H * F);
            memset(dWd_e, 0, sizeof(double) * (size_t)F * H);
            continue;
        }
        const double* Xe = Xp + (size_t)offsets[e] * H;
        double* A = (double*)malloc(sizeof(double) * (size_t)M * F);
        double* U = (double*)malloc(sizeof(double) * (size_t)M * F);
        double* Hh = (double*)malloc(sizeof(double) * (size_t)M * F);
        swiglu_forward(M, H, F, Xe, Wg + (size_t)e * H * F, Wu + (size_t)e * H * F,
                       Wd + (size_t)e * F * H, A, U, Hh, Yp + (size_t)offsets[e] * H);
        /* gate gradient and the gate-scaled output gradient of each row; a
         * dropped slot is not part of y: no output gradient, dg = 0 */
        for (int m = 0; m < M; ++m) {
            int r = offsets[e] + m;
            int t = slot_of[r] / k;
            const int kept = !keep || keep[slot_of[r]];
            double g = kept ? gates[slot_of[r]] : 0.0;
            double acc = 0.0;
            for (int h = 0; h < H; ++h) {
                acc += dY[(size_t)t * H + h] * Yp[(size_t)r * H + h];
                dYp[(size_t)r * H + h] = g * dY[(size_t)t * H + h];
            }
            dg[slot_of[r]] = kept ? acc : 0.0;
        }
        swiglu_backward(M, H, F, Xe, Wg + (size_t)e * H * F, Wu + (size_t)e * H * F,
                        Wd + (size_t)e * F * H, A, U, Hh, dYp + (size_t)offsets[e] * H,
                        dXp + (size_t)offsets[e] * H, dWg_e, dWu_e, dWd_e);
        free(A); free(U); free(Hh);
    }

    /* router: dz (dense T*E), dWr = x^T dz, dX_router = dz Wr^T */
    double* dz = (double*)calloc((size_t)T * E, sizeof(double));
    for (int t = 0; t < T; ++t) {
        double dzs[1024];
        router_dz(k, score_fn, topk + (size_t)t * k, gates + (size_t)t * k,
                  scores + (size_t)t * E, dg + (size_t)t * k, dzs);
        for (int j = 0; j < k; ++j) dz[(size_t)t * E + topk[(size_t)t * k + j]] = dzs[j];
    }
#pragma omp parallel for schedule(static)
    for (int h = 0; h < H; ++h)
        for (int e = 0; e < E; ++e) {
            double acc = 0.0;
            for (int t = 0; t < T; ++t) acc += x[(size_t)t * H + h] * dz[(size_t)t * E + e];
            dWr[(size_t)h * E + e] = acc;
        }
    /* dX = sum over the token's rows of dXp + router term */
#pragma omp parallel for schedule(static)
    for (int t = 0; t < T; ++t)
        for (int h = 0; h < H; ++h) {
            double acc = 0.0;
            for (int j = 0; j < k; ++j) acc += dXp[(size_t)row_of[(size_t)t * k + j] * H + h];
            for (int e = 0; e < E; ++e) acc += dz[(size_t)t * E + e] * Wr[(size_t)h * E + e];
            dX[(size_t)t * H + h] = acc;
        }
    /* shared expert: every token, unweighted, so its output gradient is dY */
    if (Fs > 0) {
        double* A = (double*)malloc(sizeof(double) * (size_t)T * Fs);
        double* U = (double*)malloc(sizeof(double) * (size_t)T * Fs);
        double* Hh = (double*)malloc(sizeof(double) * (size_t)T * Fs);
        double* Ys = (double*)malloc(sizeof(double) * (size_t)T * H);
        double* dXs = (double*)malloc(sizeof(double) * (size_t)T * H);
        swiglu_forward(T, H, Fs, x, Wsg, Wsu, Wsd, A, U, Hh, Ys);
        swiglu_backward(T, H, Fs, x, Wsg, Wsu, Wsd, A, U, Hh, dY, dXs, dWsg, dWsu, dWsd);
        for (size_t i = 0; i < (size_t)T * H; ++i) dX[i] += dXs[i];
        free(A); free(U); free(Hh); free(Ys); free(dXs);
    }
    if (dg_out) memcpy(dg_out, dg, sizeof(double) * (size_t)R);
    free(dz); free(Xp); free(Yp); free(dYp); free(dXp); free(dg);
    free(counts); free(offsets); free(row_of); free(slot_of);
    return 0;
}

/* ------------------------------------------------- sampled, large layers */
/*
 * The two functions below compute single outputs of the same definitions
 * without materialising the whole layer, for layers too large for the
 * functions above. Weights are read in their storage format and widened
 * exactly: wtype 0 = float32, 1 = bfloat16 bits (uint16). Per-expert weight
 * blocks are passed as pointer arrays (entries may be NULL for experts that
 * are not touched).
 */
static double ld(const void* p, int wtype, size_t i)
{
    if (wtype == 0) return (double)((const float*)p)[i];
    uint32_t bits = (uint32_t)((const uint16_t*)p)[i] << 16;
    float f;
    memcpy(&f, &bits, sizeof f);
    return (double)f;
}

/* Forward of one expert for one token: a, u, hh (F each) and y (H). */
static void token_expert_fwd(int H, int F, const double* xt, const void* Wg, const void* Wu,
                             const void* Wd, int wtype, double* a, double* u, double* hh,
                             double* y)
{
    for (int f = 0; f < F; ++f) {
        double sa = 0.0, su = 0.0;
        for (int h = 0; h < H; ++h) {
            sa += xt[h] * ld(Wg, wtype, (size_t)h * F + f);
            su += xt[h] * ld(Wu, wtype, (size_t)h * F + f);
        }
        a[f] = sa; u[f] = su; hh[f] = silu(sa) * su;
    }
    for (int h = 0; h < H; ++h) y[h] = 0.0;
    for (int f = 0; f < F; ++f)
        for (int h = 0; h < H; ++h) y[h] += hh[f] * ld(Wd, wtype, (size_t)f * H + h);
}

/* dX contribution of one expert for one token, given that row's output
 * gradient dyr (H): dh = Wd dyr, dA, dU, then dA Wg^T + dU Wu^T into dxt. */
static void token_expert_dx(int H, int F, const void* Wg, const void* Wu, const void* Wd, int wtype,
                            const double* a, const double* u, const double* dyr, double* dxt)
{
    for (int f = 0; f < F; ++f) {
        double dh = 0.0;
        for (int h = 0; h < H; ++h) dh += dyr[h] * ld(Wd, wtype, (size_t)f * H + h);
        double dA = dh * u[f] * dsilu(a[f]);
        double dU = dh * silu(a[f]);
        for (int h = 0; h < H; ++h)
            dxt[h] += dA * ld(Wg, wtype, (size_t)h * F + f) + dU * ld(Wu, wtype, (size_t)h * F + f);
    }
}

/*
 * Output rows y[t] and dX[t] (and dg[t, :]) for n listed tokens.
 * xs, dYs: n*H fp64 rows of those tokens; topk, gates: n*k; scores: n*E
 * (from oracle_route on the same rows). Wg_e/Wu_e/Wd_e: E pointers to the
 * H*F, H*F, F*H blocks; Ws*: the shared expert (Fs may be 0).
 * Outputs: y n*H, dX n*H, dg n*k.
 */
int oracle_token_rows(int n, int H, int E, int k, int F, int Fs, int score_fn, int wtype,
                      const double* xs, const double* dYs, const double* Wr,
                      const void* const* Wg_e, const void* const* Wu_e, const void* const* Wd_e,
                      const void* Wsg, const void* Wsu, const void* Wsd,
                      const int* topk, const double* gates, const double* scores,
                      double* y, double* dX, double* dg)
{
    if (n < 0 || H <= 0 || E <= 0 || k <= 0 || k > E || k > 1024 || F <= 0 || Fs < 0) return -1;
    int bad = 0;
#pragma omp parallel for schedule(dynamic, 1) reduction(| : bad)
    for (int i = 0; i < n; ++i) {
        const double* xt = xs + (size_t)i * H;
        const double* dyt = dYs + (size_t)i * H;
        int Fm = F > Fs ? F : Fs;
        double* a = (double*)malloc(sizeof(double) * Fm);
        double* u = (double*)malloc(sizeof(double) * Fm);
        double* hh = (double*)malloc(sizeof(double) * Fm);
        double* ye = (double*)malloc(sizeof(double) * H);
        double* dyr = (double*)malloc(sizeof(double) * H);
        double* yt = y + (size_t)i * H;
        double* dxt = dX + (size_t)i * H;
        const int* sel = topk + (size_t)i * k;
        const double* g = gates + (size_t)i * k;
        double dgt[1024], dz[1024];
        for (int h = 0; h < H; ++h) { yt[h] = 0.0; dxt[h] = 0.0; }
        for (int j = 0; j < k; ++j) {
            int e = sel[j];
            if (e < 0 || e >= E || !Wg_e[e] || !Wu_e[e] || !Wd_e[e]) { bad = 1; continue; }
            token_expert_fwd(H, F, xt, Wg_e[e], Wu_e[e], Wd_e[e], wtype, a, u, hh, ye);
            double acc = 0.0;
            for (int h = 0; h < H; ++h) {
                yt[h] += g[j] * ye[h];
                acc += dyt[h] * ye[h];
                dyr[h] = g[j] * dyt[h];
            }
            dgt[j] = acc;
            token_expert_dx(H, F, Wg_e[e], Wu_e[e], Wd_e[e], wtype, a, u, dyr, dxt);
        }
        router_dz(k, score_fn, sel, g, scores + (size_t)i * E, dgt, dz);
        for (int j = 0; j < k; ++j) {
            dg[(size_t)i * k + j] = dgt[j];
            for (int h = 0; h < H; ++h) dxt[h] += dz[j] * Wr[(size_t)h * E + sel[j]];
        }
        if (Fs > 0) {
            token_expert_fwd(H, Fs, xt, Wsg, Wsu, Wsd, wtype, a, u, hh, ye);
            for (int h = 0; h < H; ++h) yt[h] += ye[h];
            token_expert_dx(H, Fs, Wsg, Wsu, Wsd, wtype, a, u, dyt, dxt);
        }
        free(a); free(u); free(hh); free(ye); free(dyr);
    }
    return bad ? -1 : 0;
}

/*
 * Single weight-gradient entries. which: 0 dWg[e][i][j] (i = h, j = f),
 * 1 dWu[e][i][j], 2 dWd[e][i][j] (i = f, j = h), 3 dWsg[i][j], 4 dWsu[i][j],
 * 5 dWsd[i][j]. Each is a sum over the tokens that chose expert e (all
 * tokens for the shared expert) of that token's contribution.
 * x, dY: T*H fp64; topk, gates: T*k of the whole layer.
 */
int oracle_dw_entries(int T, int H, int E, int k, int F, int Fs, int wtype,
                      const double* x, const double* dY,
                      const void* const* Wg_e, const void* const* Wu_e, const void* const* Wd_e,
                      const void* Wsg, const void* Wsu, const void* Wsd,
                      const int* topk, const double* gates,
                      int n, const int* which, const int* ee, const int* ii, const int* jj,
                      double* out)
{
    if (T <= 0 || H <= 0 || E <= 0 || k <= 0 || F <= 0 || Fs < 0) return -1;
    int bad = 0;
#pragma omp parallel for schedule(dynamic, 1) reduction(| : bad)
    for (int q = 0; q < n; ++q) {
        int w = which[q], e = ee[q], i = ii[q], j = jj[q];
        int shared = w >= 3;
        int Fw = shared ? Fs : F;
        const void *Wg = shared ? Wsg : (e >= 0 && e < E ? Wg_e[e] : NULL);
        const void *Wu = shared ? Wsu : (e >= 0 && e < E ? Wu_e[e] : NULL);
        const void *Wd = shared ? Wsd : (e >= 0 && e < E ? Wd_e[e] : NULL);
        if (!Wg || !Wu || !Wd || Fw <= 0) { bad = 1; out[q] = NAN; continue; }
        int kind = w % 3;
        double acc = 0.0;
        for (int t = 0; t < T; ++t) {
            double g = 1.0;
            if (!shared) {
                int hit = -1;
                for (int s = 0; s < k; ++s) if (topk[(size_t)t * k + s] == e) hit = s;
                if (hit < 0) continue;
                g = gates[(size_t)t * k + hit];
            }
            const double* xt = x + (size_t)t * H;
            const double* dyt = dY + (size_t)t * H;
            int f = (kind == 2) ? i : j;
            double a = 0.0, u = 0.0;
            for (int h = 0; h < H; ++h) {
                a += xt[h] * ld(Wg, wtype, (size_t)h * Fw + f);
                u += xt[h] * ld(Wu, wtype, (size_t)h * Fw + f);
            }
            if (kind == 2) {
                acc += silu(a) * u * g * dyt[j];
            } else {
                double dh = 0.0;
                for (int h = 0; h < H; ++h) dh += g * dyt[h] * ld(Wd, wtype, (size_t)f * H + h);
                double d = (kind == 0) ? dh * u * dsilu(a) : dh * silu(a);
                acc += xt[i] * d;
            }
        }
        out[q] = acc;
    }
    return bad ? -1 : 0;
}

/* ====================================================================== */
/* Blockwise FP8 (E4M3) variant.                                           */
/*                                                                         */
/* "Scalable Training of Mixture-of-Experts Models with Megatron Core", §5 */
/* (Platform-specific recipes): blockwise FP8 scales 1x128 activation and  */
/* gradient tiles and 128x128 weight blocks; §5 (Selective precision)      */
/* keeps the router in higher precision.                                   */
/*                                                                         */
/* Readings (the pages give no formula):                                   */
/*   - E4M3 is the OCP FP8 format: 1 sign, 4 exponent (bias 7), 3 mantissa */
/*     bits, subnormals, no infinities, S.1111.111 = NaN, largest finite   */
/*     magnitude 448. Encoding rounds to nearest, ties to even, and        */
/*     saturates to +-448.                                                 */
/*   - block scale s = amax / 448 computed in fp32 (s = 1 when amax = 0);  */
/*     a value v is stored as q = E4M3(fp32(v / s)) and read as q * s.     */
/*   - in every GEMM C = A B (contraction over K), A -- whose rows are the */
/*     output rows -- is quantised in 1x128 blocks along K, and B in       */
/*     128x128 blocks. So activations and gradients feeding fprop/dgrad    */
/*     are 1x128 along their feature dimension, weights 128x128, and the   */
/*     weight-gradient GEMMs (K = the expert's tokens) quantise the left   */
/*     operand (Xp^T, h^T) per feature column over 128-token blocks and    */
/*     the right one (dA, dU, dYp) in 128x128 (tokens x features) blocks,  */
/*     token blocks counted from the start of each expert's segment.       */
/*   - the router, gates and gate gradients stay in full precision;        */
/*   - the FP8 workload fixes bf16 outputs and gradients: every GEMM       */
/*     output (a, u, y, dA, dU), h = silu(a) u (formed from the GEMM       */
/*     outputs before they are stored) and the gate-scaled output gradient */
/*     g dY are bf16 values (round to nearest even) when they are stored   */
/*     and quantised for the next GEMM; dA, dU use the stored a, u.        */
/* ====================================================================== */

double oracle_e4m3_decode(unsigned char c)
{
    int s = c >> 7, e = (c >> 3) & 15, m = c & 7;
    if (e == 15 && m == 7) return NAN;
    double v = (e == 0) ? ldexp(m / 8.0, -6) : ldexp(1.0 + m / 8.0, e - 7);
    return s ? -v : v;
}

/* Nearest E4M3 code to f (ties to the even code), saturating to +-448.
 * Below 2^-6 the values are the subnormals m 2^-9 (m = 0..7; m = 8 is the
 * smallest normal, code 8); above, a = 2^E (1 + m/8) with E = floor(log2 a),
 * the code (E + 7) << 3 | m, a mantissa that rounds up to 8 carrying into
 * the exponent. Every step is exact in double (power-of-two scaling of a
 * float), rint rounds half to even. */
unsigned char oracle_e4m3_encode(float f)
{
    if (f != f) return 0x7F;
    unsigned char sign = signbit(f) ? 0x80 : 0x00;
    double a = fabs((double)f);
    if (a >= 448.0) return sign | 0x7E;
    if (a < 0.015625) return sign | (unsigned char)rint(ldexp(a, 9));
    int p;
    frexp(a, &p);                          /* a = g 2^p, g in [0.5, 1) */
    int E = p - 1;
    int m = (int)rint((ldexp(a, -E) - 1.0) * 8.0);
    int code = ((E + 7) << 3) + m;         /* m = 8 carries into the exponent */
    if (code > 0x7E) code = 0x7E;
    return sign | (unsigned char)code;
}

/* v rounded to bfloat16 (via fp32, ties to even) */
static double bf16r(double v)
{
    float f = (float)v;
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    if ((u & 0x7f800000u) != 0x7f800000u) {
        u += 0x7fffu + ((u >> 16) & 1u);
        u &= 0xffff0000u;
        memcpy(&f, &u, sizeof f);
    }
    return (double)f;
}

/* fp32 scale of a block with largest magnitude amax */
static float block_scale(float amax) { return amax == 0.0f ? 1.0f : amax / 448.0f; }

/*
 * Quantise-dequantise the n values v[i*stride] (one block): returns the
 * values q*s in place (fp64) and optionally the codes and the scale.
 */
static void qdq_block(double* v, int n, long stride, unsigned char* codes, float* scale)
{
    float amax = 0.0f;
    for (int i = 0; i < n; ++i) {
        float f = fabsf((float)v[(long)i * stride]);
        if (f > amax) amax = f;
    }
    float s = block_scale(amax);
    for (int i = 0; i < n; ++i) {
        float f = (float)v[(long)i * stride];
        unsigned char q = oracle_e4m3_encode(f / s);
        if (codes) codes[(long)i * stride] = q;
        v[(long)i * stride] = oracle_e4m3_decode(q) * (double)s;
    }
    if (scale) *scale = s;
}

/* 1x128 blocks along the rows of an M x K matrix (K a multiple of 128). */
static void qdq_rows(int M, int K, double* X)
{
#pragma omp parallel for schedule(static)
    for (int m = 0; m < M; ++m)
        for (int k0 = 0; k0 < K; k0 += 128) qdq_block(X + (long)m * K + k0, 128, 1, NULL, NULL);
}

/* Per column, blocks of 128 consecutive rows (the last block may be short). */
static void qdq_cols(int M, int N, double* X)
{
#pragma omp parallel for schedule(static)
    for (int n = 0; n < N; ++n)
        for (int m0 = 0; m0 < M; m0 += 128) {
            int len = M - m0 < 128 ? M - m0 : 128;
            qdq_block(X + (long)m0 * N + n, len, N, NULL, NULL);
        }
}

/* 128x128 blocks of an R x C matrix (edge blocks may be smaller). */
static void qdq_tiles(int R, int C, double* X)
{
    for (int r0 = 0; r0 < R; r0 += 128)
        for (int c0 = 0; c0 < C; c0 += 128) {
            int rl = R - r0 < 128 ? R - r0 : 128, cl = C - c0 < 128 ? C - c0 : 128;
            float amax = 0.0f;
            for (int r = 0; r < rl; ++r)
                for (int c = 0; c < cl; ++c) {
                    float f = fabsf((float)X[(long)(r0 + r) * C + c0 + c]);
                    if (f > amax) amax = f;
                }
            float s = block_scale(amax);
            for (int r = 0; r < rl; ++r)
                for (int c = 0; c < cl; ++c) {
                    double* p = &X[(long)(r0 + r) * C + c0 + c];
                    *p = oracle_e4m3_decode(oracle_e4m3_encode((float)*p / s)) * (double)s;
                }
        }
}

/* Quantised bytes and scales of one matrix, for comparison with a GPU quantiser.
 * mode 0: 1x128 along rows (scales M x K/128); 1: 128x128 tiles (scales
 * ceil(M/128) x ceil(K/128)); 2: per column over 128-row blocks (scales
 * ceil(M/128) x K). Input in fp32. */
int oracle_fp8_quantize(int M, int K, int mode, const float* X, unsigned char* codes, float* scales)
{
    if (M <= 0 || K <= 0 || mode < 0 || mode > 2) return -1;
    double* v = (double*)malloc(sizeof(double) * (size_t)M * K);
    for (size_t i = 0; i < (size_t)M * K; ++i) v[i] = X[i];
    if (mode == 0) {
        if (K % 128) { free(v); return -1; }
        for (int m = 0; m < M; ++m)
            for (int k0 = 0; k0 < K; k0 += 128)
                qdq_block(v + (long)m * K + k0, 128, 1, codes + (long)m * K + k0, scales + (long)m * (K / 128) + k0 / 128);
    } else if (mode == 1) {
        int nc = (K + 127) / 128;
        for (int r0 = 0; r0 < M; r0 += 128)
            for (int c0 = 0; c0 < K; c0 += 128) {
                int rl = M - r0 < 128 ? M - r0 : 128, cl = K - c0 < 128 ? K - c0 : 128;
                float amax = 0.0f;
                for (int r = 0; r < rl; ++r)
                    for (int c = 0; c < cl; ++c) {
                        float f = fabsf(X[(long)(r0 + r) * K + c0 + c]);
                        if (f > amax) amax = f;
                    }
                float s = block_scale(amax);
                scales[(r0 / 128) * nc + c0 / 128] = s;
                for (int r = 0; r < rl; ++r)
                    for (int c = 0; c < cl; ++c)
                        codes[(long)(r0 + r) * K + c0 + c] = oracle_e4m3_encode(X[(long)(r0 + r) * K + c0 + c] / s);
            }
    } else {
        for (int n = 0; n < K; ++n)
            for (int m0 = 0; m0 < M; m0 += 128) {
                int len = M - m0 < 128 ? M - m0 : 128;
                qdq_block(v + (long)m0 * K + n, len, K, codes + (long)m0 * K + n, scales + (long)(m0 / 128) * K + n);
            }
    }
    free(v);
    return 0;
}

/* ---------------------------------------------------------------- MXFP8 */
/*
 * MXFP8 ("Scalable Training of Mixture-of-Experts Models with Megatron
 * Core", §5 Platform-specific recipes: MXFP8, the default FP8 recipe on
 * Blackwell, with 1x32 granularity). Every block of 32 consecutive values
 * along a GEMM's contraction dimension shares one power-of-two scale
 * 2^e, stored as an UE8M0 byte (e + 127); each value is stored as the
 * E4M3 code of v / 2^e (round to nearest even, saturating; the division by
 * a power of two is exact).
 * Reading of the scale (the pages give no rule): e is the smallest integer
 * with amax <= 448 * 2^e, so that no value of the block saturates, clamped
 * to the UE8M0 range [-127, 127]; an all-zero block takes e = -127.
 */
int oracle_mx_exponent(float amax)
{
    if (!(amax > 0.0f)) return -127;
    int p;
    double m = frexp((double)amax, &p);        /* amax = m 2^p, m in [0.5, 1) */
    /* 448 = 0.875 * 2^9: amax <= 448 2^e  <=>  m 2^p <= 0.875 2^(9 + e) */
    int e = (m <= 0.875) ? p - 9 : p - 8;
    if (e < -127) e = -127;
    if (e > 127) e = 127;
    return e;
}

/* Quantise-dequantise n values v[i*stride] as one MX block; optionally the
 * codes and the UE8M0 scale byte. */
static void mx_block(double* v, int n, long stride, unsigned char* codes, unsigned char* sc)
{
    float amax = 0.0f;
    for (int i = 0; i < n; ++i) {
        float f = fabsf((float)v[(long)i * stride]);
        if (f > amax) amax = f;
    }
    int e = oracle_mx_exponent(amax);
    for (int i = 0; i < n; ++i) {
        double q = ldexp((double)(float)v[(long)i * stride], -e);     /* exact */
        unsigned char c = oracle_e4m3_encode((float)q);
        if (codes) codes[(long)i * stride] = c;
        v[(long)i * stride] = ldexp(oracle_e4m3_decode(c), e);
    }
    if (sc) *sc = (unsigned char)(e + 127);
}

/* 1x32 blocks along the rows of an M x K matrix (K a multiple of 32). */
static void mx_rows(int M, int K, double* X)
{
#pragma omp parallel for schedule(static)
    for (int m = 0; m < M; ++m)
        for (int k0 = 0; k0 < K; k0 += 32) mx_block(X + (long)m * K + k0, 32, 1, NULL, NULL);
}

/* Per column, blocks of 32 consecutive rows (the last block may be short). */
static void mx_cols(int M, int N, double* X)
{
#pragma omp parallel for schedule(static)
    for (int n = 0; n < N; ++n)
        for (int m0 = 0; m0 < M; m0 += 32) {
            int len = M - m0 < 32 ? M - m0 : 32;
            mx_block(X + (long)m0 * N + n, len, N, NULL, NULL);
        }
}

/* MX codes and UE8M0 scale bytes of one fp32 matrix, for comparison with a
 * GPU quantiser. mode 0: 1x32 along rows (scales M x K/32); mode 1: per
 * column over 32-row blocks (scales ceil(M/32) x K). */
int oracle_mx_quantize(int M, int K, int mode, const float* X, unsigned char* codes, unsigned char* scales)
{
    if (M <= 0 || K <= 0 || mode < 0 || mode > 1) return -1;
    if (mode == 0 && K % 32) return -1;
    double* v = (double*)malloc(sizeof(double) * (size_t)M * K);
    for (size_t i = 0; i < (size_t)M * K; ++i) v[i] = X[i];
    if (mode == 0) {
        for (int m = 0; m < M; ++m)
            for (int k0 = 0; k0 < K; k0 += 32)
                mx_block(v + (long)m * K + k0, 32, 1, codes + (long)m * K + k0, scales + (long)m * (K / 32) + k0 / 32);
    } else {
        for (int n = 0; n < K; ++n)
            for (int m0 = 0; m0 < M; m0 += 32) {
                int len = M - m0 < 32 ? M - m0 : 32;
                mx_block(v + (long)m0 * K + n, len, K, codes + (long)m0 * K + n, scales + (long)(m0 / 32) * K + n);
            }
    }
    free(v);
    return 0;
}

/* ---------------------------------------------------------------- NVFP4 */
/*
 * NVFP4 ("Scalable Training of Mixture-of-Experts Models with Megatron
 * Core", §5 Platform-specific recipes: the framework also provides NVFP4 for
 * Blackwell; §5 Kernel and shape optimization: grouped quantisation ahead
 * of the grouped NVFP4 GEMMs). The pages give none of the recipe's
 * parameters; the reading here is the NVFP4 format itself, applied like the
 * MXFP8 recipe (1-D blocks along each GEMM's contraction dimension):
 *   - values E2M1: 1 sign, 2 exponent, 1 mantissa bit, magnitudes
 *     {0, 0.5, 1, 1.5, 2, 3, 4, 6}; encoding rounds to nearest, ties to the
 *     even code (mantissa bit 0), and saturates to +-6; every value keeps
 *     its sign bit, zero included (-0 and a negative value that rounds to
 *     zero are the code 8, as a signed-zero format conversion gives);
 *   - blocks of 16 consecutive values along K, each with an unsigned E4M3
 *     scale, plus one fp32 scale S per tensor, S = 2688 / amax (2688 =
 *     448 * 6: the tensor's largest block gets the largest E4M3 scale), S = 1
 *     for an all-zero tensor;
 *   - per block, in fp32 (each operation rounded to nearest even):
 *     a = max |v|, sb = E4M3(a * S / 6) (the product first),
 *     s = the value of sb, r = S / s, and each value is stored as
 *     E2M1(v * r) (all codes 0 when s = 0); it is read as q * s / S;
 *   - a "tensor" is one expert's operand of one grouped GEMM (grouped
 *     quantisation quantises each expert's part on its own), with the gate
 *     and up projections one tensor [Wg | Wu] and their gradients one tensor
 *     [dA | dU], as in a fused fc1 whose output is [a | u].
 */
double oracle_e2m1_decode(unsigned char c)
{
    static const double mag[8] = {0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0};
    double v = mag[c & 7];
    return (c & 8) ? -v : v;
}

/* E2M1 code (4 bits) of an fp32 value: nearest magnitude, ties to the even
 * code, saturating at 6, with the value's sign bit. */
unsigned char oracle_e2m1_encode(float f)
{
    double m = fabs((double)f);
    unsigned char c;
    if (m <= 0.25) c = 0;
    else if (m < 0.75) c = 1;
    else if (m <= 1.25) c = 2;
    else if (m < 1.75) c = 3;
    else if (m <= 2.5) c = 4;
    else if (m < 3.5) c = 5;
    else if (m <= 5.0) c = 6;
    else c = 7;
    return (unsigned char)(c | (signbit(f) ? 8 : 0));
}

/* per-tensor scale of a tensor whose largest magnitude is amax */
float oracle_nv_tensor_scale(float amax) { return amax > 0.0f ? 2688.0f / amax : 1.0f; }

/* Quantise-dequantise n values v[i*stride] as one NVFP4 block of a tensor
 * with scale S; optionally the codes (one per byte) and the E4M3 scale byte. */
static void nv_block(double* v, int n, long stride, float S, unsigned char* codes, unsigned char* sc)
{
    float a = 0.0f;
    for (int i = 0; i < n; ++i) {
        float f = fabsf((float)v[(long)i * stride]);
        if (f > a) a = f;
    }
    float t = a * S;
    float sf = t / 6.0f;
    unsigned char sb = oracle_e4m3_encode(sf);
    float s = (float)oracle_e4m3_decode(sb);
    float r = s > 0.0f ? S / s : 0.0f;
    for (int i = 0; i < n; ++i) {
        float x = (float)v[(long)i * stride];
        unsigned char c = s > 0.0f ? oracle_e2m1_encode(x * r) : (unsigned char)0;
        if (codes) codes[(long)i * stride] = c;
        v[(long)i * stride] = oracle_e2m1_decode(c) * (double)s / (double)S;
    }
    if (sc) *sc = sb;
}

static float amax_of(const double* X, size_t n)
{
    float a = 0.0f;
    for (size_t i = 0; i < n; ++i) {
        float f = fabsf((float)X[i]);
        if (f > a) a = f;
    }
    return a;
}

/* 1x16 blocks along the rows of an M x K matrix (K a multiple of 16), or
 * (by_row 0) per column over 16-row blocks (the last block may be short),
 * with the tensor scale of amax. */
static void nv_qdq(int by_row, int M, int K, double* X, float amax)
{
    const float S = oracle_nv_tensor_scale(amax);
    if (by_row) {
#pragma omp parallel for schedule(static)
        for (int m = 0; m < M; ++m)
            for (int k0 = 0; k0 < K; k0 += 16) nv_block(X + (long)m * K + k0, 16, 1, S, NULL, NULL);
    } else {
#pragma omp parallel for schedule(static)
        for (int n = 0; n < K; ++n)
            for (int m0 = 0; m0 < M; m0 += 16) {
                int len = M - m0 < 16 ? M - m0 : 16;
                nv_block(X + (long)m0 * K + n, len, K, S, NULL, NULL);
            }
    }
}

/* NVFP4 codes (one per byte, low 4 bits) and E4M3 scale bytes of one fp32
 * matrix as a single tensor, for comparison with a GPU quantiser. mode 0:
 * 1x16 along rows (scales M x K/16); mode 1: per column over 16-row blocks
 * (scales ceil(M/16) x K). *S_out receives the tensor scale. */
int oracle_nv_quantize(int M, int K, int mode, const float* X, unsigned char* codes, unsigned char* scales,
                       float* S_out)
{
    if (M <= 0 || K <= 0 || mode < 0 || mode > 1) return -1;
    if (mode == 0 && K % 16) return -1;
    double* v = (double*)malloc(sizeof(double) * (size_t)M * K);
    for (size_t i = 0; i < (size_t)M * K; ++i) v[i] = X[i];
    const float S = oracle_nv_tensor_scale(amax_of(v, (size_t)M * K));
    if (mode == 0) {
        for (int m = 0; m < M; ++m)
            for (int k0 = 0; k0 < K; k0 += 16)
                nv_block(v + (long)m * K + k0, 16, 1, S, codes + (long)m * K + k0, scales + (long)m * (K / 16) + k0 / 16);
    } else {
        for (int n = 0; n < K; ++n)
            for (int m0 = 0; m0 < M; m0 += 16) {
                int len = M - m0 < 16 ? M - m0 : 16;
                nv_block(v + (long)m0 * K + n, len, K, S, codes + (long)m0 * K + n, scales + (long)(m0 / 16) * K + n);
            }
    }
    if (S_out) *S_out = S;
    free(v);
    return 0;
}

static double* dup(const double* p, size_t n)
{
    double* q = (double*)malloc(sizeof(double) * (n ? n : 1));
    memcpy(q, p, sizeof(double) * n);
    return q;
}

/* C (M x N) = A (M x K) B (K x N), plain fp64. */
static void gemm(int M, int N, int K, const double* A, const double* B, double* C)
{
#pragma omp parallel for schedule(static)
    for (int m = 0; m < M; ++m)
        for (int n = 0; n < N; ++n) {
            double acc = 0.0;
            for (int k = 0; k < K; ++k) acc += A[(long)m * K + k] * B[(long)k * N + n];
            C[(long)m * N + n] = acc;
        }
}

/* C (M x N) = A^T B with A (K x M), B (K x N). */
static void gemm_tn(int M, int N, int K, const double* A, const double* B, double* C)
{
#pragma omp parallel for schedule(static)
    for (int m = 0; m < M; ++m)
        for (int n = 0; n < N; ++n) {
            double acc = 0.0;
            for (int k = 0; k < K; ++k) acc += A[(long)k * M + m] * B[(long)k * N + n];
            C[(long)m * N + n] = acc;
        }
}

/* C (M x N) = A B^T with A (M x K), B (N x K). */
static void gemm_nt(int M, int N, int K, const double* A, const double* B, double* C)
{
#pragma omp parallel for schedule(static)
    for (int m = 0; m < M; ++m)
        for (int n = 0; n < N; ++n) {
            double acc = 0.0;
            for (int k = 0; k < K; ++k) acc += A[(long)m * K + k] * B[(long)n * K + k];
            C[(long)m * N + n] = acc;
        }
}

/*
 * One expert (or the shared expert) in FP8, forward and -- when dYr is not
 * NULL -- backward, for its M rows X (M x H) in dispatch order. Wg, Wu: H x F;
 * Wd: F x H (unquantised). Y receives the output rows; the gradients are
 * written when dYr != NULL (dYr are the rows' output gradients, already
 * gate-scaled).
 */
/*
 * g != NULL: memory-efficient permutation ("Scalable Training of
 * Mixture-of-Experts Models with Megatron Core", §4: the routing weight is
 * folded into the activation by an algebraic rearrangement). Row r's fc2
 * input is h'_r = g_r h_r (rounded to bf16), so Y holds g_r y_r; dYr is then
 * the unweighted output gradient, dh' = dYr Wd^T, dg_r = <dh'_r, h_r> (h from
 * the bf16-stored a, u, as the backward pass recomputes it), dh = g_r dh',
 * and the fc2 weight gradient uses h' recomputed from the stored a, u.
 */
/*
 * recipe 0: blockwise FP8 (fp32 scales; 1x128 blocks along K for the operand
 * indexing output rows, 128x128 for the other). recipe 1: MXFP8 (1x32 blocks
 * along K for both operands of every GEMM, so each weight is quantised once
 * per orientation: along H for fc1 and along F for fc1's data gradient; Wd
 * along F for fc2 and along H for fc2's data gradient). recipe 2: NVFP4
 * (1x16 blocks along K like MXFP8, E4M3 block scales under one fp32 scale
 * per tensor: per expert operand, [Wg | Wu] and [dA | dU] one tensor each).
 */
#define RECIPE_BLOCK 0
#define RECIPE_MX 1
#define RECIPE_NV 2

/* the quantisation of X (rows x cols) whose contraction dimension runs along
 * its rows (by_row 1: blocks within a row) or its columns (by_row 0); amax:
 * the largest magnitude of the NVFP4 tensor X belongs to (recipe 2) */
static void q_act(int recipe, int by_row, int rows, int cols, double* X, float amax)
{
    if (recipe == RECIPE_NV) {
        nv_qdq(by_row, rows, cols, X, amax);
    } else if (recipe == RECIPE_MX) {
        if (by_row) mx_rows(rows, cols, X); else mx_cols(rows, cols, X);
    } else {
        if (by_row) qdq_rows(rows, cols, X); else qdq_cols(rows, cols, X);
    }
}
/* the second operand of a GEMM (128x128 blocks, or MX / NVFP4 blocks along K) */
static void q_other(int recipe, int by_row, int rows, int cols, double* X, float amax)
{
    if (recipe == RECIPE_NV) {
        nv_qdq(by_row, rows, cols, X, amax);
    } else if (recipe == RECIPE_MX) {
        if (by_row) mx_rows(rows, cols, X); else mx_cols(rows, cols, X);
    } else {
        qdq_tiles(rows, cols, X);
    }
}

static void swiglu_fp8(int M, int H, int F, const double* X, const double* Wg, const double* Wu,
                       const double* Wd, double* Y, const double* dYr, double* dX, double* dWg,
                       double* dWu, double* dWd, const double* g, double* dg, int recipe)
{
    size_t mf = (size_t)(M > 0 ? M : 1) * F, mh = (size_t)(M > 0 ? M : 1) * H;
    /* NVFP4 tensor maxima: x, [Wg | Wu], Wd (h, dY, [dA | dU] below) */
    const float aX = amax_of(X, (size_t)M * H);
    const float aWgu = fmaxf(amax_of(Wg, (size_t)H * F), amax_of(Wu, (size_t)H * F));
    const float aWd = amax_of(Wd, (size_t)F * H);
    double* Xq = dup(X, (size_t)M * H);
    q_act(recipe, 1, M, H, Xq, aX);                   /* fc1 A: K = H along rows */
    /* fc1 B: Wg, Wu (H x F) with K = H along their columns; fc2 B: Wd (F x H)
     * with K = F along its columns */
    double* Wgq = dup(Wg, (size_t)H * F);
    double* Wuq = dup(Wu, (size_t)H * F);
    double* Wdq = dup(Wd, (size_t)F * H);
    q_other(recipe, 0, H, F, Wgq, aWgu);
    q_other(recipe, 0, H, F, Wuq, aWgu);
    q_other(recipe, 0, F, H, Wdq, aWd);
    /* the data gradients contract the weights along their other dimension:
     * the same codes in the blockwise recipe, a second quantisation in MX
     * and NVFP4 (the same tensor scale in NVFP4) */
    double *Wgb = Wgq, *Wub = Wuq, *Wdb = Wdq;
    if (recipe != RECIPE_BLOCK && dYr) {
        Wgb = dup(Wg, (size_t)H * F);
        Wub = dup(Wu, (size_t)H * F);
        Wdb = dup(Wd, (size_t)F * H);
        q_other(recipe, 1, H, F, Wgb, aWgu);
        q_other(recipe, 1, H, F, Wub, aWgu);
        q_other(recipe, 1, F, H, Wdb, aWd);
    }
    double* A = (double*)malloc(sizeof(double) * mf);
    double* U = (double*)malloc(sizeof(double) * mf);
    double* Hh = (double*)malloc(sizeof(double) * mf);
    gemm(M, F, H, Xq, Wgq, A);
    gemm(M, F, H, Xq, Wuq, U);
    for (size_t i = 0; i < (size_t)M * F; ++i) {
        const double gr = g ? g[i / F] : 1.0;
        Hh[i] = bf16r(gr * silu(A[i]) * U[i]);   /* from the GEMM outputs themselves */
        A[i] = bf16r(A[i]);
        U[i] = bf16r(U[i]);
    }
    double* Hq = dup(Hh, (size_t)M * F);
    q_act(recipe, 1, M, F, Hq, amax_of(Hh, (size_t)M * F));   /* fc2 A: K = F */
    gemm(M, H, F, Hq, Wdq, Y);
    for (size_t i = 0; i < (size_t)M * H; ++i) Y[i] = bf16r(Y[i]);
    free(Hq);
    if (dYr) {
        /* fc2 dgrad: dh = q(dYr) q(Wd)^T, K = H */
        const float aDY = amax_of(dYr, (size_t)M * H);
        double* dYq = dup(dYr, (size_t)M * H);
        q_act(recipe, 1, M, H, dYq, aDY);
        double* dh = (double*)malloc(sizeof(double) * mf);
        gemm_nt(M, F, H, dYq, Wdb, dh);
        double* dA = (double*)malloc(sizeof(double) * mf);
        double* dU = (double*)malloc(sizeof(double) * mf);
        if (g) {
            for (int r = 0; r < M; ++r) {
                double acc = 0.0;
                for (int f = 0; f < F; ++f) {
                    const size_t i = (size_t)r * F + f;
                    const double hr = silu(A[i]) * U[i];
                    acc += dh[i] * hr;
                    dh[i] *= g[r];
                    Hh[i] = bf16r(g[r] * hr);   /* h' recomputed for the weight gradient */
                }
                dg[r] = acc;
            }
        }
        for (size_t i = 0; i < (size_t)M * F; ++i) {
            dA[i] = bf16r(dh[i] * U[i] * dsilu(A[i]));
            dU[i] = bf16r(dh[i] * silu(A[i]));
        }
        /* fc2 wgrad: dWd = q(h)^T q(dYr), K = the expert's rows (blocks along
         * the rows, counted from the segment's first row) */
        double* Hc = dup(Hh, (size_t)M * F);
        q_act(recipe, 0, M, F, Hc, amax_of(Hh, (size_t)M * F));
        double* dYt = dup(dYr, (size_t)M * H);
        q_other(recipe, 0, M, H, dYt, aDY);
        gemm_tn(F, H, M, Hc, dYt, dWd);
        /* fc1 dgrad: dX = q(dA) q(Wg)^T + q(dU) q(Wu)^T, K = F */
        const float aDAU = fmaxf(amax_of(dA, (size_t)M * F), amax_of(dU, (size_t)M * F));
        double* dAq = dup(dA, mf);
        double* dUq = dup(dU, mf);
        q_act(recipe, 1, M, F, dAq, aDAU);
        q_act(recipe, 1, M, F, dUq, aDAU);
        double* t1 = (double*)malloc(sizeof(double) * mh);
        gemm_nt(M, H, F, dAq, Wgb, dX);
        gemm_nt(M, H, F, dUq, Wub, t1);
        for (size_t i = 0; i < (size_t)M * H; ++i) dX[i] += t1[i];
        /* fc1 wgrad: dWg = q(X)^T q(dA), dWu = q(X)^T q(dU), K = rows */
        double* Xc = dup(X, (size_t)M * H);
        q_act(recipe, 0, M, H, Xc, aX);
        double* dAt = dup(dA, mf);
        double* dUt = dup(dU, mf);
        q_other(recipe, 0, M, F, dAt, aDAU);
        q_other(recipe, 0, M, F, dUt, aDAU);
        gemm_tn(H, F, M, Xc, dAt, dWg);
        gemm_tn(H, F, M, Xc, dUt, dWu);
        free(dYq); free(dh); free(dA); free(dU); free(Hc); free(dYt); free(dAq); free(dUq);
        free(t1); free(Xc); free(dAt); free(dUt);
    }
    if (Wgb != Wgq) { free(Wgb); free(Wub); free(Wdb); }
    free(Xq); free(Wgq); free(Wuq); free(Wdq); free(A); free(U); free(Hh);
}

/*
 * FP8 layer: same stages and outputs as oracle_forward / oracle_backward,
 * with every expert GEMM operand quantised as described above. dY may be
 * NULL (forward only); then only y (and dg, Yp if requested) are written.
 */
int oracle_layer_fp8(int T, int H, int E, int k, int F, int Fs, int score_fn,
                     const double* x, const double* Wr,
                     const double* Wg, const double* Wu, const double* Wd,
                     const double* Wsg, const double* Wsu, const double* Wsd,
                     const int* topk, const double* gates, const double* scores,
                     const double* dY, double* y,
                     double* dX, double* dWr, double* dWg, double* dWu, double* dWd,
                     double* dWsg, double* dWsu, double* dWsd, double* dg_out, int fold,
                     int recipe, const unsigned char* keep)
{
    if (T <= 0 || H <= 0 || H % 128 || E <= 0 || k <= 0 || k > E || k > 1024 || F <= 0 ||
        F % 128 || Fs < 0 || Fs % 128 || recipe < 0 || recipe > 2)
        return -1;
    int* counts = (int*)malloc(sizeof(int) * E);
    int* offsets = (int*)malloc(sizeof(int) * (E + 1));
    int* row_of = (int*)malloc(sizeof(int) * (size_t)T * k);
    int* slot_of = (int*)malloc(sizeof(int) * (size_t)T * k);
    if (oracle_dispatch(T, E, k, topk, counts, offsets, row_of, slot_of)) return -1;
    if (keep) {
        /* capacity-limited dropping: a dropped assignment never reaches its
         * expert, so each expert's segment holds its kept rows alone (in token
         * order) and every quantisation block along the tokens is counted from
         * the segment's first kept row; row_of of a dropped slot is -1 */
        int row = 0;
        for (int e = 0; e < E; ++e) {
            offsets[e] = row;
            for (int t = 0; t < T; ++t)
                for (int j = 0; j < k; ++j) {
                    const int sl = t * k + j;
                    if (topk[sl] != e) continue;
                    if (keep[sl]) {
                        row_of[sl] = row;
                        slot_of[row] = sl;
                        ++row;
                    } else {
                        row_of[sl] = -1;
                    }
                }
            counts[e] = row - offsets[e];
        }
        offsets[E] = row;
    }
    const int R = offsets[E];   /* rows that reach an expert */
    /* routing weight of each permuted row (folded variant) */
    double* grow = (double*)malloc(sizeof(double) * (size_t)R);
    for (int r = 0; r < R; ++r) grow[r] = gates[slot_of[r]];
    double* Xp = (double*)malloc(sizeof(double) * (size_t)R * H);
    double* Yp = (double*)malloc(sizeof(double) * (size_t)R * H);
    double* dYp = (double*)malloc(sizeof(double) * (size_t)R * H);
    double* dXp = (double*)malloc(sizeof(double) * (size_t)R * H);
    double* dg = (double*)calloc((size_t)T * k, sizeof(double));   /* per slot; 0 if dropped */
    for (int r = 0; r < R; ++r)
        memcpy(Xp + (size_t)r * H, x + (size_t)(slot_of[r] / k) * H, sizeof(double) * H);
    /* forward of every expert (Yp), then the gate-scaled output gradients */
    for (int e = 0; e < E; ++e) {
        int M = counts[e];
        if (M == 0) continue;
        swiglu_fp8(M, H, F, Xp + (size_t)offsets[e] * H, Wg + (size_t)e * H * F,
                   Wu + (size_t)e * H * F, Wd + (size_t)e * F * H, Yp + (size_t)offsets[e] * H,
                   NULL, NULL, NULL, NULL, NULL, fold ? grow + offsets[e] : NULL, NULL, recipe);
    }
    for (int t = 0; t < T; ++t)
        for (int h = 0; h < H; ++h) {
            double acc = 0.0;
            for (int j = 0; j < k; ++j) {
                const int row = row_of[(size_t)t * k + j];
                if (row < 0) continue;   /* dropped */
                acc += (fold ? 1.0 : gates[(size_t)t * k + j]) * Yp[(size_t)row * H + h];
            }
            y[(size_t)t * H + h] = acc;
        }
    double* Ys = NULL;
    if (Fs > 0) {
        Ys = (double*)malloc(sizeof(double) * (size_t)T * H);
        swiglu_fp8(T, H, Fs, x, Wsg, Wsu, Wsd, Ys, NULL, NULL, NULL, NULL, NULL, NULL, NULL, recipe);
        for (size_t i = 0; i < (size_t)T * H; ++i) y[i] += Ys[i];
    }
    if (dY) {
        for (int r = 0; r < R; ++r) {
            int t = slot_of[r] / k;
            double g = fold ? 1.0 : gates[slot_of[r]], acc = 0.0;
            for (int h = 0; h < H; ++h) {
                acc += dY[(size_t)t * H + h] * Yp[(size_t)r * H + h];
                dYp[(size_t)r * H + h] = bf16r(g * dY[(size_t)t * H + h]);
            }
            dg[slot_of[r]] = acc;   /* folded: replaced below by <dh', h> */
        }
        double* dgr = fold ? (double*)malloc(sizeof(double) * (size_t)R) : NULL;
        double* Ytmp = (double*)malloc(sizeof(double) * (size_t)(R > T ? R : T) * H);
        for (int e = 0; e < E; ++e) {
            int M = counts[e];
            double* dWg_e = dWg + (size_t)e * H * F;
            double* dWu_e = dWu + (size_t)e * H * F;
            double* dWd_e = dWd + (size_t)e * F * H;
            if (M == 0) {
                memset(dWg_e, 0, sizeof(double) * (size_t)H * F);
                memset(dWu_e, 0, sizeof(double) * (size_t)H * F);
                memset(dWd_e, 0, sizeof(double) * (size_t)F * H);
                continue;
            }
            swiglu_fp8(M, H, F, Xp + (size_t)offsets[e] * H, Wg + (size_t)e * H * F,
                       Wu + (size_t)e * H * F, Wd + (size_t)e * F * H, Ytmp,
                       dYp + (size_t)offsets[e] * H, dXp + (size_t)offsets[e] * H, dWg_e, dWu_e,
                       dWd_e, fold ? grow + offsets[e] : NULL, fold ? dgr + offsets[e] : NULL, recipe);
        }
        if (fold) {
            for (int r = 0; r < R; ++r) dg[slot_of[r]] = dgr[r];
            free(dgr);
        }
        double* dz = (double*)calloc((size_t)T * E, sizeof(double));
        for (int t = 0; t < T; ++t) {
            double dzs[1024];
            router_dz(k, score_fn, topk + (size_t)t * k, gates + (size_t)t * k,
                      scores + (size_t)t * E, dg + (size_t)t * k, dzs);
            for (int j = 0; j < k; ++j) dz[(size_t)t * E + topk[(size_t)t * k + j]] = dzs[j];
        }
#pragma omp parallel for schedule(static)
        for (int h = 0; h < H; ++h)
            for (int e = 0; e < E; ++e) {
                double acc = 0.0;
                for (int t = 0; t < T; ++t) acc += x[(size_t)t * H + h] * dz[(size_t)t * E + e];
                dWr[(size_t)h * E + e] = acc;
            }
#pragma omp parallel for schedule(static)
        for (int t = 0; t < T; ++t)
            for (int h = 0; h < H; ++h) {
                double acc = 0.0;
                for (int j = 0; j < k; ++j) {
                    const int row = row_of[(size_t)t * k + j];
                    if (row >= 0) acc += dXp[(size_t)row * H + h];
                }
                for (int e = 0; e < E; ++e) acc += dz[(size_t)t * E + e] * Wr[(size_t)h * E + e];
                dX[(size_t)t * H + h] = acc;
            }
        if (Fs > 0) {
            double* dXs = (double*)malloc(sizeof(double) * (size_t)T * H);
            swiglu_fp8(T, H, Fs, x, Wsg, Wsu, Wsd, Ytmp, dY, dXs, dWsg, dWsu, dWsd, NULL, NULL, recipe);
            for (size_t i = 0; i < (size_t)T * H; ++i) dX[i] += dXs[i];
            free(dXs);
        }
        free(Ytmp);
        free(dz);
        if (dg_out) memcpy(dg_out, dg, sizeof(double) * (size_t)T * k);
    }
    free(Ys); free(Xp); free(Yp); free(dYp); free(dXp); free(dg); free(grow);
    free(counts); free(offsets); free(row_of); free(slot_of);
    return 0;
}
