/*
 * fp64 CPU oracle for the Kimi Delta Attention (KDA) forward.
 *
 * TEST INFRASTRUCTURE ONLY.  The tests, the smoke check and the benchmark's
 * CPU-baseline leg may call this file; the product path never does, and this
 * file shares no code, header or table with the CUDA library.
 *
 * What it computes.  "Kimi K3 on Fireworks: Fast RL at frontier scale" (KDA
 * paragraph of the kernels section) describes KDA as linear attention that
 * updates a compact per-head recurrent state with channel-wise gating; its
 * speculative-decoding paragraph replays the accepted tokens' state-update
 * inputs onto a committed state (ReplaySSM).  The pages print no equation, so
 * the recurrence taken here is the gated delta rule with per-channel decay,
 * the plainest reading that matches "channel-wise gating" and "compact
 * recurrent state".  Per (sequence, head), with S in R^{dk x dv}:
 *
 *     S <- Diag(alpha_t) S                       alpha_t = exp(g_t) in [0,1]^dk
 *     S <- S - beta_t k_t (k_t^T S) + beta_t k_t v_t^T
 *     o_t = S^T (scale * q_t)
 *
 * i.e. the decay acts on the dk rows first, the delta step reads the decayed
 * state, and the output reads the state after the update (inclusive).
 *
 * Everything is evaluated token by token, row by row, in double precision,
 * exactly in that order; no chunking, blocking or reassociation.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* Return codes. */
#define KDA_ORACLE_OK 0
#define KDA_ORACLE_BAD_ARGS 1
#define KDA_ORACLE_NO_MEMORY 2

/* One (sequence, head) chain over tokens [bos, eos).
 * Layouts (token-major, packed): q,k,g [T,H,dk]; v [T,H,dv]; beta [T,H];
 * o [T,H,dv]; S [dk,dv] row-major. */
static void oracle_chain(const double *q, const double *k, const double *v, const double *g,
                         const double *beta, int64_t bos, int64_t eos, int64_t h, int64_t H,
                         int64_t dk, int64_t dv, double scale, int gate_is_alpha, double *S,
                         double *y, double *qs, double *o)
{
    for (int64_t t = bos; t < eos; ++t) {
        const double *qt = q + (t * H + h) * dk;
        const double *kt = k + (t * H + h) * dk;
        const double *gt = g + (t * H + h) * dk;
        const double *vt = v + (t * H + h) * dv;
        const double bt = beta[t * H + h];

        /* 1. channel-wise decay of the dk rows */
        for (int64_t i = 0; i < dk; ++i) {
            const double a = gate_is_alpha ? gt[i] : exp(gt[i]);
            for (int64_t j = 0; j < dv; ++j) S[i * dv + j] *= a;
        }
        /* 2. delta rule: y = S^T k, u = beta (v - y), S += k u^T */
        for (int64_t j = 0; j < dv; ++j) y[j] = 0.0;
        for (int64_t i = 0; i < dk; ++i)
            for (int64_t j = 0; j < dv; ++j) y[j] += kt[i] * S[i * dv + j];
        for (int64_t j = 0; j < dv; ++j) y[j] = bt * (vt[j] - y[j]);
        for (int64_t i = 0; i < dk; ++i)
            for (int64_t j = 0; j < dv; ++j) S[i * dv + j] += kt[i] * y[j];
        /* 3. output from the updated state with the scaled query */
        if (o) {
            double *ot = o + (t * H + h) * dv;
            for (int64_t i = 0; i < dk; ++i) qs[i] = scale * qt[i];
            for (int64_t j = 0; j < dv; ++j) ot[j] = 0.0;
            for (int64_t i = 0; i < dk; ++i)
                for (int64_t j = 0; j < dv; ++j) ot[j] += qs[i] * S[i * dv + j];
        }
    }
}

/*
 * Packed variable-length forward.
 *   cu_seqlens [N+1] (non-decreasing, cu[0] = 0): sequence n is tokens
 *     [cu[n], cu[n+1]).
 *   init_state [N,H,dk,dv] or NULL (zeros).  final_state [N,H,dk,dv] or NULL.
 *   o [T,H,dv] or NULL (state-only replay).
 *   gate_is_alpha: 0 -> g holds log-gates, alpha = exp(g);
 *                  1 -> g holds alpha itself (lets tests feed alpha = 0).
 *   nthreads: OpenMP threads over the N*H independent chains (<= 0: default).
 */
int kda_oracle_forward(const double *q, const double *k, const double *v, const double *g,
                       const double *beta, const double *init_state, const int64_t *cu_seqlens,
                       int64_t N, int64_t H, int64_t dk, int64_t dv, double scale, int gate_is_alpha,
                       double *o, double *final_state, int nthreads)
{
    if (N < 0 || H <= 0 || dk <= 0 || dv <= 0 || !cu_seqlens || !k || !v || !g || !beta)
        return KDA_ORACLE_BAD_ARGS;
    if (o && !q) return KDA_ORACLE_BAD_ARGS;
    if (N > 0 && cu_seqlens[0] != 0) return KDA_ORACLE_BAD_ARGS;
    for (int64_t n = 0; n < N; ++n)
        if (cu_seqlens[n + 1] < cu_seqlens[n]) return KDA_ORACLE_BAD_ARGS;

    const int64_t pairs = N * H;
    int failed = 0;
#ifdef _OPENMP
    if (nthreads <= 0) nthreads = omp_get_max_threads();
#pragma omp parallel for schedule(dynamic, 1) num_threads(nthreads) reduction(| : failed)
#endif
    for (int64_t p = 0; p < pairs; ++p) {
        const int64_t n = p / H, h = p % H;
        double *S = (double *)malloc(sizeof(double) * (size_t)(dk * dv + dv + dk));
        if (!S) { failed |= 1; continue; }
        double *y = S + dk * dv, *qs = y + dv;
        if (init_state)
            memcpy(S, init_state + p * dk * dv, sizeof(double) * (size_t)(dk * dv));
        else
            memset(S, 0, sizeof(double) * (size_t)(dk * dv));
        oracle_chain(q, k, v, g, beta, cu_seqlens[n], cu_seqlens[n + 1], h, H, dk, dv, scale,
                     gate_is_alpha, S, y, qs, o);
        if (final_state) memcpy(final_state + p * dk * dv, S, sizeof(double) * (size_t)(dk * dv));
        free(S);
    }
    (void)nthreads;
    return failed ? KDA_ORACLE_NO_MEMORY : KDA_ORACLE_OK;
}

/*
 * Input preprocessing, in place, for callers that pass raw projections (the
 * optional fused preprocessing of the library).  The pages do not define KDA's
 * input maps; the reading taken is the common one for delta-rule attention:
 *   flags & 1:  q_t <- q_t / sqrt(sum_i q_{t,i}^2 + eps)   per (token, head), over dk
 *   flags & 2:  k_t <- k_t / sqrt(sum_i k_{t,i}^2 + eps)
 *   flags & 4:  g   <- sigmoid(g) elementwise: the log-gate is logsigmoid(x), so the
 *               decay alpha = exp(logsigmoid(x)) = sigmoid(x) is stored directly
 *               (call kda_oracle_forward with gate_is_alpha = 1)
 *   flags & 8:  beta <- sigmoid(beta)
 * q may be NULL when flags has no bit 1.
 */
static double sigmoid(double x) { return 1.0 / (1.0 + exp(-x)); }

int kda_oracle_prep(double *q, double *k, double *g, double *beta, int64_t T, int64_t H, int64_t dk,
                    double eps, int flags)
{
    if (T < 0 || H <= 0 || dk <= 0 || eps < 0.0) return KDA_ORACLE_BAD_ARGS;
    if (((flags & 1) && !q) || ((flags & 2) && !k) || ((flags & 4) && !g) || ((flags & 8) && !beta))
        return KDA_ORACLE_BAD_ARGS;
    for (int64_t r = 0; r < T * H; ++r) {
        for (int which = 0; which < 2; ++which) {
            if (!(flags & (1 << which))) continue;
            double *x = (which == 0 ? q : k) + r * dk;
            double ss = 0.0;
            for (int64_t i = 0; i < dk; ++i) ss += x[i] * x[i];
            const double inv = 1.0 / sqrt(ss + eps);
            for (int64_t i = 0; i < dk; ++i) x[i] *= inv;
        }
        if (flags & 4)
            for (int64_t i = 0; i < dk; ++i) g[r * dk + i] = sigmoid(g[r * dk + i]);
        if (flags & 8) beta[r] = sigmoid(beta[r]);
    }
    return KDA_ORACLE_OK;
}

/*
 * Backward (reverse mode) of kda_oracle_forward, for training: given the
 * gradients of a loss with respect to the outputs o (d_o, [T,H,dv]) and to the
 * final states (d_final, [N,H,dk,dv] or NULL = zero), the gradients with
 * respect to q, k, v, g (log-gates; with gate_is_alpha, alpha itself), beta and
 * the initial states.  The KDA paragraph quotes a backward kernel (its speedup
 * over FLA) but no formula; this is the adjoint of exactly the three steps the
 * forward takes per token, applied in reverse token order:
 *
 *   forward   S' = Diag(a) S_prev;  y = S'^T k;  u = beta (v - y);  S = S' + k u^T;
 *             o = S^T (scale q)
 *   reverse   dS += (scale q) do^T;   dq = scale S do
 *             du = dS^T k;  dk = dS u;  dbeta = du . (v - y);  dv = beta du;  dy = -beta du
 *             dS' = dS + k dy^T;  dk += S' dy
 *             da_i = sum_j dS'_ij S_prev,ij;  dg_i = da_i a_i (log-gates);  dS_prev = Diag(a) dS'
 *
 * The state before every token's decay is kept (stored on the way forward), so
 * each reverse step recomputes S', y, u and S from it in double precision.
 * Outputs dq, dk, dg [T,H,dk], dv [T,H,dv], dbeta [T,H] are written for every
 * token; d_init [N,H,dk,dv] may be NULL.
 */
static void oracle_chain_bwd(const double *q, const double *k, const double *v, const double *g,
                             const double *beta, int64_t bos, int64_t eos, int64_t h, int64_t H,
                             int64_t dk, int64_t dv, double scale, int gate_is_alpha, const double *d_o,
                             double *Sall, double *dS, double *Sp, double *dSp, double *y, double *u,
                             double *du, double *dy, double *dq, double *dkk, double *dvv, double *dg,
                             double *dbeta)
{
    const int64_t L = eos - bos, sz = dk * dv;
    /* forward, keeping the state before each token: Sall[l] = S before token bos + l */
    for (int64_t l = 0; l < L; ++l) {
        const int64_t t = bos + l;
        const double *kt = k + (t * H + h) * dk, *gt = g + (t * H + h) * dk, *vt = v + (t * H + h) * dv;
        const double bt = beta[t * H + h];
        double *S = Sall + (l + 1) * sz;
        memcpy(S, Sall + l * sz, sizeof(double) * (size_t)sz);
        for (int64_t i = 0; i < dk; ++i) {
            const double a = gate_is_alpha ? gt[i] : exp(gt[i]);
            for (int64_t j = 0; j < dv; ++j) S[i * dv + j] *= a;
        }
        for (int64_t j = 0; j < dv; ++j) y[j] = 0.0;
        for (int64_t i = 0; i < dk; ++i)
            for (int64_t j = 0; j < dv; ++j) y[j] += kt[i] * S[i * dv + j];
        for (int64_t j = 0; j < dv; ++j) u[j] = bt * (vt[j] - y[j]);
        for (int64_t i = 0; i < dk; ++i)
            for (int64_t j = 0; j < dv; ++j) S[i * dv + j] += kt[i] * u[j];
    }
    /* reverse; dS holds the gradient with respect to the state after token t */
    for (int64_t l = L - 1; l >= 0; --l) {
        const int64_t t = bos + l;
        const double *qt = q + (t * H + h) * dk, *kt = k + (t * H + h) * dk, *gt = g + (t * H + h) * dk;
        const double *vt = v + (t * H + h) * dv, *dot = d_o + (t * H + h) * dv;
        const double bt = beta[t * H + h];
        const double *Sprev = Sall + l * sz, *S = Sall + (l + 1) * sz;
        double *dqt = dq + (t * H + h) * dk, *dkt = dkk + (t * H + h) * dk, *dgt = dg + (t * H + h) * dk;
        double *dvt = dvv + (t * H + h) * dv;
        /* recompute S' = Diag(a) S_prev, y, u */
        for (int64_t i = 0; i < dk; ++i) {
            const double a = gate_is_alpha ? gt[i] : exp(gt[i]);
            for (int64_t j = 0; j < dv; ++j) Sp[i * dv + j] = a * Sprev[i * dv + j];
        }
        for (int64_t j = 0; j < dv; ++j) y[j] = 0.0;
        for (int64_t i = 0; i < dk; ++i)
            for (int64_t j = 0; j < dv; ++j) y[j] += kt[i] * Sp[i * dv + j];
        for (int64_t j = 0; j < dv; ++j) u[j] = bt * (vt[j] - y[j]);
        /* o = S^T (scale q) */
        for (int64_t i = 0; i < dk; ++i) {
            double acc = 0.0;
            for (int64_t j = 0; j < dv; ++j) acc += S[i * dv + j] * dot[j];
            dqt[i] = scale * acc;
            for (int64_t j = 0; j < dv; ++j) dS[i * dv + j] += scale * qt[i] * dot[j];
        }
        /* S = S' + k u^T */
        for (int64_t j = 0; j < dv; ++j) du[j] = 0.0;
        for (int64_t i = 0; i < dk; ++i) {
            double acc = 0.0;
            for (int64_t j = 0; j < dv; ++j) {
                acc += dS[i * dv + j] * u[j];
                du[j] += dS[i * dv + j] * kt[i];
            }
            dkt[i] = acc;
        }
        /* u = beta (v - y) */
        double db = 0.0;
        for (int64_t j = 0; j < dv; ++j) {
            db += du[j] * (vt[j] - y[j]);
            dvt[j] = bt * du[j];
            dy[j] = -bt * du[j];
        }
        dbeta[t * H + h] = db;
        /* y = S'^T k:  dS' = dS + k dy^T,  dk += S' dy */
        for (int64_t i = 0; i < dk; ++i) {
            double acc = 0.0;
            for (int64_t j = 0; j < dv; ++j) {
                dSp[i * dv + j] = dS[i * dv + j] + kt[i] * dy[j];
                acc += Sp[i * dv + j] * dy[j];
            }
            dkt[i] += acc;
        }
        /* S' = Diag(a) S_prev */
        for (int64_t i = 0; i < dk; ++i) {
            const double a = gate_is_alpha ? gt[i] : exp(gt[i]);
            double da = 0.0;
            for (int64_t j = 0; j < dv; ++j) {
                da += dSp[i * dv + j] * Sprev[i * dv + j];
                dS[i * dv + j] = a * dSp[i * dv + j];
            }
            dgt[i] = gate_is_alpha ? da : da * a;
        }
    }
}

int kda_oracle_backward(const double *q, const double *k, const double *v, const double *g,
                        const double *beta, const double *init_state, const int64_t *cu_seqlens,
                        int64_t N, int64_t H, int64_t dk, int64_t dv, double scale, int gate_is_alpha,
                        const double *d_o, const double *d_final, double *dq, double *dk_out,
                        double *dv_out, double *dg, double *dbeta, double *d_init, int nthreads)
{
    if (N < 0 || H <= 0 || dk <= 0 || dv <= 0 || !cu_seqlens || !q || !k || !v || !g || !beta || !d_o ||
        !dq || !dk_out || !dv_out || !dg || !dbeta)
        return KDA_ORACLE_BAD_ARGS;
    if (N > 0 && cu_seqlens[0] != 0) return KDA_ORACLE_BAD_ARGS;
    for (int64_t n = 0; n < N; ++n)
        if (cu_seqlens[n + 1] < cu_seqlens[n]) return KDA_ORACLE_BAD_ARGS;

    const int64_t pairs = N * H, sz = dk * dv;
    int failed = 0;
#ifdef _OPENMP
    if (nthreads <= 0) nthreads = omp_get_max_threads();
#pragma omp parallel for schedule(dynamic, 1) num_threads(nthreads) reduction(| : failed)
#endif
    for (int64_t p = 0; p < pairs; ++p) {
        const int64_t n = p / H, h = p % H;
        const int64_t L = cu_seqlens[n + 1] - cu_seqlens[n];
        double *Sall = (double *)malloc(sizeof(double) * (size_t)((L + 1) * sz));
        double *work = (double *)malloc(sizeof(double) * (size_t)(3 * sz + 4 * dv));
        if (!Sall || !work) {
            free(Sall);
            free(work);
            failed |= 1;
            continue;
        }
        double *dS = work, *Sp = work + sz, *dSp = work + 2 * sz, *y = work + 3 * sz, *u = y + dv, *du = u + dv,
               *dy = du + dv;
        if (init_state)
            memcpy(Sall, init_state + p * sz, sizeof(double) * (size_t)sz);
        else
            memset(Sall, 0, sizeof(double) * (size_t)sz);
        if (d_final)
            memcpy(dS, d_final + p * sz, sizeof(double) * (size_t)sz);
        else
            memset(dS, 0, sizeof(double) * (size_t)sz);
        oracle_chain_bwd(q, k, v, g, beta, cu_seqlens[n], cu_seqlens[n + 1], h, H, dk, dv, scale, gate_is_alpha,
                         d_o, Sall, dS, Sp, dSp, y, u, du, dy, dq, dk_out, dv_out, dg, dbeta);
        if (d_init) memcpy(d_init + p * sz, dS, sizeof(double) * (size_t)sz);
        free(Sall);
        free(work);
    }
    (void)nthreads;
    return failed ? KDA_ORACLE_NO_MEMORY : KDA_ORACLE_OK;
}

/*
 * Short causal convolution of the input projections, with the convolution state
 * carried across calls.  "Kimi K3 on Fireworks: Fast RL at frontier scale"
 * (disaggregated-serving paragraph) says a handoff must move KDA's recurrent
 * and convolution state; the pages define neither.  The reading taken: a
 * depthwise causal 1-D convolution of width W over the tokens of each sequence,
 * one weight vector per channel, followed by SiLU:
 *
 *   pre_t[c] = sum_{i=0}^{W-1} w[h][c][i] * x_{t-(W-1)+i}[c],   y_t[c] = pre / (1 + exp(-pre))
 *
 * where tokens before the sequence's first come from its convolution state, the
 * W-1 previous inputs oldest first (zeros when state_in is NULL).  state_out
 * receives the last W-1 inputs of (state ++ tokens).
 * Layouts: x, y [T, H, C]; w [H, C, W]; state [N, W-1, H, C].
 */
int kda_oracle_conv(const double *x, const double *w, const double *state_in, const int64_t *cu_seqlens,
                    int64_t N, int64_t H, int64_t C, int64_t W, double *y, double *state_out)
{
    if (N < 0 || H <= 0 || C <= 0 || W < 1 || !x || !w || !y || !cu_seqlens) return KDA_ORACLE_BAD_ARGS;
    for (int64_t n = 0; n < N; ++n) {
        const int64_t bos = cu_seqlens[n], eos = cu_seqlens[n + 1];
        if (eos < bos) return KDA_ORACLE_BAD_ARGS;
        for (int64_t h = 0; h < H; ++h) {
            for (int64_t c = 0; c < C; ++c) {
                /* value of input j positions back from token t (j >= 1 may reach into the state) */
                for (int64_t t = bos; t < eos; ++t) {
                    double pre = 0.0;
                    for (int64_t i = 0; i < W; ++i) {
                        const int64_t src = t - (W - 1) + i;
                        double xv;
                        if (src >= bos)
                            xv = x[(src * H + h) * C + c];
                        else {
                            const int64_t back = bos - src; /* 1 .. W-1 positions before the first token */
                            xv = state_in ? state_in[((n * (W - 1) + (W - 1 - back)) * H + h) * C + c] : 0.0;
                        }
                        pre += w[(h * C + c) * W + i] * xv;
                    }
                    y[(t * H + h) * C + c] = pre / (1.0 + exp(-pre));
                }
                if (state_out) {
                    for (int64_t j = 0; j < W - 1; ++j) {
                        /* slot j of the new state: the input W-1-j positions before the end */
                        const int64_t src = eos - (W - 1) + j;
                        double xv;
                        if (src >= bos)
                            xv = x[(src * H + h) * C + c];
                        else {
                            const int64_t back = bos - src;
                            xv = state_in ? state_in[((n * (W - 1) + (W - 1 - back)) * H + h) * C + c] : 0.0;
                        }
                        state_out[((n * (W - 1) + j) * H + h) * C + c] = xv;
                    }
                }
            }
        }
    }
    return KDA_ORACLE_OK;
}

/* Threads the OpenMP runtime would use by default (1 without OpenMP). */
int kda_oracle_max_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
