/*
 * lro_oracle.c -- plain, sequential float64 CPU oracle for the three gated
 * linear-recurrence scans  h_t = a_t (.) h_{t-1} + b_t  with a readout.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the correctness reference for the
 * CUDA library in selective_state_space_chunked_gb300/.  It shares no code,
 * header, table or constant with that library and includes nothing from it.
 * Only the test suite, the smoke check and the benchmark's CPU-baseline /
 * reference arm may load it; no product code path calls it.
 *
 * Every loop below is the recurrence written out one time step at a time, in
 * float64, in the order the source pages state it.  No chunking, blocking,
 * fusion or reordering.  Inputs arrive as float64 arrays that hold exactly the
 * values handed to the GPU (bf16 or fp32 values widened to double).
 *
 * Sources (web pages, cited by title and section):
 *   [SSM]   cortexnet 3.2.1, cortexnet/ssm.py: module docstring (ZOH
 *           discretisation), MultiScaleSSM.__init__ (A_log, D), forward
 *           (A = -exp(A_log), dt = softplus(dt_proj(x)), D skip, silu(z) gate),
 *           MultiScaleSSM._selective_scan (the sequential float32 loop).
 *   [RGLRU] lrnnx, lrnnx.models.ltv.rglru module source: RGLRU.step, the
 *           non-Triton fallback branch (a_bar = a^(c*r), sqrt(1 - a_bar^2),
 *           state update, readout = sum over dstate).
 *   [HGRN2] frankenstein-transformer API docs, HGRN2 Attention page: the
 *           state update S_t = diag(g_t) S_{t-1} + v_t k_t^T and the
 *           token-by-token forward description.
 *   [MINMAX] minmaxrnc 0.1.0 wheel: minmax_neuron.py (MinMaxNeuron class
 *           docstring, x_{t+1} = max(min(r_t, x_t), s_t); forward, which
 *           returns the states after every step and the last state) and
 *           minmax_operator.py (apply: f(x) = max(min(a, x), b)).
 *
 * Parity pins (closed forms, brute force, library special cases) live in
 * tests/test_oracle_pins.py.  All four functions are pinned there.
 *
 * Layouts (row-major, contiguous):
 *   selective: x, dt, z, y: (B, L, D); Bm, Cm: (B, L, N); A_log: (D, N);
 *              Dskip: (D); h0, h_final: (B, D, N)
 *   rglru:     x, r, ig, y: (B, L, D); a_log: (D); h0, h_final: (B, D)
 *   hgrn2:     q, k: (B, L, H*dk); v, g, o: (B, L, H*dv);
 *              S0, S_final: (B, H, dv, dk)   (row i = value channel,
 *              column j = key channel)
 *   minmax:    r, s, y: (B, L, D); x0, x_final: (B, D)
 *
 * Return value: 0 on success, -1 on an invalid argument (nothing written).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#ifdef _OPENMP
#include <omp.h>
#endif

/* torch.nn.functional.softplus with beta = 1, threshold = 20: the input is
 * returned unchanged above the threshold, else log(1 + exp(v)). [SSM] forward
 * applies it to dt_proj(x). */
static double softplus_thresholded(double v)
{
    return v > 20.0 ? v : log1p(exp(v));
}

static double logistic(double v) { return 1.0 / (1.0 + exp(-v)); }

static void set_threads(int nthreads)
{
#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
#else
    (void)nthreads;
#endif
}

int lro_max_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/*
 * Selective SSM scan, [SSM] MultiScaleSSM._selective_scan followed by the
 * D skip and silu(z) gate of MultiScaleSSM.forward.  For each (b, d):
 *
 *   h[n] = h0[b,d,n]                       (zero when h0 == NULL)
 *   for t in 0..L-1:
 *     delta = softplus(dt[b,t,d])  if dt_softplus, else dt[b,t,d]
 *     for n: A     = -exp(A_log[d,n])
 *            a     = exp(delta * A)                    (A_bar, ZOH)
 *            h[n]  = a * h[n] + delta * Bm[b,t,n] * x[b,t,d]
 *     yv = sum_n Cm[b,t,n] * h[n]                      (readout after update)
 *     yv = yv + Dskip[d] * x[b,t,d]                    (when Dskip != NULL)
 *     yv = yv * z * logistic(z)                        (when z != NULL)
 *     y[b,t,d] = yv
 *   h_final[b,d,:] = h                                 (when h_final != NULL)
 *
 * The page clamps delta*A at 20 from above before the exp; with delta >= 0
 * and A < 0 that clamp never binds, so it is not written here.
 */
int lro_selective_scan_ref(const double *x, const double *dt, const double *z,
                           const double *Bm, const double *Cm,
                           const double *A_log, const double *Dskip,
                           const double *h0, int dt_softplus,
                           int64_t B, int64_t L, int64_t D, int64_t N,
                           double *y, double *h_final, int nthreads)
{
    if (!x || !dt || !Bm || !Cm || !A_log || !y) return -1;
    if (B < 0 || L < 0 || D < 0 || N <= 0 || N > 256) return -1;
    set_threads(nthreads);
    int64_t bd;
#pragma omp parallel for schedule(static)
    for (bd = 0; bd < B * D; ++bd) {
        const int64_t b = bd / D, d = bd % D;
        double h[256];
        double A[256];
        for (int64_t n = 0; n < N; ++n) {
            h[n] = h0 ? h0[(b * D + d) * N + n] : 0.0;
            A[n] = -exp(A_log[d * N + n]);
        }
        for (int64_t t = 0; t < L; ++t) {
            const int64_t i_bld = (b * L + t) * D + d;
            const int64_t i_bln = (b * L + t) * N;
            const double xv = x[i_bld];
            const double delta = dt_softplus ? softplus_thresholded(dt[i_bld]) : dt[i_bld];
            double yv = 0.0;
            for (int64_t n = 0; n < N; ++n) {
                const double a = exp(delta * A[n]);
                h[n] = a * h[n] + delta * Bm[i_bln + n] * xv;
                yv += Cm[i_bln + n] * h[n];
            }
            if (Dskip) yv += Dskip[d] * xv;
            if (z) {
                const double zv = z[i_bld];
                yv *= zv * logistic(zv);
            }
            y[i_bld] = yv;
        }
        if (h_final)
            for (int64_t n = 0; n < N; ++n) h_final[(b * D + d) * N + n] = h[n];
    }
    return 0;
}

/*
 * RG-LRU scalar-state scan, [RGLRU] RGLRU.step fallback, applied at every
 * time step of the sequence.  For each (b, d):
 *
 *   h = h0[b,d]                            (zero when h0 == NULL)
 *   for t in 0..L-1:
 *     eps  = c * r[b,t,d] * a_log[d]       so that a_t = exp(eps) = a^(c*r)
 *                                          with the per-channel base a = exp(a_log)
 *     a_t  = exp(eps)
 *     mult = sqrt(1 - a_t^2)  computed as sqrt(-expm1(2*eps)), the same
 *            number without the cancellation of 1 - a_t*a_t near a_t = 1
 *     h    = a_t * h + mult * (ig[b,t,d] * x[b,t,d])
 *     y[b,t,d] = h                         (dstate = 1: the readout sums one term)
 *   h_final[b,d] = h
 */
int lro_rglru_scan_ref(const double *x, const double *r, const double *ig,
                       const double *a_log, double c, const double *h0,
                       int64_t B, int64_t L, int64_t D,
                       double *y, double *h_final, int nthreads)
{
    if (!x || !r || !ig || !a_log || !y) return -1;
    if (B < 0 || L < 0 || D < 0) return -1;
    set_threads(nthreads);
    int64_t bd;
#pragma omp parallel for schedule(static)
    for (bd = 0; bd < B * D; ++bd) {
        const int64_t b = bd / D, d = bd % D;
        double h = h0 ? h0[b * D + d] : 0.0;
        for (int64_t t = 0; t < L; ++t) {
            const int64_t i = (b * L + t) * D + d;
            const double eps = c * r[i] * a_log[d];
            const double a_t = exp(eps);
            const double mult = sqrt(-expm1(2.0 * eps));
            h = a_t * h + mult * (ig[i] * x[i]);
            y[i] = h;
        }
        if (h_final) h_final[b * D + d] = h;
    }
    return 0;
}

/*
 * HGRN2 matrix-state recurrence, [HGRN2] class docstring and forward
 * description, one token at a time.  For each (b, head):
 *
 *   S = S0[b,head]  (dv x dk; zero when S0 == NULL)
 *   for t in 0..L-1:
 *     for i < dv, j < dk:  S[i][j] = g_t[i] * S[i][j] + v_t[i] * k_t[j]
 *                          (diag(g_t) scales the rows of S = sum v k^T)
 *     for i < dv:          o_t[i] = sum_j S[i][j] * q_t[j]
 *                          (readout o_t = S_t q_t, after the update at t)
 *   S_final[b,head] = S
 */
int lro_hgrn2_ref(const double *q, const double *k, const double *v,
                  const double *g, const double *S0,
                  int64_t B, int64_t L, int64_t H, int64_t dk, int64_t dv,
                  double *o, double *S_final, int nthreads)
{
    if (!q || !k || !v || !g || !o) return -1;
    if (B < 0 || L < 0 || H <= 0 || dk <= 0 || dv <= 0) return -1;
    set_threads(nthreads);
    int64_t bh;
    int failed = 0;
#pragma omp parallel for schedule(static)
    for (bh = 0; bh < B * H; ++bh) {
        const int64_t b = bh / H, hd = bh % H;
        double *S = (double *)malloc((size_t)(dv * dk) * sizeof(double));
        if (!S) {
#pragma omp atomic write
            failed = 1;
            continue;
        }
        const double *S0bh = S0 ? S0 + bh * dv * dk : NULL;
        for (int64_t e = 0; e < dv * dk; ++e) S[e] = S0bh ? S0bh[e] : 0.0;
        for (int64_t t = 0; t < L; ++t) {
            const double *qt = q + (b * L + t) * H * dk + hd * dk;
            const double *kt = k + (b * L + t) * H * dk + hd * dk;
            const double *vt = v + (b * L + t) * H * dv + hd * dv;
            const double *gt = g + (b * L + t) * H * dv + hd * dv;
            double *ot = o + (b * L + t) * H * dv + hd * dv;
            for (int64_t i = 0; i < dv; ++i) {
                double acc = 0.0;
                for (int64_t j = 0; j < dk; ++j) {
                    S[i * dk + j] = gt[i] * S[i * dk + j] + vt[i] * kt[j];
                    acc += S[i * dk + j] * qt[j];
                }
                ot[i] = acc;
            }
        }
        if (S_final)
            memcpy(S_final + bh * dv * dk, S, (size_t)(dv * dk) * sizeof(double));
        free(S);
    }
    return failed ? -1 : 0;
}

/*
 * MinMax recurrence, [MINMAX] MinMaxNeuron, one step at a time.  For each
 * (b, d):
 *
 *   x = x0[b,d]  (zero when x0 == NULL: the neuron's default initial state)
 *   for t in 0..L-1:
 *     x = max(min(r[b,t,d], x), s[b,t,d])   (the operator f(x) = max(min(a, x), b)
 *                                           with a = r_t, b = s_t)
 *     y[b,t,d] = x                          (forward returns the states after
 *                                           every step)
 *   x_final[b,d] = x
 *
 * min and max return one of their arguments exactly, so the result is
 * exact: every output equals one of the inputs or x0.  As torch.minimum and
 * torch.maximum in the page's apply, a NaN argument gives NaN.
 */
static double min_nan(double a, double b) { return isnan(a) || isnan(b) ? NAN : (a < b ? a : b); }
static double max_nan(double a, double b) { return isnan(a) || isnan(b) ? NAN : (a > b ? a : b); }

int lro_minmax_scan_ref(const double *r, const double *s, const double *x0,
                        int64_t B, int64_t L, int64_t D,
                        double *y, double *x_final, int nthreads)
{
    if (!r || !s || !y) return -1;
    if (B < 0 || L < 0 || D < 0) return -1;
    set_threads(nthreads);
    int64_t bd;
#pragma omp parallel for schedule(static)
    for (bd = 0; bd < B * D; ++bd) {
        const int64_t b = bd / D, d = bd % D;
        double x = x0 ? x0[b * D + d] : 0.0;
        for (int64_t t = 0; t < L; ++t) {
            const int64_t i = (b * L + t) * D + d;
            x = max_nan(min_nan(r[i], x), s[i]);
            y[i] = x;
        }
        if (x_final) x_final[b * D + d] = x;
    }
    return 0;
}
