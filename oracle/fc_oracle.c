/*
 * fc_oracle.c -- the oracle: a plain, slow, fp64 CPU statement of the three
 * fused operator chains.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may call, link or
 * execute this file; only the tests, the package's smoke check and the
 * benchmark's CPU-baseline leg do.  It shares no code, header or constant
 * table with the CUDA library.
 *
 * Every function is the plain definition written out, in double precision,
 * with one fixed summation order per output.  Inputs arrive as fp32 arrays
 * holding the exact stored values (bf16 inputs are widened exactly to fp32 by
 * the input generator), and every product and sum is taken in double.
 *
 * Sources (the pages are three reasoning traces titled by their problem):
 *  - Conv2d -> GELU -> adaptive_avg_pool2d(1) -> squeeze (page "Kimi-K2.6 l2_p67"):
 *    problem statement; "exact GELU vs tanh approximation" discussion; the
 *    global average over the OH x OW plane.
 *  - Conv2d -> Mish -> Mish (page "Kimi-K2.6 l2_p4"): problem statement; the
 *    numerically stable softplus max(x,0) + log1p(exp(-|x|)).
 *  - Linear -> *scale -> x + x -> clamp -> logsumexp(dim 1) -> x * mish(x)
 *    (page "Kimi-K2.6 l2_p22"): problem statement (the module's forward); the
 *    stable "max + log sum exp(x - max)" logsumexp discussion.
 *
 * Parity pins for every function live in tests/test_oracle_pins.py.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#ifdef _OPENMP
#include <omp.h>
#endif

enum { ORACLE_ACT_NONE = -1, ORACLE_ACT_GELU = 0, ORACLE_ACT_MISH = 1, ORACLE_ACT_MISH_MISH = 2, ORACLE_ACT_GELU_TANH = 3 };

/* ---------------------------------------------------------------- pointwise */

/* Exact GELU, torch's default approximate='none': 0.5 v (1 + erf(v / sqrt 2)).
 * Conv->GELU->pool page: the trace settles on the erf form after rejecting
 * the tanh approximation as a mismatch. */
double oracle_gelu(double v) { return 0.5 * v * (1.0 + erf(v / sqrt(2.0))); }

/* tanh-approximate GELU, torch's approximate='tanh':
 * 0.5 v (1 + tanh(sqrt(2/pi) (v + 0.044715 v^3))) -- the variant the Conv->GELU->pool
 * page's trace weighs (and rejects for that module) against the exact form. */
double oracle_gelu_tanh(double v)
{
    return 0.5 * v * (1.0 + tanh(sqrt(2.0 / 3.14159265358979323846) * (v + 0.044715 * v * v * v)));
}

/* softplus(z) = log(1 + e^z), in the overflow-safe form the Mish page uses:
 * max(z, 0) + log1p(exp(-|z|)). */
double oracle_softplus(double z) { return fmax(z, 0.0) + log1p(exp(-fabs(z))); }

/* Mish(z) = z * tanh(softplus(z)) (Conv->Mish->Mish page, problem statement). */
double oracle_mish(double z) { return z * tanh(oracle_softplus(z)); }

double oracle_act(int act, double v)
{
    switch (act) {
    case ORACLE_ACT_GELU: return oracle_gelu(v);
    case ORACLE_ACT_MISH: return oracle_mish(v);
    case ORACLE_ACT_MISH_MISH: return oracle_mish(oracle_mish(v));
    case ORACLE_ACT_GELU_TANH: return oracle_gelu_tanh(v);
    default: return v;
    }
}

/* ------------------------------------------------------------------- conv */

/* Pre-activation of Conv2d(k=3, stride 1, padding p, dilation 1, groups 1)
 * with bias at one output point: cross-correlation (no kernel flip) over the
 * input extended by p zero rows / columns on every side (padding_mode zeros),
 *   v = b[co] + sum_{ci} sum_{kh<3} sum_{kw<3} x[n,ci,oh+kh-p,ow+kw-p] * w[co,ci,kh,kw],
 * terms outside the input omitted.  x is NCHW, w is OIHW, both contiguous.
 * The pages' operators use p = 0 (output (H-2) x (W-2)); p > 0 is the general
 * padding variant (output (H+2p-2) x (W+2p-2)). */
double oracle_conv3x3_point(const float* x, const float* w, const float* b,
                            int Cin, int H, int W, int pad, int n, int co, int oh, int ow)
{
    double acc = (double)b[co];
    for (int ci = 0; ci < Cin; ++ci) {
        const float* xp = x + ((int64_t)n * Cin + ci) * H * (int64_t)W;
        const float* wp = w + ((int64_t)co * Cin + ci) * 9;
        for (int kh = 0; kh < 3; ++kh) {
            const int ih = oh + kh - pad;
            if (ih < 0 || ih >= H) continue;
            for (int kw = 0; kw < 3; ++kw) {
                const int iw = ow + kw - pad;
                if (iw < 0 || iw >= W) continue;
                acc += (double)xp[(int64_t)ih * W + iw] * (double)wp[kh * 3 + kw];
            }
        }
    }
    return acc;
}

/* Full pre-activation output, (N, Cout, H+2p-2, W+2p-2). */
void oracle_conv3x3_preact(const float* x, const float* w, const float* b, double* out,
                           int N, int Cin, int H, int W, int Cout, int pad)
{
    const int OH = H + 2 * pad - 2, OW = W + 2 * pad - 2;
#pragma omp parallel for collapse(2) schedule(static)
    for (int n = 0; n < N; ++n)
        for (int co = 0; co < Cout; ++co) {
            double* o = out + ((int64_t)n * Cout + co) * OH * (int64_t)OW;
            for (int oh = 0; oh < OH; ++oh)
                for (int ow = 0; ow < OW; ++ow)
                    o[(int64_t)oh * OW + ow] = oracle_conv3x3_point(x, w, b, Cin, H, W, pad, n, co, oh, ow);
        }
}

/* act(conv + bias), full output (N, Cout, H+2p-2, W+2p-2).  With act = Mish twice
 * and p = 0 this is the Conv->Mish->Mish chain. */
void oracle_conv3x3_act(const float* x, const float* w, const float* b, double* out,
                        int N, int Cin, int H, int W, int Cout, int pad, int act)
{
    const int OH = H + 2 * pad - 2, OW = W + 2 * pad - 2;
#pragma omp parallel for collapse(2) schedule(static)
    for (int n = 0; n < N; ++n)
        for (int co = 0; co < Cout; ++co) {
            double* o = out + ((int64_t)n * Cout + co) * OH * (int64_t)OW;
            for (int oh = 0; oh < OH; ++oh)
                for (int ow = 0; ow < OW; ++ow)
                    o[(int64_t)oh * OW + ow] =
                        oracle_act(act, oracle_conv3x3_point(x, w, b, Cin, H, W, pad, n, co, oh, ow));
        }
}

/* The same chain at a list of flat output indices into (N, Cout, H+2p-2, W+2p-2). */
void oracle_conv3x3_act_at(const float* x, const float* w, const float* b,
                           int N, int Cin, int H, int W, int Cout, int pad, int act,
                           const int64_t* idx, int64_t count, double* out)
{
    const int64_t OH = H + 2 * pad - 2, OW = W + 2 * pad - 2;
    (void)N;
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < count; ++i) {
        int64_t f = idx[i];
        int ow = (int)(f % OW); f /= OW;
        int oh = (int)(f % OH); f /= OH;
        int co = (int)(f % Cout);
        int n = (int)(f / Cout);
        out[i] = oracle_act(act, oracle_conv3x3_point(x, w, b, Cin, H, W, pad, n, co, oh, ow));
    }
}

/* Global average pool of act(conv + bias) over the OH x OW plane (adaptive
 * average pool to 1x1, then squeeze), y (N, Cout):
 *   y[n,co] = (sum_{oh,ow} act(v[n,co,oh,ow])) / (OH OW),  OH = H+2p-2, OW = W+2p-2,
 * summed in row-major (oh, ow) order. */
static double pool_one(const float* x, const float* w, const float* b,
                       int Cin, int H, int W, int pad, int act, int n, int co)
{
    const int OH = H + 2 * pad - 2, OW = W + 2 * pad - 2;
    double s = 0.0;
    for (int oh = 0; oh < OH; ++oh)
        for (int ow = 0; ow < OW; ++ow)
            s += oracle_act(act, oracle_conv3x3_point(x, w, b, Cin, H, W, pad, n, co, oh, ow));
    return s / ((double)OH * (double)OW);
}

void oracle_conv3x3_act_pool(const float* x, const float* w, const float* b, double* y,
                             int N, int Cin, int H, int W, int Cout, int pad, int act)
{
#pragma omp parallel for collapse(2) schedule(dynamic, 1)
    for (int n = 0; n < N; ++n)
        for (int co = 0; co < Cout; ++co)
            y[(int64_t)n * Cout + co] = pool_one(x, w, b, Cin, H, W, pad, act, n, co);
}

/* The pool at a list of flat (n * Cout + co) indices. */
void oracle_conv3x3_act_pool_at(const float* x, const float* w, const float* b,
                                int N, int Cin, int H, int W, int Cout, int pad, int act,
                                const int64_t* idx, int64_t count, double* out)
{
    (void)N;
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t i = 0; i < count; ++i)
        out[i] = pool_one(x, w, b, Cin, H, W, pad, act, (int)(idx[i] / Cout), (int)(idx[i] % Cout));
}

/* ----------------------------------------------------------------- linear */

/* logsumexp of a row, the two-pass stable form of the Linear page:
 * m = max_j t_j, then m + log(sum_j exp(t_j - m)). */
double oracle_logsumexp(const double* t, int64_t n)
{
    double m = t[0];
    for (int64_t j = 1; j < n; ++j) m = fmax(m, t[j]);
    double s = 0.0;
    for (int64_t j = 0; j < n; ++j) s += exp(t[j] - m);
    return m + log(s);
}

/* One row of the Linear chain (Linear page, the module's forward):
 *   t_j = b_j + sum_k x[m,k] W[j,k]        (nn.Linear: x W^T + b)
 *   t = t * scale;  t = t + t;             (the two scalings, in this order)
 *   t = min(max(t, lo), hi)                (torch.clamp, inclusive bounds)
 *   l = logsumexp_j t_j                    (dim 1, keepdim)
 *   y = l * mish(l).
 * `t` is caller scratch of Nout doubles.  Returns y; writes l to *lse_out. */
static double linear_row(const float* x, const float* Wt, const float* b, int K, int Nout,
                         double scale, double lo, double hi, int m, double* t, double* lse_out)
{
    const float* xr = x + (int64_t)m * K;
    for (int j = 0; j < Nout; ++j) {
        const float* wr = Wt + (int64_t)j * K;
        double acc = (double)b[j];
        for (int k = 0; k < K; ++k) acc += (double)xr[k] * (double)wr[k];
        double u = acc * scale;
        u = u + u;
        t[j] = fmin(fmax(u, lo), hi);
    }
    double l = oracle_logsumexp(t, Nout);
    if (lse_out) *lse_out = l;
    return l * oracle_mish(l);
}

/* y (M) and optionally lse (M) for a list of rows (all rows when rows == NULL). */
int oracle_linear_lse_mish_rows(const float* x, const float* Wt, const float* b,
                                int M, int K, int Nout, double scale, double lo, double hi,
                                const int64_t* rows, int64_t count, double* y, double* lse)
{
    int failed = 0;
    if (rows == NULL) count = M;
#pragma omp parallel reduction(| : failed)
    {
        double* t = (double*)malloc(sizeof(double) * (size_t)Nout);
        if (t == NULL) {
            failed = 1;
        } else {
#pragma omp for schedule(dynamic, 1)
            for (int64_t i = 0; i < count; ++i) {
                int m = rows ? (int)rows[i] : (int)i;
                y[i] = linear_row(x, Wt, b, K, Nout, scale, lo, hi, m, t, lse ? &lse[i] : NULL);
            }
            free(t);
        }
    }
    return failed ? -1 : 0;
}

/* ------------------------------------------------ standalone epilogues
 * The pages' own deliverables are epilogue kernels over an already computed
 * contraction output: GELU + global mean over each (n, c) plane (Conv->GELU->pool
 * page, its fused epilogue kernel), Mish twice elementwise (Conv->Mish->Mish page,
 * its elementwise kernel), and the scale / clamp / logsumexp / x*mish(x) row kernel
 * (Linear page, its row kernel).  Plain definitions over fp32 inputs, fp64 math. */

/* out[i] = act(v[i]). */
void oracle_act_map(const float* v, double* out, int64_t n, int act)
{
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < n; ++i) out[i] = oracle_act(act, (double)v[i]);
}

/* out[p] = (sum_{i < plane} act(v[p * plane + i])) / plane for each of `planes` planes. */
void oracle_act_mean(const float* v, double* out, int64_t planes, int64_t plane, int act)
{
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t p = 0; p < planes; ++p) {
        const float* q = v + p * plane;
        double s = 0.0;
        for (int64_t i = 0; i < plane; ++i) s += oracle_act(act, (double)q[i]);
        out[p] = s / (double)plane;
    }
}

/* The Linear chain's tail on an already computed row y (bias included):
 * t = y * scale; t = t + t; t = clamp(t, lo, hi); l = logsumexp(t); out = l * mish(l). */
int oracle_scale_clamp_lse_mish_rows(const float* y, int M, int N, double scale, double lo, double hi, double* out)
{
    int failed = 0;
#pragma omp parallel reduction(| : failed)
    {
        double* t = (double*)malloc(sizeof(double) * (size_t)N);
        if (t == NULL) {
            failed = 1;
        } else {
#pragma omp for schedule(dynamic, 1)
            for (int m = 0; m < M; ++m) {
                const float* r = y + (int64_t)m * N;
                for (int j = 0; j < N; ++j) {
                    double u = (double)r[j] * scale;
                    u = u + u;
                    t[j] = fmin(fmax(u, lo), hi);
                }
                const double l = oracle_logsumexp(t, N);
                out[m] = l * oracle_mish(l);
            }
            free(t);
        }
    }
    return failed ? -1 : 0;
}

int oracle_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* Threads for the following calls (n >= 1).  Every unit (image and channel, pixel, row)
 * is summed in a fixed order by one thread, so the results do not depend on it. */
void oracle_set_threads(int n)
{
#ifdef _OPENMP
    if (n >= 1) omp_set_num_threads(n);
#else
    (void)n;
#endif
}
