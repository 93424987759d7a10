/*
 * Oracle for the logsumexp hot path: plain, slow, obviously correct CPU code.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the bench's
 * CPU-baseline leg may load this library.  The product (the CUDA library under
 * log_softmax_gb300/) shares no code with it and never calls it.
 *
 * Every value is computed in double from the fp32 inputs and returned in
 * double, so the comparison against the GPU's fp32 results sees the GPU's
 * error alone.  No blocking, fusion or reordering: each function is the
 * definition of its operation written out as nested loops.
 *
 * Sources (web pages on the POPCORNBENCH site, cited by title and passage):
 *  [P1] "FW-GLM-5-1 / l1_p29": custom kernel for torch.logsumexp(x, dim=0) on
 *       an (R,B,D) tensor; the task analysis states
 *       logsumexp(x) = max(x) + log(sum(exp(x - max(x)))) along dim 0.
 *  [P2] "Kimi-K2.6 / l1_p24": custom kernel for LogSoftmax over dim=1 of a
 *       (4096, 393216) tensor; the opening analysis states
 *       LogSoftmax(x_i) = x_i - max(x) - log(sum_j exp(x_j - max(x))).
 *  [P3] "Kimi-K2.6 / l2_p92": Conv2d -> GroupNorm -> Tanh -> HardSwish ->
 *       residual add (conv output + hardswish output) -> LogSumExp over the
 *       channel axis, keepdim.  Its GroupNorm discussion fixes the statistics:
 *       per (sample, group) mean and population variance (unbiased=False) over
 *       the group's C/G channels and all H*W positions, normalised as
 *       (x - mean) / sqrt(var + eps), then the per-channel affine weight and
 *       bias; HardSwish(t) = t * min(max(t + 3, 0), 6) / 6.  The chain's input
 *       is a Conv2d with 8 input and 64 output channels, kernel 3, stride 1,
 *       no padding (128 x 128 input planes give 126 x 126 outputs), with bias.
 *
 * Special values (the pages are silent; the readings taken here):
 *  - a NaN anywhere in the reduced set gives NaN;
 *  - else a +inf gives +inf;
 *  - else a set that is entirely -inf gives -inf (the limit of log 0);
 *  - -inf entries among finite ones contribute exp(-inf) = 0.
 * log_softmax is x_j - lse computed in IEEE double, so +inf rows give NaN at
 * the +inf entries and -inf elsewhere, and all -inf rows give NaN.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>

/* logsumexp of n doubles read at a stride: the identity of [P1] task analysis,
 * with the special-value readings above. */
static double lse_strided_double(const double* v, int64_t n, int64_t stride)
{
    int has_nan = 0, has_pinf = 0;
    double m = -INFINITY;
    for (int64_t k = 0; k < n; ++k) {
        double a = v[k * stride];
        if (isnan(a)) has_nan = 1;
        else if (a == INFINITY) has_pinf = 1;
        else if (a > m) m = a;
    }
    if (has_nan) return NAN;
    if (has_pinf) return INFINITY;
    if (m == -INFINITY) return -INFINITY;
    double s = 0.0;
    for (int64_t k = 0; k < n; ++k) s += exp(v[k * stride] - m);
    return m + log(s);
}

/* Same for float inputs, widened to double element by element. */
static double lse_strided_float(const float* v, int64_t n, int64_t stride)
{
    int has_nan = 0, has_pinf = 0;
    double m = -INFINITY;
    for (int64_t k = 0; k < n; ++k) {
        double a = (double)v[k * stride];
        if (isnan(a)) has_nan = 1;
        else if (a == INFINITY) has_pinf = 1;
        else if (a > m) m = a;
    }
    if (has_nan) return NAN;
    if (has_pinf) return INFINITY;
    if (m == -INFINITY) return -INFINITY;
    double s = 0.0;
    for (int64_t k = 0; k < n; ++k) s += exp((double)v[k * stride] - m);
    return m + log(s);
}

/* [P1]: out[o, i] = logsumexp over r of x[o, r, i], x contiguous (outer, R, inner).
 * Returns 0, or -1 on a bad argument. */
int oracle_lse_reduce(const float* x, double* out, int64_t outer, int64_t R, int64_t inner)
{
    if (!x || !out || outer < 0 || R <= 0 || inner < 0) return -1;
    for (int64_t o = 0; o < outer; ++o)
        for (int64_t i = 0; i < inner; ++i)
            out[o * inner + i] = lse_strided_float(x + o * R * inner + i, R, inner);
    return 0;
}

/* [P2]: per row, lse = logsumexp of the row; out[row, j] = x[row, j] - lse. */
int oracle_log_softmax(const float* x, double* out, int64_t rows, int64_t cols)
{
    if (!x || !out || rows < 0 || cols <= 0) return -1;
    for (int64_t r = 0; r < rows; ++r) {
        const float* row = x + r * cols;
        double lse = lse_strided_float(row, cols, 1);
        for (int64_t j = 0; j < cols; ++j) out[r * cols + j] = (double)row[j] - lse;
    }
    return 0;
}

/* [P2] row statistic alone: lse[row] = logsumexp of the row. */
int oracle_row_lse(const float* x, double* lse, int64_t rows, int64_t cols)
{
    if (!x || !lse || rows < 0 || cols <= 0) return -1;
    for (int64_t r = 0; r < rows; ++r) lse[r] = lse_strided_float(x + r * cols, cols, 1);
    return 0;
}

/* [P3] GroupNorm statistics for one (n, g): mean and population variance of the
 * count = (C/G)*HW contiguous values starting at p. */
static void group_stats(const float* p, int64_t count, double* mean_out, double* var_out)
{
    double sum = 0.0;
    for (int64_t k = 0; k < count; ++k) sum += (double)p[k];
    double mean = sum / (double)count;
    double sq = 0.0;
    for (int64_t k = 0; k < count; ++k) {
        double d = (double)p[k] - mean;
        sq += d * d;
    }
    *mean_out = mean;
    *var_out = sq / (double)count;
}

/* [P3] HardSwish as the page writes it: t * clamp(t + 3, 0, 6) / 6. */
static double hardswish(double t)
{
    double c = t + 3.0;
    if (c < 0.0) c = 0.0;
    if (c > 6.0) c = 6.0;
    return t * c / 6.0;
}

/* [P3]: y is [N, C, HW] (NCHW with H*W flattened); gamma, beta are [C];
 * out is [N, HW] (= [N, 1, H, W]).  For each (n, p):
 *   z_c = (y - mean_g) / sqrt(var_g + eps) * gamma_c + beta_c
 *   r_c = y_c + hardswish(tanh(z_c))
 *   out = logsumexp over c of r_c.
 * Also writes the statistics when mean_out / rstd_out are non-null ([N, G]). */
int oracle_gn_act_lse(const float* y, const float* gamma, const float* beta, double* out,
                      int64_t N, int64_t C, int64_t HW, int64_t G, double eps,
                      double* mean_out, double* rstd_out)
{
    if (!y || !gamma || !beta || !out || N < 0 || C <= 0 || HW < 0 || G <= 0 || C % G != 0)
        return -1;
    const int64_t cpg = C / G;
    double* mean = (double*)malloc(sizeof(double) * (size_t)(G > 0 ? G : 1));
    double* rstd = (double*)malloc(sizeof(double) * (size_t)(G > 0 ? G : 1));
    double* r = (double*)malloc(sizeof(double) * (size_t)C);
    if (!mean || !rstd || !r) { free(mean); free(rstd); free(r); return -2; }
    for (int64_t n = 0; n < N; ++n) {
        const float* yn = y + n * C * HW;
        for (int64_t g = 0; g < G; ++g) {
            double mu, var;
            group_stats(yn + g * cpg * HW, cpg * HW, &mu, &var);
            mean[g] = mu;
            rstd[g] = 1.0 / sqrt(var + eps);
            if (mean_out) mean_out[n * G + g] = mean[g];
            if (rstd_out) rstd_out[n * G + g] = rstd[g];
        }
        for (int64_t p = 0; p < HW; ++p) {
            for (int64_t c = 0; c < C; ++c) {
                int64_t g = c / cpg;
                double v = (double)yn[c * HW + p];
                double z = (v - mean[g]) * rstd[g] * (double)gamma[c] + (double)beta[c];
                r[c] = v + hardswish(tanh(z));
            }
            out[n * HW + p] = lse_strided_double(r, C, 1);
        }
    }
    free(mean);
    free(rstd);
    free(r);
    return 0;
}

/* ------------------------------------------------------------------------
 * Neighbouring operations of the same method.
 * ------------------------------------------------------------------------ */

/* Softmax of each row ([P2] describes it beside LogSoftmax as exp(x - m)
 * scaled by 1 / sum): out[row, j] = exp(x[row, j] - lse(row)). */
int oracle_softmax(const float* x, double* out, int64_t rows, int64_t cols)
{
    if (!x || !out || rows < 0 || cols <= 0) return -1;
    for (int64_t r = 0; r < rows; ++r) {
        const float* row = x + r * cols;
        double lse = lse_strided_float(row, cols, 1);
        for (int64_t j = 0; j < cols; ++j) out[r * cols + j] = exp((double)row[j] - lse);
    }
    return 0;
}

/* LogSoftmax along the middle axis of a contiguous (outer, R, inner) tensor:
 * out[o, r, i] = x[o, r, i] - lse over r' of x[o, r', i]. */
int oracle_log_softmax_dim(const float* x, double* out, int64_t outer, int64_t R, int64_t inner)
{
    if (!x || !out || outer < 0 || R <= 0 || inner < 0) return -1;
    for (int64_t o = 0; o < outer; ++o)
        for (int64_t i = 0; i < inner; ++i) {
            const float* col = x + o * R * inner + i;
            double lse = lse_strided_float(col, R, inner);
            for (int64_t r = 0; r < R; ++r)
                out[(o * R + r) * inner + i] = (double)col[r * inner] - lse;
        }
    return 0;
}

/* [P3] GroupNorm alone (act = 0): out = (y - mean_g) / sqrt(var_g + eps) * gamma_c + beta_c,
 * or the chain without the channel reduction (act = 1):
 * out = y + hardswish(tanh(GroupNorm(y))).  y, out are [N, C, HW]. */
static int group_norm_impl(const float* y, const float* gamma, const float* beta, double* out,
                           int64_t N, int64_t C, int64_t HW, int64_t G, double eps, int act)
{
    if (!y || !gamma || !beta || !out || N < 0 || C <= 0 || HW < 0 || G <= 0 || C % G != 0)
        return -1;
    const int64_t cpg = C / G;
    for (int64_t n = 0; n < N; ++n)
        for (int64_t g = 0; g < G; ++g) {
            const float* span = y + (n * C + g * cpg) * HW;
            double mu, var;
            group_stats(span, cpg * HW, &mu, &var);
            double rs = 1.0 / sqrt(var + eps);
            for (int64_t cc = 0; cc < cpg; ++cc) {
                int64_t c = g * cpg + cc;
                for (int64_t p = 0; p < HW; ++p) {
                    double v = (double)y[(n * C + c) * HW + p];
                    double z = (v - mu) * rs * (double)gamma[c] + (double)beta[c];
                    out[(n * C + c) * HW + p] = act ? v + hardswish(tanh(z)) : z;
                }
            }
        }
    return 0;
}

int oracle_group_norm(const float* y, const float* gamma, const float* beta, double* out,
                      int64_t N, int64_t C, int64_t HW, int64_t G, double eps)
{
    return group_norm_impl(y, gamma, beta, out, N, C, HW, G, eps, 0);
}

int oracle_gn_act_residual(const float* y, const float* gamma, const float* beta, double* out,
                           int64_t N, int64_t C, int64_t HW, int64_t G, double eps)
{
    return group_norm_impl(y, gamma, beta, out, N, C, HW, G, eps, 1);
}

/* [P3] Conv2d as the chain's first layer: valid cross-correlation, stride 1,
 * no padding, with bias.  x is [N, Cin, H, W], w is [Cout, Cin, KH, KW], b is
 * [Cout]; y is [N, Cout, H - KH + 1, W - KW + 1]:
 *   y[n,co,i,j] = b[co] + sum over ci, u, v of w[co,ci,u,v] * x[n,ci,i+u,j+v]
 * accumulated in double. */
int oracle_conv2d(const float* x, const float* w, const float* b, double* y, int64_t N, int64_t Cin,
                  int64_t H, int64_t W, int64_t Cout, int64_t KH, int64_t KW)
{
    if (!x || !w || !b || !y || N < 0 || Cin <= 0 || Cout <= 0 || KH <= 0 || KW <= 0 || H < KH || W < KW)
        return -1;
    const int64_t OH = H - KH + 1, OW = W - KW + 1;
    for (int64_t n = 0; n < N; ++n)
        for (int64_t co = 0; co < Cout; ++co)
            for (int64_t i = 0; i < OH; ++i)
                for (int64_t j = 0; j < OW; ++j) {
                    double acc = (double)b[co];
                    for (int64_t ci = 0; ci < Cin; ++ci)
                        for (int64_t u = 0; u < KH; ++u)
                            for (int64_t v = 0; v < KW; ++v)
                                acc += (double)w[((co * Cin + ci) * KH + u) * KW + v] *
                                       (double)x[((n * Cin + ci) * H + i + u) * W + j + v];
                    y[((n * Cout + co) * OH + i) * OW + j] = acc;
                }
    return 0;
}

/* [P3] the whole chain from the convolution's input: y = Conv2d(x) (3 x 3,
 * valid, bias) kept in double, then the GroupNorm -> tanh -> hardswish ->
 * residual -> channel logsumexp steps of oracle_gn_act_lse on that y.
 * out is [N, OH * OW]. */
int oracle_conv_gn_act_lse(const float* x, const float* w, const float* b, const float* gamma,
                           const float* beta, double* out, int64_t N, int64_t Cin, int64_t H,
                           int64_t W, int64_t Cout, int64_t G, double eps)
{
    if (!gamma || !beta || !out || G <= 0 || Cout % G != 0 || H < 3 || W < 3) return -1;
    const int64_t OH = H - 2, OW = W - 2, HW = OH * OW, C = Cout, cpg = C / G;
    double* y = (double*)malloc(sizeof(double) * (size_t)(N * C * HW > 0 ? N * C * HW : 1));
    double* r = (double*)malloc(sizeof(double) * (size_t)C);
    double* mean = (double*)malloc(sizeof(double) * (size_t)G);
    double* rstd = (double*)malloc(sizeof(double) * (size_t)G);
    if (!y || !r || !mean || !rstd) { free(y); free(r); free(mean); free(rstd); return -2; }
    int rc = oracle_conv2d(x, w, b, y, N, Cin, H, W, Cout, 3, 3);
    for (int64_t n = 0; rc == 0 && n < N; ++n) {
        const double* yn = y + n * C * HW;
        for (int64_t g = 0; g < G; ++g) {
            const double* span = yn + g * cpg * HW;
            const int64_t count = cpg * HW;
            double sum = 0.0;
            for (int64_t k = 0; k < count; ++k) sum += span[k];
            const double mu = sum / (double)count;
            double sq = 0.0;
            for (int64_t k = 0; k < count; ++k) sq += (span[k] - mu) * (span[k] - mu);
            mean[g] = mu;
            rstd[g] = 1.0 / sqrt(sq / (double)count + eps);
        }
        for (int64_t p = 0; p < HW; ++p) {
            for (int64_t c = 0; c < C; ++c) {
                const int64_t g = c / cpg;
                const double v = yn[c * HW + p];
                const double z = (v - mean[g]) * rstd[g] * (double)gamma[c] + (double)beta[c];
                r[c] = v + hardswish(tanh(z));
            }
            out[n * HW + p] = lse_strided_double(r, C, 1);
        }
    }
    free(y);
    free(r);
    free(mean);
    free(rstd);
    return rc;
}
