/*
 * Row-normalisation oracle: plain, single-threaded FP64 C.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the checker the CUDA library is
 * compared against; it is loaded only by the tests, by the smoke check and by
 * the benchmark's CPU-baseline leg.  The library itself never calls it, shares
 * no header, helper or constant with it, and has no CPU fallback.
 *
 * Every function is the textbook definition written out, one row at a time:
 * inputs are the exact FP32 values given to the GPU, widened to double; every
 * sum is a left-to-right FP64 loop; nothing is blocked, fused or reordered.
 * Outputs are FP64.  Layout: row-major, row i starts at element i*width.
 *
 * Sources (pages of the "tile_compiler_row" engineering notes):
 *  - residual LayerNorm: "Residual LayerNorm shared-Tile materialization
 *    search", section "Structural finding" -- c = x + residual,
 *    mean = sum(c)/width, centered = c - mean,
 *    variance = sum(centered^2)/width, y = centered / sqrt(variance + 1e-5).
 *  - LayerNorm (no affine): the same map without the residual term
 *    ("Cooperating-program packing", section "Validation": no-affine
 *    LayerNorm; "Immutable input reuse in Metal reductions", section
 *    "What the transformation actually preserves").
 *  - RMSNorm and softmax: named on "Immutable input reuse in Metal
 *    reductions" (fixed-width results table) without a printed formula.
 *    Readings taken: RMSNorm y = x / sqrt(mean(x^2) + eps) with no weight;
 *    softmax subtracts the row maximum (the max collective listed in
 *    "Cooperating-program packing", section "Implementation boundary")
 *    before exponentiating: y = exp(x - max) / sum(exp(x - max)).
 *
 * Build: gcc -O2 -std=c11 -ffp-contract=off -fPIC -shared oracle.c -lm
 * (no fused multiply-add contraction, so x86 and Arm hosts agree bit for bit).
 */
#include <math.h>

/* y = (c - mean) / sqrt(var + eps), c = x + r, centred biased variance. */
void oracle_residual_layernorm(const float *x, const float *r, double *y,
                               long rows, long width, double eps)
{
    for (long i = 0; i < rows; ++i) {
        const float *xi = x + i * width;
        const float *ri = r + i * width;
        double *yi = y + i * width;

        double sum = 0.0;
        for (long j = 0; j < width; ++j)
            sum += (double)xi[j] + (double)ri[j];
        double mean = sum / (double)width;

        double sq = 0.0;
        for (long j = 0; j < width; ++j) {
            double centered = ((double)xi[j] + (double)ri[j]) - mean;
            sq += centered * centered;
        }
        double variance = sq / (double)width;

        double denom = sqrt(variance + eps);
        for (long j = 0; j < width; ++j)
            yi[j] = (((double)xi[j] + (double)ri[j]) - mean) / denom;
    }
}

/* y = (x - mean) / sqrt(var + eps), centred biased variance, no affine. */
void oracle_layernorm(const float *x, double *y, long rows, long width, double eps)
{
    for (long i = 0; i < rows; ++i) {
        const float *xi = x + i * width;
        double *yi = y + i * width;

        double sum = 0.0;
        for (long j = 0; j < width; ++j)
            sum += (double)xi[j];
        double mean = sum / (double)width;

        double sq = 0.0;
        for (long j = 0; j < width; ++j) {
            double centered = (double)xi[j] - mean;
            sq += centered * centered;
        }
        double variance = sq / (double)width;

        double denom = sqrt(variance + eps);
        for (long j = 0; j < width; ++j)
            yi[j] = ((double)xi[j] - mean) / denom;
    }
}

/* y = x / sqrt(mean(x^2) + eps), no weight. */
void oracle_rmsnorm(const float *x, double *y, long rows, long width, double eps)
{
    for (long i = 0; i < rows; ++i) {
        const float *xi = x + i * width;
        double *yi = y + i * width;

        double sq = 0.0;
        for (long j = 0; j < width; ++j)
            sq += (double)xi[j] * (double)xi[j];
        double mean_square = sq / (double)width;

        double denom = sqrt(mean_square + eps);
        for (long j = 0; j < width; ++j)
            yi[j] = (double)xi[j] / denom;
    }
}

/* y = exp(x - max) / sum(exp(x - max)). */
void oracle_softmax(const float *x, double *y, long rows, long width)
{
    for (long i = 0; i < rows; ++i) {
        const float *xi = x + i * width;
        double *yi = y + i * width;

        double m = (double)xi[0];
        for (long j = 1; j < width; ++j)
            if ((double)xi[j] > m)
                m = (double)xi[j];

        double total = 0.0;
        for (long j = 0; j < width; ++j)
            total += exp((double)xi[j] - m);

        for (long j = 0; j < width; ++j)
            yi[j] = exp((double)xi[j] - m) / total;
    }
}

/* ------------------------------------------------------------------------
 * Further operations named on the pages.
 *
 *  - affine LayerNorm: the runner's tolerance table of "Cooperating-program
 *    packing", section "Predeclared comparison and measurement", lists
 *    affine LayerNorm; the formula is not printed.  Reading taken: the
 *    LayerNorm above, then y * gamma[j] + beta[j] (beta optional), with the
 *    residual added first when one is given.  Weighted RMSNorm likewise:
 *    x / sqrt(mean(x^2) + eps) * gamma[j].
 *  - row sum and paired row min/max: the operators "sum" and "paired min/max"
 *    of "Cooperating-program packing", section "Validation" (sum is also the
 *    identical-source control of "Immutable input reuse in Metal
 *    reductions").
 *  - sigmoid and tanh-approximate GELU, each with its derivative:
 *    "Multi-output pointwise fusion: evidence and limits", section
 *    "Measurement definitions and population".  sigmoid(x) = 1/(1+exp(-x)),
 *    derivative s(1-s).  tanh GELU (Hendrycks and Gimpel 2016):
 *    g(x) = x/2 (1 + tanh(u)), u = sqrt(2/pi) (x + 0.044715 x^3), derivative
 *    g'(x) = (1 + tanh(u))/2 + x/2 (1 - tanh(u)^2) sqrt(2/pi) (1 + 3*0.044715 x^2).
 * ------------------------------------------------------------------------ */

/* y = LayerNorm(x [+ r]) * gamma + beta; r and beta may be NULL. */
void oracle_layernorm_affine(const float *x, const float *r, const float *gamma,
                             const float *beta, double *y, long rows, long width, double eps)
{
    for (long i = 0; i < rows; ++i) {
        const float *xi = x + i * width;
        const float *ri = r ? r + i * width : 0;
        double *yi = y + i * width;

        double sum = 0.0;
        for (long j = 0; j < width; ++j)
            sum += (double)xi[j] + (ri ? (double)ri[j] : 0.0);
        double mean = sum / (double)width;

        double sq = 0.0;
        for (long j = 0; j < width; ++j) {
            double centered = ((double)xi[j] + (ri ? (double)ri[j] : 0.0)) - mean;
            sq += centered * centered;
        }
        double variance = sq / (double)width;

        double denom = sqrt(variance + eps);
        for (long j = 0; j < width; ++j) {
            double normed = (((double)xi[j] + (ri ? (double)ri[j] : 0.0)) - mean) / denom;
            yi[j] = normed * (double)gamma[j] + (beta ? (double)beta[j] : 0.0);
        }
    }
}

/* y = x / sqrt(mean(x^2) + eps) * gamma. */
void oracle_rmsnorm_weighted(const float *x, const float *gamma, double *y, long rows,
                             long width, double eps)
{
    for (long i = 0; i < rows; ++i) {
        const float *xi = x + i * width;
        double *yi = y + i * width;

        double sq = 0.0;
        for (long j = 0; j < width; ++j)
            sq += (double)xi[j] * (double)xi[j];
        double mean_square = sq / (double)width;

        double denom = sqrt(mean_square + eps);
        for (long j = 0; j < width; ++j)
            yi[j] = (double)xi[j] / denom * (double)gamma[j];
    }
}

/* s[i] = sum_j x[i][j]. */
void oracle_row_sum(const float *x, double *s, long rows, long width)
{
    for (long i = 0; i < rows; ++i) {
        const float *xi = x + i * width;
        double sum = 0.0;
        for (long j = 0; j < width; ++j)
            sum += (double)xi[j];
        s[i] = sum;
    }
}

/* mn[i] = min_j x[i][j], mx[i] = max_j x[i][j]. */
void oracle_row_minmax(const float *x, double *mn, double *mx, long rows, long width)
{
    for (long i = 0; i < rows; ++i) {
        const float *xi = x + i * width;
        double lo = (double)xi[0], hi = (double)xi[0];
        for (long j = 1; j < width; ++j) {
            if ((double)xi[j] < lo)
                lo = (double)xi[j];
            if ((double)xi[j] > hi)
                hi = (double)xi[j];
        }
        mn[i] = lo;
        mx[i] = hi;
    }
}

/* y = sigmoid(x), dy = sigmoid'(x), elementwise over n values. */
void oracle_sigmoid_pair(const float *x, double *y, double *dy, long n)
{
    for (long k = 0; k < n; ++k) {
        double s = 1.0 / (1.0 + exp(-(double)x[k]));
        y[k] = s;
        dy[k] = s * (1.0 - s);
    }
}

/* y = tanh-approximate GELU(x), dy = its derivative, elementwise. */
void oracle_gelu_tanh_pair(const float *x, double *y, double *dy, long n)
{
    const double c = sqrt(2.0 / 3.14159265358979323846);
    const double a = 0.044715;
    for (long k = 0; k < n; ++k) {
        double v = (double)x[k];
        double u = c * (v + a * v * v * v);
        double t = tanh(u);
        y[k] = 0.5 * v * (1.0 + t);
        dy[k] = 0.5 * (1.0 + t) + 0.5 * v * (1.0 - t * t) * c * (1.0 + 3.0 * a * v * v);
    }
}

/* ------------------------------------------------------------------------
 * Backward passes (gradients with respect to the inputs and the per-column
 * parameters).  The pages do not cover backward normalisation ("Residual
 * LayerNorm shared-Tile materialization search", last paragraph); these are
 * the chain rule applied to the forward definitions above, with
 * xhat = (x - mean) * rstd (LayerNorm) or x * rstd (RMSNorm),
 * rstd = 1/sqrt(var + eps) or 1/sqrt(mean(x^2) + eps), and g = dy * gamma
 * (gamma = 1 when NULL):
 *   LayerNorm:  dx = rstd * (g - mean(g) - xhat * mean(g * xhat))
 *   RMSNorm:    dx = rstd * (g - xhat * mean(g * xhat))
 *   softmax:    dx = y * (dy - sum(dy * y))        (from the forward output y)
 *   parameters: dgamma[j] = sum_rows dy * xhat,  dbeta[j] = sum_rows dy.
 * ------------------------------------------------------------------------ */

/* dx of y = LayerNorm(x) * gamma (+ beta); gamma may be NULL. */
void oracle_layernorm_backward(const float *x, const float *gamma, const float *dy, double *dx,
                               long rows, long width, double eps)
{
    for (long i = 0; i < rows; ++i) {
        const float *xi = x + i * width;
        const float *di = dy + i * width;
        double *out = dx + i * width;

        double sum = 0.0;
        for (long j = 0; j < width; ++j)
            sum += (double)xi[j];
        double mean = sum / (double)width;
        double sq = 0.0;
        for (long j = 0; j < width; ++j)
            sq += ((double)xi[j] - mean) * ((double)xi[j] - mean);
        double rstd = 1.0 / sqrt(sq / (double)width + eps);

        double sum_g = 0.0, sum_gx = 0.0;
        for (long j = 0; j < width; ++j) {
            double g = (double)di[j] * (gamma ? (double)gamma[j] : 1.0);
            double xhat = ((double)xi[j] - mean) * rstd;
            sum_g += g;
            sum_gx += g * xhat;
        }
        double mean_g = sum_g / (double)width;
        double mean_gx = sum_gx / (double)width;
        for (long j = 0; j < width; ++j) {
            double g = (double)di[j] * (gamma ? (double)gamma[j] : 1.0);
            double xhat = ((double)xi[j] - mean) * rstd;
            out[j] = rstd * (g - mean_g - xhat * mean_gx);
        }
    }
}

/* dx of y = RMSNorm(x) * gamma; gamma may be NULL. */
void oracle_rmsnorm_backward(const float *x, const float *gamma, const float *dy, double *dx,
                             long rows, long width, double eps)
{
    for (long i = 0; i < rows; ++i) {
        const float *xi = x + i * width;
        const float *di = dy + i * width;
        double *out = dx + i * width;

        double sq = 0.0;
        for (long j = 0; j < width; ++j)
            sq += (double)xi[j] * (double)xi[j];
        double rstd = 1.0 / sqrt(sq / (double)width + eps);

        double sum_gx = 0.0;
        for (long j = 0; j < width; ++j)
            sum_gx += (double)di[j] * (gamma ? (double)gamma[j] : 1.0) * ((double)xi[j] * rstd);
        double mean_gx = sum_gx / (double)width;
        for (long j = 0; j < width; ++j) {
            double g = (double)di[j] * (gamma ? (double)gamma[j] : 1.0);
            out[j] = rstd * (g - (double)xi[j] * rstd * mean_gx);
        }
    }
}

/* dx of y = softmax(x), given y and dy. */
void oracle_softmax_backward(const float *y, const float *dy, double *dx, long rows, long width)
{
    for (long i = 0; i < rows; ++i) {
        const float *yi = y + i * width;
        const float *di = dy + i * width;
        double *out = dx + i * width;

        double dot = 0.0;
        for (long j = 0; j < width; ++j)
            dot += (double)di[j] * (double)yi[j];
        for (long j = 0; j < width; ++j)
            out[j] = (double)yi[j] * ((double)di[j] - dot);
    }
}

/* dgamma[j] = sum_i dy[i][j] * xhat[i][j]; dbeta[j] = sum_i dy[i][j] (LayerNorm;
 * dbeta may be NULL).  rms != 0 uses the RMSNorm xhat = x * rstd instead. */
void oracle_norm_param_grad(const float *x, const float *dy, double *dgamma, double *dbeta,
                            long rows, long width, double eps, int rms)
{
    for (long j = 0; j < width; ++j) {
        dgamma[j] = 0.0;
        if (dbeta)
            dbeta[j] = 0.0;
    }
    for (long i = 0; i < rows; ++i) {
        const float *xi = x + i * width;
        const float *di = dy + i * width;
        double mean = 0.0;
        if (!rms) {
            for (long j = 0; j < width; ++j)
                mean += (double)xi[j];
            mean /= (double)width;
        }
        double sq = 0.0;
        for (long j = 0; j < width; ++j)
            sq += ((double)xi[j] - mean) * ((double)xi[j] - mean);
        double rstd = 1.0 / sqrt(sq / (double)width + eps);
        for (long j = 0; j < width; ++j) {
            dgamma[j] += (double)di[j] * (((double)xi[j] - mean) * rstd);
            if (dbeta)
                dbeta[j] += (double)di[j];
        }
    }
}
