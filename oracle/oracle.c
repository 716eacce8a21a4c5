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
