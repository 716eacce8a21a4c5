/*
 * tile_rows.h -- C ABI of the fused FP32 row-normalisation library for
 * NVIDIA GB300 (sm_103a).
 *
 * Four operations, each applied independently to every row of a row-major
 * FP32 matrix [rows][width] (row i starts at element i*width):
 *
 *   residual LayerNorm  y = (c - mean(c)) / sqrt(var(c) + eps),  c = x + r
 *   LayerNorm           y = (x - mean(x)) / sqrt(var(x) + eps)
 *   RMSNorm             y = x / sqrt(mean(x^2) + eps)
 *   softmax             y = exp(x - max(x)) / sum(exp(x - max(x)))
 *
 * var is the centred, biased variance (divided by width); there are no
 * affine weights.  The definitions follow the notes "Residual LayerNorm
 * shared-Tile materialization search" (section "Structural finding": the
 * residual LayerNorm expression, eps = 1e-5 inside the square root) and
 * "Immutable input reuse in Metal reductions" (softmax, RMSNorm and
 * LayerNorm rows; each input element read once and kept in worker-private
 * stripes across the reduction phases).  Several rows may be packed into one
 * CTA as cooperating programs, as in "Cooperating-program packing",
 * section "Implementation boundary".
 *
 * Common contract of the four compute entry points
 * ------------------------------------------------
 *  - Pointers are DEVICE pointers (or managed/host-mapped memory the device
 *    can read), FP32, 4-byte aligned.  16-byte alignment is not required:
 *    rows whose start is not 16-byte aligned take a scalar head and tail.
 *  - The caller owns every buffer.  The library allocates nothing, writes
 *    exactly rows*width elements of `out` and nothing else, and never writes
 *    `in` or `residual`.
 *  - `out` must not overlap `in` or `residual` (the caller guarantees
 *    no aliasing; an overlap that the library can see from the address
 *    ranges is rejected with TILE_ERR_ALIAS).  `in` and `residual` may
 *    overlap each other.
 *  - Work is enqueued on `stream` (0 = the legacy default stream); the call
 *    returns without synchronising.  Results are bitwise reproducible for a
 *    given (op, rows, width, pointer alignment) on the same GPU.
 *  - rows == 0 is a no-op returning TILE_OK.  1 <= width <= tile_max_width().
 *  - Return value: TILE_OK (0) or a negative TILE_ERR_* code; on error
 *    nothing is launched, except TILE_ERR_CUDA, which reports the launch
 *    error returned by the CUDA runtime.
 */
#ifndef TILE_ROWS_H
#define TILE_ROWS_H

#include <stddef.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ---- status codes ------------------------------------------------------ */
#define TILE_OK               0
#define TILE_ERR_NULL        -1  /* a required pointer is NULL (rows > 0)       */
#define TILE_ERR_SHAPE       -2  /* rows < 0, width < 1 or width > max width   */
#define TILE_ERR_ALIAS       -3  /* out overlaps in or residual               */
#define TILE_ERR_EPS         -4  /* eps negative or not finite (normalisers)  */
#define TILE_ERR_CUDA        -5  /* the CUDA runtime reported a launch error  */
#define TILE_ERR_OP          -6  /* unknown operation code                    */
#define TILE_ERR_ALIGN       -7  /* a pointer is not 4-byte aligned           */
#define TILE_ERR_PLAN        -8  /* an explicit plan is not one of the built  */
#define TILE_ERR_DEVICE      -9  /* a kernel recorded an error on the device  */
#define TILE_ERR_WORKSPACE  -10  /* device workspace too small for one row    */
#define TILE_ERR_DTYPE      -11  /* unknown element type code                 */

/* ---- element types of row data (tile_row_args_t, tile_*_ex) ------------ */
#define TILE_DTYPE_F32  0   /* IEEE binary32                                  */
#define TILE_DTYPE_BF16 1   /* bfloat16: the high 16 bits of a binary32       */
#define TILE_DTYPE_F16  2   /* IEEE binary16                                  */

/* ---- operation codes (tile_describe_plan, tile_run_plan_*) ------------- */
#define TILE_OP_RESIDUAL_LAYERNORM 0
#define TILE_OP_LAYERNORM          1
#define TILE_OP_RMSNORM            2
#define TILE_OP_SOFTMAX            3
#define TILE_OP_ROW_SUM            4
#define TILE_OP_ROW_MINMAX         5
#define TILE_OP_LAYERNORM_AFFINE   6
#define TILE_OP_RMSNORM_WEIGHTED   7

/* ---- launch paths ------------------------------------------------------ */
#define TILE_PATH_CTA      0  /* P programs x S warps per CTA, one row each  */
#define TILE_PATH_CLUSTER  1  /* one row split over a cluster of C CTAs,     */
                              /* partials exchanged through DSMEM            */
#define TILE_PATH_STAGED   2  /* persistent CTAs; whole rows copied into a   */
                              /* ring of shared-memory stages by the bulk-   */
                              /* copy engine (mbarrier completion), several  */
                              /* rows in flight per CTA; 16-byte aligned     */
                              /* rows of whole vectors; normalisers, softmax */
#define TILE_PATH_ROWS     3  /* one CTA normalises R rows, each thread      */
                              /* owning the same columns of all R (one       */
                              /* reduction round and one gamma/beta load     */
                              /* serve R rows); 16-byte aligned rows of      */
                              /* whole vectors; normalisers, softmax;        */
                              /* programs_per_cta reports R                  */

/*
 * A launch plan: how rows map onto the GPU.  Worker w of program p in a CTA
 * owns the row elements e = (chunk * W * C + rank * W + w) * V + v of its
 * row (chunk < K, v < V; rank = CTA rank in the cluster), keeps them in
 * registers across every reduction phase, and reduces with warp shuffles,
 * then P*S shared partials, then (C > 1) the C CTA partials of the cluster.
 */
typedef struct tile_plan {
    int op;                 /* TILE_OP_*                                      */
    int rows, width;        /* the shape the plan was made for                */
    int id;                 /* index in the built plan table                  */
    int path;               /* TILE_PATH_*                                    */
    int vec;                /* elements per access: a 16-byte vector (4 FP32  */
                            /* or 8 BF16/FP16, + scalar head/tail), or 1      */
    int warps_per_program;  /* S                                              */
    int programs_per_cta;   /* P                                              */
    int chunks;             /* K: V-vectors per worker                        */
    int cluster;            /* C: CTAs per row (1 = no cluster)               */
    int threads;            /* T = 32 * S * P                                 */
    int workers;            /* W = 32 * S                                     */
    int stripe_floats;      /* K * vec FP32 registers of row data per thread  */
    int max_width;          /* widest row this plan covers                    */
    int smem_bytes;         /* static shared memory per CTA                   */
    int barriers_per_row;   /* CTA or cluster barriers on a row's path        */
    long long grid;         /* CTAs launched for `rows` (0 for staged plans:  */
                            /* persistent, min(rows, SMs x resident CTAs))    */
    int dtype;              /* TILE_DTYPE_* the plan was described for        */
} tile_plan_t;

/* ---- compute entry points --------------------------------------------- */

/* Residual LayerNorm, no affine: c = in + residual, then LayerNorm of c.
 * "Residual LayerNorm shared-Tile materialization search", "Structural
 * finding".  in, residual, out: [rows][width] FP32 on the device. */
int tile_residual_layernorm_f32(const float *in, const float *residual, float *out,
                                int rows, int width, float eps, cudaStream_t stream);

/* LayerNorm, no affine.  "Cooperating-program packing", "Validation"
 * (no-affine LayerNorm); "Immutable input reuse in Metal reductions". */
int tile_layernorm_f32(const float *in, float *out, int rows, int width, float eps,
                       cudaStream_t stream);

/* RMSNorm, no weight: y = x / sqrt(mean(x^2) + eps).  Named in "Immutable
 * input reuse in Metal reductions" (fixed-width results table). */
int tile_rmsnorm_f32(const float *in, float *out, int rows, int width, float eps,
                     cudaStream_t stream);

/* softmax over each row with the row maximum subtracted first (the max
 * collective of "Cooperating-program packing", "Implementation boundary").
 * `eps` is accepted for a uniform signature and ignored. */
int tile_softmax_f32(const float *in, float *out, int rows, int width, float eps,
                     cudaStream_t stream);

/* ---- more row operations ---------------------------------------------- */

/* Affine LayerNorm: y = LayerNorm(in [+ residual]) * gamma + beta.  The
 * pages list affine LayerNorm (tolerance atol 1e-5) in "Cooperating-program
 * packing", "Predeclared comparison and measurement"; the formula is the
 * LayerNorm above followed by the per-column scale and shift.  residual and
 * beta may be NULL; gamma, beta: [width] FP32 device vectors (read through
 * the read-only cache; any 4-byte alignment).  Same contract otherwise. */
int tile_layernorm_affine_f32(const float *in, const float *residual, const float *gamma,
                              const float *beta, float *out, int rows, int width, float eps,
                              cudaStream_t stream);

/* Weighted RMSNorm: y = in / sqrt(mean(in^2) + eps) * gamma, gamma [width]. */
int tile_rmsnorm_weighted_f32(const float *in, const float *gamma, float *out, int rows,
                              int width, float eps, cudaStream_t stream);

/* Row sums: sums[i] = sum_j in[i][j], sums: [rows] FP32 on the device.  The
 * "sum" operator of "Cooperating-program packing", "Validation".  Each
 * thread and every reduction level keeps a compensated (TwoSum) pair, so the
 * result is close to the correctly rounded sum even when terms cancel. */
int tile_row_sum_f32(const float *in, float *sums, int rows, int width, cudaStream_t stream);

/* Paired row min/max in one pass: mins[i] = min_j in[i][j], maxs[i] =
 * max_j in[i][j] (exact).  The "paired min/max" operator of
 * "Cooperating-program packing", "Validation".  Inputs must not be NaN. */
int tile_row_minmax_f32(const float *in, float *mins, float *maxs, int rows, int width,
                        cudaStream_t stream);

/* Operands of a row operation for tile_run_plan_args_f32.  Unused pointers
 * are ignored (set them NULL). */
typedef struct tile_row_args {
    const void *in;         /* [rows][width] of `dtype`                         */
    const void *residual;   /* residual LayerNorm; optional for affine LN       */
    const float *gamma;     /* affine LN / weighted RMSNorm: [width] FP32       */
    const float *beta;      /* affine LN: [width] FP32 or NULL                  */
    void *out;              /* [rows][width] of `dtype`, or [rows] FP32 sums /  */
                            /* minima                                            */
    float *out2;            /* [rows] FP32 maxima (TILE_OP_ROW_MINMAX)          */
    int rows, width;
    float eps;              /* normalisers only                                  */
    int dtype;              /* TILE_DTYPE_F32, TILE_DTYPE_BF16 or TILE_DTYPE_F16 */
} tile_row_args_t;

/* Any row operation with the built plan `plan_id` forced (plan sweeps,
 * per-plan tests).  Errors as tile_run_plan_f32. */
int tile_run_plan_args_f32(int op, int plan_id, const tile_row_args_t *args, cudaStream_t stream);

/* ---- BF16 rows ----------------------------------------------------------
 * The row operations on BF16 data (2 bytes per element; the pages cover FP32
 * only and name low precision as not covered, "Residual LayerNorm
 * shared-Tile materialization search", "Exact command").  Each element is
 * widened exactly to FP32, every reduction and map runs in FP32 as for the
 * FP32 entry points (except that the row statistics multiply by 1/width
 * and take rsqrtf, at most 2 ulp, where the FP32 rows divide and take a
 * correctly rounded 1/sqrt: a few FP32 ulp, far inside half a BF16 ulp),
 * and outputs are rounded to nearest-even BF16.  gamma,
 * beta and the row outputs of sum and min/max stay FP32.  Pointers to BF16
 * data must be 2-byte aligned; 16-byte vectors (8 elements) are used when
 * in, residual and out share a 16-byte phase.  Everything else is the
 * contract of the FP32 entry point of the same name. */
int tile_residual_layernorm_bf16(const void *in, const void *residual, void *out, int rows,
                                 int width, float eps, cudaStream_t stream);
int tile_layernorm_bf16(const void *in, void *out, int rows, int width, float eps,
                        cudaStream_t stream);
int tile_rmsnorm_bf16(const void *in, void *out, int rows, int width, float eps,
                      cudaStream_t stream);
int tile_softmax_bf16(const void *in, void *out, int rows, int width, float eps,
                      cudaStream_t stream);
int tile_layernorm_affine_bf16(const void *in, const void *residual, const float *gamma,
                               const float *beta, void *out, int rows, int width, float eps,
                               cudaStream_t stream);
int tile_rmsnorm_weighted_bf16(const void *in, const float *gamma, void *out, int rows,
                               int width, float eps, cudaStream_t stream);
int tile_row_sum_bf16(const void *in, float *sums, int rows, int width, cudaStream_t stream);
int tile_row_minmax_bf16(const void *in, float *mins, float *maxs, int rows, int width,
                         cudaStream_t stream);

/* ---- FP16 rows ----------------------------------------------------------
 * The same row operations on IEEE binary16 data (the "FP16 I/O" of low
 * precision the pages name as not covered, same section as above): each
 * element is widened exactly to FP32, every reduction and map runs in FP32
 * (row statistics as for BF16 rows), outputs are rounded to nearest-even
 * binary16 (an output beyond 65504
 * becomes +-inf, as a binary16 rounding does; normalised rows stay far below
 * it).  Layout, alignment, vectors, plans and errors as the BF16 entry
 * points; gamma, beta and the row outputs of sum and min/max stay FP32. */
int tile_residual_layernorm_f16(const void *in, const void *residual, void *out, int rows,
                                int width, float eps, cudaStream_t stream);
int tile_layernorm_f16(const void *in, void *out, int rows, int width, float eps,
                       cudaStream_t stream);
int tile_rmsnorm_f16(const void *in, void *out, int rows, int width, float eps,
                     cudaStream_t stream);
int tile_softmax_f16(const void *in, void *out, int rows, int width, float eps,
                     cudaStream_t stream);
int tile_layernorm_affine_f16(const void *in, const void *residual, const float *gamma,
                              const float *beta, void *out, int rows, int width, float eps,
                              cudaStream_t stream);
int tile_rmsnorm_weighted_f16(const void *in, const float *gamma, void *out, int rows,
                              int width, float eps, cudaStream_t stream);
int tile_row_sum_f16(const void *in, float *sums, int rows, int width, cudaStream_t stream);
int tile_row_minmax_f16(const void *in, float *mins, float *maxs, int rows, int width,
                        cudaStream_t stream);

/* ---- backward passes ---------------------------------------------------
 * Input gradients of LayerNorm, RMSNorm and softmax, FP32.  The pages do
 * not cover backward normalisation ("Residual LayerNorm shared-Tile
 * materialization search", last paragraph); these are the chain rule of the
 * forward maps above:
 *   LayerNorm  dx = rstd (g - mean(g) - xhat mean(g xhat)),  xhat = (x - mean) rstd
 *   RMSNorm    dx = rstd (g - xhat mean(g xhat)),            xhat = x rstd
 *   softmax    dx = y (dy - sum(dy y))
 * with g = dy * gamma (gamma = 1 when NULL).  `in` is the forward input
 * (x, or x + residual for residual LayerNorm); the statistics are recomputed
 * from it exactly as the forward kernels compute them.  Each row of in and
 * dy is read once into registers, dx written once.  If row_stats is not
 * NULL, (mean, rstd) of every row is written to row_stats[2*i], [2*i+1]
 * (mean 0 for RMSNorm) for tile_norm_param_grad_f32.  dx and row_stats must
 * not overlap any input.  Other rules as the forward entry points. */
int tile_layernorm_backward_f32(const float *in, const float *gamma, const float *dy, float *dx,
                                float *row_stats, int rows, int width, float eps,
                                cudaStream_t stream);
int tile_rmsnorm_backward_f32(const float *in, const float *gamma, const float *dy, float *dx,
                              float *row_stats, int rows, int width, float eps,
                              cudaStream_t stream);
/* y: the forward softmax output. */
int tile_softmax_backward_f32(const float *y, const float *dy, float *dx, int rows, int width,
                              cudaStream_t stream);

/* A backward call with the built plan `plan_id` forced (op: TILE_OP_LAYERNORM,
 * TILE_OP_RMSNORM or TILE_OP_SOFTMAX).  TILE_ERR_PLAN if the plan is not built
 * for backward (two stripes of at most 32 floats), cannot cover the width, or
 * needs co-aligned pointers. */
int tile_run_backward_plan_f32(int op, int plan_id, const float *in, const float *gamma,
                               const float *dy, float *dx, float *row_stats, int rows, int width,
                               float eps, cudaStream_t stream);

/* Parameter gradients, summed over rows:
 *   dgamma[j] = sum_i dy[i][j] (in[i][j] - mean_i) rstd_i,  dbeta[j] = sum_i dy[i][j]
 * from the row statistics a backward call wrote (RMSNorm: mean 0, pass
 * dbeta = NULL).  Deterministic: rows are split into fixed blocks whose
 * column partials (compensated sums) go to the caller's device `workspace`
 * of at least tile_norm_param_grad_workspace_bytes(rows, width) bytes,
 * then are summed in block order.  rows == 0 writes zeros. */
size_t tile_norm_param_grad_workspace_bytes(int rows, int width);
int tile_norm_param_grad_f32(const float *in, const float *dy, const float *row_stats,
                             float *dgamma, float *dbeta, int rows, int width, void *workspace,
                             size_t workspace_bytes, cudaStream_t stream);

/* The backward passes with BF16 or FP16 in / y, dy and dx (2 bytes per
 * element, 2-byte aligned): every element is widened exactly to FP32, the
 * statistics, sums and maps run in FP32 as above (row statistics as for the
 * 2-byte forward rows), and dx is rounded to
 * nearest-even of its type.  gamma, row_stats, dgamma, dbeta and the
 * workspace stay FP32; tile_norm_param_grad_* uses the same workspace size.
 * 16-byte vectors (8 elements) are used when in, dy and dx share a 16-byte
 * phase.  Everything else is the contract of the FP32 entry point. */
int tile_layernorm_backward_bf16(const void *in, const float *gamma, const void *dy, void *dx,
                                 float *row_stats, int rows, int width, float eps,
                                 cudaStream_t stream);
int tile_rmsnorm_backward_bf16(const void *in, const float *gamma, const void *dy, void *dx,
                               float *row_stats, int rows, int width, float eps,
                               cudaStream_t stream);
int tile_softmax_backward_bf16(const void *y, const void *dy, void *dx, int rows, int width,
                               cudaStream_t stream);
int tile_norm_param_grad_bf16(const void *in, const void *dy, const float *row_stats,
                              float *dgamma, float *dbeta, int rows, int width, void *workspace,
                              size_t workspace_bytes, cudaStream_t stream);
int tile_layernorm_backward_f16(const void *in, const float *gamma, const void *dy, void *dx,
                                float *row_stats, int rows, int width, float eps,
                                cudaStream_t stream);
int tile_rmsnorm_backward_f16(const void *in, const float *gamma, const void *dy, void *dx,
                              float *row_stats, int rows, int width, float eps,
                              cudaStream_t stream);
int tile_softmax_backward_f16(const void *y, const void *dy, void *dx, int rows, int width,
                              cudaStream_t stream);
int tile_norm_param_grad_f16(const void *in, const void *dy, const float *row_stats,
                             float *dgamma, float *dbeta, int rows, int width, void *workspace,
                             size_t workspace_bytes, cudaStream_t stream);

/* tile_run_backward_plan_f32 for an element type (TILE_DTYPE_*; in, dy, dx
 * of that type).  For BF16 / FP16, plans whose stripes would pass 32 floats
 * (K above 4 with 16-byte vectors) return TILE_ERR_PLAN; an unknown type
 * TILE_ERR_DTYPE. */
int tile_run_backward_plan_ex(int op, int plan_id, int dtype, const void *in, const float *gamma,
                              const void *dy, void *dx, float *row_stats, int rows, int width,
                              float eps, cudaStream_t stream);

/* The plan the backward entry points launch for (op, dtype, rows, width)
 * with 16-byte co-aligned in, dy and dx (op: TILE_OP_LAYERNORM,
 * TILE_OP_RMSNORM or TILE_OP_SOFTMAX; the choice depends on the width, not
 * on the rows).  Host only; touches no GPU.  Returns TILE_OK, TILE_ERR_OP,
 * TILE_ERR_DTYPE, TILE_ERR_SHAPE or TILE_ERR_NULL; `plan` is written on
 * success only. */
int tile_describe_backward_plan(int op, int dtype, int rows, int width, tile_plan_t *plan);

/* ---- pointwise value/derivative pairs ---------------------------------- */

/* value[k] = sigmoid(in[k]) and derivative[k] = sigmoid'(in[k]) for k < n,
 * one read and two writes per element in one kernel ("Multi-output
 * pointwise fusion: evidence and limits", "Measurement definitions and
 * population").  Device buffers of n floats, 4-byte aligned; the outputs
 * must not overlap the input or each other.  n == 0 is a no-op. */
int tile_sigmoid_pair_f32(const float *in, float *value, float *derivative, long long n,
                          cudaStream_t stream);

/* The same for tanh-approximate GELU, g(x) = x/2 (1 + tanh(sqrt(2/pi)
 * (x + 0.044715 x^3))), and its derivative. */
int tile_gelu_tanh_pair_f32(const float *in, float *value, float *derivative, long long n,
                            cudaStream_t stream);

/* ---- end to end on host buffers ---------------------------------------- */
/* The notes time single calls in two phases, GPU time and end to end with
 * the host's part included ("Immutable input reuse in Metal reductions",
 * "Fixed-width GPU and dispatch results"); on a GPU whose inputs start in
 * host memory the end-to-end phase also moves the rows across the host
 * link, which these entry points pipeline.  The notes have no interface of
 * this kind: its arguments and schedule are this library's own. */

/* Run `op` on HOST buffers h_in[, h_residual] -> h_out ([rows][width] FP32
 * each).  Rows stream through the caller's device workspace `d_work`
 * (`work_bytes` bytes, 256-byte aligned) in chunks of about rows/16 rows (at
 * least 1 MiB of a tensor, at most what fits twice in the workspace), held in
 * a ring of 2 to 4 workspace buffers (as many as fit): the host->device copy
 * of one chunk, the kernel on an earlier chunk and the device->host copy of
 * one before that overlap on three streams (the caller's
 * `stream` runs the kernels; two internal non-blocking streams per device,
 * created on first use, run the copies).  Host buffers should be pinned
 * (cudaHostAlloc / cudaHostRegister) for the copies to overlap; pageable
 * memory gives the same results more slowly.  When h_out is pinned the
 * kernels store the results straight into it through its device address
 * (NVLink-C2C on Grace systems) and no device->host copies are made.  When
 * h_in, h_residual and h_out are all pinned and device-addressable, there is
 * no pipeline: one launch of the selected kernel reads and writes the host
 * buffers directly (d_work is then not touched).  Ownership: the caller owns all
 * buffers and must keep them alive and untouched until `stream` has passed
 * this call (the call returns once everything is enqueued; `stream` is
 * ordered after the last copy or the kernel).  Results meet the same tolerance
 * as the device entry points, and are bitwise equal to those of a device
 * call on the whole matrix when width is a multiple of 4: every chunk runs
 * the whole matrix's plan (chunks start 256-byte aligned in the workspace,
 * so row start phases can differ from the full matrix otherwise).  `h_residual` is read only by
 * TILE_OP_RESIDUAL_LAYERNORM.  Errors: as the compute entry points, plus
 * TILE_ERR_NULL for a NULL d_work, TILE_ERR_ALIGN for a misaligned d_work and
 * TILE_ERR_WORKSPACE when not even one row fits twice.  Calls from several
 * host threads on one device are serialised inside the library. */
int tile_run_host_f32(int op, const float *h_in, const float *h_residual, float *h_out,
                      int rows, int width, float eps, void *d_work, size_t work_bytes,
                      cudaStream_t stream);

/* Workspace bytes tile_run_host_f32 needs to move `chunk_rows` rows per
 * chunk (0 for invalid arguments).  Host only. */
size_t tile_host_workspace_bytes(int op, int width, int chunk_rows);

/* The schedule tile_run_host_f32 uses for these arguments: rows per full
 * chunk (the first and the last chunk are a quarter of that when a quarter
 * still holds 1 MiB of an input and there are more than two chunks; the
 * last may otherwise be shorter) and the number of workspace buffers in the
 * ring.  `direct_output` != 0 describes a call whose h_out is pinned and
 * device-addressable (results stored straight into it), 0 one whose results
 * are copied out.  Host only: no CUDA call.  Returns TILE_OK, TILE_ERR_OP,
 * TILE_ERR_SHAPE (rows < 1 or width outside 1..tile_max_width()),
 * TILE_ERR_NULL for a NULL output pointer, or TILE_ERR_WORKSPACE as
 * tile_run_host_f32 would. */
int tile_host_schedule(int op, int rows, int width, size_t work_bytes, int direct_output,
                       int *chunk_rows, int *slots);

/* Size of the library's own device staging area used by
 * tile_run_host_static_f32: 64 MiB, held by every GPU that loads the library
 * until the process exits. */
#define TILE_STATIC_STAGING_BYTES (64u << 20)

/* tile_run_host_f32 for callers that cannot allocate device memory.  (The
 * notes this library follows have no counterpart of this call.)
 *
 * Some callers cannot call cudaMalloc where they run: code that runs after
 * an application has fixed its device memory budget, plugin code inside a
 * framework that owns the device allocator, or latency-critical code where a
 * device allocation (which can synchronise the device) is not allowed.  This
 * call allocates nothing: rows are staged through a static device array of
 * TILE_STATIC_STAGING_BYTES inside the library instead of a caller
 * workspace (pinned, device-addressable buffers are processed in place, as
 * by tile_run_host_f32).  Arguments, results, errors and ownership are those of
 * tile_run_host_f32 without d_work/work_bytes.
 *
 * Limits: any number of rows (they stream through the area in chunks);
 * 1 <= width <= tile_max_width() (one row of every tensor, 3 x 4 x 131072
 * bytes at most, fits the area twice).  A width beyond that maximum returns
 * TILE_ERR_SHAPE, and TILE_ERR_WORKSPACE would report a row that cannot fit.
 *
 * Set-up: the first call on each device looks up the array's device address
 * (cudaGetSymbolAddress, which may load the library's device code) and
 * creates one event; make that first call before any stream capture.
 *
 * Sharing: every call on a device uses the same array, and the array keeps
 * the last call's contents (nothing in it needs to start at zero: each
 * chunk is copied in before the kernel reads it).  Calls that overlapped on
 * the GPU would race on the array, so the library orders each call's work
 * on the GPU after the previous call's end (an event), whatever stream it
 * was given; calls on different streams therefore run one after another.
 * A call that fails part-way (TILE_ERR_CUDA after some chunks were
 * enqueued) still marks its end after everything it enqueued, so the next
 * call waits for that work too.  Argument errors are returned before any
 * CUDA call. */
int tile_run_host_static_f32(int op, const float *h_in, const float *h_residual, float *h_out,
                             int rows, int width, float eps, cudaStream_t stream);

/* ---- plans and diagnostics -------------------------------------------- */

/* The plan the library would launch for (op, rows, width) with 16-byte
 * co-aligned pointers (the common case).  Host only; touches no GPU.
 * Returns TILE_OK, TILE_ERR_OP or TILE_ERR_SHAPE.  `plan` is written on
 * success only. */
int tile_describe_plan(int op, int rows, int width, tile_plan_t *plan);

/* tile_describe_plan for an element type (TILE_DTYPE_*); TILE_ERR_DTYPE for
 * an unknown one.  For large problems (rows * width above 2^22) the answer
 * may be a plan that needs rows of whole 16-byte vectors -- a
 * shared-memory-staged plan (path TILE_PATH_STAGED) or an R-rows-per-CTA
 * plan (TILE_PATH_ROWS) -- which a call takes only when every pointer is
 * 16-byte aligned and width is a multiple of the vector (4 FP32, 8 BF16 /
 * FP16 elements); other calls of that shape take the register plan of the
 * same width.  For TILE_OP_LAYERNORM_AFFINE the answer is that of a call
 * without a residual (a call with a residual has its own measured table). */
int tile_describe_plan_ex(int op, int dtype, int rows, int width, tile_plan_t *plan);

/* Number of plans built into the library, and plan `id` of that table
 * described for (op, rows, width).  Returns TILE_ERR_PLAN for a bad id and
 * TILE_ERR_SHAPE if the plan cannot cover `width`.  Host only. */
int tile_plan_count(void);
int tile_plan_info(int id, int op, int rows, int width, tile_plan_t *plan);

/* tile_plan_info for an element type; TILE_ERR_PLAN also when plan `id` is
 * not built for that type (BF16 / FP16 plans whose stripe would pass 64 floats), or
 * is a shared-memory-staged plan and `op` a row reduction (sum, min/max),
 * which only the register plans implement. */
int tile_plan_info_ex(int id, int op, int dtype, int rows, int width, tile_plan_t *plan);

/* Test hook for failure detection without a GPU fault (the notes have no
 * counterpart: their runner has no error path to test).  After `skip` more
 * launch attempts that proceed normally, the next `count` kernel launch
 * attempts of the library's entry points fail on the host with the CUDA
 * error `cuda_error` (a nonzero cudaError_t value) instead of launching:
 * the entry point returns TILE_ERR_CUDA and tile_last_cuda_error() on that
 * thread gives `cuda_error`.  Argument errors are still reported first.
 * Nothing reaches the GPU for an injected failure; work the same call
 * enqueued before it (copies and kernels of earlier chunks of
 * tile_run_host_f32 / tile_run_host_static_f32) stays enqueued, and the
 * caller's stream stays ordered after it.  count = 0 disarms.  Process-wide,
 * thread-safe, host only.  Returns TILE_OK, or TILE_ERR_SHAPE for a negative
 * skip or count, or a zero error with count > 0. */
int tile_inject_launch_failure(int cuda_error, int skip, int count);

/* Test hook for the whole-vector kernels (the notes have no counterpart).
 * 2-byte rows that are 16-byte aligned and hold whole 16-byte vectors run
 * a form of the row kernel (and, on the S = 4, P = 1, K = 4 shape, of the
 * LayerNorm backward kernel) without a scalar head and tail; its results
 * are bitwise those of the general form, where a head and tail of no
 * elements add exact +0 terms (which can change only the sign of a zero
 * result, after a partial sum of exactly -0).  With `on` nonzero every
 * later launch takes the general form instead, so a test can compare the
 * two on the same rows; 0 restores the default.  Process-wide, host only;
 * returns TILE_OK. */
int tile_test_force_general_kernels(int on);

/* Test hook for the bounded waits of the shared-memory-staged kernel (the
 * notes have no counterpart: their kernels have no copy engine to wait on).
 * Runs the staged plan `plan_id` (path TILE_PATH_STAGED) of `op` on `args`
 * as tile_run_plan_args_f32 would, except that no CTA issues the bulk copy
 * of its first row and every barrier wait gives up after `spin_limit` polls
 * (0 counts as 1).  The first wait of every CTA therefore runs out: the
 * kernel sets its wait-timeout bit in the device status word, stops
 * waiting and copying, waits (bounded) for the copies it did issue, and
 * returns with its outputs invalid.  tile_check_device_status then returns
 * TILE_ERR_DEVICE and clears the word.  Nothing is left in flight (the
 * withheld copy is never issued).  No other entry point withholds a copy;
 * library calls wait up to 2^20 polls.  Errors as tile_run_plan_args_f32;
 * TILE_ERR_PLAN also for a plan that is not staged. */
int tile_test_staged_wait_timeout(int op, int plan_id, const tile_row_args_t *args,
                                  unsigned int spin_limit, cudaStream_t stream);

/* Run `op` (one of the first four op codes) with the built plan `plan_id`
 * instead of the selector's choice (used by the measured plan sweep and by
 * tests that check every plan; tile_run_plan_args_f32 covers every op).
 * Same contract as the compute entry points; `residual` is used only by
 * TILE_OP_RESIDUAL_LAYERNORM.  Returns TILE_ERR_PLAN if the plan does not
 * exist, cannot cover `width`, or needs 16-byte co-alignment (V = 4) that
 * the pointers do not have. */
int tile_run_plan_f32(int op, int plan_id, const float *in, const float *residual,
                      float *out, int rows, int width, float eps, cudaStream_t stream);

/* Widest row any built plan covers. */
int tile_max_width(void);

/* The cudaError_t value behind the last TILE_ERR_CUDA returned on this host
 * thread (0 if none). */
int tile_last_cuda_error(void);

/* A static, human-readable description of a status code. */
const char *tile_status_string(int status);

/* Synchronise `stream`, then read and clear the device error word that
 * kernels set instead of trapping.  Returns TILE_OK, TILE_ERR_DEVICE (a
 * kernel recorded an error since the last check) or TILE_ERR_CUDA. */
int tile_check_device_status(cudaStream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* TILE_ROWS_H */
