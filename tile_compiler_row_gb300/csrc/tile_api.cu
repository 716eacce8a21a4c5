// C ABI of the row-normalisation library: argument checks, the width->plan
// selector and dispatch to the per-op launchers.  See include/tile_rows.h for
// the contract of every entry point.
#include "../../include/tile_rows.h"

#include <atomic>
#include <cmath>
#include <cstdint>
#include <mutex>

#include "launch.h"
#include "plans.h"

namespace {

struct PlanDesc {
    int id, V, S, P, K, C;
    bool staged;   // shared-memory-staged persistent kernel (staged_kernel.cuh)
    int stage_kb;  // staged plans: shared memory budget of the ring of stages
    int R;         // rows per CTA sharing each thread's columns (multi_kernel.cuh); 1 else
};

constexpr int kAllPlans = TILE_PLAN_COUNT + TILE_STAGED_COUNT + TILE_MULTI_COUNT;

constexpr PlanDesc kPlans[kAllPlans] = {
#define TILE_ROW(id, V, S, P, K, C) {id, V, S, P, K, C, false, 0, 1},
    TILE_PLAN_LIST(TILE_ROW)
#undef TILE_ROW
#define TILE_STAGED_ROW(id, S, K, KB) {id, 4, S, 1, K, 1, true, KB, 1},
    TILE_STAGED_LIST(TILE_STAGED_ROW)
#undef TILE_STAGED_ROW
#define TILE_MULTI_ROW(id, S, K, R) {id, 4, S, 1, K, 1, false, 0, R},
    TILE_MULTI_LIST(TILE_MULTI_ROW)
#undef TILE_MULTI_ROW
};

// Plans that run on 16-byte aligned rows of whole vectors only: the staged
// plans and the R-rows-per-CTA plans.
constexpr bool whole_vectors(const PlanDesc &p) { return p.staged || p.R > 1; }

// Vector slots a plan's workers own for one row.
constexpr long long capacity(const PlanDesc &p) {
    return static_cast<long long>(p.K) * 32 * p.S * p.C;
}

// Elements per access of a plan for an element type: a 16-byte vector
// (4 FP32 or 8 BF16 / FP16) for V = 4 plans, one element for V = 1 plans.
bool two_byte(int dtype) { return dtype == TILE_DTYPE_BF16 || dtype == TILE_DTYPE_F16; }
bool valid_dtype(int dtype) { return dtype == TILE_DTYPE_F32 || two_byte(dtype); }

int elems_per_vec(const PlanDesc &p, int dtype) {
    return p.V == 4 ? (two_byte(dtype) ? 8 : 4) : 1;
}

// 2-byte plans whose stripe would exceed the register budget are not built,
// nor R-row plans whose R stripes would (for any element type).
bool built(const PlanDesc &p, int dtype) {
    if (p.R > 1) return p.R * p.K * elems_per_vec(p, dtype) <= 64;
    return !two_byte(dtype) || p.K * elems_per_vec(p, dtype) <= tile::kMaxStripeBf16;
}

bool covers(const PlanDesc &p, int width, int dtype = TILE_DTYPE_F32) {
    if (width < 1 || !built(p, dtype)) return false;
    const int ev = elems_per_vec(p, dtype);
    if (whole_vectors(p))   // whole 16-byte vectors only: no head or tail
        return width % ev == 0 && width / ev <= capacity(p);
    return (width / ev) <= capacity(p);
}

// A staged plan copies whole rows with the bulk-copy engine: every row
// pointer (and gamma/beta) must be 16-byte aligned.
bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int max_width_of(const PlanDesc &p, int dtype = TILE_DTYPE_F32) {
    const int ev = elems_per_vec(p, dtype);
    const long long w = capacity(p) * ev + (whole_vectors(p) ? 0 : ev - 1);
    return w > TILE_MAX_WIDTH ? TILE_MAX_WIDTH : static_cast<int>(w);
}

// Selector: for each op, the first entry whose width bound covers the row.
// The tables (16-byte co-aligned pointers) are generated from a measured
// plan sweep on GB300 (selector_tables.py: every built plan timed at each
// width of a ladder, about 2^26 FP32 / 2^27 2-byte elements per tensor,
// plus the small workload shapes), so measurement, not a score, picks each
// mapping; profiles/selector_sweep.md holds an independent sweep of every
// bucket.  Pointers with different 16-byte phases use the scalar plans.
struct Bucket {
    int max_width;
    int plan;
};

#include "selector_tables.h"

struct Table {
    const Bucket *b;
    int n;
};
#define TILE_TABLE(name) Table{name, static_cast<int>(sizeof(name) / sizeof(Bucket))}
#define TILE_TABLES(fam, kind)                                                              \
    {TILE_TABLE(k##fam##kind##ResidualLN), TILE_TABLE(k##fam##kind##LN),                     \
     TILE_TABLE(k##fam##kind##RMS),        TILE_TABLE(k##fam##kind##Softmax),                \
     TILE_TABLE(k##fam##kind##RowSum),     TILE_TABLE(k##fam##kind##RowMinmax),              \
     TILE_TABLE(k##fam##kind##Affine),     TILE_TABLE(k##fam##kind##Weighted),               \
     TILE_TABLE(k##fam##kind##ResidualAffine)}
// Indexed by table op: the TILE_OP_* code, and 8 for affine LayerNorm with
// a residual (three row streams instead of two).
constexpr Table kRegF32[9] = TILE_TABLES(F32, Reg);
constexpr Table kStagedF32[9] = TILE_TABLES(F32, Staged);
constexpr Table kRegB16[9] = TILE_TABLES(B16, Reg);        // BF16 and FP16 rows
constexpr Table kStagedB16[9] = TILE_TABLES(B16, Staged);
constexpr Table kTinyF32[9] = TILE_TABLES(F32, Tiny);
constexpr Table kSmallF32[9] = TILE_TABLES(F32, Small);
#undef TILE_TABLES
#undef TILE_TABLE

// Small problems: rows * width <= kSmallElems (L2 resident), in two tiers
// (up to kTinyElems, and above).
constexpr long long kSmallElems = 1LL << 22;
constexpr long long kTinyElems = 1LL << 19;

constexpr Bucket kVec1[] = {
    {128, 25}, {1024, 26}, {4096, 27}, {16384, 28}, {TILE_MAX_WIDTH, 29},
};

template <int N>
int pick(const Bucket (&table)[N], int width) {
    for (int i = 0; i < N; ++i)
        if (width <= table[i].max_width) return table[i].plan;
    return -1;
}

int pick(const Table &t, int width) {
    for (int i = 0; i < t.n; ++i)
        if (width <= t.b[i].max_width) return t.b[i].plan;
    return -1;
}

int table_op(int op, bool residual) {
    return (op == TILE_OP_LAYERNORM_AFFINE && residual) ? 8 : op;
}

// staged_eligible: every pointer 16-byte aligned (rows of whole vectors are
// checked by covers()); residual: affine LayerNorm called with a residual.
int select_plan(int op, long long rows, int width, bool vec4, int dtype,
                bool staged_eligible = false, bool residual = false) {
    if (!vec4) return pick(kVec1, width);
    const int t = table_op(op, residual);
    const bool b16 = two_byte(dtype);      // FP16 rows share the BF16 tables
    const long long elems = rows * static_cast<long long>(width);
    const bool small = elems <= kSmallElems;
    if (staged_eligible && !small) {
        const int sid = pick(b16 ? kStagedB16[t] : kStagedF32[t], width);
        if (sid >= 0 && covers(kPlans[sid], width, dtype)) return sid;
    }
    if (small && !b16) {
        const int id = pick(elems <= kTinyElems ? kTinyF32[t] : kSmallF32[t], width);
        if (id >= 0 && covers(kPlans[id], width, dtype)) return id;
    }
    const int id = pick(b16 ? kRegB16[t] : kRegF32[t], width);
    return (id >= 0 && covers(kPlans[id], width, dtype)) ? id : -1;
}

long long grid_of(const PlanDesc &p, long long rows) {
    const long long per_cta = static_cast<long long>(p.P) * p.R;
    return ((rows + per_cta - 1) / per_cta) * p.C;
}

void fill_plan(const PlanDesc &p, int op, int dtype, int rows, int width, tile_plan_t *out) {
    out->op = op;
    out->rows = rows;
    out->width = width;
    out->id = p.id;
    out->path = p.staged  ? TILE_PATH_STAGED
                : p.R > 1 ? TILE_PATH_ROWS
                : p.C > 1 ? TILE_PATH_CLUSTER
                          : TILE_PATH_CTA;
    out->vec = elems_per_vec(p, dtype);
    out->warps_per_program = p.S;
    out->programs_per_cta = p.P * p.R;
    out->chunks = p.K;
    out->cluster = p.C;
    out->threads = 32 * p.S * p.P;       // R-row plans: R rows on the same threads
    out->workers = 32 * p.S;
    out->stripe_floats = p.K * elems_per_vec(p, dtype);
    out->max_width = max_width_of(p, dtype);
    out->dtype = dtype;
    const int part = p.S > 1 ? 3 * p.P * p.S * p.R : 0;
    out->smem_bytes = 4 * (part + (p.C > 1 ? 4 : 0));
    if (p.staged) {
        // the launcher's stage count: the plan's budget, 1..8 stages
        const int nin = (op == TILE_OP_RESIDUAL_LAYERNORM) ? 2 : 1;
        const long long stage = static_cast<long long>(width) *
                                (two_byte(dtype) ? 2 : 4) * nin;
        long long nst = (static_cast<long long>(p.stage_kb) << 10) / stage;
        nst = nst > 8 ? 8 : nst < 1 ? 1 : nst;
        out->smem_bytes = static_cast<int>(stage * nst) + 4 * 8 * p.S + 80;
    }
    const int phases = (op == TILE_OP_RESIDUAL_LAYERNORM || op == TILE_OP_LAYERNORM ||
                        op == TILE_OP_LAYERNORM_AFFINE || op == TILE_OP_SOFTMAX) ? 2 : 1;
    out->barriers_per_row = (p.S > 1 ? phases : 0) + (p.C > 1 ? phases + 1 : 0);
    out->grid = rows > 0 ? grid_of(p, rows) : 0;
    if (p.staged) out->grid = 0;   // persistent: min(rows, SMs x resident CTAs), device dependent
}

bool overlaps(const void *a, size_t abytes, const void *b, size_t bbytes) {
    if (a == nullptr || b == nullptr) return false;
    const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
    return x < y + bbytes && y < x + abytes;
}

bool misaligned(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 3u) != 0; }

bool valid_op(int op) { return op >= TILE_OP_RESIDUAL_LAYERNORM && op <= TILE_OP_RMSNORM_WEIGHTED; }

bool is_normaliser(int op) {
    return op == TILE_OP_RESIDUAL_LAYERNORM || op == TILE_OP_LAYERNORM || op == TILE_OP_RMSNORM ||
           op == TILE_OP_LAYERNORM_AFFINE || op == TILE_OP_RMSNORM_WEIGHTED;
}

bool row_output(int op) { return op == TILE_OP_ROW_SUM || op == TILE_OP_ROW_MINMAX; }

// One call of a row operation with its operands normalised: pointers an op
// does not use are cleared, so the kernel never sees them.
struct Call {
    int op;
    int dtype;
    const void *in, *res;
    const float *gamma, *beta;
    void *out;
    float *out2;
    int rows, width;
    float eps;
};

Call make_call(int op, const tile_row_args_t &a) {
    Call c{op, a.dtype, a.in, nullptr, nullptr, nullptr, a.out, nullptr, a.rows, a.width, a.eps};
    if (op == TILE_OP_RESIDUAL_LAYERNORM || op == TILE_OP_LAYERNORM_AFFINE) c.res = a.residual;
    if (op == TILE_OP_LAYERNORM_AFFINE || op == TILE_OP_RMSNORM_WEIGHTED) c.gamma = a.gamma;
    if (op == TILE_OP_LAYERNORM_AFFINE) c.beta = a.beta;
    if (op == TILE_OP_ROW_MINMAX) c.out2 = a.out2;
    if (!is_normaliser(op)) c.eps = 0.0f;
    return c;
}

bool coaligned16(const Call &c) {
    const uintptr_t a = reinterpret_cast<uintptr_t>(c.in);
    if (!row_output(c.op) && ((a ^ reinterpret_cast<uintptr_t>(c.out)) & 15u) != 0) return false;
    if (c.res != nullptr && ((a ^ reinterpret_cast<uintptr_t>(c.res)) & 15u) != 0) return false;
    return true;
}

// Checks shared by every row entry point.  Returns TILE_OK with *noop set
// when there is nothing to launch.  No CUDA call is made.
size_t elem_size(int dtype) { return two_byte(dtype) ? 2 : 4; }

bool misaligned_to(const void *p, size_t bytes) {
    return (reinterpret_cast<uintptr_t>(p) & (bytes - 1)) != 0;
}

int validate(const Call &c, bool *noop) {
    *noop = false;
    if (!valid_op(c.op)) return TILE_ERR_OP;
    if (!valid_dtype(c.dtype)) return TILE_ERR_DTYPE;
    if (c.rows < 0 || c.width < 1 || c.width > TILE_MAX_WIDTH) return TILE_ERR_SHAPE;
    if (is_normaliser(c.op) && !(std::isfinite(c.eps) && c.eps >= 0.0f)) return TILE_ERR_EPS;
    if (c.rows == 0) {
        *noop = true;
        return TILE_OK;
    }
    if (c.in == nullptr || c.out == nullptr) return TILE_ERR_NULL;
    if (c.op == TILE_OP_RESIDUAL_LAYERNORM && c.res == nullptr) return TILE_ERR_NULL;
    if ((c.op == TILE_OP_LAYERNORM_AFFINE || c.op == TILE_OP_RMSNORM_WEIGHTED) && c.gamma == nullptr)
        return TILE_ERR_NULL;
    if (c.op == TILE_OP_ROW_MINMAX && c.out2 == nullptr) return TILE_ERR_NULL;
    const size_t es = elem_size(c.dtype);
    if (misaligned_to(c.in, es) || misaligned_to(c.res, es) ||
        misaligned_to(c.out, row_output(c.op) ? sizeof(float) : es))
        return TILE_ERR_ALIGN;
    for (const void *p : {static_cast<const void *>(c.gamma), static_cast<const void *>(c.beta),
                          static_cast<const void *>(c.out2)})
        if (misaligned(p)) return TILE_ERR_ALIGN;
    const size_t mat = static_cast<size_t>(c.rows) * static_cast<size_t>(c.width) * es;
    const size_t vec = static_cast<size_t>(c.width) * sizeof(float);
    const size_t out_bytes = row_output(c.op) ? static_cast<size_t>(c.rows) * sizeof(float) : mat;
    const size_t out2_bytes = static_cast<size_t>(c.rows) * sizeof(float);
    if (overlaps(c.out, out_bytes, c.in, mat) || overlaps(c.out, out_bytes, c.res, mat) ||
        overlaps(c.out, out_bytes, c.gamma, vec) || overlaps(c.out, out_bytes, c.beta, vec) ||
        overlaps(c.out2, out2_bytes, c.in, mat) || overlaps(c.out2, out2_bytes, c.out, out_bytes))
        return TILE_ERR_ALIAS;
    return TILE_OK;
}

int kernel_op_of(const Call &c) {
    switch (c.op) {
        case TILE_OP_RESIDUAL_LAYERNORM: return tile::OP_RESLN;
        case TILE_OP_LAYERNORM: return tile::OP_LN;
        case TILE_OP_LAYERNORM_AFFINE: return c.res != nullptr ? tile::OP_RESLN : tile::OP_LN;
        case TILE_OP_RMSNORM:
        case TILE_OP_RMSNORM_WEIGHTED: return tile::OP_RMS;
        case TILE_OP_SOFTMAX: return tile::OP_SOFTMAX;
        case TILE_OP_ROW_SUM: return tile::OP_SUM;
        default: return tile::OP_MINMAX;
    }
}

// Staged plans serve the normalisers and softmax, with every pointer
// 16-byte aligned.
bool staged_ok(const Call &c) {
    const int k = kernel_op_of(c);
    if (k == tile::OP_SUM || k == tile::OP_MINMAX) return false;
    return aligned16(c.in) && aligned16(c.out) && (c.res == nullptr || aligned16(c.res)) &&
           (c.gamma == nullptr || aligned16(c.gamma)) && (c.beta == nullptr || aligned16(c.beta));
}

// A launch failure injected on the host for tests: TILE_ERR_CUDA with the
// injected error, nothing launched.
#define TILE_INJECTED_FAILURE()                                              \
    do {                                                                     \
        const cudaError_t inj = tile::injected_launch_failure();             \
        if (inj != cudaSuccess) {                                            \
            tile::set_last_cuda_error(static_cast<int>(inj));                \
            return TILE_ERR_CUDA;                                            \
        }                                                                    \
    } while (0)

int launch(const Call &c, int plan_id, cudaStream_t stream) {
    const PlanDesc &p = kPlans[plan_id];
    if (grid_of(p, c.rows) > 0x7fffffffLL) return TILE_ERR_SHAPE;
    TILE_INJECTED_FAILURE();
    tile::RowArgs a{c.in, c.res, c.gamma, c.beta, c.out, c.out2, c.rows, c.width, c.eps, nullptr,
                    1.0f / static_cast<float>(c.width)};
    cudaError_t err;
    if (whole_vectors(p)) {
        err = p.staged ? tile::launch_staged(kernel_op_of(c), c.dtype, plan_id, a, stream)
                       : tile::launch_multi(kernel_op_of(c), c.dtype, plan_id, a, stream);
        if (err != cudaSuccess) {
            tile::set_last_cuda_error(static_cast<int>(err));
            return TILE_ERR_CUDA;
        }
        return TILE_OK;
    }
    // the launcher of each row-kernel op, per element type
    using Launch = cudaError_t (*)(int, tile::RowArgs, cudaStream_t);
    struct Launchers {
        Launch resln, ln, rms, softmax, sum, minmax;
    };
    static const Launchers kF32 = {tile::launch_residual_layernorm, tile::launch_layernorm,
                                   tile::launch_rmsnorm, tile::launch_softmax,
                                   tile::launch_row_sum, tile::launch_row_minmax};
    static const Launchers kBf16 = {tile::launch_residual_layernorm_bf16,
                                    tile::launch_layernorm_bf16, tile::launch_rmsnorm_bf16,
                                    tile::launch_softmax_bf16, tile::launch_row_sum_bf16,
                                    tile::launch_row_minmax_bf16};
    static const Launchers kF16 = {tile::launch_residual_layernorm_f16,
                                   tile::launch_layernorm_f16, tile::launch_rmsnorm_f16,
                                   tile::launch_softmax_f16, tile::launch_row_sum_f16,
                                   tile::launch_row_minmax_f16};
    const Launchers &L =
        c.dtype == TILE_DTYPE_BF16 ? kBf16 : c.dtype == TILE_DTYPE_F16 ? kF16 : kF32;
    switch (kernel_op_of(c)) {
        case tile::OP_RESLN: err = L.resln(plan_id, a, stream); break;
        case tile::OP_LN: err = L.ln(plan_id, a, stream); break;
        case tile::OP_RMS: err = L.rms(plan_id, a, stream); break;
        case tile::OP_SUM: err = L.sum(plan_id, a, stream); break;
        case tile::OP_MINMAX: err = L.minmax(plan_id, a, stream); break;
        default: err = L.softmax(plan_id, a, stream); break;
    }
    if (err != cudaSuccess) {
        tile::set_last_cuda_error(static_cast<int>(err));
        return TILE_ERR_CUDA;
    }
    return TILE_OK;
}

// select_rows > 0: choose the plan as for a call of that many rows (a chunk
// of a larger matrix takes the whole matrix's plan, so its results are
// bitwise those of one call on the whole matrix).
int run_call(const Call &c, cudaStream_t stream, long long select_rows = 0) {
    bool noop = false;
    const int st = validate(c, &noop);
    if (st != TILE_OK || noop) return st;
    const int plan = select_plan(c.op, select_rows > 0 ? select_rows : c.rows, c.width,
                                 coaligned16(c), c.dtype, staged_ok(c), c.res != nullptr);
    if (plan < 0) return TILE_ERR_SHAPE;
    return launch(c, plan, stream);
}

int run_call_plan(const Call &c, int plan_id, cudaStream_t stream) {
    bool noop = false;
    const int st = validate(c, &noop);
    if (st != TILE_OK) return st;
    if (plan_id < 0 || plan_id >= kAllPlans || !covers(kPlans[plan_id], c.width, c.dtype))
        return TILE_ERR_PLAN;
    if (noop) return TILE_OK;
    if (kPlans[plan_id].V == 4 && !coaligned16(c)) return TILE_ERR_PLAN;
    if (whole_vectors(kPlans[plan_id]) && !staged_ok(c)) return TILE_ERR_PLAN;
    return launch(c, plan_id, stream);
}

tile_row_args_t args_of(const void *in, const void *res, const float *gamma, const float *beta,
                        void *out, float *out2, int rows, int width, float eps,
                        int dtype = TILE_DTYPE_F32) {
    tile_row_args_t a;
    a.dtype = dtype;
    a.in = in;
    a.residual = res;
    a.gamma = gamma;
    a.beta = beta;
    a.out = out;
    a.out2 = out2;
    a.rows = rows;
    a.width = width;
    a.eps = eps;
    return a;
}

// Backward plans hold two stripes (input and upstream gradient): a plan is
// built for backward when K * (elements per vector) <= 32 floats per stripe
// (2-byte rows of 16-byte vectors use the raw-word kernel: stripes of up to
// 8 vectors of 8).  The per-op tables in selector_tables.h are generated
// from a measured backward sweep (every built plan at each ladder width).
bool built_backward(const PlanDesc &p, int dtype = TILE_DTYPE_F32) {
    const bool raw = two_byte(dtype) && p.V == 4;     // raw-word stripes (bwd_kernel.cuh)
    return p.K * elems_per_vec(p, dtype) <= (raw ? tile::kMaxStripeBwdRaw : tile::kMaxStripeBwd);
}

// The backward plan for a call: 16-byte vectors when x, dy and dx share a
// 16-byte phase (the generated per-op tables, FP16 sharing BF16's), else the
// scalar plans.
int select_backward_plan(int op, int dtype, int width, bool vec4) {
    if (!vec4) return pick(kVec1, width);
    const bool b16 = two_byte(dtype);
    const int id = op == TILE_OP_LAYERNORM ? (b16 ? pick(kB16RegBwdLN, width)
                                                  : pick(kF32RegBwdLN, width))
                   : op == TILE_OP_RMSNORM ? (b16 ? pick(kB16RegBwdRMS, width)
                                                  : pick(kF32RegBwdRMS, width))
                                           : (b16 ? pick(kB16RegBwdSoftmax, width)
                                                  : pick(kF32RegBwdSoftmax, width));
    return (id >= 0 && built_backward(kPlans[id], dtype) && covers(kPlans[id], width, dtype))
               ? id : -1;
}

int bwd_kernel_op(int op) {
    return op == TILE_OP_LAYERNORM ? tile::BWD_LN_OP : op == TILE_OP_RMSNORM ? tile::BWD_RMS_OP
                                                                             : tile::BWD_SOFTMAX_OP;
}

// Checks and launch of a backward call; plan_id < 0 selects a plan.  x, dy,
// dx are [rows][width] of element type dtype; gamma and stats are FP32.
int run_backward(int op, int plan_id, int dtype, const void *x, const float *gamma,
                 const void *dy, void *dx, float *stats, int rows, int width, float eps,
                 cudaStream_t stream) {
    if (op != TILE_OP_LAYERNORM && op != TILE_OP_RMSNORM && op != TILE_OP_SOFTMAX)
        return TILE_ERR_OP;
    if (!valid_dtype(dtype)) return TILE_ERR_DTYPE;
    if (rows < 0 || width < 1 || width > TILE_MAX_WIDTH) return TILE_ERR_SHAPE;
    if (op != TILE_OP_SOFTMAX && !(std::isfinite(eps) && eps >= 0.0f)) return TILE_ERR_EPS;
    if (plan_id >= TILE_PLAN_COUNT) return TILE_ERR_PLAN;   // register plans only
    if (plan_id >= 0 &&
        (!built_backward(kPlans[plan_id], dtype) || !covers(kPlans[plan_id], width, dtype)))
        return TILE_ERR_PLAN;
    if (rows == 0) return TILE_OK;
    if (op == TILE_OP_SOFTMAX) {
        gamma = nullptr;
        stats = nullptr;
    }
    if (x == nullptr || dy == nullptr || dx == nullptr) return TILE_ERR_NULL;
    const size_t es = elem_size(dtype);
    if (misaligned_to(x, es) || misaligned_to(dy, es) || misaligned_to(dx, es) ||
        misaligned(gamma) || misaligned(stats))
        return TILE_ERR_ALIGN;
    const size_t mat = static_cast<size_t>(rows) * static_cast<size_t>(width) * es;
    const size_t vec = static_cast<size_t>(width) * sizeof(float);
    const size_t st = static_cast<size_t>(rows) * 2 * sizeof(float);
    if (overlaps(dx, mat, x, mat) || overlaps(dx, mat, dy, mat) || overlaps(dx, mat, gamma, vec) ||
        overlaps(stats, st, x, mat) || overlaps(stats, st, dy, mat) || overlaps(stats, st, dx, mat) ||
        overlaps(stats, st, gamma, vec))
        return TILE_ERR_ALIAS;
    const uintptr_t a = reinterpret_cast<uintptr_t>(x);
    const bool vec4 = ((a ^ reinterpret_cast<uintptr_t>(dy)) & 15u) == 0 &&
                      ((a ^ reinterpret_cast<uintptr_t>(dx)) & 15u) == 0;
    if (plan_id < 0) plan_id = select_backward_plan(op, dtype, width, vec4);
    if (plan_id < 0) return TILE_ERR_SHAPE;
    if (kPlans[plan_id].V == 4 && !vec4) return TILE_ERR_PLAN;
    if (grid_of(kPlans[plan_id], rows) > 0x7fffffffLL) return TILE_ERR_SHAPE;
    TILE_INJECTED_FAILURE();
    tile::BwdArgs args{x, dy, gamma, dx, stats, rows, width, eps, nullptr,
                       1.0f / static_cast<float>(width)};
    const int kop = bwd_kernel_op(op);
    const cudaError_t err =
        dtype == TILE_DTYPE_BF16  ? tile::launch_backward_bf16(kop, plan_id, args, stream)
        : dtype == TILE_DTYPE_F16 ? tile::launch_backward_f16(kop, plan_id, args, stream)
                                  : tile::launch_backward(kop, plan_id, args, stream);
    if (err != cudaSuccess) {
        tile::set_last_cuda_error(static_cast<int>(err));
        return TILE_ERR_CUDA;
    }
    return TILE_OK;
}

// Checks and launch of the parameter gradients; in and dy of element type
// dtype.
int run_param_grad(int dtype, const void *in, const void *dy, const float *row_stats,
                   float *dgamma, float *dbeta, int rows, int width, void *workspace,
                   size_t workspace_bytes, cudaStream_t stream) {
    if (!valid_dtype(dtype)) return TILE_ERR_DTYPE;
    if (rows < 0 || width < 1 || width > TILE_MAX_WIDTH) return TILE_ERR_SHAPE;
    if (in == nullptr || dy == nullptr || dgamma == nullptr) return TILE_ERR_NULL;
    if (rows > 0 && (row_stats == nullptr || workspace == nullptr)) return TILE_ERR_NULL;
    const size_t es = elem_size(dtype);
    if (misaligned_to(in, es) || misaligned_to(dy, es))
        return TILE_ERR_ALIGN;
    for (const void *p : {static_cast<const void *>(row_stats), static_cast<const void *>(dgamma),
                          static_cast<const void *>(dbeta), static_cast<const void *>(workspace)})
        if (misaligned(p)) return TILE_ERR_ALIGN;
    const size_t vec = static_cast<size_t>(width) * sizeof(float);
    if (rows == 0) {
        // no rows: the sums are zero
        cudaError_t err = cudaMemsetAsync(dgamma, 0, vec, stream);
        if (err == cudaSuccess && dbeta != nullptr) err = cudaMemsetAsync(dbeta, 0, vec, stream);
        if (err != cudaSuccess) {
            tile::set_last_cuda_error(static_cast<int>(err));
            return TILE_ERR_CUDA;
        }
        return TILE_OK;
    }
    const size_t need = tile_norm_param_grad_workspace_bytes(rows, width);
    if (workspace_bytes < need) return TILE_ERR_WORKSPACE;
    const size_t mat = static_cast<size_t>(rows) * static_cast<size_t>(width) * es;
    const size_t st = static_cast<size_t>(rows) * 2 * sizeof(float);
    for (const void *o : {static_cast<const void *>(dgamma), static_cast<const void *>(dbeta)})
        if (overlaps(o, vec, in, mat) || overlaps(o, vec, dy, mat) || overlaps(o, vec, row_stats, st) ||
            overlaps(o, vec, workspace, need))
            return TILE_ERR_ALIAS;
    if (overlaps(dgamma, vec, dbeta, vec) || overlaps(workspace, need, in, mat) ||
        overlaps(workspace, need, dy, mat) || overlaps(workspace, need, row_stats, st))
        return TILE_ERR_ALIAS;
    TILE_INJECTED_FAILURE();
    const cudaError_t err = tile::launch_param_grad(dtype, in, dy, row_stats, dgamma, dbeta, rows,
                                                    width, static_cast<float *>(workspace), stream);
    if (err != cudaSuccess) {
        tile::set_last_cuda_error(static_cast<int>(err));
        return TILE_ERR_CUDA;
    }
    return TILE_OK;
}

}  // namespace

namespace tile {

namespace {
thread_local int t_last_cuda_error = 0;

// Launch failures injected on the host (tile_inject_launch_failure).
std::mutex g_inject_mu;
std::atomic<int> g_inject_armed{0};
int g_inject_skip = 0, g_inject_count = 0, g_inject_code = 0;

// tile_test_force_general_kernels: nonzero while the general kernel forms
// are forced.
std::atomic<int> g_force_general{0};
}  // namespace

bool whole_vector_kernels() { return g_force_general.load(std::memory_order_relaxed) == 0; }

void set_last_cuda_error(int err) { t_last_cuda_error = err; }
int last_cuda_error() { return t_last_cuda_error; }

cudaError_t injected_launch_failure() {
    if (g_inject_armed.load(std::memory_order_acquire) == 0) return cudaSuccess;
    std::lock_guard<std::mutex> lock(g_inject_mu);
    if (g_inject_count <= 0) return cudaSuccess;
    if (g_inject_skip > 0) {
        --g_inject_skip;
        return cudaSuccess;
    }
    if (--g_inject_count == 0) g_inject_armed.store(0, std::memory_order_release);
    return static_cast<cudaError_t>(g_inject_code);
}

int run_selected(int op, const float *in, const float *res, float *out, int rows, int width,
                 float eps, cudaStream_t stream, long long select_rows) {
    return run_call(make_call(op, args_of(in, res, nullptr, nullptr, out, nullptr, rows, width, eps)),
                    stream, select_rows);
}

int run_pairs(int kind, const float *in, float *value, float *derivative, long long n,
              cudaStream_t stream) {
    if (n < 0) return TILE_ERR_SHAPE;
    if (n == 0) return TILE_OK;
    if (in == nullptr || value == nullptr || derivative == nullptr) return TILE_ERR_NULL;
    if (misaligned(in) || misaligned(value) || misaligned(derivative)) return TILE_ERR_ALIGN;
    const size_t bytes = static_cast<size_t>(n) * sizeof(float);
    if (overlaps(value, bytes, in, bytes) || overlaps(derivative, bytes, in, bytes) ||
        overlaps(value, bytes, derivative, bytes))
        return TILE_ERR_ALIAS;
    TILE_INJECTED_FAILURE();
    const cudaError_t err = launch_pairs(kind, in, value, derivative, n, stream);
    if (err != cudaSuccess) {
        set_last_cuda_error(static_cast<int>(err));
        return TILE_ERR_CUDA;
    }
    return TILE_OK;
}

}  // namespace tile

extern "C" {

int tile_residual_layernorm_f32(const float *in, const float *residual, float *out, int rows,
                                int width, float eps, cudaStream_t stream) {
    return tile::run_selected(TILE_OP_RESIDUAL_LAYERNORM, in, residual, out, rows, width, eps, stream);
}

int tile_layernorm_f32(const float *in, float *out, int rows, int width, float eps,
                       cudaStream_t stream) {
    return tile::run_selected(TILE_OP_LAYERNORM, in, nullptr, out, rows, width, eps, stream);
}

int tile_rmsnorm_f32(const float *in, float *out, int rows, int width, float eps,
                     cudaStream_t stream) {
    return tile::run_selected(TILE_OP_RMSNORM, in, nullptr, out, rows, width, eps, stream);
}

int tile_softmax_f32(const float *in, float *out, int rows, int width, float eps,
                     cudaStream_t stream) {
    return tile::run_selected(TILE_OP_SOFTMAX, in, nullptr, out, rows, width, eps, stream);
}

int tile_layernorm_affine_f32(const float *in, const float *residual, const float *gamma,
                              const float *beta, float *out, int rows, int width, float eps,
                              cudaStream_t stream) {
    return run_call(make_call(TILE_OP_LAYERNORM_AFFINE,
                              args_of(in, residual, gamma, beta, out, nullptr, rows, width, eps)),
                    stream);
}

int tile_rmsnorm_weighted_f32(const float *in, const float *gamma, float *out, int rows,
                              int width, float eps, cudaStream_t stream) {
    return run_call(make_call(TILE_OP_RMSNORM_WEIGHTED,
                              args_of(in, nullptr, gamma, nullptr, out, nullptr, rows, width, eps)),
                    stream);
}

int tile_row_sum_f32(const float *in, float *sums, int rows, int width, cudaStream_t stream) {
    return run_call(make_call(TILE_OP_ROW_SUM,
                              args_of(in, nullptr, nullptr, nullptr, sums, nullptr, rows, width, 0.0f)),
                    stream);
}

int tile_row_minmax_f32(const float *in, float *mins, float *maxs, int rows, int width,
                        cudaStream_t stream) {
    return run_call(make_call(TILE_OP_ROW_MINMAX,
                              args_of(in, nullptr, nullptr, nullptr, mins, maxs, rows, width, 0.0f)),
                    stream);
}

int tile_residual_layernorm_bf16(const void *in, const void *residual, void *out, int rows,
                                 int width, float eps, cudaStream_t stream) {
    return run_call(make_call(TILE_OP_RESIDUAL_LAYERNORM,
                              args_of(in, residual, nullptr, nullptr, out, nullptr, rows, width,
                                      eps, TILE_DTYPE_BF16)),
                    stream);
}

int tile_layernorm_bf16(const void *in, void *out, int rows, int width, float eps,
                        cudaStream_t stream) {
    return run_call(make_call(TILE_OP_LAYERNORM, args_of(in, nullptr, nullptr, nullptr, out,
                                                         nullptr, rows, width, eps,
                                                         TILE_DTYPE_BF16)),
                    stream);
}

int tile_rmsnorm_bf16(const void *in, void *out, int rows, int width, float eps,
                      cudaStream_t stream) {
    return run_call(make_call(TILE_OP_RMSNORM, args_of(in, nullptr, nullptr, nullptr, out,
                                                       nullptr, rows, width, eps,
                                                       TILE_DTYPE_BF16)),
                    stream);
}

int tile_softmax_bf16(const void *in, void *out, int rows, int width, float eps,
                      cudaStream_t stream) {
    return run_call(make_call(TILE_OP_SOFTMAX, args_of(in, nullptr, nullptr, nullptr, out,
                                                       nullptr, rows, width, eps,
                                                       TILE_DTYPE_BF16)),
                    stream);
}

int tile_layernorm_affine_bf16(const void *in, const void *residual, const float *gamma,
                               const float *beta, void *out, int rows, int width, float eps,
                               cudaStream_t stream) {
    return run_call(make_call(TILE_OP_LAYERNORM_AFFINE,
                              args_of(in, residual, gamma, beta, out, nullptr, rows, width, eps,
                                      TILE_DTYPE_BF16)),
                    stream);
}

int tile_rmsnorm_weighted_bf16(const void *in, const float *gamma, void *out, int rows,
                               int width, float eps, cudaStream_t stream) {
    return run_call(make_call(TILE_OP_RMSNORM_WEIGHTED,
                              args_of(in, nullptr, gamma, nullptr, out, nullptr, rows, width, eps,
                                      TILE_DTYPE_BF16)),
                    stream);
}

int tile_row_sum_bf16(const void *in, float *sums, int rows, int width, cudaStream_t stream) {
    return run_call(make_call(TILE_OP_ROW_SUM, args_of(in, nullptr, nullptr, nullptr, sums,
                                                       nullptr, rows, width, 0.0f,
                                                       TILE_DTYPE_BF16)),
                    stream);
}

int tile_row_minmax_bf16(const void *in, float *mins, float *maxs, int rows, int width,
                         cudaStream_t stream) {
    return run_call(make_call(TILE_OP_ROW_MINMAX, args_of(in, nullptr, nullptr, nullptr, mins,
                                                          maxs, rows, width, 0.0f,
                                                          TILE_DTYPE_BF16)),
                    stream);
}

int tile_residual_layernorm_f16(const void *in, const void *residual, void *out, int rows,
                                 int width, float eps, cudaStream_t stream) {
    return run_call(make_call(TILE_OP_RESIDUAL_LAYERNORM,
                              args_of(in, residual, nullptr, nullptr, out, nullptr, rows, width,
                                      eps, TILE_DTYPE_F16)),
                    stream);
}

int tile_layernorm_f16(const void *in, void *out, int rows, int width, float eps,
                        cudaStream_t stream) {
    return run_call(make_call(TILE_OP_LAYERNORM, args_of(in, nullptr, nullptr, nullptr, out,
                                                         nullptr, rows, width, eps,
                                                         TILE_DTYPE_F16)),
                    stream);
}

int tile_rmsnorm_f16(const void *in, void *out, int rows, int width, float eps,
                      cudaStream_t stream) {
    return run_call(make_call(TILE_OP_RMSNORM, args_of(in, nullptr, nullptr, nullptr, out,
                                                       nullptr, rows, width, eps,
                                                       TILE_DTYPE_F16)),
                    stream);
}

int tile_softmax_f16(const void *in, void *out, int rows, int width, float eps,
                      cudaStream_t stream) {
    return run_call(make_call(TILE_OP_SOFTMAX, args_of(in, nullptr, nullptr, nullptr, out,
                                                       nullptr, rows, width, eps,
                                                       TILE_DTYPE_F16)),
                    stream);
}

int tile_layernorm_affine_f16(const void *in, const void *residual, const float *gamma,
                               const float *beta, void *out, int rows, int width, float eps,
                               cudaStream_t stream) {
    return run_call(make_call(TILE_OP_LAYERNORM_AFFINE,
                              args_of(in, residual, gamma, beta, out, nullptr, rows, width, eps,
                                      TILE_DTYPE_F16)),
                    stream);
}

int tile_rmsnorm_weighted_f16(const void *in, const float *gamma, void *out, int rows,
                               int width, float eps, cudaStream_t stream) {
    return run_call(make_call(TILE_OP_RMSNORM_WEIGHTED,
                              args_of(in, nullptr, gamma, nullptr, out, nullptr, rows, width, eps,
                                      TILE_DTYPE_F16)),
                    stream);
}

int tile_row_sum_f16(const void *in, float *sums, int rows, int width, cudaStream_t stream) {
    return run_call(make_call(TILE_OP_ROW_SUM, args_of(in, nullptr, nullptr, nullptr, sums,
                                                       nullptr, rows, width, 0.0f,
                                                       TILE_DTYPE_F16)),
                    stream);
}

int tile_row_minmax_f16(const void *in, float *mins, float *maxs, int rows, int width,
                         cudaStream_t stream) {
    return run_call(make_call(TILE_OP_ROW_MINMAX, args_of(in, nullptr, nullptr, nullptr, mins,
                                                          maxs, rows, width, 0.0f,
                                                          TILE_DTYPE_F16)),
                    stream);
}

int tile_run_plan_args_f32(int op, int plan_id, const tile_row_args_t *args, cudaStream_t stream) {
    if (args == nullptr) return TILE_ERR_NULL;
    return run_call_plan(make_call(op, *args), plan_id, stream);
}

int tile_test_staged_wait_timeout(int op, int plan_id, const tile_row_args_t *args,
                                  unsigned int spin_limit, cudaStream_t stream) {
    if (args == nullptr) return TILE_ERR_NULL;
    const Call c = make_call(op, *args);
    bool noop = false;
    const int st = validate(c, &noop);
    if (st != TILE_OK) return st;
    if (plan_id < 0 || plan_id >= kAllPlans || !kPlans[plan_id].staged ||
        !covers(kPlans[plan_id], c.width, c.dtype) || !staged_ok(c))
        return TILE_ERR_PLAN;
    if (noop) return TILE_OK;
    if (grid_of(kPlans[plan_id], c.rows) > 0x7fffffffLL) return TILE_ERR_SHAPE;
    TILE_INJECTED_FAILURE();
    tile::RowArgs a{c.in, c.res, c.gamma, c.beta, c.out, c.out2, c.rows, c.width, c.eps, nullptr,
                    1.0f / static_cast<float>(c.width)};
    const cudaError_t err = tile::launch_staged_withheld(kernel_op_of(c), c.dtype, plan_id, a,
                                                         spin_limit < 1 ? 1u : spin_limit, stream);
    if (err != cudaSuccess) {
        tile::set_last_cuda_error(static_cast<int>(err));
        return TILE_ERR_CUDA;
    }
    return TILE_OK;
}

int tile_run_plan_f32(int op, int plan_id, const float *in, const float *residual, float *out,
                      int rows, int width, float eps, cudaStream_t stream) {
    if (op > TILE_OP_SOFTMAX) return TILE_ERR_OP;
    return run_call_plan(make_call(op, args_of(in, residual, nullptr, nullptr, out, nullptr, rows,
                                               width, eps)),
                         plan_id, stream);
}

int tile_describe_plan_ex(int op, int dtype, int rows, int width, tile_plan_t *plan) {
    if (!valid_op(op)) return TILE_ERR_OP;
    if (!valid_dtype(dtype)) return TILE_ERR_DTYPE;
    if (rows < 0 || width < 1 || width > TILE_MAX_WIDTH) return TILE_ERR_SHAPE;
    if (plan == nullptr) return TILE_ERR_NULL;
    const int id = select_plan(op, rows, width, true, dtype, true);
    if (id < 0) return TILE_ERR_SHAPE;
    fill_plan(kPlans[id], op, dtype, rows, width, plan);
    return TILE_OK;
}

int tile_describe_plan(int op, int rows, int width, tile_plan_t *plan) {
    return tile_describe_plan_ex(op, TILE_DTYPE_F32, rows, width, plan);
}

int tile_plan_count(void) { return kAllPlans; }

int tile_plan_info_ex(int id, int op, int dtype, int rows, int width, tile_plan_t *plan) {
    if (id < 0 || id >= kAllPlans) return TILE_ERR_PLAN;
    if (!valid_op(op)) return TILE_ERR_OP;
    if (!valid_dtype(dtype)) return TILE_ERR_DTYPE;
    if (!built(kPlans[id], dtype)) return TILE_ERR_PLAN;
    // the staged and R-row kernels have no row-reduction (sum, min/max) variant
    if (whole_vectors(kPlans[id]) && (op == TILE_OP_ROW_SUM || op == TILE_OP_ROW_MINMAX))
        return TILE_ERR_PLAN;
    if (rows < 0 || width < 1 || width > TILE_MAX_WIDTH || !covers(kPlans[id], width, dtype))
        return TILE_ERR_SHAPE;
    if (plan == nullptr) return TILE_ERR_NULL;
    fill_plan(kPlans[id], op, dtype, rows, width, plan);
    return TILE_OK;
}

int tile_plan_info(int id, int op, int rows, int width, tile_plan_t *plan) {
    return tile_plan_info_ex(id, op, TILE_DTYPE_F32, rows, width, plan);
}

int tile_max_width(void) { return TILE_MAX_WIDTH; }

int tile_last_cuda_error(void) { return tile::last_cuda_error(); }

int tile_inject_launch_failure(int cuda_error, int skip, int count) {
    if (skip < 0 || count < 0 || (count > 0 && cuda_error == 0)) return TILE_ERR_SHAPE;
    std::lock_guard<std::mutex> lock(tile::g_inject_mu);
    tile::g_inject_code = cuda_error;
    tile::g_inject_skip = skip;
    tile::g_inject_count = count;
    tile::g_inject_armed.store(count > 0 ? 1 : 0, std::memory_order_release);
    return TILE_OK;
}

int tile_test_force_general_kernels(int on) {
    tile::g_force_general.store(on != 0 ? 1 : 0, std::memory_order_relaxed);
    return TILE_OK;
}

const char *tile_status_string(int status) {
    switch (status) {
        case TILE_OK: return "ok";
        case TILE_ERR_NULL: return "a required pointer is NULL";
        case TILE_ERR_SHAPE: return "rows < 0, width < 1, width above the maximum, or grid too large";
        case TILE_ERR_ALIAS: return "an output overlaps an input or the other output";
        case TILE_ERR_EPS: return "eps is negative or not finite";
        case TILE_ERR_CUDA: return "the CUDA runtime reported an error (see tile_last_cuda_error)";
        case TILE_ERR_OP: return "unknown operation code";
        case TILE_ERR_ALIGN: return "a pointer is not 4-byte aligned (workspace: 256-byte)";
        case TILE_ERR_PLAN: return "the plan does not exist, cannot cover the width, or needs 16-byte co-aligned pointers";
        case TILE_ERR_DEVICE: return "a kernel recorded an error in the device status word";
        case TILE_ERR_WORKSPACE: return "the device workspace cannot hold one row chunk twice";
        case TILE_ERR_DTYPE: return "unknown element type code";
        default: return "unknown status";
    }
}

int tile_check_device_status(cudaStream_t stream) {
    unsigned int word = 0, v = 0;
    cudaError_t (*fetch[])(unsigned int *, cudaStream_t) = {
        tile::status_residual_layernorm, tile::status_layernorm, tile::status_rmsnorm,
        tile::status_softmax, tile::status_row_sum, tile::status_row_minmax,
        tile::status_residual_layernorm_bf16, tile::status_layernorm_bf16,
        tile::status_rmsnorm_bf16, tile::status_softmax_bf16, tile::status_row_sum_bf16,
        tile::status_row_minmax_bf16, tile::status_residual_layernorm_f16,
        tile::status_layernorm_f16, tile::status_rmsnorm_f16, tile::status_softmax_f16,
        tile::status_row_sum_f16, tile::status_row_minmax_f16, tile::status_pairs,
        tile::status_backward, tile::status_backward_bf16, tile::status_backward_f16,
        tile::status_param_grad, tile::status_staged, tile::status_multi};
    for (auto f : fetch) {
        v = 0;
        const cudaError_t err = f(&v, stream);
        if (err != cudaSuccess) {
            tile::set_last_cuda_error(static_cast<int>(err));
            return TILE_ERR_CUDA;
        }
        word |= v;
    }
    return word ? TILE_ERR_DEVICE : TILE_OK;
}

int tile_layernorm_backward_f32(const float *in, const float *gamma, const float *dy, float *dx,
                                float *row_stats, int rows, int width, float eps,
                                cudaStream_t stream) {
    return run_backward(TILE_OP_LAYERNORM, -1, TILE_DTYPE_F32, in, gamma, dy, dx, row_stats, rows,
                        width, eps, stream);
}

int tile_rmsnorm_backward_f32(const float *in, const float *gamma, const float *dy, float *dx,
                              float *row_stats, int rows, int width, float eps,
                              cudaStream_t stream) {
    return run_backward(TILE_OP_RMSNORM, -1, TILE_DTYPE_F32, in, gamma, dy, dx, row_stats, rows,
                        width, eps, stream);
}

int tile_softmax_backward_f32(const float *y, const float *dy, float *dx, int rows, int width,
                              cudaStream_t stream) {
    return run_backward(TILE_OP_SOFTMAX, -1, TILE_DTYPE_F32, y, nullptr, dy, dx, nullptr, rows,
                        width, 0.0f, stream);
}

int tile_run_backward_plan_f32(int op, int plan_id, const float *in, const float *gamma,
                               const float *dy, float *dx, float *row_stats, int rows, int width,
                               float eps, cudaStream_t stream) {
    if (plan_id < 0) return TILE_ERR_PLAN;
    return run_backward(op, plan_id, TILE_DTYPE_F32, in, gamma, dy, dx, row_stats, rows, width,
                        eps, stream);
}

int tile_describe_backward_plan(int op, int dtype, int rows, int width, tile_plan_t *plan) {
    if (op != TILE_OP_LAYERNORM && op != TILE_OP_RMSNORM && op != TILE_OP_SOFTMAX)
        return TILE_ERR_OP;
    if (!valid_dtype(dtype)) return TILE_ERR_DTYPE;
    if (rows < 0 || width < 1 || width > TILE_MAX_WIDTH) return TILE_ERR_SHAPE;
    if (plan == nullptr) return TILE_ERR_NULL;
    const int id = select_backward_plan(op, dtype, width, true);
    if (id < 0) return TILE_ERR_SHAPE;
    fill_plan(kPlans[id], op, dtype, rows, width, plan);
    return TILE_OK;
}

int tile_run_backward_plan_ex(int op, int plan_id, int dtype, const void *in, const float *gamma,
                              const void *dy, void *dx, float *row_stats, int rows, int width,
                              float eps, cudaStream_t stream) {
    if (plan_id < 0) return TILE_ERR_PLAN;
    return run_backward(op, plan_id, dtype, in, gamma, dy, dx, row_stats, rows, width, eps,
                        stream);
}

#define TILE_BWD_2BYTE(suffix, dtype)                                                           \
    int tile_layernorm_backward_##suffix(const void *in, const float *gamma, const void *dy,     \
                                         void *dx, float *row_stats, int rows, int width,       \
                                         float eps, cudaStream_t stream) {                      \
        return run_backward(TILE_OP_LAYERNORM, -1, dtype, in, gamma, dy, dx, row_stats, rows,    \
                            width, eps, stream);                                                \
    }                                                                                           \
    int tile_rmsnorm_backward_##suffix(const void *in, const float *gamma, const void *dy,       \
                                       void *dx, float *row_stats, int rows, int width,         \
                                       float eps, cudaStream_t stream) {                        \
        return run_backward(TILE_OP_RMSNORM, -1, dtype, in, gamma, dy, dx, row_stats, rows,      \
                            width, eps, stream);                                                \
    }                                                                                           \
    int tile_softmax_backward_##suffix(const void *y, const void *dy, void *dx, int rows,        \
                                       int width, cudaStream_t stream) {                        \
        return run_backward(TILE_OP_SOFTMAX, -1, dtype, y, nullptr, dy, dx, nullptr, rows,       \
                            width, 0.0f, stream);                                               \
    }                                                                                           \
    int tile_norm_param_grad_##suffix(const void *in, const void *dy, const float *row_stats,    \
                                      float *dgamma, float *dbeta, int rows, int width,         \
                                      void *workspace, size_t workspace_bytes,                  \
                                      cudaStream_t stream) {                                    \
        return run_param_grad(dtype, in, dy, row_stats, dgamma, dbeta, rows, width, workspace,   \
                              workspace_bytes, stream);                                         \
    }
TILE_BWD_2BYTE(bf16, TILE_DTYPE_BF16)
TILE_BWD_2BYTE(f16, TILE_DTYPE_F16)
#undef TILE_BWD_2BYTE

size_t tile_norm_param_grad_workspace_bytes(int rows, int width) {
    if (rows < 1 || width < 1) return 0;
    return static_cast<size_t>(tile::param_blocks(rows)) * 2 * static_cast<size_t>(width) *
           sizeof(float);
}

int tile_norm_param_grad_f32(const float *in, const float *dy, const float *row_stats,
                             float *dgamma, float *dbeta, int rows, int width, void *workspace,
                             size_t workspace_bytes, cudaStream_t stream) {
    return run_param_grad(TILE_DTYPE_F32, in, dy, row_stats, dgamma, dbeta, rows, width,
                          workspace, workspace_bytes, stream);
}

int tile_sigmoid_pair_f32(const float *in, float *value, float *derivative, long long n,
                          cudaStream_t stream) {
    return tile::run_pairs(tile::PAIR_SIGMOID, in, value, derivative, n, stream);
}

int tile_gelu_tanh_pair_f32(const float *in, float *value, float *derivative, long long n,
                            cudaStream_t stream) {
    return tile::run_pairs(tile::PAIR_GELU_TANH, in, value, derivative, n, stream);
}

}  // extern "C"
