"""Host-only checks of the C ABI: the library loads, exports every function
declared in include/*.h, and rejects bad arguments before any CUDA call.

The argument tests pass fake device addresses that every call must reject
before launching anything.  As a second guard they run only where no GPU is
visible, so a mistake in a test can never launch a kernel on fake pointers."""

import ctypes
import glob
import os
import re

import pytest

import tile_compiler_row_gb300 as tile
from tile_compiler_row_gb300 import _build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

OK, NULL, SHAPE, ALIAS, EPS, CUDA, OP, ALIGN, PLAN, DEVICE, WORKSPACE = 0, -1, -2, -3, -4, -5, -6, -7, -8, -9, -10


@pytest.fixture(scope="module")
def lib():
    _build.build()
    return tile.load()


def declared_functions():
    names = set()
    for hdr in glob.glob(os.path.join(ROOT, "include", "*.h")):
        text = open(hdr).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        for m in re.finditer(r"\b(tile_\w+)\s*\(", text):
            names.add(m.group(1))
    return sorted(names)


def test_header_declares_the_four_ops():
    names = declared_functions()
    for n in ("tile_residual_layernorm_f32", "tile_layernorm_f32", "tile_rmsnorm_f32",
              "tile_softmax_f32", "tile_describe_plan", "tile_status_string",
              "tile_check_device_status"):
        assert n in names


def test_every_declared_symbol_is_exported(lib):
    for name in declared_functions():
        assert hasattr(lib, name), f"{name} declared in include/ but not exported"


def test_python_binding_has_the_same_names():
    for name in declared_functions():
        assert hasattr(tile, name), f"binding lacks {name}"


def test_status_strings(lib):
    for code in (OK, NULL, SHAPE, ALIAS, EPS, CUDA, OP, ALIGN, PLAN, DEVICE, WORKSPACE):
        s = tile.tile_status_string(code)
        assert s and s != "unknown status"
    assert tile.tile_status_string(12345) == "unknown status"


A = 0x10000000      # fake, never dereferenced: every call below fails validation
B = 0x20000000


def _no_gpu():
    try:
        import torch
        return not torch.cuda.is_available()
    except Exception:
        return True


fake_pointers = pytest.mark.skipif(not _no_gpu(), reason="fake device pointers: CPU-only test")


def _resln(lib, x, r, y, rows, width, eps=1e-5):
    return lib.tile_residual_layernorm_f32(x, r, y, rows, width, eps, None)


@fake_pointers
def test_shape_errors(lib):
    assert _resln(lib, A, A, B, -1, 8) == SHAPE
    assert _resln(lib, A, A, B, 4, 0) == SHAPE
    assert _resln(lib, A, A, B, 4, tile.tile_max_width() + 1) == SHAPE
    assert lib.tile_softmax_f32(A, B, 1, -3, 0.0, None) == SHAPE


@fake_pointers
def test_rows_zero_is_a_noop(lib):
    assert _resln(lib, None, None, None, 0, 8) == OK
    assert lib.tile_softmax_f32(None, None, 0, 8, 0.0, None) == OK


@fake_pointers
def test_null_pointers(lib):
    assert _resln(lib, None, A, B, 2, 8) == NULL
    assert _resln(lib, A, None, B, 2, 8) == NULL
    assert _resln(lib, A, A, None, 2, 8) == NULL
    assert lib.tile_layernorm_f32(None, B, 2, 8, 1e-5, None) == NULL


@fake_pointers
def test_eps_checked_for_normalisers_only(lib):
    assert lib.tile_rmsnorm_f32(A, B, 2, 8, -1.0, None) == EPS
    assert lib.tile_layernorm_f32(A, B, 2, 8, float("nan"), None) == EPS
    assert _resln(lib, A, A, B, 2, 8, float("inf")) == EPS


@fake_pointers
def test_alignment(lib):
    assert lib.tile_rmsnorm_f32(A + 2, B, 2, 8, 1e-5, None) == ALIGN
    assert lib.tile_rmsnorm_f32(A, B + 1, 2, 8, 1e-5, None) == ALIGN


@fake_pointers
def test_alias(lib):
    # out overlaps in: [A, A+64) vs [A+32, A+96)
    assert lib.tile_layernorm_f32(A, A + 32, 2, 8, 1e-5, None) == ALIAS
    assert _resln(lib, A, B, B + 60, 2, 8) == ALIAS
    assert lib.tile_softmax_f32(A, A, 1, 1, 0.0, None) == ALIAS


@fake_pointers
def test_run_plan_rejects_bad_plans(lib):
    n = lib.tile_plan_count()
    assert lib.tile_run_plan_f32(0, -1, A, A, B, 2, 8, 1e-5, None) == PLAN
    assert lib.tile_run_plan_f32(0, n, A, A, B, 2, 8, 1e-5, None) == PLAN
    # plan 0 covers at most 131 columns
    assert lib.tile_run_plan_f32(1, 0, A, None, B, 2, 4096, 1e-5, None) == PLAN
    # a float4 plan needs co-aligned pointers (A and B+4 differ mod 16)
    assert lib.tile_run_plan_f32(1, 0, A, None, B + 4, 2, 8, 1e-5, None) == PLAN
    assert lib.tile_run_plan_f32(9, 0, A, None, B, 2, 8, 1e-5, None) == OP


def test_every_width_has_a_covering_plan(lib):
    widths = list(range(1, 600)) + [1023, 1024, 1025, 1537, 4095, 4096, 4097, 8192, 8195,
                                      16384, 16388, 32768, 32772, 65536, 65540, 131071, 131072]
    for op in range(4):
        for w in widths:
            p = tile.tile_describe_plan(op, 5, w)
            assert p["max_width"] >= w
            assert p["threads"] == 32 * p["warps_per_program"] * p["programs_per_cta"] <= 1024
            cap = p["chunks"] * p["workers"] * p["cluster"]
            assert (w // 4 if p["vec"] == 4 else w) <= cap
            assert p["grid"] == -(-5 // p["programs_per_cta"]) * p["cluster"]


def test_plan_info_table(lib):
    n = tile.tile_plan_count()
    assert n >= 20
    seen_vec1 = False
    for pid in range(n):
        info = tile.tile_plan_info(pid, 0, 3, 1)
        if info is None:                 # staged and R-row plans: whole vectors only
            info = tile.tile_plan_info(pid, 0, 3, 4)
            assert info is not None and info["path"] in (2, 3) and info["id"] == pid
            if info["path"] == 3:        # R rows per CTA on the same threads
                r = info["programs_per_cta"]
                assert r > 1 and info["grid"] == -(-3 // r)
            assert tile.tile_plan_info(pid, 0, 3, 6) is None
            continue
        assert info["id"] == pid
        assert tile.tile_plan_info(pid, 0, 3, info["max_width"]) is not None
        if info["max_width"] < tile.tile_max_width():
            assert tile.tile_plan_info(pid, 0, 3, info["max_width"] + 1) is None
        seen_vec1 |= info["vec"] == 1
        if info["cluster"] > 1:
            assert info["programs_per_cta"] == 1 and info["cluster"] <= 8
    assert seen_vec1


def test_describe_plan_errors(lib):
    plan = tile.TilePlan()
    assert lib.tile_describe_plan(8, 4, 8, ctypes.byref(plan)) == OP
    assert lib.tile_describe_plan(0, 4, 0, ctypes.byref(plan)) == SHAPE
    assert lib.tile_describe_plan(0, 4, 8, None) == NULL


def test_binding_rejects_cpu_tensors():
    import torch
    x = torch.zeros(2, 8)
    with pytest.raises(ValueError):
        tile.tile_rmsnorm_f32(x, torch.zeros(2, 8))


@fake_pointers
def test_host_entry_rejects_bad_arguments(lib):
    ws = 1 << 20
    W = 0x30000000                       # fake device workspace, 256-aligned
    f = lib.tile_run_host_f32
    assert f(0, A, A, B, 0, 8, 1e-5, None, 0, None) == OK          # rows == 0
    assert f(5, A, A, B, 2, 8, 1e-5, W, ws, None) == OP
    assert f(0, A, A, B, 2, 0, 1e-5, W, ws, None) == SHAPE
    assert f(1, A, None, B, 2, 8, -1.0, W, ws, None) == EPS
    assert f(0, A, None, B, 2, 8, 1e-5, W, ws, None) == NULL
    assert f(1, A, None, B, 2, 8, 1e-5, None, ws, None) == NULL
    assert f(1, A, None, B, 2, 8, 1e-5, W + 16, ws, None) == ALIGN
    assert f(1, A, None, A + 8, 2, 8, 1e-5, W, ws, None) == ALIAS
    # one row of 4096 floats needs 2 x 2 x 16 KiB for a unary op
    assert f(1, A, None, B, 2, 4096, 1e-5, W, 65535, None) == -10


@fake_pointers
def test_static_host_entry_rejects_bad_arguments_before_any_cuda_call(lib):
    """The entry point without a workspace finds argument errors on the host,
    before it looks up its device array (this container has no GPU, so any
    CUDA call would fail with TILE_ERR_CUDA instead)."""
    f = lib.tile_run_host_static_f32
    assert f(0, A, A, B, 0, 8, 1e-5, None) == OK            # rows == 0
    assert f(5, A, A, B, 2, 8, 1e-5, None) == OP
    assert f(0, A, A, B, 2, 0, 1e-5, None) == SHAPE
    assert f(1, A, None, B, 2, 8, -1.0, None) == EPS
    assert f(0, A, None, B, 2, 8, 1e-5, None) == NULL          # residual LN without r
    assert f(1, None, None, B, 2, 8, 1e-5, None) == NULL
    assert f(1, A, None, None, 2, 8, 1e-5, None) == NULL
    assert f(1, A, None, A + 8, 2, 8, 1e-5, None) == ALIAS
    assert f(0, A, B, B + 16, 2, 8, 1e-5, None) == ALIAS        # out overlaps r


@fake_pointers
def test_injected_launch_failures_are_reported_without_a_cuda_call(lib):
    """tile_inject_launch_failure: the armed launch attempts of every kind of
    entry point return TILE_ERR_CUDA with the injected error, before any
    CUDA call (this container has no GPU, so a CUDA call would report
    something else); argument errors still come first; skip and count are
    honoured and the hook disarms itself."""
    code = 719                                   # cudaErrorLaunchFailure
    assert lib.tile_inject_launch_failure(code, -1, 1) == SHAPE
    assert lib.tile_inject_launch_failure(code, 0, -1) == SHAPE
    assert lib.tile_inject_launch_failure(0, 0, 1) == SHAPE
    try:
        assert lib.tile_inject_launch_failure(code, 0, 6) == OK
        assert lib.tile_rmsnorm_f32(None, B, 2, 8, 1e-5, None) == NULL      # arguments first
        assert lib.tile_rmsnorm_f32(A, B, 2, 8, 1e-5, None) == CUDA
        assert lib.tile_last_cuda_error() == code
        assert lib.tile_residual_layernorm_bf16(A, A + 64, B, 2, 8, 1e-5, None) == CUDA
        assert lib.tile_softmax_backward_f32(A, A + 64, B, 2, 8, None) == CUDA
        assert lib.tile_sigmoid_pair_f32(A, B, B + 64, 16, None) == CUDA
        a = tile.TileRowArgs()
        a.in_, a.out, a.rows, a.width, a.eps, a.dtype = A, B, 4, 256, 1e-5, 1
        assert lib.tile_test_staged_wait_timeout(1, 45, ctypes.byref(a), 16, None) == CUDA
        ws, dg, db, st = 0x40000000, 0x50000000, 0x50001000, 0x60000000
        need = lib.tile_norm_param_grad_workspace_bytes(2, 8)
        assert lib.tile_norm_param_grad_f32(A, A + 64, st, dg, db, 2, 8, ws, need, None) == CUDA
        # the six armed attempts are used up: disarmed
        assert lib.tile_inject_launch_failure(code, 0, 0) == OK
        # skip: two attempts proceed (here they reach CUDA and fail otherwise),
        # the third reports the injected error
        assert lib.tile_inject_launch_failure(700, 2, 1) == OK
        assert lib.tile_rmsnorm_f32(A, B, 2, 8, 1e-5, None) != OK
        assert lib.tile_rmsnorm_f32(A, B, 2, 8, 1e-5, None) != OK
        assert lib.tile_rmsnorm_f32(A, B, 2, 8, 1e-5, None) == CUDA
        assert lib.tile_last_cuda_error() == 700
    finally:
        assert lib.tile_inject_launch_failure(0, 0, 0) == OK


def test_general_kernel_hook_is_host_only(lib):
    """tile_test_force_general_kernels sets a process-wide host flag: TILE_OK
    for any value on a machine without a GPU, and 0 restores the default
    (its effect on the launches is tested on the GPU)."""
    try:
        assert lib.tile_test_force_general_kernels(1) == OK
        assert lib.tile_test_force_general_kernels(7) == OK
    finally:
        assert lib.tile_test_force_general_kernels(0) == OK


@fake_pointers
def test_staged_wait_hook_rejects_bad_arguments(lib):
    a = tile.TileRowArgs()
    a.in_, a.out, a.rows, a.width, a.eps, a.dtype = A, B, 4, 256, 1e-5, 1
    f = lib.tile_test_staged_wait_timeout
    assert f(1, 45, None, 16, None) == NULL
    assert f(1, 7, ctypes.byref(a), 16, None) == PLAN           # a register plan
    assert f(1, 99, ctypes.byref(a), 16, None) == PLAN
    assert f(4, 45, ctypes.byref(a), 16, None) == PLAN          # row sum: no staged kernel
    a.rows = 0
    assert f(1, 45, ctypes.byref(a), 16, None) == OK            # nothing to launch


def test_host_workspace_bytes(lib):
    assert tile.tile_host_workspace_bytes("layernorm", 4096, 1) == 2 * 2 * 16384
    assert tile.tile_host_workspace_bytes("residual_layernorm", 100, 3) == 2 * 3 * 1280
    assert tile.tile_host_workspace_bytes("softmax", 0, 3) == 0
    assert tile.tile_host_workspace_bytes(9, 10, 3) == 0


@pytest.mark.parametrize("op", ["residual_layernorm", "layernorm", "rmsnorm", "softmax"])
@pytest.mark.parametrize("rows,width", [(1, 1), (3, 127), (37, 1537), (65536, 4096),
                                        (20000, 257), (5, 131072)])
@pytest.mark.parametrize("ws_rows", [1, 7, 1 << 20])
@pytest.mark.parametrize("direct", [False, True])
def test_host_schedule_fits_the_workspace(lib, op, rows, width, ws_rows, direct):
    """The host pipeline's chunking: every slot of the ring fits the
    workspace, chunks never exceed the rows, there are 2 to 4 slots, and a
    roomy workspace gives about 16 chunks of at least 1 MiB each."""
    ws = tile.tile_host_workspace_bytes(op, width, min(ws_rows, rows))
    chunk, slots = tile.tile_host_schedule(op, rows, width, ws, direct_output=direct)
    row_bytes = 4 * width
    per_slot = (2 if op == "residual_layernorm" else 1) + (0 if direct else 1)
    buf = -(-chunk * row_bytes // 256) * 256
    assert 1 <= chunk <= rows and 2 <= slots <= 4
    assert slots * per_slot * buf <= ws
    nchunks = -(-rows // chunk)
    if nchunks >= 2:
        assert slots <= nchunks
    if ws_rows >= rows:
        assert chunk == min(rows, max(-(-rows // 16), -(-(1 << 20) // row_bytes)))


def test_host_schedule_rejects_bad_arguments(lib):
    c, k = ctypes.c_int(), ctypes.c_int()
    f = lib.tile_host_schedule
    assert f(7, 4, 8, 1 << 20, 1, ctypes.byref(c), ctypes.byref(k)) == -6
    assert f(1, 0, 8, 1 << 20, 1, ctypes.byref(c), ctypes.byref(k)) == SHAPE
    assert f(1, 4, 0, 1 << 20, 1, ctypes.byref(c), ctypes.byref(k)) == SHAPE
    assert f(1, 4, 8, 1 << 20, 1, None, ctypes.byref(k)) == NULL
    assert f(1, 4, 4096, 65535, 1, ctypes.byref(c), ctypes.byref(k)) == -10


@fake_pointers
def test_new_row_ops_reject_bad_arguments(lib):
    f = lib.tile_layernorm_affine_f32
    assert f(A, None, None, None, B, 2, 8, 1e-5, None) == NULL            # gamma required
    assert f(A, None, A + 64, None, B, 2, 8, -1.0, None) == EPS
    assert f(A, None, B + 8, None, B, 2, 8, 1e-5, None) == ALIAS          # out overlaps gamma
    assert f(A, None, A + 64, B + 40, B, 2, 8, 1e-5, None) == ALIAS       # out overlaps beta
    assert f(A, None, A + 66, None, B, 2, 8, 1e-5, None) == ALIGN
    assert f(A, None, None, None, B, 0, 8, 1e-5, None) == OK              # rows == 0
    g = lib.tile_rmsnorm_weighted_f32
    assert g(A, None, B, 2, 8, 1e-5, None) == NULL
    assert g(A, A + 64, B, 2, 8, float("nan"), None) == EPS
    s = lib.tile_row_sum_f32
    assert s(A, None, 2, 8, None) == NULL
    assert s(A, A + 4, 2, 8, None) == ALIAS                               # sums inside x
    assert s(A, B, 2, 0, None) == SHAPE
    m = lib.tile_row_minmax_f32
    assert m(A, B, None, 2, 8, None) == NULL
    assert m(A, B, B + 4, 2, 8, None) == ALIAS                            # mins/maxs overlap
    assert m(A, B, A + 8, 2, 8, None) == ALIAS                            # maxs inside x
    assert m(A, B, B + 4096, 0, 8, None) == OK


@fake_pointers
def test_run_plan_args(lib):
    a = tile.TileRowArgs()
    a.in_, a.out, a.rows, a.width, a.eps = A, B, 2, 8, 1e-5
    assert lib.tile_run_plan_args_f32(4, 10**6, ctypes.byref(a), None) == PLAN
    assert lib.tile_run_plan_args_f32(42, 0, ctypes.byref(a), None) == OP
    assert lib.tile_run_plan_args_f32(0, 0, None, None) == NULL
    assert lib.tile_run_plan_args_f32(0, 0, ctypes.byref(a), None) == NULL  # residual missing


@fake_pointers
def test_pair_entry_points_reject_bad_arguments(lib):
    for f in (lib.tile_sigmoid_pair_f32, lib.tile_gelu_tanh_pair_f32):
        assert f(A, B, B + 4096, 0, None) == OK
        assert f(A, B, B + 4096, -1, None) == SHAPE
        assert f(None, B, B + 4096, 8, None) == NULL
        assert f(A, A + 4, B, 8, None) == ALIAS
        assert f(A, B, B + 16, 8, None) == ALIAS
        assert f(A, B + 2, B + 4096, 8, None) == ALIGN


def test_describe_plan_covers_the_new_ops(lib):
    for op in ("row_sum", "row_minmax", "layernorm_affine", "rmsnorm_weighted"):
        for w in (1, 127, 4096, 65536, 131072):
            p = tile.tile_describe_plan(op, 3, w)
            assert p["max_width"] >= w


@fake_pointers
def test_bf16_entry_points_reject_bad_arguments(lib):
    assert lib.tile_layernorm_bf16(A, B, 2, 0, 1e-5, None) == SHAPE
    assert lib.tile_layernorm_bf16(A + 1, B, 2, 8, 1e-5, None) == ALIGN     # odd address
    assert lib.tile_rmsnorm_bf16(A, A + 16, 2, 8, 1e-5, None) == ALIAS      # 2 x 8 x 2 bytes
    assert lib.tile_residual_layernorm_bf16(A, None, B, 2, 8, 1e-5, None) == NULL
    assert lib.tile_row_sum_bf16(A, B + 2, 2, 8, None) == ALIGN             # FP32 output
    a = tile.TileRowArgs()
    a.in_, a.out, a.rows, a.width, a.eps, a.dtype = A, B, 2, 8, 1e-5, 7
    assert lib.tile_run_plan_args_f32(1, 0, ctypes.byref(a), None) == -11


def test_bf16_plans(lib):
    for op in ("residual_layernorm", "layernorm", "rmsnorm", "softmax", "row_sum"):
        for w in (1, 127, 4096, 8192, 65536, 131072):
            p = tile.tile_describe_plan_ex(op, "bf16", 9, w)
            assert p["dtype"] == 1 and p["max_width"] >= w
            assert p["stripe_floats"] <= 64
    # K = 16 plans are not built for BF16
    k16 = [pid for pid in range(tile.tile_plan_count())
           if tile.tile_plan_info(pid, 0, 1, 4)["chunks"] == 16 and
           tile.tile_plan_info(pid, 0, 1, 4)["vec"] == 4]
    assert k16 and all(tile.tile_plan_info_ex(pid, 0, "bf16", 1, 1) is None for pid in k16)


def test_staged_plans_have_no_row_reductions(lib):
    staged = [pid for pid in range(tile.tile_plan_count())
              if (tile.tile_plan_info(pid, "layernorm", 8, 4096) or {}).get("path") in (2, 3)]
    assert staged
    for pid in staged:
        for op in ("row_sum", "row_minmax"):
            assert tile.tile_plan_info(pid, op, 8, 4096) is None
            assert tile.tile_plan_info_ex(pid, op, "bf16", 8, 4096) is None


@fake_pointers
def test_f16_entry_points_reject_bad_arguments(lib):
    assert lib.tile_layernorm_f16(A, B, 2, 0, 1e-5, None) == SHAPE
    assert lib.tile_layernorm_f16(A + 1, B, 2, 8, 1e-5, None) == ALIGN      # odd address
    assert lib.tile_softmax_f16(A, A + 16, 2, 8, 1e-5, None) == ALIAS       # 2 x 8 x 2 bytes
    assert lib.tile_residual_layernorm_f16(A, None, B, 2, 8, 1e-5, None) == NULL
    assert lib.tile_layernorm_affine_f16(A, None, None, None, B, 2, 8, 1e-5, None) == NULL
    assert lib.tile_row_minmax_f16(A, B + 2, B + 64, 2, 8, None) == ALIGN    # FP32 outputs
    assert lib.tile_rmsnorm_f16(A, B, 2, 8, -1.0, None) == EPS


def test_f16_plans_are_the_bf16_plans(lib):
    """FP16 rows have the BF16 geometry (2-byte elements, 8 per vector) and
    share its selector tables."""
    for op in ("residual_layernorm", "layernorm", "rmsnorm", "softmax", "row_sum",
               "row_minmax", "layernorm_affine", "rmsnorm_weighted"):
        for rows, w in ((9, 1), (9, 127), (65536, 4096), (4096, 8192), (1024, 16384),
                        (64, 65536), (9, 131072)):
            a = tile.tile_describe_plan_ex(op, "f16", rows, w)
            b = tile.tile_describe_plan_ex(op, "bf16", rows, w)
            assert a["dtype"] == 2
            assert {k: v for k, v in a.items() if k != "dtype"} == \
                {k: v for k, v in b.items() if k != "dtype"}
    for pid in range(tile.tile_plan_count()):
        a = tile.tile_plan_info_ex(pid, "layernorm", "f16", 4, 1024)
        b = tile.tile_plan_info_ex(pid, "layernorm", "bf16", 4, 1024)
        assert (a is None) == (b is None)


@fake_pointers
def test_backward_entry_points_reject_bad_arguments(lib):
    """Backward and parameter-gradient calls check their arguments on the
    host like the forward ones (rows == 0 is a no-op for the input
    gradients; the parameter gradients then write zeros, so that case is
    left to the GPU tests)."""
    X, DY, DX = A, A + 4096, B
    ln = lib.tile_layernorm_backward_f32        # (in, gamma, dy, dx, stats, rows, width, eps, s)
    assert ln(None, None, DY, DX, None, 2, 8, 1e-5, None) == NULL
    assert ln(X, None, None, DX, None, 2, 8, 1e-5, None) == NULL
    assert ln(X, None, DY, None, None, 2, 8, 1e-5, None) == NULL
    assert ln(X, None, DY, DX, None, -1, 8, 1e-5, None) == SHAPE
    assert ln(X, None, DY, DX, None, 2, 0, 1e-5, None) == SHAPE
    assert ln(X, None, DY, DX, None, 2, 8, -1.0, None) == EPS
    assert ln(X, None, DY, X + 32, None, 2, 8, 1e-5, None) == ALIAS      # dx overlaps in
    assert ln(X, None, DY, DX, X + 4, 2, 8, 1e-5, None) == ALIAS         # stats inside in
    assert ln(X, None, DY, DX + 2, None, 2, 8, 1e-5, None) == ALIGN
    assert ln(None, None, None, None, None, 0, 8, 1e-5, None) == OK
    rms = lib.tile_rmsnorm_backward_f32
    assert rms(X, None, DY, DX, None, 2, 8, float("nan"), None) == EPS
    assert rms(X, DX, DY, DX, None, 2, 8, 1e-5, None) == ALIAS           # dx overlaps gamma
    sm = lib.tile_softmax_backward_f32          # (y, dy, dx, rows, width, s)
    assert sm(X, None, DX, 2, 8, None) == NULL
    assert sm(X, DY, X, 2, 8, None) == ALIAS
    assert sm(X, DY, DX, 2, 0, None) == SHAPE
    bf = lib.tile_layernorm_backward_bf16
    assert bf(X, None, None, DX, None, 2, 8, 1e-5, None) == NULL
    assert bf(X, None, DY, DX + 1, None, 2, 8, 1e-5, None) == ALIGN     # 2-byte alignment
    pg = lib.tile_norm_param_grad_f32           # (in, dy, stats, dg, db, rows, width, ws, bytes, s)
    need = lib.tile_norm_param_grad_workspace_bytes(2, 8)
    assert need > 0
    WS, DG, ST = B + 65536, B + 8192, B + 16384
    assert pg(X, DY, ST, DG, None, 2, 8, WS, need - 1, None) == WORKSPACE
    assert pg(X, DY, None, DG, None, 2, 8, WS, need, None) == NULL
    assert pg(X, DY, ST, None, None, 2, 8, WS, need, None) == NULL
    assert pg(X, DY, ST, DG, None, -1, 8, WS, need, None) == SHAPE
    ex = lib.tile_run_backward_plan_ex          # (op, plan, dtype, in, gamma, dy, dx, stats, ...)
    assert ex(1, 0, 7, X, None, DY, DX, None, 2, 8, 1e-5, None) == -11  # TILE_ERR_DTYPE
    assert ex(1, 10 ** 6, 0, X, None, DY, DX, None, 2, 8, 1e-5, None) == PLAN
    assert ex(9, 0, 0, X, None, DY, DX, None, 2, 8, 1e-5, None) == OP
