"""Python binding of ``libtile_rows.so``: fused FP32 row normalisation on GB300.

Argument marshalling only.  Every function here checks tensor metadata, takes
device pointers and the current CUDA stream from PyTorch, and calls the C ABI
of the same name (declared in ``include/tile_rows.h``); all arithmetic runs in
the library's CUDA kernels.  There is no CPU path: CPU tensors are rejected,
and importing the binding without the built library raises.

    import torch, tile_compiler_row_gb300 as tile
    y = torch.empty_like(x)
    tile.tile_residual_layernorm_f32(x, r, y, eps=1e-5)
"""

from __future__ import annotations

import ctypes
import os

from ._build import LIBRARY

__all__ = [
    "TileError", "OPS", "load", "library_path",
    "tile_residual_layernorm_f32", "tile_layernorm_f32", "tile_rmsnorm_f32",
    "tile_softmax_f32", "tile_run_plan_f32", "tile_describe_plan", "tile_plan_info",
    "tile_plan_count", "tile_max_width", "tile_status_string",
    "tile_check_device_status", "tile_last_cuda_error", "tile_run_host_f32",
    "tile_host_workspace_bytes", "tile_host_schedule", "tile_run_host_static_f32", "tile_layernorm_affine_f32",
    "tile_rmsnorm_weighted_f32", "tile_row_sum_f32", "tile_row_minmax_f32",
    "tile_run_plan_args_f32", "tile_sigmoid_pair_f32", "tile_gelu_tanh_pair_f32",
    "tile_residual_layernorm_bf16", "tile_layernorm_bf16", "tile_rmsnorm_bf16",
    "tile_softmax_bf16", "tile_layernorm_affine_bf16", "tile_rmsnorm_weighted_bf16",
    "tile_row_sum_bf16", "tile_row_minmax_bf16", "tile_residual_layernorm_f16",
    "tile_layernorm_f16", "tile_rmsnorm_f16", "tile_softmax_f16", "tile_layernorm_affine_f16",
    "tile_rmsnorm_weighted_f16", "tile_row_sum_f16", "tile_row_minmax_f16",
    "tile_describe_plan_ex", "tile_plan_info_ex",
    "tile_layernorm_backward_f32", "tile_rmsnorm_backward_f32", "tile_softmax_backward_f32",
    "tile_run_backward_plan_f32", "tile_norm_param_grad_workspace_bytes",
    "tile_norm_param_grad_f32", "tile_run_backward_plan_ex",
    "tile_layernorm_backward_bf16", "tile_rmsnorm_backward_bf16", "tile_softmax_backward_bf16",
    "tile_norm_param_grad_bf16", "tile_layernorm_backward_f16", "tile_rmsnorm_backward_f16",
    "tile_softmax_backward_f16", "tile_norm_param_grad_f16", "tile_test_staged_wait_timeout",
    "tile_inject_launch_failure", "tile_describe_backward_plan", "tile_test_force_general_kernels",
    "residual_layernorm", "layernorm", "rmsnorm", "softmax", "run",
]

#: Library operation codes, by name.
OPS = {"residual_layernorm": 0, "layernorm": 1, "rmsnorm": 2, "softmax": 3, "row_sum": 4,
       "row_minmax": 5, "layernorm_affine": 6, "rmsnorm_weighted": 7}

TILE_OK = 0

#: Element type codes (TILE_DTYPE_*).
DTYPES = {"f32": 0, "bf16": 1, "f16": 2}


class TileError(RuntimeError):
    """A non-zero status returned by the C ABI."""

    def __init__(self, status: int, where: str):
        self.status = status
        msg = f"{where}: status {status} ({tile_status_string(status)})"
        if status == -5:
            msg += f", cudaError {tile_last_cuda_error()}"
        super().__init__(msg)


class TilePlan(ctypes.Structure):
    _fields_ = [
        ("op", ctypes.c_int), ("rows", ctypes.c_int), ("width", ctypes.c_int),
        ("id", ctypes.c_int), ("path", ctypes.c_int), ("vec", ctypes.c_int),
        ("warps_per_program", ctypes.c_int), ("programs_per_cta", ctypes.c_int),
        ("chunks", ctypes.c_int), ("cluster", ctypes.c_int), ("threads", ctypes.c_int),
        ("workers", ctypes.c_int), ("stripe_floats", ctypes.c_int),
        ("max_width", ctypes.c_int), ("smem_bytes", ctypes.c_int),
        ("barriers_per_row", ctypes.c_int), ("grid", ctypes.c_longlong),
        ("dtype", ctypes.c_int),
    ]

    def as_dict(self):
        return {name: getattr(self, name) for name, _ in self._fields_}


class TileRowArgs(ctypes.Structure):
    _fields_ = [
        ("in_", ctypes.c_void_p), ("residual", ctypes.c_void_p), ("gamma", ctypes.c_void_p),
        ("beta", ctypes.c_void_p), ("out", ctypes.c_void_p), ("out2", ctypes.c_void_p),
        ("rows", ctypes.c_int), ("width", ctypes.c_int), ("eps", ctypes.c_float),
        ("dtype", ctypes.c_int),
    ]


_lib = None


def library_path() -> str:
    return LIBRARY


def load():
    """Load the shared library (raises if it has not been built)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIBRARY):
        raise RuntimeError(
            f"{LIBRARY} is not built: run `python -c 'import __graft_entry__ as g; g.build()'` "
            "(the library has no CPU fallback)")
    lib = ctypes.CDLL(LIBRARY)
    P, I, F = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
    sigs = {
        "tile_residual_layernorm_f32": [P, P, P, I, I, F, P],
        "tile_layernorm_f32": [P, P, I, I, F, P],
        "tile_rmsnorm_f32": [P, P, I, I, F, P],
        "tile_softmax_f32": [P, P, I, I, F, P],
        "tile_run_plan_f32": [I, I, P, P, P, I, I, F, P],
        "tile_describe_plan": [I, I, I, ctypes.POINTER(TilePlan)],
        "tile_plan_info": [I, I, I, I, ctypes.POINTER(TilePlan)],
        "tile_plan_count": [],
        "tile_max_width": [],
        "tile_check_device_status": [P],
        "tile_last_cuda_error": [],
        "tile_run_host_f32": [I, P, P, P, I, I, F, P, ctypes.c_size_t, P],
        "tile_host_schedule": [I, I, I, ctypes.c_size_t, I, ctypes.POINTER(ctypes.c_int),
                               ctypes.POINTER(ctypes.c_int)],
        "tile_run_host_static_f32": [I, P, P, P, I, I, F, P],
        "tile_layernorm_affine_f32": [P, P, P, P, P, I, I, F, P],
        "tile_rmsnorm_weighted_f32": [P, P, P, I, I, F, P],
        "tile_row_sum_f32": [P, P, I, I, P],
        "tile_row_minmax_f32": [P, P, P, I, I, P],
        "tile_run_plan_args_f32": [I, I, ctypes.POINTER(TileRowArgs), P],
        "tile_sigmoid_pair_f32": [P, P, P, ctypes.c_longlong, P],
        "tile_gelu_tanh_pair_f32": [P, P, P, ctypes.c_longlong, P],
        "tile_residual_layernorm_bf16": [P, P, P, I, I, F, P],
        "tile_layernorm_bf16": [P, P, I, I, F, P],
        "tile_rmsnorm_bf16": [P, P, I, I, F, P],
        "tile_softmax_bf16": [P, P, I, I, F, P],
        "tile_layernorm_affine_bf16": [P, P, P, P, P, I, I, F, P],
        "tile_rmsnorm_weighted_bf16": [P, P, P, I, I, F, P],
        "tile_row_sum_bf16": [P, P, I, I, P],
        "tile_row_minmax_bf16": [P, P, P, I, I, P],
        "tile_residual_layernorm_f16": [P, P, P, I, I, F, P],
        "tile_layernorm_f16": [P, P, I, I, F, P],
        "tile_rmsnorm_f16": [P, P, I, I, F, P],
        "tile_softmax_f16": [P, P, I, I, F, P],
        "tile_layernorm_affine_f16": [P, P, P, P, P, I, I, F, P],
        "tile_rmsnorm_weighted_f16": [P, P, P, I, I, F, P],
        "tile_row_sum_f16": [P, P, I, I, P],
        "tile_row_minmax_f16": [P, P, P, I, I, P],
        "tile_describe_plan_ex": [I, I, I, I, ctypes.POINTER(TilePlan)],
        "tile_layernorm_backward_f32": [P, P, P, P, P, I, I, F, P],
        "tile_rmsnorm_backward_f32": [P, P, P, P, P, I, I, F, P],
        "tile_softmax_backward_f32": [P, P, P, I, I, P],
        "tile_run_backward_plan_f32": [I, I, P, P, P, P, P, I, I, F, P],
        "tile_norm_param_grad_f32": [P, P, P, P, P, I, I, P, ctypes.c_size_t, P],
        "tile_run_backward_plan_ex": [I, I, I, P, P, P, P, P, I, I, F, P],
        "tile_layernorm_backward_bf16": [P, P, P, P, P, I, I, F, P],
        "tile_rmsnorm_backward_bf16": [P, P, P, P, P, I, I, F, P],
        "tile_softmax_backward_bf16": [P, P, P, I, I, P],
        "tile_norm_param_grad_bf16": [P, P, P, P, P, I, I, P, ctypes.c_size_t, P],
        "tile_layernorm_backward_f16": [P, P, P, P, P, I, I, F, P],
        "tile_rmsnorm_backward_f16": [P, P, P, P, P, I, I, F, P],
        "tile_softmax_backward_f16": [P, P, P, I, I, P],
        "tile_norm_param_grad_f16": [P, P, P, P, P, I, I, P, ctypes.c_size_t, P],
        "tile_plan_info_ex": [I, I, I, I, I, ctypes.POINTER(TilePlan)],
        "tile_test_staged_wait_timeout": [I, I, ctypes.POINTER(TileRowArgs), ctypes.c_uint, P],
        "tile_inject_launch_failure": [I, I, I],
        "tile_test_force_general_kernels": [I],
        "tile_describe_backward_plan": [I, I, I, I, ctypes.POINTER(TilePlan)],
    }
    for name, argtypes in sigs.items():
        fn = getattr(lib, name)
        fn.argtypes = argtypes
        fn.restype = ctypes.c_int
    lib.tile_norm_param_grad_workspace_bytes.argtypes = [I, I]
    lib.tile_norm_param_grad_workspace_bytes.restype = ctypes.c_size_t
    lib.tile_host_workspace_bytes.argtypes = [I, I, I]
    lib.tile_host_workspace_bytes.restype = ctypes.c_size_t
    lib.tile_status_string.argtypes = [I]
    lib.tile_status_string.restype = ctypes.c_char_p
    _lib = lib
    return lib


# ---------------------------------------------------------------------------
# marshalling helpers
# ---------------------------------------------------------------------------

def _stream(stream):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _matrix(t, name, dtype="f32"):
    """(pointer, rows, width) of a CUDA row-major matrix tensor of ``dtype``."""
    import torch
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor (there is no CPU path)")
    want = {"f32": torch.float32, "bf16": torch.bfloat16, "f16": torch.float16}[dtype]
    if t.dtype != want:
        raise ValueError(f"{name} must be {want}")
    if t.dim() != 2:
        raise ValueError(f"{name} must be 2-D [rows, width]")
    rows, width = t.shape
    if rows > 1 and t.stride(0) != width or width > 1 and t.stride(1) != 1:
        raise ValueError(f"{name} must be row-major with row stride == width")
    return t.data_ptr(), rows, width


def _check(status, where):
    if status != TILE_OK:
        raise TileError(status, where)


def _same_shape(a, b, names):
    if tuple(a.shape) != tuple(b.shape):
        raise ValueError(f"{names}: shapes {tuple(a.shape)} and {tuple(b.shape)} differ")


# ---------------------------------------------------------------------------
# the C ABI, one Python function per entry point
# ---------------------------------------------------------------------------

def tile_residual_layernorm_f32(x, residual, out, eps=1e-5, stream=None):
    px, rows, width = _matrix(x, "x")
    pr, _, _ = _matrix(residual, "residual")
    po, _, _ = _matrix(out, "out")
    _same_shape(x, residual, "x/residual")
    _same_shape(x, out, "x/out")
    _check(load().tile_residual_layernorm_f32(px, pr, po, rows, width, eps, _stream(stream)),
           "tile_residual_layernorm_f32")


def _unary(name):
    def fn(x, out, eps=1e-5, stream=None):
        px, rows, width = _matrix(x, "x")
        po, _, _ = _matrix(out, "out")
        _same_shape(x, out, "x/out")
        _check(getattr(load(), name)(px, po, rows, width, eps, _stream(stream)), name)
    fn.__name__ = name
    fn.__doc__ = f"Calls ``{name}`` (see include/tile_rows.h)."
    return fn


tile_layernorm_f32 = _unary("tile_layernorm_f32")
tile_rmsnorm_f32 = _unary("tile_rmsnorm_f32")
tile_softmax_f32 = _unary("tile_softmax_f32")


def tile_run_plan_f32(op, plan_id, x, residual, out, eps=1e-5, stream=None):
    op = OPS[op] if isinstance(op, str) else op
    px, rows, width = _matrix(x, "x")
    po, _, _ = _matrix(out, "out")
    _same_shape(x, out, "x/out")
    pr = None
    if residual is not None:
        pr, _, _ = _matrix(residual, "residual")
        _same_shape(x, residual, "x/residual")
    _check(load().tile_run_plan_f32(op, plan_id, px, pr, po, rows, width, eps, _stream(stream)),
           "tile_run_plan_f32")


def _vector(t, n, name):
    """Pointer of a CUDA FP32 contiguous tensor of n elements (None -> NULL)."""
    import torch
    if t is None:
        return None
    if not isinstance(t, torch.Tensor) or not t.is_cuda or t.dtype != torch.float32:
        raise ValueError(f"{name} must be a CUDA float32 tensor")
    if not t.is_contiguous() or t.numel() != n:
        raise ValueError(f"{name} must be contiguous with {n} elements")
    return t.data_ptr()


def tile_layernorm_affine_f32(x, residual, gamma, beta, out, eps=1e-5, stream=None):
    """LayerNorm(x [+ residual]) * gamma + beta; residual and beta may be None."""
    px, rows, width = _matrix(x, "x")
    po, _, _ = _matrix(out, "out")
    _same_shape(x, out, "x/out")
    pr = None
    if residual is not None:
        pr, _, _ = _matrix(residual, "residual")
        _same_shape(x, residual, "x/residual")
    pg = _vector(gamma, width, "gamma")
    pb = _vector(beta, width, "beta")
    _check(load().tile_layernorm_affine_f32(px, pr, pg, pb, po, rows, width, eps, _stream(stream)),
           "tile_layernorm_affine_f32")


def tile_rmsnorm_weighted_f32(x, gamma, out, eps=1e-5, stream=None):
    px, rows, width = _matrix(x, "x")
    po, _, _ = _matrix(out, "out")
    _same_shape(x, out, "x/out")
    pg = _vector(gamma, width, "gamma")
    _check(load().tile_rmsnorm_weighted_f32(px, pg, po, rows, width, eps, _stream(stream)),
           "tile_rmsnorm_weighted_f32")


def tile_row_sum_f32(x, sums, stream=None):
    px, rows, width = _matrix(x, "x")
    ps = _vector(sums, rows, "sums")
    _check(load().tile_row_sum_f32(px, ps, rows, width, _stream(stream)), "tile_row_sum_f32")


def tile_row_minmax_f32(x, mins, maxs, stream=None):
    px, rows, width = _matrix(x, "x")
    pmn = _vector(mins, rows, "mins")
    pmx = _vector(maxs, rows, "maxs")
    _check(load().tile_row_minmax_f32(px, pmn, pmx, rows, width, _stream(stream)),
           "tile_row_minmax_f32")


def _row_args(x, out, residual, gamma, beta, out2, eps):
    import torch
    dt = {torch.bfloat16: "bf16", torch.float16: "f16"}.get(
        x.dtype if isinstance(x, torch.Tensor) else None, "f32")
    px, rows, width = _matrix(x, "x", dt)
    a = TileRowArgs()
    a.in_ = px
    a.dtype = DTYPES[dt]
    a.residual = _matrix(residual, "residual", dt)[0] if residual is not None else None
    a.gamma = _vector(gamma, width, "gamma")
    a.beta = _vector(beta, width, "beta")
    a.out = out.data_ptr()
    a.out2 = out2.data_ptr() if out2 is not None else None
    a.rows, a.width, a.eps = rows, width, eps
    return a


def tile_run_plan_args_f32(op, plan_id, x, out, residual=None, gamma=None, beta=None, out2=None,
                           eps=1e-5, stream=None):
    """Any row op with a forced plan (``out``: matrix, or [rows] for row_sum/row_minmax).
    ``x`` may be float32, bfloat16 or float16; the element type follows it."""
    op = OPS[op] if isinstance(op, str) else op
    a = _row_args(x, out, residual, gamma, beta, out2, eps)
    _check(load().tile_run_plan_args_f32(op, plan_id, ctypes.byref(a), _stream(stream)),
           "tile_run_plan_args_f32")


def tile_inject_launch_failure(cuda_error, skip=0, count=1):
    """Test hook: after ``skip`` launch attempts, the next ``count`` fail on
    the host with ``cuda_error`` (``count=0`` disarms)."""
    _check(load().tile_inject_launch_failure(int(cuda_error), int(skip), int(count)),
           "tile_inject_launch_failure")


def tile_test_force_general_kernels(on):
    """Test hook: with ``on`` true, 2-byte launches take the general kernel
    forms instead of the whole-vector ones (bitwise the same results)."""
    _check(load().tile_test_force_general_kernels(int(bool(on))),
           "tile_test_force_general_kernels")


def tile_test_staged_wait_timeout(op, plan_id, x, out, spin_limit, residual=None, gamma=None,
                                  beta=None, eps=1e-5, stream=None):
    """Test hook: the staged plan with every CTA's first copy withheld and
    waits limited to ``spin_limit`` polls (the outputs are invalid; the
    device status word reports the timeout)."""
    op = OPS[op] if isinstance(op, str) else op
    a = _row_args(x, out, residual, gamma, beta, None, eps)
    _check(load().tile_test_staged_wait_timeout(op, plan_id, ctypes.byref(a), int(spin_limit),
                                                _stream(stream)),
           "tile_test_staged_wait_timeout")


def _flat(t, name):
    import torch
    if not isinstance(t, torch.Tensor) or not t.is_cuda or t.dtype != torch.float32:
        raise ValueError(f"{name} must be a CUDA float32 tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return t.data_ptr(), t.numel()


def _pair_fn(name):
    def fn(x, value, derivative, stream=None):
        px, n = _flat(x, "x")
        pv, nv = _flat(value, "value")
        pd, nd = _flat(derivative, "derivative")
        if nv != n or nd != n:
            raise ValueError("value and derivative must have as many elements as x")
        _check(getattr(load(), name)(px, pv, pd, n, _stream(stream)), name)
    fn.__name__ = name
    fn.__doc__ = f"Calls ``{name}`` (see include/tile_rows.h)."
    return fn


tile_sigmoid_pair_f32 = _pair_fn("tile_sigmoid_pair_f32")
tile_gelu_tanh_pair_f32 = _pair_fn("tile_gelu_tanh_pair_f32")


# ---- backward passes ----------------------------------------------------------

def _bwd(name, dtype="f32"):
    def fn(x, gamma, dy, dx, row_stats=None, eps=1e-5, stream=None):
        px, rows, width = _matrix(x, "x", dtype)
        pd, _, _ = _matrix(dy, "dy", dtype)
        po, _, _ = _matrix(dx, "dx", dtype)
        _same_shape(x, dy, "x/dy")
        _same_shape(x, dx, "x/dx")
        ps = _vector(row_stats, 2 * rows, "row_stats") if row_stats is not None else None
        _check(getattr(load(), name)(px, _vector(gamma, width, "gamma"), pd, po, ps, rows, width,
                                     eps, _stream(stream)), name)
    fn.__name__ = name
    fn.__doc__ = f"Calls ``{name}`` (see include/tile_rows.h)."
    return fn


tile_layernorm_backward_f32 = _bwd("tile_layernorm_backward_f32")
tile_rmsnorm_backward_f32 = _bwd("tile_rmsnorm_backward_f32")


def tile_softmax_backward_f32(y, dy, dx, stream=None):
    py, rows, width = _matrix(y, "y")
    pd, _, _ = _matrix(dy, "dy")
    po, _, _ = _matrix(dx, "dx")
    _same_shape(y, dy, "y/dy")
    _same_shape(y, dx, "y/dx")
    _check(load().tile_softmax_backward_f32(py, pd, po, rows, width, _stream(stream)),
           "tile_softmax_backward_f32")


def tile_run_backward_plan_f32(op, plan_id, x, gamma, dy, dx, row_stats=None, eps=1e-5,
                               stream=None):
    op = OPS[op] if isinstance(op, str) else op
    px, rows, width = _matrix(x, "x")
    pd, _, _ = _matrix(dy, "dy")
    po, _, _ = _matrix(dx, "dx")
    ps = _vector(row_stats, 2 * rows, "row_stats") if row_stats is not None else None
    _check(load().tile_run_backward_plan_f32(op, plan_id, px, _vector(gamma, width, "gamma"), pd,
                                             po, ps, rows, width, eps, _stream(stream)),
           "tile_run_backward_plan_f32")


def _softmax_bwd(name, dtype):
    def fn(y, dy, dx, stream=None):
        py, rows, width = _matrix(y, "y", dtype)
        pd, _, _ = _matrix(dy, "dy", dtype)
        po, _, _ = _matrix(dx, "dx", dtype)
        _same_shape(y, dy, "y/dy")
        _same_shape(y, dx, "y/dx")
        _check(getattr(load(), name)(py, pd, po, rows, width, _stream(stream)), name)
    fn.__name__ = name
    fn.__doc__ = f"Calls ``{name}`` (see include/tile_rows.h)."
    return fn


def _param_grad(name, dtype):
    def fn(x, dy, row_stats, dgamma, dbeta, workspace, stream=None):
        px, rows, width = _matrix(x, "x", dtype)
        pd, _, _ = _matrix(dy, "dy", dtype)
        if not workspace.is_cuda:
            raise ValueError("workspace must be a CUDA tensor")
        _check(getattr(load(), name)(
            px, pd, _vector(row_stats, 2 * rows, "row_stats"), _vector(dgamma, width, "dgamma"),
            _vector(dbeta, width, "dbeta"), rows, width, workspace.data_ptr(),
            workspace.numel() * workspace.element_size(), _stream(stream)), name)
    fn.__name__ = name
    fn.__doc__ = f"Calls ``{name}`` (see include/tile_rows.h)."
    return fn


tile_layernorm_backward_bf16 = _bwd("tile_layernorm_backward_bf16", "bf16")
tile_rmsnorm_backward_bf16 = _bwd("tile_rmsnorm_backward_bf16", "bf16")
tile_softmax_backward_bf16 = _softmax_bwd("tile_softmax_backward_bf16", "bf16")
tile_norm_param_grad_bf16 = _param_grad("tile_norm_param_grad_bf16", "bf16")
tile_layernorm_backward_f16 = _bwd("tile_layernorm_backward_f16", "f16")
tile_rmsnorm_backward_f16 = _bwd("tile_rmsnorm_backward_f16", "f16")
tile_softmax_backward_f16 = _softmax_bwd("tile_softmax_backward_f16", "f16")
tile_norm_param_grad_f16 = _param_grad("tile_norm_param_grad_f16", "f16")


def tile_run_backward_plan_ex(op, plan_id, x, gamma, dy, dx, row_stats=None, eps=1e-5,
                              stream=None):
    """tile_run_backward_plan_f32 for the element type of ``x`` (float32,
    bfloat16 or float16)."""
    import torch
    op = OPS[op] if isinstance(op, str) else op
    dt = {torch.bfloat16: "bf16", torch.float16: "f16"}.get(x.dtype, "f32")
    px, rows, width = _matrix(x, "x", dt)
    pd, _, _ = _matrix(dy, "dy", dt)
    po, _, _ = _matrix(dx, "dx", dt)
    ps = _vector(row_stats, 2 * rows, "row_stats") if row_stats is not None else None
    _check(load().tile_run_backward_plan_ex(op, plan_id, DTYPES[dt], px,
                                            _vector(gamma, width, "gamma"), pd, po, ps, rows,
                                            width, eps, _stream(stream)),
           "tile_run_backward_plan_ex")


def tile_norm_param_grad_workspace_bytes(rows, width):
    return load().tile_norm_param_grad_workspace_bytes(rows, width)


def tile_norm_param_grad_f32(x, dy, row_stats, dgamma, dbeta, workspace, stream=None):
    px, rows, width = _matrix(x, "x")
    pd, _, _ = _matrix(dy, "dy")
    if not workspace.is_cuda:
        raise ValueError("workspace must be a CUDA tensor")
    _check(load().tile_norm_param_grad_f32(
        px, pd, _vector(row_stats, 2 * rows, "row_stats"), _vector(dgamma, width, "dgamma"),
        _vector(dbeta, width, "dbeta"), rows, width, workspace.data_ptr(),
        workspace.numel() * workspace.element_size(), _stream(stream)), "tile_norm_param_grad_f32")


# ---- BF16 rows ---------------------------------------------------------------

def tile_residual_layernorm_bf16(x, residual, out, eps=1e-5, stream=None):
    px, rows, width = _matrix(x, "x", "bf16")
    pr, _, _ = _matrix(residual, "residual", "bf16")
    po, _, _ = _matrix(out, "out", "bf16")
    _same_shape(x, residual, "x/residual")
    _same_shape(x, out, "x/out")
    _check(load().tile_residual_layernorm_bf16(px, pr, po, rows, width, eps, _stream(stream)),
           "tile_residual_layernorm_bf16")


def _unary_bf16(name):
    def fn(x, out, eps=1e-5, stream=None):
        px, rows, width = _matrix(x, "x", "bf16")
        po, _, _ = _matrix(out, "out", "bf16")
        _same_shape(x, out, "x/out")
        _check(getattr(load(), name)(px, po, rows, width, eps, _stream(stream)), name)
    fn.__name__ = name
    fn.__doc__ = f"Calls ``{name}`` (see include/tile_rows.h)."
    return fn


tile_layernorm_bf16 = _unary_bf16("tile_layernorm_bf16")
tile_rmsnorm_bf16 = _unary_bf16("tile_rmsnorm_bf16")
tile_softmax_bf16 = _unary_bf16("tile_softmax_bf16")


def tile_layernorm_affine_bf16(x, residual, gamma, beta, out, eps=1e-5, stream=None):
    px, rows, width = _matrix(x, "x", "bf16")
    po, _, _ = _matrix(out, "out", "bf16")
    _same_shape(x, out, "x/out")
    pr = None
    if residual is not None:
        pr, _, _ = _matrix(residual, "residual", "bf16")
        _same_shape(x, residual, "x/residual")
    _check(load().tile_layernorm_affine_bf16(px, pr, _vector(gamma, width, "gamma"),
                                             _vector(beta, width, "beta"), po, rows, width, eps,
                                             _stream(stream)), "tile_layernorm_affine_bf16")


def tile_rmsnorm_weighted_bf16(x, gamma, out, eps=1e-5, stream=None):
    px, rows, width = _matrix(x, "x", "bf16")
    po, _, _ = _matrix(out, "out", "bf16")
    _same_shape(x, out, "x/out")
    _check(load().tile_rmsnorm_weighted_bf16(px, _vector(gamma, width, "gamma"), po, rows, width,
                                             eps, _stream(stream)), "tile_rmsnorm_weighted_bf16")


def tile_row_sum_bf16(x, sums, stream=None):
    px, rows, width = _matrix(x, "x", "bf16")
    _check(load().tile_row_sum_bf16(px, _vector(sums, rows, "sums"), rows, width, _stream(stream)),
           "tile_row_sum_bf16")


def tile_row_minmax_bf16(x, mins, maxs, stream=None):
    px, rows, width = _matrix(x, "x", "bf16")
    _check(load().tile_row_minmax_bf16(px, _vector(mins, rows, "mins"), _vector(maxs, rows, "maxs"),
                                       rows, width, _stream(stream)), "tile_row_minmax_bf16")


def tile_residual_layernorm_f16(x, residual, out, eps=1e-5, stream=None):
    px, rows, width = _matrix(x, "x", "f16")
    pr, _, _ = _matrix(residual, "residual", "f16")
    po, _, _ = _matrix(out, "out", "f16")
    _same_shape(x, residual, "x/residual")
    _same_shape(x, out, "x/out")
    _check(load().tile_residual_layernorm_f16(px, pr, po, rows, width, eps, _stream(stream)),
           "tile_residual_layernorm_f16")


def _unary_f16(name):
    def fn(x, out, eps=1e-5, stream=None):
        px, rows, width = _matrix(x, "x", "f16")
        po, _, _ = _matrix(out, "out", "f16")
        _same_shape(x, out, "x/out")
        _check(getattr(load(), name)(px, po, rows, width, eps, _stream(stream)), name)
    fn.__name__ = name
    fn.__doc__ = f"Calls ``{name}`` (see include/tile_rows.h)."
    return fn


tile_layernorm_f16 = _unary_f16("tile_layernorm_f16")
tile_rmsnorm_f16 = _unary_f16("tile_rmsnorm_f16")
tile_softmax_f16 = _unary_f16("tile_softmax_f16")


def tile_layernorm_affine_f16(x, residual, gamma, beta, out, eps=1e-5, stream=None):
    px, rows, width = _matrix(x, "x", "f16")
    po, _, _ = _matrix(out, "out", "f16")
    _same_shape(x, out, "x/out")
    pr = None
    if residual is not None:
        pr, _, _ = _matrix(residual, "residual", "f16")
        _same_shape(x, residual, "x/residual")
    _check(load().tile_layernorm_affine_f16(px, pr, _vector(gamma, width, "gamma"),
                                             _vector(beta, width, "beta"), po, rows, width, eps,
                                             _stream(stream)), "tile_layernorm_affine_f16")


def tile_rmsnorm_weighted_f16(x, gamma, out, eps=1e-5, stream=None):
    px, rows, width = _matrix(x, "x", "f16")
    po, _, _ = _matrix(out, "out", "f16")
    _same_shape(x, out, "x/out")
    _check(load().tile_rmsnorm_weighted_f16(px, _vector(gamma, width, "gamma"), po, rows, width,
                                             eps, _stream(stream)), "tile_rmsnorm_weighted_f16")


def tile_row_sum_f16(x, sums, stream=None):
    px, rows, width = _matrix(x, "x", "f16")
    _check(load().tile_row_sum_f16(px, _vector(sums, rows, "sums"), rows, width, _stream(stream)),
           "tile_row_sum_f16")


def tile_row_minmax_f16(x, mins, maxs, stream=None):
    px, rows, width = _matrix(x, "x", "f16")
    _check(load().tile_row_minmax_f16(px, _vector(mins, rows, "mins"), _vector(maxs, rows, "maxs"),
                                       rows, width, _stream(stream)), "tile_row_minmax_f16")


def _host_matrix(t, name):
    """(pointer, rows, width) of a CPU FP32 row-major matrix tensor."""
    import torch
    if not isinstance(t, torch.Tensor) or t.is_cuda:
        raise ValueError(f"{name} must be a CPU tensor (ideally pinned)")
    if t.dtype != torch.float32 or t.dim() != 2:
        raise ValueError(f"{name} must be a 2-D float32 tensor")
    rows, width = t.shape
    if rows > 1 and t.stride(0) != width or width > 1 and t.stride(1) != 1:
        raise ValueError(f"{name} must be row-major with row stride == width")
    return t.data_ptr(), rows, width


def tile_run_host_f32(op, x, residual, out, workspace, eps=1e-5, stream=None):
    """``op`` on host tensors: in place when every tensor is pinned (one kernel
    reads and writes them over the host link), otherwise through the device
    ``workspace`` (a CUDA tensor) in chunks."""
    op = OPS[op] if isinstance(op, str) else op
    px, rows, width = _host_matrix(x, "x")
    po, _, _ = _host_matrix(out, "out")
    _same_shape(x, out, "x/out")
    pr = None
    if residual is not None:
        pr, _, _ = _host_matrix(residual, "residual")
        _same_shape(x, residual, "x/residual")
    if not workspace.is_cuda:
        raise ValueError("workspace must be a CUDA tensor")
    nbytes = workspace.numel() * workspace.element_size()
    _check(load().tile_run_host_f32(op, px, pr, po, rows, width, eps, workspace.data_ptr(),
                                    nbytes, _stream(stream)), "tile_run_host_f32")


def tile_run_host_static_f32(op, x, residual, out, eps=1e-5, stream=None):
    """``op`` on host tensors through the library's static device staging
    area: for callers that cannot allocate device memory."""
    op = OPS[op] if isinstance(op, str) else op
    px, rows, width = _host_matrix(x, "x")
    po, _, _ = _host_matrix(out, "out")
    _same_shape(x, out, "x/out")
    pr = None
    if residual is not None:
        pr, _, _ = _host_matrix(residual, "residual")
        _same_shape(x, residual, "x/residual")
    _check(load().tile_run_host_static_f32(op, px, pr, po, rows, width, eps, _stream(stream)),
           "tile_run_host_static_f32")


def tile_host_workspace_bytes(op, width, chunk_rows):
    op = OPS[op] if isinstance(op, str) else op
    return load().tile_host_workspace_bytes(op, width, chunk_rows)


def tile_host_schedule(op, rows, width, work_bytes, direct_output=True):
    """(chunk rows, ring slots) that tile_run_host_f32 uses for these
    arguments; `direct_output` describes a pinned output buffer."""
    op = OPS[op] if isinstance(op, str) else op
    chunk, slots = ctypes.c_int(0), ctypes.c_int(0)
    _check(load().tile_host_schedule(op, rows, width, work_bytes, int(bool(direct_output)),
                                     ctypes.byref(chunk), ctypes.byref(slots)),
           "tile_host_schedule")
    return chunk.value, slots.value


def tile_describe_plan(op, rows, width):
    op = OPS[op] if isinstance(op, str) else op
    plan = TilePlan()
    _check(load().tile_describe_plan(op, rows, width, ctypes.byref(plan)), "tile_describe_plan")
    return plan.as_dict()


def tile_describe_plan_ex(op, dtype, rows, width):
    op = OPS[op] if isinstance(op, str) else op
    dtype = DTYPES[dtype] if isinstance(dtype, str) else dtype
    plan = TilePlan()
    _check(load().tile_describe_plan_ex(op, dtype, rows, width, ctypes.byref(plan)),
           "tile_describe_plan_ex")
    return plan.as_dict()


def tile_describe_backward_plan(op, dtype, rows, width):
    """The plan the backward entry points launch for (op, dtype, rows, width)
    on 16-byte co-aligned tensors."""
    op = OPS[op] if isinstance(op, str) else op
    dtype = DTYPES[dtype] if isinstance(dtype, str) else dtype
    plan = TilePlan()
    _check(load().tile_describe_backward_plan(op, dtype, rows, width, ctypes.byref(plan)),
           "tile_describe_backward_plan")
    return plan.as_dict()


def tile_plan_info_ex(plan_id, op, dtype, rows, width):
    """Plan ``plan_id`` for (op, dtype, rows, width), or None if not built, not
    covering, or without a variant for ``op``."""
    op = OPS[op] if isinstance(op, str) else op
    dtype = DTYPES[dtype] if isinstance(dtype, str) else dtype
    plan = TilePlan()
    st = load().tile_plan_info_ex(plan_id, op, dtype, rows, width, ctypes.byref(plan))
    if st in (-2, -8):
        return None
    _check(st, "tile_plan_info_ex")
    return plan.as_dict()


def tile_plan_info(plan_id, op, rows, width):
    """The built plan ``plan_id`` for (op, rows, width), or None if it cannot
    cover ``width`` or has no variant for ``op``."""
    op = OPS[op] if isinstance(op, str) else op
    plan = TilePlan()
    st = load().tile_plan_info(plan_id, op, rows, width, ctypes.byref(plan))
    if st in (-2, -8):
        return None
    _check(st, "tile_plan_info")
    return plan.as_dict()


def tile_plan_count():
    return load().tile_plan_count()


def tile_max_width():
    return load().tile_max_width()


def tile_status_string(status):
    return load().tile_status_string(status).decode()


def tile_check_device_status(stream=None):
    return load().tile_check_device_status(_stream(stream))


def tile_last_cuda_error():
    return load().tile_last_cuda_error()


# ---------------------------------------------------------------------------
# convenience wrappers (allocate the output with torch when not given)
# ---------------------------------------------------------------------------

def residual_layernorm(x, residual, out=None, eps=1e-5, stream=None):
    import torch
    out = torch.empty_like(x) if out is None else out
    tile_residual_layernorm_f32(x, residual, out, eps, stream)
    return out


def layernorm(x, out=None, eps=1e-5, stream=None):
    import torch
    out = torch.empty_like(x) if out is None else out
    tile_layernorm_f32(x, out, eps, stream)
    return out


def rmsnorm(x, out=None, eps=1e-5, stream=None):
    import torch
    out = torch.empty_like(x) if out is None else out
    tile_rmsnorm_f32(x, out, eps, stream)
    return out


def softmax(x, out=None, stream=None):
    import torch
    out = torch.empty_like(x) if out is None else out
    tile_softmax_f32(x, out, 0.0, stream)
    return out


def run(op, x, residual=None, out=None, eps=1e-5, stream=None):
    """Dispatch by op name."""
    if op == "residual_layernorm":
        return residual_layernorm(x, residual, out, eps, stream)
    if op == "softmax":
        return softmax(x, out, stream)
    return {"layernorm": layernorm, "rmsnorm": rmsnorm}[op](x, out, eps, stream)
