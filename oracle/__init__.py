"""FP64 CPU oracle for the row-normalisation kernels (ctypes over ``oracle.c``).

TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the benchmark's
CPU-baseline / reference leg import this package.  The CUDA library never
imports, links or calls it, and there is no CPU fallback anywhere in the
product path.

The C source (``oracle.c``) is the authority; this module only compiles it
with gcc, loads it and marshals numpy arrays.  Every function takes the exact
FP32 inputs given to the GPU and returns FP64 outputs.
"""

from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
SOURCE = os.path.join(HERE, "oracle.c")
LIBRARY = os.path.join(HERE, "liboracle.so")

#: gcc flags: IEEE FP64, no FMA contraction, so x86 and Arm agree bit for bit.
CFLAGS = ["-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared"]

_lock = threading.Lock()
_default = None


def build(source: str = SOURCE, output: str = LIBRARY, force: bool = False) -> str:
    """Compile ``source`` into the shared library ``output`` (if stale)."""
    if (not force and os.path.exists(output)
            and os.path.getmtime(output) >= os.path.getmtime(source)):
        return output
    tmp = output + f".tmp{os.getpid()}"
    subprocess.run(["gcc", *CFLAGS, "-o", tmp, source, "-lm"], check=True)
    os.replace(tmp, output)
    return output


class Oracle:
    """One loaded copy of the oracle library."""

    def __init__(self, path: str):
        self.path = path
        lib = ctypes.CDLL(path)
        f32p = ctypes.POINTER(ctypes.c_float)
        f64p = ctypes.POINTER(ctypes.c_double)
        L, D = ctypes.c_long, ctypes.c_double
        lib.oracle_residual_layernorm.argtypes = [f32p, f32p, f64p, L, L, D]
        lib.oracle_layernorm.argtypes = [f32p, f64p, L, L, D]
        lib.oracle_rmsnorm.argtypes = [f32p, f64p, L, L, D]
        lib.oracle_softmax.argtypes = [f32p, f64p, L, L]
        lib.oracle_layernorm_affine.argtypes = [f32p, f32p, f32p, f32p, f64p, L, L, D]
        lib.oracle_rmsnorm_weighted.argtypes = [f32p, f32p, f64p, L, L, D]
        lib.oracle_row_sum.argtypes = [f32p, f64p, L, L]
        lib.oracle_row_minmax.argtypes = [f32p, f64p, f64p, L, L]
        lib.oracle_sigmoid_pair.argtypes = [f32p, f64p, f64p, L]
        lib.oracle_gelu_tanh_pair.argtypes = [f32p, f64p, f64p, L]
        lib.oracle_layernorm_backward.argtypes = [f32p, f32p, f32p, f64p, L, L, D]
        lib.oracle_rmsnorm_backward.argtypes = [f32p, f32p, f32p, f64p, L, L, D]
        lib.oracle_softmax_backward.argtypes = [f32p, f32p, f64p, L, L]
        lib.oracle_norm_param_grad.argtypes = [f32p, f32p, f64p, f64p, L, L, D, ctypes.c_int]
        for fn in (lib.oracle_layernorm_backward, lib.oracle_rmsnorm_backward,
                   lib.oracle_softmax_backward, lib.oracle_norm_param_grad):
            fn.restype = None
        for fn in (lib.oracle_residual_layernorm, lib.oracle_layernorm,
                   lib.oracle_rmsnorm, lib.oracle_softmax, lib.oracle_layernorm_affine,
                   lib.oracle_rmsnorm_weighted, lib.oracle_row_sum, lib.oracle_row_minmax,
                   lib.oracle_sigmoid_pair, lib.oracle_gelu_tanh_pair):
            fn.restype = None
        self._lib = lib

    @staticmethod
    def _f32(a):
        a = np.ascontiguousarray(a, dtype=np.float32)
        if a.ndim != 2:
            raise ValueError("oracle inputs are 2-D [rows, width]")
        return a

    @staticmethod
    def _p(a, ct):
        return a.ctypes.data_as(ctypes.POINTER(ct))

    def residual_layernorm(self, x, r, eps=1e-5):
        x, r = self._f32(x), self._f32(r)
        if x.shape != r.shape:
            raise ValueError("x and residual shapes differ")
        y = np.empty(x.shape, dtype=np.float64)
        if x.size:
            self._lib.oracle_residual_layernorm(
                self._p(x, ctypes.c_float), self._p(r, ctypes.c_float),
                self._p(y, ctypes.c_double), x.shape[0], x.shape[1], float(eps))
        return y

    def layernorm(self, x, eps=1e-5):
        x = self._f32(x)
        y = np.empty(x.shape, dtype=np.float64)
        if x.size:
            self._lib.oracle_layernorm(self._p(x, ctypes.c_float), self._p(y, ctypes.c_double),
                                       x.shape[0], x.shape[1], float(eps))
        return y

    def rmsnorm(self, x, eps=1e-5):
        x = self._f32(x)
        y = np.empty(x.shape, dtype=np.float64)
        if x.size:
            self._lib.oracle_rmsnorm(self._p(x, ctypes.c_float), self._p(y, ctypes.c_double),
                                     x.shape[0], x.shape[1], float(eps))
        return y

    def softmax(self, x, eps=None):
        x = self._f32(x)
        y = np.empty(x.shape, dtype=np.float64)
        if x.size:
            self._lib.oracle_softmax(self._p(x, ctypes.c_float), self._p(y, ctypes.c_double),
                                     x.shape[0], x.shape[1])
        return y

    @staticmethod
    def _vec(a, n, name):
        a = np.ascontiguousarray(a, dtype=np.float32).reshape(-1)
        if a.size != n:
            raise ValueError(f"{name} must have {n} elements")
        return a

    def layernorm_affine(self, x, gamma, beta=None, r=None, eps=1e-5):
        """LayerNorm of x (+ r) times gamma plus beta (r, beta optional)."""
        x = self._f32(x)
        rows, width = x.shape
        g = self._vec(gamma, width, "gamma")
        b = self._vec(beta, width, "beta") if beta is not None else None
        rr = self._f32(r) if r is not None else None
        if rr is not None and rr.shape != x.shape:
            raise ValueError("x and residual shapes differ")
        y = np.empty(x.shape, dtype=np.float64)
        if x.size:
            f32 = ctypes.c_float
            self._lib.oracle_layernorm_affine(
                self._p(x, f32), self._p(rr, f32) if rr is not None else None,
                self._p(g, f32), self._p(b, f32) if b is not None else None,
                self._p(y, ctypes.c_double), rows, width, float(eps))
        return y

    def rmsnorm_weighted(self, x, gamma, eps=1e-5):
        x = self._f32(x)
        rows, width = x.shape
        g = self._vec(gamma, width, "gamma")
        y = np.empty(x.shape, dtype=np.float64)
        if x.size:
            self._lib.oracle_rmsnorm_weighted(self._p(x, ctypes.c_float), self._p(g, ctypes.c_float),
                                              self._p(y, ctypes.c_double), rows, width, float(eps))
        return y

    def row_sum(self, x):
        x = self._f32(x)
        s = np.empty(x.shape[0], dtype=np.float64)
        if x.size:
            self._lib.oracle_row_sum(self._p(x, ctypes.c_float), self._p(s, ctypes.c_double),
                                     x.shape[0], x.shape[1])
        return s

    def row_minmax(self, x):
        x = self._f32(x)
        mn = np.empty(x.shape[0], dtype=np.float64)
        mx = np.empty(x.shape[0], dtype=np.float64)
        if x.size:
            self._lib.oracle_row_minmax(self._p(x, ctypes.c_float), self._p(mn, ctypes.c_double),
                                        self._p(mx, ctypes.c_double), x.shape[0], x.shape[1])
        return mn, mx

    def _pair(self, fn, x):
        x = np.ascontiguousarray(x, dtype=np.float32)
        y = np.empty(x.shape, dtype=np.float64)
        dy = np.empty(x.shape, dtype=np.float64)
        if x.size:
            fn(self._p(x, ctypes.c_float), self._p(y, ctypes.c_double),
               self._p(dy, ctypes.c_double), x.size)
        return y, dy

    def sigmoid_pair(self, x):
        """(sigmoid(x), sigmoid'(x)) elementwise, any shape."""
        return self._pair(self._lib.oracle_sigmoid_pair, x)

    def gelu_tanh_pair(self, x):
        """(tanh-GELU(x), its derivative) elementwise, any shape."""
        return self._pair(self._lib.oracle_gelu_tanh_pair, x)

    def layernorm_backward(self, x, dy, gamma=None, eps=1e-5):
        """dx of LayerNorm(x) * gamma (gamma optional) for upstream gradient dy."""
        return self._backward(self._lib.oracle_layernorm_backward, x, dy, gamma, eps)

    def rmsnorm_backward(self, x, dy, gamma=None, eps=1e-5):
        return self._backward(self._lib.oracle_rmsnorm_backward, x, dy, gamma, eps)

    def _backward(self, fn, x, dy, gamma, eps):
        x, dy = self._f32(x), self._f32(dy)
        if x.shape != dy.shape:
            raise ValueError("x and dy shapes differ")
        g = self._vec(gamma, x.shape[1], "gamma") if gamma is not None else None
        out = np.empty(x.shape, dtype=np.float64)
        if x.size:
            fn(self._p(x, ctypes.c_float), self._p(g, ctypes.c_float) if g is not None else None,
               self._p(dy, ctypes.c_float), self._p(out, ctypes.c_double), x.shape[0], x.shape[1],
               float(eps))
        return out

    def softmax_backward(self, y, dy):
        """dx of softmax given its output y and upstream gradient dy."""
        y, dy = self._f32(y), self._f32(dy)
        if y.shape != dy.shape:
            raise ValueError("y and dy shapes differ")
        out = np.empty(y.shape, dtype=np.float64)
        if y.size:
            self._lib.oracle_softmax_backward(self._p(y, ctypes.c_float), self._p(dy, ctypes.c_float),
                                              self._p(out, ctypes.c_double), y.shape[0], y.shape[1])
        return out

    def norm_param_grad(self, x, dy, eps=1e-5, rms=False):
        """(dgamma, dbeta) summed over rows (dbeta None for RMSNorm)."""
        x, dy = self._f32(x), self._f32(dy)
        width = x.shape[1]
        dg = np.empty(width, dtype=np.float64)
        db = None if rms else np.empty(width, dtype=np.float64)
        self._lib.oracle_norm_param_grad(
            self._p(x, ctypes.c_float), self._p(dy, ctypes.c_float), self._p(dg, ctypes.c_double),
            self._p(db, ctypes.c_double) if db is not None else None, x.shape[0], width,
            float(eps), int(bool(rms)))
        return dg, db

    def run(self, op: str, x, r=None, eps=1e-5):
        """Dispatch by library op name."""
        if op == "residual_layernorm":
            return self.residual_layernorm(x, r, eps)
        return getattr(self, op)(x, eps)


def get() -> Oracle:
    """The oracle built from ``oracle.c`` (compiled on first use)."""
    global _default
    with _lock:
        if _default is None:
            _default = Oracle(build())
        return _default


def kernel_eps(eps: float = 1e-5) -> float:
    """The FP32 value of ``eps`` widened to FP64: what the kernel receives."""
    return float(np.float32(eps))
