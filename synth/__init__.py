"""Seeded synthetic inputs for the row-normalisation workloads.

This module is shared by the tests, the benchmark and the oracle harness.  It
holds no arithmetic of the normalisation method itself: only a counter-based
random number generator and the recipes (shape, distribution, special rows)
of the workloads the kernels are checked and timed on.

Generator: SplitMix64 (G. L. Steele, D. Lea, C. H. Flood, "Fast splittable
pseudorandom number generators", OOPSLA 2014).  Element ``i`` of the stream
with seed ``s`` is the ``i``-th output of the sequential SplitMix64 generator
whose state starts at ``s``:

    z  = s + (i + 1) * 0x9E3779B97F4A7C15          (mod 2**64)
    z  = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9
    z  = (z ^ (z >> 27)) * 0x94D049BB133111EB
    h  = z ^ (z >> 31)

Because every element is a pure function of ``(s, i)``, any slice of rows can
be generated without producing the rows before it.

Value maps:
  * uniform on [-1, 1):  k = h >> 40 (24 bits), x = (k - 2**23) / 2**23,
    which is exact in FP32;
  * normal N(0, sigma**2): Box-Muller in FP64 on the pair (h[2j], h[2j+1]),
    u1 = ((h >> 11) + 1) / 2**53 in (0, 1], u2 = (h >> 11) / 2**53,
    z = sqrt(-2 ln u1) cos(2 pi u2), rounded to FP32 after scaling.
"""

from __future__ import annotations

import concurrent.futures as cf
import os

import numpy as np

GOLDEN_GAMMA = np.uint64(0x9E3779B97F4A7C15)
_MIX1 = np.uint64(0xBF58476D1CE4E5B9)
_MIX2 = np.uint64(0x94D049BB133111EB)

_CHUNK = 1 << 22


def splitmix64(seed: int, start: int, count: int) -> np.ndarray:
    """Outputs ``start .. start+count-1`` of the SplitMix64 stream ``seed``."""
    with np.errstate(over="ignore"):
        idx = np.arange(start + 1, start + count + 1, dtype=np.uint64)
        z = np.uint64(seed & 0xFFFFFFFFFFFFFFFF) + idx * GOLDEN_GAMMA
        z = (z ^ (z >> np.uint64(30))) * _MIX1
        z = (z ^ (z >> np.uint64(27))) * _MIX2
        return z ^ (z >> np.uint64(31))


def _chunked(count: int, fill) -> None:
    """Call ``fill(lo, n)`` over chunks of ``count``; large requests use a
    thread pool (numpy releases the GIL inside these array operations)."""
    spans = [(lo, min(_CHUNK, count - lo)) for lo in range(0, count, _CHUNK)]
    if len(spans) <= 2:
        for lo, n in spans:
            fill(lo, n)
        return
    workers = max(1, min(16, os.cpu_count() or 1))
    with cf.ThreadPoolExecutor(max_workers=workers) as pool:
        list(pool.map(lambda s: fill(*s), spans))


def uniform_pm1(seed: int, count: int, start: int = 0) -> np.ndarray:
    """``count`` FP32 values on [-1, 1), elements ``start..`` of stream ``seed``."""
    out = np.empty(count, dtype=np.float32)

    def fill(lo, n):
        k = (splitmix64(seed, start + lo, n) >> np.uint64(40)).astype(np.int64)
        out[lo:lo + n] = (k - (1 << 23)).astype(np.float32) * np.float32(2.0 ** -23)

    _chunked(count, fill)
    return out


def normal(seed: int, count: int, sigma: float, start: int = 0) -> np.ndarray:
    """``count`` FP32 draws of N(0, sigma**2); element ``j`` uses outputs 2j, 2j+1."""
    out = np.empty(count, dtype=np.float32)

    def fill(lo, n):
        h = splitmix64(seed, 2 * (start + lo), 2 * n)
        u1 = ((h[0::2] >> np.uint64(11)).astype(np.float64) + 1.0) * 2.0 ** -53
        u2 = (h[1::2] >> np.uint64(11)).astype(np.float64) * 2.0 ** -53
        z = np.sqrt(-2.0 * np.log(u1)) * np.cos(2.0 * np.pi * u2)
        out[lo:lo + n] = (sigma * z).astype(np.float32)

    _chunked(count, fill)
    return out


# ---------------------------------------------------------------------------
# Workload recipes
# ---------------------------------------------------------------------------

#: Ops and shapes of the five workloads.  ``ops`` names use the library's
#: operation names.
WORKLOADS = {
    1: dict(name="residual LayerNorm 17x257",
            ops=("residual_layernorm",), shapes=((17, 257),), dist="uniform"),
    2: dict(name="softmax/RMSNorm/LayerNorm 1024x4096",
            ops=("softmax", "rmsnorm", "layernorm"), shapes=((1024, 4096),),
            dist="uniform"),
    3: dict(name="narrow/ragged row-packing sweep",
            ops=("residual_layernorm", "rmsnorm", "softmax"),
            shapes=((1, 127), (7, 1537), (17, 257), (64, 4096)), dist="uniform"),
    4: dict(name="wide rows, N(0,3^2) with a constant row and a +40 outlier",
            ops=("softmax", "rmsnorm", "layernorm"),
            shapes=((128, 8192), (32, 65536)), dist="normal3"),
    5: dict(name="HBM roofline 65536x4096",
            ops=("residual_layernorm", "rmsnorm", "softmax"),
            shapes=((65536, 4096),), dist="uniform"),
}


def x_seed(cfg: int) -> int:
    return 1000 + cfg


def r_seed(cfg: int) -> int:
    return 2000 + cfg


def rows_of(cfg: int, rows: int, width: int, row_ids=None, which: str = "x") -> np.ndarray:
    """FP32 input rows of workload ``cfg`` at shape ``rows x width``.

    ``which`` is ``"x"`` (the input) or ``"r"`` (the residual).  ``row_ids``
    selects rows (default: all), returned as a ``[len(row_ids), width]`` array
    equal to the same rows of the full tensor.
    """
    if row_ids is None:
        row_ids = range(rows)
    row_ids = [int(i) for i in row_ids]
    for i in row_ids:
        if not 0 <= i < rows:
            raise IndexError(f"row {i} outside [0, {rows})")
    seed = x_seed(cfg) if which == "x" else r_seed(cfg)
    dist = WORKLOADS[cfg]["dist"] if cfg in WORKLOADS else "uniform"
    out = np.empty((len(row_ids), width), dtype=np.float32)
    if row_ids and row_ids == list(range(row_ids[0], row_ids[0] + len(row_ids))):
        flat = _draw(dist, seed, len(row_ids) * width, row_ids[0] * width)
        out[:] = flat.reshape(len(row_ids), width)
    else:
        for k, i in enumerate(row_ids):
            out[k] = _draw(dist, seed, width, i * width)
    if dist == "normal3" and which == "x":
        first = _draw(dist, seed, 1, 0)[0]
        for k, i in enumerate(row_ids):
            if i == 0:
                out[k, :] = first                      # one row of constants
            elif i == 1:
                out[k, outlier_column(width)] = np.float32(40.0)   # one +40 outlier
    return out


def outlier_column(width: int) -> int:
    """Column of row 1 that holds the +40 outlier in the wide-row workload."""
    return (width // 2 + 3) % width


def _draw(dist: str, seed: int, count: int, start: int) -> np.ndarray:
    if dist == "uniform":
        return uniform_pm1(seed, count, start)
    if dist == "normal3":
        return normal(seed, count, 3.0, start)
    raise ValueError(dist)


def workload_inputs(cfg: int, rows: int, width: int, op: str):
    """``(x, r)`` for one op/shape of a workload; ``r`` is None unless the op is
    residual LayerNorm."""
    x = rows_of(cfg, rows, width, which="x")
    r = rows_of(cfg, rows, width, which="r") if op == "residual_layernorm" else None
    return x, r
