"""GPU parity of the backward kernels (input gradients, row statistics and
parameter gradients) against the FP64 oracle.

The pages print no tolerance for gradients.  dx is a difference of O(1)
terms, dx_j = rstd (g_j - mean(g) - xhat_j mean(g xhat)), so its FP32 error
scales with the terms, not with dx:

    |dx - ref| <= 2e-6 + 2e-5 |ref| + 16 u rstd (|g_j| + mean|g| + |xhat_j| mean|g xhat|)

with u = 2^-24 and the term magnitudes taken in FP64 from the inputs.
Parameter gradients are sums over rows, bounded by the compensated-sum
error:  |d - ref| <= 2e-6 + 2e-5 |ref| + 2^-22 sum_i |term_i|."""

from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
import synth
import tile_compiler_row_gb300 as tile
from parity import ATOL, EPS, RTOL, ref_eps

pytestmark = pytest.mark.gpu

U = 2.0 ** -24


@pytest.fixture(scope="module", autouse=True)
def device():
    from tile_compiler_row_gb300 import _build
    _build.build()
    torch.cuda.set_device(0)
    yield
    assert tile.tile_check_device_status() == 0


def _dev(a, offset=0):
    a = np.ascontiguousarray(a, dtype=np.float32)
    buf = torch.empty(a.size + 8, dtype=torch.float32, device="cuda")
    view = buf[offset:offset + a.size].view(a.shape)
    view.copy_(torch.from_numpy(a))
    return view


def _stats64(x, rms):
    x = x.astype(np.float64)
    mean = np.zeros(x.shape[0]) if rms else x.mean(axis=1)
    rstd = 1.0 / np.sqrt(((x - mean[:, None]) ** 2).mean(axis=1) + ref_eps())
    return mean, rstd


def _dx_bound(x, dy, gamma, ref, rms):
    mean, rstd = _stats64(x, rms)
    xhat = (x.astype(np.float64) - mean[:, None]) * rstd[:, None]
    g = dy.astype(np.float64) * (gamma.astype(np.float64) if gamma is not None else 1.0)
    terms = (np.abs(g) + np.abs(g).mean(axis=1, keepdims=True)
             + np.abs(xhat) * np.abs(g * xhat).mean(axis=1, keepdims=True))
    return ATOL + RTOL * np.abs(ref) + 16 * U * rstd[:, None] * terms


def _check(got, ref, bound, what):
    got = np.asarray(got, np.float64)
    assert got.shape == ref.shape and np.all(np.isfinite(got)), what
    err = np.abs(got - ref)
    bad = err > bound
    assert not bad.any(), f"{what}: {int(bad.sum())} beyond the bound, max err {err.max():.3e}"


SHAPES = [(1, 127), (17, 257), (7, 1537), (64, 4096), (1024, 4096), (128, 8192), (32, 65536)]


@pytest.mark.parametrize("rows,width", SHAPES)
@pytest.mark.parametrize("op", ["layernorm", "rmsnorm"])
@pytest.mark.parametrize("with_gamma", [False, True])
def test_norm_backward(op, rows, width, with_gamma):
    cfg = 4 if width in (8192, 65536) else 3
    x = synth.rows_of(cfg, rows, width, which="x")
    dy = synth.rows_of(3, rows, width, which="r")
    gamma = synth.uniform_pm1(3001, width) * np.float32(2.0) if with_gamma else None
    dx = torch.full((rows, width), float("nan"), device="cuda")
    stats = torch.full((2 * rows,), float("nan"), device="cuda")
    getattr(tile, f"tile_{op}_backward_f32")(_dev(x), _dev(gamma) if with_gamma else None, _dev(dy),
                                             dx, stats, EPS)
    orc = oracle.get()
    ref = getattr(orc, f"{op}_backward")(x, dy, gamma, ref_eps())
    _check(dx.cpu().numpy(), ref, _dx_bound(x, dy, gamma, ref, op == "rmsnorm"),
           f"{op} backward {rows}x{width} gamma={with_gamma}")
    mean, rstd = _stats64(x, op == "rmsnorm")
    st = stats.cpu().numpy().reshape(rows, 2).astype(np.float64)
    assert np.all(np.abs(st[:, 0] - mean) <= 1e-6 * (1 + np.abs(x).max()))
    assert np.all(np.abs(st[:, 1] - rstd) <= 2e-6 * rstd)


@pytest.mark.parametrize("rows,width", SHAPES)
def test_softmax_backward(rows, width):
    cfg = 4 if width in (8192, 65536) else 3
    x = synth.rows_of(cfg, rows, width, which="x")
    y = oracle.get().softmax(x).astype(np.float32)          # a forward output
    dy = synth.rows_of(3, rows, width, which="r")
    dx = torch.full((rows, width), float("nan"), device="cuda")
    tile.tile_softmax_backward_f32(_dev(y), _dev(dy), dx)
    ref = oracle.get().softmax_backward(y, dy)
    dot = np.abs((dy.astype(np.float64) * y).sum(axis=1, keepdims=True))
    bound = ATOL + RTOL * np.abs(ref) + 16 * U * np.abs(y) * (np.abs(dy) + dot)
    _check(dx.cpu().numpy(), ref, bound, f"softmax backward {rows}x{width}")


@pytest.mark.parametrize("rows,width", [(17, 257), (1024, 4096), (3000, 1537), (64, 65536),
                                        (1, 1), (3, 131072), (100000, 5)])
@pytest.mark.parametrize("op", ["layernorm", "rmsnorm"])
def test_param_grad(op, rows, width):
    x = synth.rows_of(3, rows, width, which="x")
    dy = synth.rows_of(3, rows, width, which="r")
    tx, tdy = _dev(x), _dev(dy)
    dx = torch.empty(rows, width, device="cuda")
    stats = torch.empty(2 * rows, device="cuda")
    getattr(tile, f"tile_{op}_backward_f32")(tx, None, tdy, dx, stats, EPS)
    dg = torch.full((width,), float("nan"), device="cuda")
    db = torch.full((width,), float("nan"), device="cuda") if op == "layernorm" else None
    ws = torch.empty(tile.tile_norm_param_grad_workspace_bytes(rows, width), dtype=torch.uint8,
                     device="cuda")
    tile.tile_norm_param_grad_f32(tx, tdy, stats, dg, db, ws)
    rg, rb = oracle.get().norm_param_grad(x, dy, ref_eps(), rms=op == "rmsnorm")
    mean, rstd = _stats64(x, op == "rmsnorm")
    xhat = (x.astype(np.float64) - mean[:, None]) * rstd[:, None]
    mag_g = np.abs(dy * xhat).sum(axis=0)
    _check(dg.cpu().numpy(), rg, ATOL + RTOL * np.abs(rg) + 2.0 ** -22 * mag_g, f"{op} dgamma")
    if db is not None:
        mag_b = np.abs(dy.astype(np.float64)).sum(axis=0)
        _check(db.cpu().numpy(), rb, ATOL + RTOL * np.abs(rb) + 2.0 ** -22 * mag_b, f"{op} dbeta")
    # deterministic: a second call gives the same bits
    dg2 = torch.empty_like(dg)
    tile.tile_norm_param_grad_f32(tx, tdy, stats, dg2, None, ws)
    assert torch.equal(dg, dg2)


def _bwd_plan_cases():
    from tile_compiler_row_gb300 import _build
    _build.build()
    out = []
    for pid in range(tile.tile_plan_count()):
        info = tile.tile_plan_info(pid, 0, 1, 1)
        if info is None or info["chunks"] * info["vec"] > 32:
            continue
        maxw = info["max_width"]
        rows = 3 if maxw > 16384 else 2 * info["programs_per_cta"] + 1
        for op in ("layernorm", "rmsnorm", "softmax"):
            out.append((pid, op, rows, sorted({1, 6, min(maxw, 41), maxw}), info["vec"]))
    return out


@pytest.mark.parametrize("pid,op,rows,widths,vec", _bwd_plan_cases(),
                         ids=lambda v: str(v) if not isinstance(v, list) else "w")
def test_every_backward_plan(pid, op, rows, widths, vec):
    orc = oracle.get()
    for w in widths:
        x = synth.rows_of(3, rows, w, which="x")
        dy = synth.rows_of(3, rows, w, which="r")
        gamma = synth.uniform_pm1(3001, w) + np.float32(1.0)
        for off in (0, 1):
            dx = _dev(np.zeros((rows, w), np.float32), off if vec == 4 else (off + 2) % 4)
            if op == "softmax":
                y = orc.softmax(x).astype(np.float32)
                tile.tile_run_backward_plan_f32(op, pid, _dev(y, off), None, _dev(dy, off), dx)
                ref = orc.softmax_backward(y, dy)
                dot = np.abs((dy.astype(np.float64) * y).sum(axis=1, keepdims=True))
                bound = ATOL + RTOL * np.abs(ref) + 16 * U * np.abs(y) * (np.abs(dy) + dot)
            else:
                tile.tile_run_backward_plan_f32(op, pid, _dev(x, off), _dev(gamma), _dev(dy, off),
                                                dx, None, EPS)
                ref = getattr(orc, f"{op}_backward")(x, dy, gamma, ref_eps())
                bound = _dx_bound(x, dy, gamma, ref, op == "rmsnorm")
            _check(dx.cpu().numpy(), ref, bound, f"plan {pid} {op} w={w} off={off}")


def test_backward_errors_on_device_buffers():
    t = torch.zeros(4, 64, device="cuda")
    with pytest.raises(tile.TileError) as e:
        tile.tile_layernorm_backward_f32(t, None, torch.zeros_like(t), t)
    assert e.value.status == -3
    x = torch.zeros(4, 64, device="cuda")
    ws = torch.empty(8, dtype=torch.uint8, device="cuda")
    with pytest.raises(tile.TileError) as e:
        tile.tile_norm_param_grad_f32(x, x.clone(), torch.zeros(8, device="cuda"),
                                      torch.empty(64, device="cuda"), None, ws)
    assert e.value.status == -10
