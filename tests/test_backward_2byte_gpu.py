"""GPU parity of the backward kernels on BF16 and FP16 rows (x or y, dy and dx
of the 2-byte type; row statistics, gamma and parameter gradients FP32)
against the FP64 oracle, run on the exact widened 2-byte inputs.

dx is computed in FP32 and rounded to the output type, so the bound is the
FP32 backward bound (its terms scale with the O(1) quantities dx is a
difference of, see test_backward_gpu.py) plus half an ulp of the type,
h |ref| with h = 2^-8 (BF16) or 2^-11 (FP16).  Row statistics and parameter
gradients are FP32 outputs with the FP32 bounds."""

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
TYPES = {"bf16": (torch.bfloat16, 2.0 ** -8), "f16": (torch.float16, 2.0 ** -11)}


@pytest.fixture(scope="module", autouse=True)
def device():
    from tile_compiler_row_gb300 import _build
    _build.build()
    torch.cuda.set_device(0)
    yield
    assert tile.tile_check_device_status() == 0


def _rows(cfg, rows, width, which, dt):
    """(device tensor of type dt, its exact values as FP32 numpy)."""
    t = torch.from_numpy(synth.rows_of(cfg, rows, width, which=which)).to(TYPES[dt][0])
    return t, t.float().numpy()


def _placed(t, offset=0):
    buf = torch.empty(t.numel() + 16, dtype=t.dtype, device="cuda")
    view = buf[offset:offset + t.numel()].view(t.shape)
    view.copy_(t)
    return view


def _stats64(x, rms):
    x = x.astype(np.float64)
    mean = np.zeros(x.shape[0]) if rms else x.mean(axis=1)
    rstd = 1.0 / np.sqrt(((x - mean[:, None]) ** 2).mean(axis=1) + ref_eps())
    return mean, rstd


def _dx_bound(x, dy, gamma, ref, rms, h):
    mean, rstd = _stats64(x, rms)
    xhat = (x.astype(np.float64) - mean[:, None]) * rstd[:, None]
    g = dy.astype(np.float64) * (gamma.astype(np.float64) if gamma is not None else 1.0)
    terms = (np.abs(g) + np.abs(g).mean(axis=1, keepdims=True)
             + np.abs(xhat) * np.abs(g * xhat).mean(axis=1, keepdims=True))
    fp32 = ATOL + RTOL * np.abs(ref) + 16 * U * rstd[:, None] * terms
    return fp32 + h * (np.abs(ref) + fp32)


def _softmax_bound(y, dy, ref, h):
    dot = np.abs((dy.astype(np.float64) * y).sum(axis=1, keepdims=True))
    fp32 = ATOL + RTOL * np.abs(ref) + 16 * U * np.abs(y) * (np.abs(dy) + dot)
    return fp32 + h * (np.abs(ref) + fp32)


def _check(got, ref, bound, what):
    got = np.asarray(got, np.float64)
    assert got.shape == ref.shape and np.all(np.isfinite(got)), what
    err = np.abs(got - ref)
    bad = err > bound
    assert not bad.any(), f"{what}: {int(bad.sum())} beyond the bound, max err {err.max():.3e}"


SHAPES = [(1, 127), (17, 257), (7, 1537), (64, 4096), (256, 4096), (128, 8192), (32, 65536)]


@pytest.mark.parametrize("dt", ["bf16", "f16"])
@pytest.mark.parametrize("rows,width", SHAPES)
@pytest.mark.parametrize("op", ["layernorm", "rmsnorm"])
@pytest.mark.parametrize("with_gamma", [False, True])
def test_norm_backward(dt, op, rows, width, with_gamma):
    cfg = 4 if width in (8192, 65536) else 3
    x, xf = _rows(cfg, rows, width, "x", dt)
    dy, dyf = _rows(3, rows, width, "r", dt)
    gamma = synth.uniform_pm1(3001, width) * np.float32(2.0) if with_gamma else None
    dx = torch.full((rows, width), float("nan"), dtype=TYPES[dt][0], device="cuda")
    stats = torch.full((2 * rows,), float("nan"), device="cuda")
    getattr(tile, f"tile_{op}_backward_{dt}")(
        _placed(x), torch.from_numpy(gamma).cuda() if with_gamma else None, _placed(dy), dx,
        stats, EPS)
    ref = getattr(oracle.get(), f"{op}_backward")(xf, dyf, gamma, ref_eps())
    _check(dx.float().cpu().numpy(), ref,
           _dx_bound(xf, dyf, gamma, ref, op == "rmsnorm", TYPES[dt][1]),
           f"{dt} {op} backward {rows}x{width} gamma={with_gamma}")
    mean, rstd = _stats64(xf, op == "rmsnorm")
    st = stats.cpu().numpy().reshape(rows, 2).astype(np.float64)
    assert np.all(np.abs(st[:, 0] - mean) <= 1e-6 * (1 + np.abs(xf).max()))
    assert np.all(np.abs(st[:, 1] - rstd) <= 2e-6 * rstd)


@pytest.mark.parametrize("dt", ["bf16", "f16"])
@pytest.mark.parametrize("rows,width", SHAPES)
def test_softmax_backward(dt, rows, width):
    cfg = 4 if width in (8192, 65536) else 3
    x = synth.rows_of(cfg, rows, width, which="x")
    y = torch.from_numpy(oracle.get().softmax(x).astype(np.float32)).to(TYPES[dt][0])
    yf = y.float().numpy()
    dy, dyf = _rows(3, rows, width, "r", dt)
    dx = torch.full((rows, width), float("nan"), dtype=TYPES[dt][0], device="cuda")
    getattr(tile, f"tile_softmax_backward_{dt}")(_placed(y), _placed(dy), dx)
    ref = oracle.get().softmax_backward(yf, dyf)
    _check(dx.float().cpu().numpy(), ref, _softmax_bound(yf, dyf, ref, TYPES[dt][1]),
           f"{dt} softmax backward {rows}x{width}")


@pytest.mark.parametrize("dt", ["bf16", "f16"])
@pytest.mark.parametrize("rows,width,offset", [(17, 257, 0), (1024, 4096, 0), (3000, 1537, 1),
                                               (64, 65536, 0), (100, 1030, 2)])
@pytest.mark.parametrize("op", ["layernorm", "rmsnorm"])
def test_param_grad(dt, op, rows, width, offset):
    x, xf = _rows(3, rows, width, "x", dt)
    dy, dyf = _rows(3, rows, width, "r", dt)
    tx, tdy = _placed(x, offset), _placed(dy, offset)
    dx = torch.empty(rows, width, dtype=TYPES[dt][0], device="cuda")
    stats = torch.empty(2 * rows, device="cuda")
    getattr(tile, f"tile_{op}_backward_{dt}")(tx, None, tdy, dx, stats, EPS)
    dg = torch.full((width,), float("nan"), device="cuda")
    db = torch.full((width,), float("nan"), device="cuda") if op == "layernorm" else None
    ws = torch.empty(tile.tile_norm_param_grad_workspace_bytes(rows, width), dtype=torch.uint8,
                     device="cuda")
    getattr(tile, f"tile_norm_param_grad_{dt}")(tx, tdy, stats, dg, db, ws)
    rg, rb = oracle.get().norm_param_grad(xf, dyf, ref_eps(), rms=op == "rmsnorm")
    mean, rstd = _stats64(xf, op == "rmsnorm")
    xhat = (xf.astype(np.float64) - mean[:, None]) * rstd[:, None]
    mag_g = np.abs(dyf * xhat).sum(axis=0)
    _check(dg.cpu().numpy(), rg, ATOL + RTOL * np.abs(rg) + 2.0 ** -22 * mag_g,
           f"{dt} {op} dgamma")
    if db is not None:
        mag_b = np.abs(dyf.astype(np.float64)).sum(axis=0)
        _check(db.cpu().numpy(), rb, ATOL + RTOL * np.abs(rb) + 2.0 ** -22 * mag_b,
               f"{dt} {op} dbeta")


def _plan_cases():
    from tile_compiler_row_gb300 import _build
    _build.build()
    out = []
    for pid in range(tile.tile_plan_count()):
        info = tile.tile_plan_info_ex(pid, 0, "bf16", 1, 1)
        # raw-word stripes: up to 64 elements for 16-byte vectors, 32 scalar
        budget = 64 if info is not None and info["vec"] == 8 else 32
        if info is None or info["path"] == 2 or info["chunks"] * info["vec"] > budget:
            continue
        maxw = info["max_width"]
        rows = 3 if maxw > 16384 else 2 * info["programs_per_cta"] + 1
        for op in ("layernorm", "rmsnorm", "softmax"):
            out.append((pid, op, rows, sorted({1, 6, min(maxw, 41), maxw}), info["vec"]))
    return out


@pytest.mark.parametrize("dt", ["bf16", "f16"])
@pytest.mark.parametrize("pid,op,rows,widths,vec", _plan_cases(),
                         ids=lambda v: str(v) if not isinstance(v, list) else "w")
def test_every_2byte_backward_plan(dt, pid, op, rows, widths, vec):
    orc = oracle.get()
    h = TYPES[dt][1]
    for w in widths:
        x, xf = _rows(3, rows, w, "x", dt)
        dy, dyf = _rows(3, rows, w, "r", dt)
        gamma = synth.uniform_pm1(3001, w) + np.float32(1.0)
        tg = torch.from_numpy(gamma).cuda()
        for off in (0, 3):
            dx = _placed(torch.zeros(rows, w, dtype=TYPES[dt][0]), off if vec > 1 else off + 1)
            if op == "softmax":
                y = torch.from_numpy(orc.softmax(xf).astype(np.float32)).to(TYPES[dt][0])
                yf = y.float().numpy()
                tile.tile_run_backward_plan_ex(op, pid, _placed(y, off), None, _placed(dy, off),
                                               dx)
                ref = orc.softmax_backward(yf, dyf)
                bound = _softmax_bound(yf, dyf, ref, h)
            else:
                tile.tile_run_backward_plan_ex(op, pid, _placed(x, off), tg, _placed(dy, off), dx,
                                               None, EPS)
                ref = getattr(orc, f"{op}_backward")(xf, dyf, gamma, ref_eps())
                bound = _dx_bound(xf, dyf, gamma, ref, op == "rmsnorm", h)
            _check(dx.float().cpu().numpy(), ref, bound, f"{dt} plan {pid} {op} w={w} off={off}")


def test_2byte_plans_above_the_stripe_budget_are_rejected():
    # K = 16 plans exist for FP32 only; K = 8 is the 2-byte backward limit
    big = [pid for pid in range(tile.tile_plan_count())
           if (tile.tile_plan_info(pid, 0, 1, 4) or {}).get("chunks", 0) == 16
           and tile.tile_plan_info(pid, 0, 1, 4)["vec"] == 4]
    assert big
    t = torch.zeros(2, 64, dtype=torch.bfloat16, device="cuda")   # (not built for 2-byte)
    with pytest.raises(tile.TileError) as e:
        tile.tile_run_backward_plan_ex("layernorm", big[0], t, None, t.clone(),
                                       torch.empty_like(t))
    assert e.value.status == -8
