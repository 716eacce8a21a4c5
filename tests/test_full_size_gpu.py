"""Every forward and backward entry point at the benchmark's 65536 x 4096
shape, every output element against the FP64 oracle.

The benchmark's own launches (FP32 residual LayerNorm, RMSNorm, softmax and
BF16 residual LayerNorm) are compared in full in test_parity_gpu.py and
test_parity_bf16_gpu.py; here are the other forward operations and element
types at the same size (268,435,456 outputs each, 1 GiB per FP32 tensor),
through the selector's plan for that shape.  The oracle runs over row
blocks on every host core and each block is compared in its thread, so
host memory stays bounded.

Bounds per element (ref = oracle, FP64): 2e-6 + 2e-5 |ref| for FP32
outputs (atol 1e-5 for affine LayerNorm, the pages' affine tolerance),
plus half an ulp of the output type (2^-8 |ref| BF16, 2^-11 |ref| FP16) for
2-byte outputs; row minima and maxima exact."""

from __future__ import annotations

from concurrent.futures import ThreadPoolExecutor

import numpy as np
import pytest
import torch

import oracle
import synth
import tile_compiler_row_gb300 as tile
from parity import ATOL, EPS, RTOL, host_threads, ref_eps

pytestmark = pytest.mark.gpu

ROWS, WIDTH = 65536, 4096
BLOCK = 2048
HALF_ULP = {"f32": 0.0, "bf16": 2.0 ** -8, "f16": 2.0 ** -11}
TORCH = {"f32": torch.float32, "bf16": torch.bfloat16, "f16": torch.float16}


@pytest.fixture(scope="module", autouse=True)
def device():
    from tile_compiler_row_gb300 import _build
    _build.build()
    torch.cuda.set_device(0)
    yield
    assert tile.tile_check_device_status() == 0


@pytest.fixture(scope="module")
def data():
    x = synth.rows_of(5, ROWS, WIDTH, which="x")
    r = synth.rows_of(5, ROWS, WIDTH, which="r")
    g = synth.uniform_pm1(3001, WIDTH) * np.float32(2.0)
    b = synth.uniform_pm1(3002, WIDTH)
    return x, r, g, b


def _typed(a, dtype):
    """(device tensor of `dtype`, the exact FP32 values it holds, on the host)."""
    t = torch.from_numpy(a).to(TORCH[dtype])
    return t.cuda(), (t.float().numpy() if dtype != "f32" else a)


def _blocks(ref_fn, check_fn):
    """ref_fn(a, b) -> oracle output for rows [a, b); check_fn(a, b, ref)
    asserts the bound; blocks run on every host core."""
    spans = [(a, min(ROWS, a + BLOCK)) for a in range(0, ROWS, BLOCK)]

    def one(ab):
        a, b = ab
        check_fn(a, b, ref_fn(a, b))

    with ThreadPoolExecutor(max_workers=host_threads()) as ex:
        list(ex.map(one, spans))


def _bound_check(got, atol, rtol, what):
    def check(a, b, ref):
        g = got[a:b].astype(np.float64)
        assert np.all(np.isfinite(g)), f"{what} rows {a}..{b - 1}: non-finite"
        err = np.abs(g - ref)
        bad = ~(err <= atol + rtol * np.abs(ref))
        assert not bad.any(), (f"{what} rows {a}..{b - 1}: {int(bad.sum())} beyond the bound, "
                               f"max err {float(err.max()):.3e}")
    return check


NORMALISERS = [
    ("layernorm", "f32"), ("layernorm_affine", "f32"), ("layernorm_affine_residual", "f32"),
    ("rmsnorm_weighted", "f32"),
    ("residual_layernorm", "f16"), ("layernorm", "bf16"), ("layernorm", "f16"),
    ("rmsnorm", "bf16"), ("rmsnorm", "f16"), ("softmax", "bf16"), ("softmax", "f16"),
    ("layernorm_affine", "bf16"), ("layernorm_affine_residual", "bf16"),
    ("rmsnorm_weighted", "bf16"),
]


@pytest.mark.parametrize("op,dtype", NORMALISERS)
def test_normaliser_every_element(op, dtype, data):
    x, r, g, b = data
    xd, xf = _typed(x, dtype)
    residual = op in ("residual_layernorm", "layernorm_affine_residual")
    rd, rf = _typed(r, dtype) if residual else (None, None)
    gd, bd = torch.from_numpy(g).cuda(), torch.from_numpy(b).cuda()
    out = torch.full((ROWS, WIDTH), float("nan"), dtype=TORCH[dtype], device="cuda")
    orc = oracle.get()
    e = ref_eps()
    if op == "residual_layernorm":
        getattr(tile, f"tile_residual_layernorm_{dtype}")(xd, rd, out, EPS)
        ref_fn = lambda a, c: orc.residual_layernorm(xf[a:c], rf[a:c], e)          # noqa: E731
    elif op in ("layernorm", "rmsnorm", "softmax"):
        getattr(tile, f"tile_{op}_{dtype}")(xd, out, EPS)
        ref_fn = lambda a, c: orc.run(op, xf[a:c], eps=e)                          # noqa: E731
    elif op.startswith("layernorm_affine"):
        getattr(tile, f"tile_layernorm_affine_{dtype}")(xd, rd, gd, bd, out, EPS)
        ref_fn = lambda a, c: orc.layernorm_affine(                                # noqa: E731
            xf[a:c], g, b, r=rf[a:c] if residual else None, eps=e)
    else:
        getattr(tile, f"tile_rmsnorm_weighted_{dtype}")(xd, gd, out, EPS)
        ref_fn = lambda a, c: orc.rmsnorm_weighted(xf[a:c], g, eps=e)              # noqa: E731
    torch.cuda.synchronize()
    got = out.float().cpu().numpy()
    del out, xd, rd
    atol = 1e-5 if op.startswith("layernorm_affine") else ATOL
    _blocks(ref_fn, _bound_check(got, atol, RTOL + HALF_ULP[dtype], f"{op} {dtype}"))


def test_row_sum_and_minmax_every_row(data):
    x = data[0]
    xd = torch.from_numpy(x).cuda()
    s = torch.full((ROWS,), float("nan"), device="cuda")
    mn = torch.full((ROWS,), float("nan"), device="cuda")
    mx = torch.full((ROWS,), float("nan"), device="cuda")
    tile.tile_row_sum_f32(xd, s)
    tile.tile_row_minmax_f32(xd, mn, mx)
    torch.cuda.synchronize()
    orc = oracle.get()
    ref_s = np.concatenate([orc.row_sum(x[a:a + BLOCK]) for a in range(0, ROWS, BLOCK)])
    err = np.abs(s.cpu().numpy().astype(np.float64) - ref_s)
    assert np.all(err <= ATOL + RTOL * np.abs(ref_s)), f"row sums: max err {err.max():.3e}"
    ref_mn, ref_mx = orc.row_minmax(x)
    assert np.array_equal(mn.cpu().numpy().astype(np.float64), ref_mn)
    assert np.array_equal(mx.cpu().numpy().astype(np.float64), ref_mx)


@pytest.mark.parametrize("kind", ["sigmoid", "gelu_tanh"])
def test_pair_every_element(kind, data):
    x = data[0]
    xd = torch.from_numpy(x).cuda()
    y = torch.full_like(xd, float("nan"))
    dy = torch.full_like(xd, float("nan"))
    getattr(tile, f"tile_{kind}_pair_f32")(xd, y, dy)
    torch.cuda.synchronize()
    got_y, got_dy = y.cpu().numpy(), dy.cpu().numpy()
    del y, dy, xd
    fn = getattr(oracle.get(), f"{kind}_pair")
    check_y = _bound_check(got_y, ATOL, RTOL, f"{kind} value")
    check_dy = _bound_check(got_dy, ATOL, RTOL, f"{kind} derivative")

    def check(a, b, ref):
        check_y(a, b, ref[0])
        check_dy(a, b, ref[1])

    _blocks(lambda a, b: fn(x[a:b]), check)


# ---------------------------------------------------------------------------
# backward passes at the same shape, with the bounds of test_backward_gpu.py:
# dx within 2e-6 + 2e-5 |ref| + 16 u rstd (|g_j| + mean|g| + |xhat_j|
# mean|g xhat|) (softmax: 16 u |y_j| (|dy_j| + |sum dy y|)), plus half an
# ulp of a 2-byte output; parameter gradients within 2e-6 + 2e-5 |ref| +
# 2^-22 sum_i |term_i|.
# ---------------------------------------------------------------------------

U = 2.0 ** -24


def _dx_bound_rows(x, dy, gamma, ref, rms):
    x = x.astype(np.float64)
    mean = np.zeros(x.shape[0]) if rms else x.mean(axis=1)
    rstd = 1.0 / np.sqrt(((x - mean[:, None]) ** 2).mean(axis=1) + ref_eps())
    xhat = (x - mean[:, None]) * rstd[:, None]
    g = dy.astype(np.float64) * (gamma.astype(np.float64) if gamma is not None else 1.0)
    terms = (np.abs(g) + np.abs(g).mean(axis=1, keepdims=True)
             + np.abs(xhat) * np.abs(g * xhat).mean(axis=1, keepdims=True))
    return ATOL + RTOL * np.abs(ref) + 16 * U * rstd[:, None] * terms


def _check_against(got, bound_fn, what):
    def check(a, b, ref):
        g = got[a:b].astype(np.float64)
        assert np.all(np.isfinite(g)), f"{what} rows {a}..{b - 1}: non-finite"
        err = np.abs(g - ref)
        bad = ~(err <= bound_fn(a, b, ref))
        assert not bad.any(), (f"{what} rows {a}..{b - 1}: {int(bad.sum())} beyond the bound, "
                               f"max err {float(err.max()):.3e}")
    return check


@pytest.mark.parametrize("op,dtype", [("layernorm", "f32"), ("rmsnorm", "f32"),
                                      ("layernorm", "bf16"), ("rmsnorm", "bf16")])
def test_norm_backward_every_element(op, dtype, data):
    x, dyh, g, _ = data
    xd, xf = _typed(x, dtype)
    dyd, dyf = _typed(dyh, dtype)
    dx = torch.full((ROWS, WIDTH), float("nan"), dtype=TORCH[dtype], device="cuda")
    stats = torch.empty(2 * ROWS, device="cuda")
    getattr(tile, f"tile_{op}_backward_{dtype}")(xd, torch.from_numpy(g).cuda(), dyd, dx, stats,
                                                 EPS)
    torch.cuda.synchronize()
    got = dx.float().cpu().numpy()
    del dx, xd, dyd
    orc = oracle.get()
    fn = getattr(orc, f"{op}_backward")
    half = HALF_ULP[dtype]
    _blocks(lambda a, b: fn(xf[a:b], dyf[a:b], g, ref_eps()),
            _check_against(got, lambda a, b, ref: _dx_bound_rows(
                xf[a:b], dyf[a:b], g, ref, op == "rmsnorm") + half * np.abs(ref),
                f"{op} backward {dtype}"))


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_softmax_backward_every_element(dtype, data):
    x, dyh = data[0], data[1]
    orc = oracle.get()
    y = np.concatenate([orc.softmax(x[a:a + BLOCK]) for a in range(0, ROWS, BLOCK)]).astype(
        np.float32)                                           # a forward output
    yd, yf = _typed(y, dtype)
    dyd, dyf = _typed(dyh, dtype)
    dx = torch.full((ROWS, WIDTH), float("nan"), dtype=TORCH[dtype], device="cuda")
    getattr(tile, f"tile_softmax_backward_{dtype}")(yd, dyd, dx)
    torch.cuda.synchronize()
    got = dx.float().cpu().numpy()
    del dx, yd, dyd
    half = HALF_ULP[dtype]

    def bound(a, b, ref):
        yy, dd = yf[a:b].astype(np.float64), dyf[a:b].astype(np.float64)
        dot = np.abs((dd * yy).sum(axis=1, keepdims=True))
        return ATOL + (RTOL + half) * np.abs(ref) + 16 * U * np.abs(yy) * (np.abs(dd) + dot)

    _blocks(lambda a, b: orc.softmax_backward(yf[a:b], dyf[a:b]),
            _check_against(got, bound, f"softmax backward {dtype}"))


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_param_grad_every_column(dtype, data):
    x, dyh = data[0], data[1]
    xd, xf = _typed(x, dtype)
    dyd, dyf = _typed(dyh, dtype)
    dx = torch.empty((ROWS, WIDTH), dtype=TORCH[dtype], device="cuda")
    stats = torch.empty(2 * ROWS, device="cuda")
    getattr(tile, f"tile_layernorm_backward_{dtype}")(xd, None, dyd, dx, stats, EPS)
    del dx
    dg = torch.full((WIDTH,), float("nan"), device="cuda")
    db = torch.full((WIDTH,), float("nan"), device="cuda")
    ws = torch.empty(tile.tile_norm_param_grad_workspace_bytes(ROWS, WIDTH), dtype=torch.uint8,
                     device="cuda")
    getattr(tile, f"tile_norm_param_grad_{dtype}")(xd, dyd, stats, dg, db, ws)
    torch.cuda.synchronize()
    rg, rb = oracle.get().norm_param_grad(xf, dyf, ref_eps(), rms=False)
    x64 = xf.astype(np.float64)
    mean = x64.mean(axis=1)
    rstd = 1.0 / np.sqrt(((x64 - mean[:, None]) ** 2).mean(axis=1) + ref_eps())
    mag_g = np.abs(dyf * ((x64 - mean[:, None]) * rstd[:, None])).sum(axis=0)
    mag_b = np.abs(dyf.astype(np.float64)).sum(axis=0)
    for got, ref, mag, what in ((dg, rg, mag_g, "dgamma"), (db, rb, mag_b, "dbeta")):
        err = np.abs(got.cpu().numpy().astype(np.float64) - ref)
        bound = ATOL + RTOL * np.abs(ref) + 2.0 ** -22 * mag
        assert np.all(err <= bound), f"{what} {dtype}: max err {err.max():.3e}"
