"""GPU parity of the further row operations and the pointwise pairs against
the FP64 oracle.

Tolerances (the pages' runner, "Cooperating-program packing", "Predeclared
comparison and measurement"; "Multi-output pointwise fusion: evidence and
limits"): affine LayerNorm atol 1e-5, everything else atol 2e-6; rtol 2e-5
for all.  Row min/max are exact."""

from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
import synth
import tile_compiler_row_gb300 as tile
from parity import ATOL, EPS, RTOL, ref_eps

pytestmark = pytest.mark.gpu

ATOL_AFFINE = 1e-5


@pytest.fixture(scope="module", autouse=True)
def device():
    from tile_compiler_row_gb300 import _build
    _build.build()
    torch.cuda.set_device(0)
    yield
    assert tile.tile_check_device_status() == 0


def _placed(a, offset=0):
    """A device copy of ``a`` starting ``offset`` floats into its buffer."""
    a = np.ascontiguousarray(a, dtype=np.float32)
    buf = torch.empty(a.size + 8, dtype=torch.float32, device="cuda")
    view = buf[offset:offset + a.size].view(a.shape)
    view.copy_(torch.from_numpy(a))
    return view


def _out(shape, offset=0):
    n = int(np.prod(shape))
    buf = torch.full((n + 8,), float("nan"), device="cuda")
    return buf[offset:offset + n].view(shape)


def _check_bound(got, ref, atol, what):
    got = np.asarray(got, np.float64)
    assert got.shape == ref.shape, what
    assert np.all(np.isfinite(got)), what
    err = np.abs(got - ref)
    bad = err > atol + RTOL * np.abs(ref)
    assert not bad.any(), f"{what}: {int(bad.sum())} beyond tolerance, max err {err.max():.3e}"


def _gamma_beta(width):
    g = synth.uniform_pm1(3001, width) * np.float32(2.0)
    b = synth.uniform_pm1(3002, width)
    return g, b


# ---------------------------------------------------------------------------
# affine LayerNorm / weighted RMSNorm
# ---------------------------------------------------------------------------

SHAPES = [(1, 127), (7, 1537), (17, 257), (64, 4096), (1024, 4096), (128, 8192), (32, 65536)]


@pytest.mark.parametrize("rows,width", SHAPES)
@pytest.mark.parametrize("residual", [False, True])
@pytest.mark.parametrize("with_beta", [False, True])
def test_layernorm_affine(rows, width, residual, with_beta):
    x = synth.rows_of(3, rows, width, which="x")
    r = synth.rows_of(3, rows, width, which="r") if residual else None
    g, b = _gamma_beta(width)
    b = b if with_beta else None
    out = _out((rows, width))
    tile.tile_layernorm_affine_f32(_placed(x), _placed(r) if residual else None, _placed(g),
                                   _placed(b) if with_beta else None, out, EPS)
    ref = oracle.get().layernorm_affine(x, g, b, r=r, eps=ref_eps())
    _check_bound(out.cpu().numpy(), ref, ATOL_AFFINE, f"affine LN {rows}x{width}")


@pytest.mark.parametrize("rows,width", SHAPES)
def test_rmsnorm_weighted(rows, width):
    x = synth.rows_of(3, rows, width, which="x")
    g, _ = _gamma_beta(width)
    out = _out((rows, width))
    tile.tile_rmsnorm_weighted_f32(_placed(x), _placed(g), out, EPS)
    ref = oracle.get().rmsnorm_weighted(x, g, eps=ref_eps())
    _check_bound(out.cpu().numpy(), ref, ATOL, f"weighted RMSNorm {rows}x{width}")


@pytest.mark.parametrize("x_off,g_off", [(1, 0), (0, 1), (2, 3), (3, 3)])
def test_affine_with_unaligned_rows_and_vectors(x_off, g_off):
    """Row starts and gamma/beta at different 16-byte phases take the scalar
    gamma/beta loads; ragged widths give every row a different phase."""
    for rows, width in [(9, 1537), (4, 4099), (3, 258)]:
        x = synth.rows_of(3, rows, width, which="x")
        r = synth.rows_of(3, rows, width, which="r")
        g, b = _gamma_beta(width)
        out = _out((rows, width), x_off)
        tile.tile_layernorm_affine_f32(_placed(x, x_off), _placed(r, x_off), _placed(g, g_off),
                                       _placed(b, g_off), out, EPS)
        ref = oracle.get().layernorm_affine(x, g, b, r=r, eps=ref_eps())
        _check_bound(out.cpu().numpy(), ref, ATOL_AFFINE, f"affine LN offsets {x_off}/{g_off}")
        out = _out((rows, width), x_off)
        tile.tile_rmsnorm_weighted_f32(_placed(x, x_off), _placed(g, g_off), out, EPS)
        ref = oracle.get().rmsnorm_weighted(x, g, eps=ref_eps())
        _check_bound(out.cpu().numpy(), ref, ATOL, f"weighted RMS offsets {x_off}/{g_off}")


def test_affine_with_unit_gamma_matches_the_plain_ops_bitwise():
    """gamma = 1, beta = 0 on the same plan gives the plain op's bits."""
    x = synth.rows_of(3, 33, 4096, which="x")
    ones = np.ones(4096, np.float32)
    zeros = np.zeros(4096, np.float32)
    tx = _placed(x)
    for plain, affine in (("layernorm", "layernorm_affine"), ("rmsnorm", "rmsnorm_weighted")):
        pid = tile.tile_describe_plan(plain, 33, 4096)["id"]
        a = _out((33, 4096))
        b = _out((33, 4096))
        tile.tile_run_plan_args_f32(affine, pid, tx, a, gamma=_placed(ones),
                                    beta=_placed(zeros) if affine == "layernorm_affine" else None,
                                    eps=EPS)
        tile.tile_run_plan_args_f32(plain, pid, tx, b, eps=EPS)
        assert torch.equal(a, b)


# ---------------------------------------------------------------------------
# row sum and paired min/max
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("rows,width", SHAPES + [(3, 131072), (1000, 1)])
@pytest.mark.parametrize("offset", [0, 1])
def test_row_sum(rows, width, offset):
    x = synth.rows_of(3, rows, width, which="x")
    sums = _out((rows,))
    tile.tile_row_sum_f32(_placed(x, offset), sums)
    _check_bound(sums.cpu().numpy(), oracle.get().row_sum(x), ATOL, f"row sum {rows}x{width}")


def test_row_sum_with_cancellation():
    """Rows whose terms cancel: x, then -x reversed, then a small tail; the
    exact sum is the tail's.  An uncompensated FP32 sum misses it badly."""
    rows, width = 8, 8192
    half = synth.uniform_pm1(3100, rows * 4000).reshape(rows, 4000) * np.float32(1000.0)
    tail = synth.uniform_pm1(3101, rows * 192).reshape(rows, 192) * np.float32(1e-3)
    x = np.concatenate([half, -half[:, ::-1], tail], axis=1)
    sums = _out((rows,))
    tile.tile_row_sum_f32(_placed(x), sums)
    _check_bound(sums.cpu().numpy(), oracle.get().row_sum(x), ATOL, "row sum cancellation")


@pytest.mark.parametrize("rows,width", SHAPES + [(3, 131072), (1000, 1)])
@pytest.mark.parametrize("offset", [0, 3])
def test_row_minmax_exact(rows, width, offset):
    x = synth.rows_of(4 if width in (8192, 65536) else 3, rows, width, which="x")
    mins, maxs = _out((rows,)), _out((rows,))
    tile.tile_row_minmax_f32(_placed(x, offset), mins, maxs)
    mn, mx = oracle.get().row_minmax(x)
    assert np.array_equal(mins.cpu().numpy().astype(np.float64), mn)
    assert np.array_equal(maxs.cpu().numpy().astype(np.float64), mx)


# ---------------------------------------------------------------------------
# every built plan for the new row ops
# ---------------------------------------------------------------------------

def _plan_cases():
    from tile_compiler_row_gb300 import _build
    _build.build()
    cases = []
    for pid in range(tile.tile_plan_count()):
        info = tile.tile_plan_info(pid, 0, 1, 1)
        if info is None:          # staged plans: tests/test_staged_gpu.py
            continue
        maxw = info["max_width"]
        rows = 3 if maxw > 16384 else 2 * info["programs_per_cta"] + 1
        widths = sorted({1, 5, min(maxw, 37), maxw})
        for op in ("row_sum", "row_minmax", "layernorm_affine", "rmsnorm_weighted"):
            cases.append((pid, op, rows, widths, info["vec"]))
    return cases


@pytest.mark.parametrize("pid,op,rows,widths,vec", _plan_cases(),
                         ids=lambda v: str(v) if not isinstance(v, list) else "w")
def test_every_plan_new_ops(pid, op, rows, widths, vec):
    orc = oracle.get()
    for w in widths:
        x = synth.rows_of(3, rows, w, which="x")
        g, b = _gamma_beta(w)
        for off in (0, 1):
            tx = _placed(x, off)
            if op == "row_sum":
                out = _out((rows,))
                tile.tile_run_plan_args_f32(op, pid, tx, out)
                _check_bound(out.cpu().numpy(), orc.row_sum(x), ATOL, f"plan {pid} sum w={w}")
            elif op == "row_minmax":
                mn_t, mx_t = _out((rows,)), _out((rows,))
                tile.tile_run_plan_args_f32(op, pid, tx, mn_t, out2=mx_t)
                mn, mx = orc.row_minmax(x)
                assert np.array_equal(mn_t.cpu().numpy().astype(np.float64), mn)
                assert np.array_equal(mx_t.cpu().numpy().astype(np.float64), mx)
            else:
                out = _out((rows, w), off if vec == 4 else (off + 1) % 4)
                if op == "layernorm_affine":
                    r = synth.rows_of(3, rows, w, which="r")
                    tile.tile_run_plan_args_f32(op, pid, tx, out, residual=_placed(r, off),
                                                gamma=_placed(g), beta=_placed(b), eps=EPS)
                    ref = orc.layernorm_affine(x, g, b, r=r, eps=ref_eps())
                    _check_bound(out.cpu().numpy(), ref, ATOL_AFFINE, f"plan {pid} affine w={w}")
                else:
                    tile.tile_run_plan_args_f32(op, pid, tx, out, gamma=_placed(g), eps=EPS)
                    ref = orc.rmsnorm_weighted(x, g, eps=ref_eps())
                    _check_bound(out.cpu().numpy(), ref, ATOL, f"plan {pid} weighted w={w}")


# ---------------------------------------------------------------------------
# pointwise value/derivative pairs
# ---------------------------------------------------------------------------

PAIR_SHAPES = [(1, 127), (37, 1537), (1024, 4096), (4096, 4096)]


@pytest.mark.parametrize("kind", ["sigmoid", "gelu_tanh"])
@pytest.mark.parametrize("rows,width", PAIR_SHAPES)
def test_pairs_uniform(kind, rows, width):
    x = synth.rows_of(3, rows, width, which="x")
    y, dy = _out((rows, width)), _out((rows, width))
    getattr(tile, f"tile_{kind}_pair_f32")(_placed(x), y, dy)
    ref_y, ref_dy = getattr(oracle.get(), f"{kind}_pair")(x)
    _check_bound(y.cpu().numpy(), ref_y, ATOL, f"{kind} value {rows}x{width}")
    _check_bound(dy.cpu().numpy(), ref_dy, ATOL, f"{kind} derivative {rows}x{width}")


@pytest.mark.parametrize("kind", ["sigmoid", "gelu_tanh"])
def test_pairs_wide_range_and_offsets(kind):
    """N(0, 8^2) values (saturated tails on both sides) and the three
    pointers at different 16-byte phases."""
    n = 100003
    x = synth.normal(3200, n, 8.0)
    x[:4] = [0.0, -0.0, 80.0, -80.0]
    ref_y, ref_dy = getattr(oracle.get(), f"{kind}_pair")(x)
    for xo, yo, do in [(0, 0, 0), (1, 1, 1), (0, 1, 2), (3, 0, 0)]:
        y, dy = _out((n,), yo), _out((n,), do)
        getattr(tile, f"tile_{kind}_pair_f32")(_placed(x, xo), y, dy)
        _check_bound(y.cpu().numpy(), ref_y, ATOL, f"{kind} value offsets {xo}{yo}{do}")
        _check_bound(dy.cpu().numpy(), ref_dy, ATOL, f"{kind} derivative offsets {xo}{yo}{do}")


def test_pairs_empty_is_a_noop():
    x = torch.empty(0, device="cuda")
    tile.tile_sigmoid_pair_f32(x, torch.empty(0, device="cuda"), torch.empty(0, device="cuda"))
