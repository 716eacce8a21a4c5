"""GPU invariants that need no oracle: permutation equivariance within a row,
shift invariance of softmax and LayerNorm, the symmetry of residual
LayerNorm in (x, r), and residual LayerNorm with r = 0 being LayerNorm.

Exact identities are checked bit for bit: softmax of x + k on inputs whose
binary grid keeps x + k exact (then (x + k) - max(x + k) = x - max x), and
residual LayerNorm's x + r = r + x.  Identities that change the reduction
order (a permuted row, a shifted mean) are checked within twice the oracle
bound, 2 (2e-6 + 2e-5 |y|)."""

from __future__ import annotations

import numpy as np
import pytest
import torch

import synth
import tile_compiler_row_gb300 as tile
from parity import ATOL, EPS, RTOL

pytestmark = pytest.mark.gpu

OPS = ("residual_layernorm", "layernorm", "rmsnorm", "softmax")
SHAPES = [(33, 257), (64, 4096), (8, 1537)]


@pytest.fixture(scope="module", autouse=True)
def device():
    from tile_compiler_row_gb300 import _build
    _build.build()
    torch.cuda.set_device(0)
    yield
    assert tile.tile_check_device_status() == 0


def _run(op, x, r=None):
    y = torch.empty_like(x)
    tile.run(op, x, r, y, EPS)
    torch.cuda.synchronize()
    return y


def _close(a, b, what):
    a = a.double().cpu().numpy()
    b = b.double().cpu().numpy()
    bound = 2 * (ATOL + RTOL * np.abs(b))
    assert np.all(np.abs(a - b) <= bound), f"{what}: max diff {np.abs(a - b).max():.3e}"


@pytest.mark.parametrize("op", OPS)
@pytest.mark.parametrize("rows,width", SHAPES)
def test_permutation_equivariance(op, rows, width):
    x = torch.from_numpy(synth.rows_of(3, rows, width, which="x")).cuda()
    r = torch.from_numpy(synth.rows_of(3, rows, width, which="r")).cuda() \
        if op == "residual_layernorm" else None
    g = torch.Generator().manual_seed(rows * 7 + width)
    perm = torch.randperm(width, generator=g).cuda()
    y = _run(op, x, r)
    yp = _run(op, x[:, perm].contiguous(), r[:, perm].contiguous() if r is not None else None)
    _close(yp, y[:, perm], f"{op} {rows}x{width} permuted")


@pytest.mark.parametrize("rows,width", SHAPES + [(128, 8192), (4, 65536)])
@pytest.mark.parametrize("k", [8.0, -4.0, 1024.0])
def test_softmax_shift_is_exact_on_a_coarse_grid(rows, width, k):
    # inputs on a 2^-10 grid in [-1, 1): x + k stays exact in FP32
    x = torch.from_numpy(synth.rows_of(3, rows, width, which="x")).cuda()
    x = torch.round(x * 1024.0) / 1024.0
    assert torch.equal((x + k) - k, x)
    y = _run("softmax", x)
    ys = _run("softmax", x + k)
    assert torch.equal(y, ys), f"softmax {rows}x{width} shifted by {k}"


@pytest.mark.parametrize("op", ["layernorm", "residual_layernorm"])
@pytest.mark.parametrize("rows,width", SHAPES)
def test_layernorm_shift_invariance(op, rows, width):
    x = torch.from_numpy(synth.rows_of(3, rows, width, which="x")).cuda()
    x = torch.round(x * 1024.0) / 1024.0
    r = torch.from_numpy(synth.rows_of(3, rows, width, which="r")).cuda() \
        if op == "residual_layernorm" else None
    if r is not None:
        r = torch.round(r * 1024.0) / 1024.0
    y = _run(op, x, r)
    ys = _run(op, x + 16.0, r)
    _close(ys, y, f"{op} {rows}x{width} shifted by 16")


@pytest.mark.parametrize("rows,width", SHAPES)
def test_residual_layernorm_is_symmetric(rows, width):
    x = torch.from_numpy(synth.rows_of(3, rows, width, which="x")).cuda()
    r = torch.from_numpy(synth.rows_of(3, rows, width, which="r")).cuda()
    assert torch.equal(_run("residual_layernorm", x, r), _run("residual_layernorm", r, x))


@pytest.mark.parametrize("rows,width", SHAPES)
def test_residual_layernorm_with_zero_residual_is_layernorm(rows, width):
    x = torch.from_numpy(synth.rows_of(3, rows, width, which="x")).cuda()
    pid = tile.tile_describe_plan("layernorm", rows, width)["id"]
    a, b = torch.empty_like(x), torch.empty_like(x)
    tile.tile_run_plan_f32("layernorm", pid, x, None, a, EPS)
    tile.tile_run_plan_f32("residual_layernorm", pid, x, torch.zeros_like(x), b, EPS)
    torch.cuda.synchronize()
    assert torch.equal(a, b)
