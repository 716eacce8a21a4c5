"""GPU parity past 2^31 elements: the kernels index rows with 64-bit offsets,
so a matrix of more than 2^31 elements (here 524305 x 4096 = 2^31 + 69632,
8 GiB per FP32 tensor) must work end to end.  The inputs are an integer hash
of the flat element index, filled on the GPU in row blocks and recomputed
exactly in numpy for the sampled rows, which sit on both sides of element
2^31 and at the ends of the matrix; those rows are checked against the FP64
oracle with the usual bound."""

from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
import tile_compiler_row_gb300 as tile
from parity import ATOL, EPS, RTOL, ref_eps

pytestmark = pytest.mark.gpu

ROWS, WIDTH = (1 << 19) + 17, 4096                 # 2^31 + 69632 elements
BOUNDARY_ROW = (1 << 31) // WIDTH                  # first row past element 2^31
SAMPLE = [0, 1, BOUNDARY_ROW - 1, BOUNDARY_ROW, BOUNDARY_ROW + 1, ROWS - 2, ROWS - 1]
MULT = 2654435761                                  # Knuth's multiplicative hash constant


@pytest.fixture(scope="module", autouse=True)
def device():
    from tile_compiler_row_gb300 import _build
    _build.build()
    torch.cuda.set_device(0)
    yield
    torch.cuda.empty_cache()
    assert tile.tile_check_device_status() == 0


def _fill(t, salt):
    """t[i][j] = hash(i * width + j): uniform on [-1, 1) over a 2^-23 grid,
    exact in FP32."""
    rows, width = t.shape
    step = 8192
    for r0 in range(0, rows, step):
        r1 = min(rows, r0 + step)
        idx = torch.arange(r0 * width, r1 * width, device="cuda", dtype=torch.int64)
        h = ((idx + salt) * MULT) & 0xFFFFFF
        t[r0:r1] = (h.to(torch.float32) / float(1 << 23) - 1.0).view(r1 - r0, width).to(t.dtype)
        del idx, h


def _host_rows(rows, width, salt):
    idx = (np.asarray(rows, np.int64)[:, None] * width + np.arange(width, dtype=np.int64)[None, :])
    h = ((idx + salt) * MULT) & 0xFFFFFF
    return (h.astype(np.float32) / np.float32(1 << 23) - np.float32(1.0)).astype(np.float32)


def _check(got, ref, what, extra_rel=0.0):
    got = np.asarray(got, np.float64)
    err = np.abs(got - ref)
    bound = ATOL + (RTOL + extra_rel) * np.abs(ref)
    assert np.all(np.isfinite(got)), what
    assert np.all(err <= bound), f"{what}: max err {err.max():.3e}"


@pytest.mark.parametrize("op", ["residual_layernorm", "layernorm", "rmsnorm", "softmax"])
def test_fp32_rows_past_2_31_elements(op):
    assert ROWS * WIDTH > (1 << 31)
    x = torch.empty(ROWS, WIDTH, device="cuda")
    _fill(x, 11)
    r = None
    if op == "residual_layernorm":
        r = torch.empty_like(x)
        _fill(r, 23)
    y = torch.full_like(x, float("nan"))
    tile.run(op, x, r, y, EPS)
    torch.cuda.synchronize()
    got = y[SAMPLE].cpu().numpy()
    xh = _host_rows(SAMPLE, WIDTH, 11)
    assert np.array_equal(x[SAMPLE].cpu().numpy(), xh)        # the generators agree
    orc = oracle.get()
    if op == "residual_layernorm":
        ref = orc.residual_layernorm(xh, _host_rows(SAMPLE, WIDTH, 23), ref_eps())
    else:
        ref = orc.run(op, xh, eps=ref_eps())
    _check(got, ref, f"{op} {ROWS}x{WIDTH}")
    assert not torch.isnan(y[-1]).any() and not torch.isnan(y[0]).any()
    del x, r, y


def test_bf16_residual_layernorm_past_2_31_elements():
    """The selector takes the shared-memory-staged kernel for this shape."""
    assert tile.tile_describe_plan_ex("residual_layernorm", "bf16", ROWS, WIDTH)["path"] == 2
    x = torch.empty(ROWS, WIDTH, device="cuda", dtype=torch.bfloat16)
    r = torch.empty_like(x)
    _fill(x, 11)
    _fill(r, 23)
    y = torch.empty_like(x)
    tile.tile_residual_layernorm_bf16(x, r, y, EPS)
    torch.cuda.synchronize()
    xh = x[SAMPLE].float().cpu().numpy()
    rh = r[SAMPLE].float().cpu().numpy()
    ref = oracle.get().residual_layernorm(xh, rh, ref_eps())
    _check(y[SAMPLE].float().cpu().numpy(), ref, "bf16 residual LayerNorm", 2.0 ** -8)
    del x, r, y


def test_pairs_past_2_31_elements():
    n = (1 << 31) + 5
    x = torch.empty(n, device="cuda")
    # filled as rows of 4096, the last 5 elements (past the rows) from numpy
    body = x[: (n // WIDTH) * WIDTH].view(-1, WIDTH)
    _fill(body, 37)
    tail_idx = np.arange((n // WIDTH) * WIDTH, n, dtype=np.int64)
    tail = ((((tail_idx + 37) * MULT) & 0xFFFFFF).astype(np.float32) / np.float32(1 << 23)
            - np.float32(1.0))
    x[(n // WIDTH) * WIDTH:] = torch.from_numpy(tail).cuda()
    y = torch.empty_like(x)
    dy = torch.empty_like(x)
    tile.tile_sigmoid_pair_f32(x, y, dy)
    torch.cuda.synchronize()
    picks = np.array([0, 1, (1 << 31) - 1, 1 << 31, (1 << 31) + 1, n - 1], np.int64)
    xs = x[torch.from_numpy(picks).cuda()].cpu().numpy()
    vy, vd = oracle.get().sigmoid_pair(xs)
    _check(y[torch.from_numpy(picks).cuda()].cpu().numpy(), vy, "sigmoid value")
    _check(dy[torch.from_numpy(picks).cuda()].cpu().numpy(), vd, "sigmoid derivative")
    del x, y, dy
