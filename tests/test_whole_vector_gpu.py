"""The whole-vector kernel forms against the general ones, bit for bit.

2-byte rows that are 16-byte aligned and hold whole 16-byte vectors run a
form of the register row kernel without a scalar head and tail (and
LayerNorm backward on the S = 4, P = 1, K = 4 shape a raw backward kernel
without one).  A head and tail of no elements add exact +0 terms, which
can change only the sign of a partial sum that is exactly -0; none is on
these random rows, so the results must be bitwise those of the general
form.  The test hook
tile_test_force_general_kernels makes the same calls take the general form,
and every output of both runs is compared with torch.equal, for every
forward op on forced register plans (packed, single-row and cluster plans)
and for LayerNorm backward with gamma and row statistics."""

from __future__ import annotations

import pytest
import torch

import synth
import tile_compiler_row_gb300 as tile

pytestmark = pytest.mark.gpu

TYPES = {"bf16": torch.bfloat16, "f16": torch.float16}
OPS = ("residual_layernorm", "layernorm", "rmsnorm", "softmax", "row_sum", "row_minmax",
       "layernorm_affine", "rmsnorm_weighted")
# (rows, width) of whole 16-byte vectors, and register plans to force there
CASES = [((64, 4096), (6, 5, 8)), ((17, 1024), (2, 4)), ((300, 2048), (4, 39)),
         ((9, 8192), (8, 10)), ((3, 65536), (19, 33))]


@pytest.fixture(scope="module", autouse=True)
def device():
    from tile_compiler_row_gb300 import _build
    _build.build()
    torch.cuda.set_device(0)
    yield
    tile.tile_test_force_general_kernels(False)
    assert tile.tile_check_device_status() == 0


def _inputs(rows, width, dt):
    x = torch.from_numpy(synth.rows_of(3, rows, width, which="x")).to(TYPES[dt]).cuda()
    r = torch.from_numpy(synth.rows_of(3, rows, width, which="r")).to(TYPES[dt]).cuda()
    g = torch.from_numpy(synth.uniform_pm1(3001, width) * 2).cuda()
    b = torch.from_numpy(synth.uniform_pm1(3002, width)).cuda()
    return x, r, g, b


def _forced(op, pid, x, r, g, b):
    rows = x.shape[0]
    if op in ("row_sum", "row_minmax"):
        out = torch.full((rows,), float("nan"), device="cuda")
        out2 = torch.full((rows,), float("nan"), device="cuda") if op == "row_minmax" else None
    else:
        out, out2 = torch.full_like(x, float("nan")), None
    tile.tile_run_plan_args_f32(
        op, pid, x, out, residual=r if op == "residual_layernorm" else None,
        gamma=g if op in ("layernorm_affine", "rmsnorm_weighted") else None,
        beta=b if op == "layernorm_affine" else None, out2=out2)
    torch.cuda.synchronize()
    return out, out2


@pytest.mark.parametrize("dt", ["bf16", "f16"])
@pytest.mark.parametrize("shape,plans", CASES)
def test_forward_whole_vector_form_is_bitwise_the_general_form(dt, shape, plans):
    rows, width = shape
    x, r, g, b = _inputs(rows, width, dt)
    ran = 0
    for op in OPS:
        for pid in plans:
            info = tile.tile_plan_info_ex(pid, op, dt, rows, width)
            if info is None or info["path"] not in (0, 1):     # register or cluster plans
                continue
            tile.tile_test_force_general_kernels(False)
            a1, a2 = _forced(op, pid, x, r, g, b)
            tile.tile_test_force_general_kernels(True)
            g1, g2 = _forced(op, pid, x, r, g, b)
            tile.tile_test_force_general_kernels(False)
            assert torch.equal(a1, g1), f"{op} {dt} {rows}x{width} plan {pid}"
            if a2 is not None:
                assert torch.equal(a2, g2), f"{op} {dt} {rows}x{width} plan {pid} (second output)"
            ran += 1
    assert ran >= len(OPS)


@pytest.mark.parametrize("dt", ["bf16", "f16"])
@pytest.mark.parametrize("rows", [1, 64, 257])
def test_layernorm_backward_whole_vector_form_is_bitwise_the_general_form(dt, rows):
    width = 4096                      # plan 6's shape: the whole-vector backward kernel
    assert tile.tile_describe_backward_plan("layernorm", dt, rows, width)["id"] == 6
    x, dy, g, _ = _inputs(rows, width, dt)
    outs = []
    for force in (False, True):
        tile.tile_test_force_general_kernels(force)
        dx = torch.full_like(x, float("nan"))
        stats = torch.full((2 * rows,), float("nan"), device="cuda")
        getattr(tile, f"tile_layernorm_backward_{dt}")(x, g, dy, dx, stats)
        torch.cuda.synchronize()
        outs.append((dx, stats))
    tile.tile_test_force_general_kernels(False)
    assert torch.equal(outs[0][0], outs[1][0])
    assert torch.equal(outs[0][1], outs[1][1])
