"""GPU parity of the plans that need 16-byte aligned rows of whole vectors
against the FP64 oracle: the shared-memory-staged plans (bulk row copies
into a ring of shared-memory stages, persistent CTAs) and the
R-rows-per-CTA plans (each thread owning the same columns of R rows).

Row counts are chosen so every staged CTA walks several times round its
ring of stages (stage reuse, barrier phase flips) and so the last R-row CTA
replays a row.  Bounds as for the register plans: 2e-6 + 2e-5 |ref| (affine
LayerNorm atol 1e-5), BF16 and FP16 outputs plus half an ulp of their type.
Anything but aligned rows of whole vectors is rejected with TILE_ERR_PLAN.
An R-row plan gives bitwise the results of the register plan with the same
warps and vectors per row."""

from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
import synth
import tile_compiler_row_gb300 as tile
from parity import ATOL, EPS, RTOL, ref_eps

pytestmark = pytest.mark.gpu

HALF_ULP_REL = {"f32": 0.0, "bf16": 2.0 ** -8, "f16": 2.0 ** -11}


@pytest.fixture(scope="module", autouse=True)
def device():
    from tile_compiler_row_gb300 import _build
    _build.build()
    torch.cuda.set_device(0)
    yield
    assert tile.tile_check_device_status() == 0


def _staged_plans():
    from tile_compiler_row_gb300 import _build
    _build.build()
    out = []
    for pid in range(tile.tile_plan_count()):
        info = tile.tile_plan_info(pid, 0, 1, 8)
        if info is not None and info["path"] in (2, 3):
            out.append(pid)
    return out


STAGED = _staged_plans()
OPS = ("residual_layernorm", "layernorm", "rmsnorm", "softmax", "layernorm_affine",
       "rmsnorm_weighted")


def _reference(op, x, r, g, b):
    orc = oracle.get()
    if op == "residual_layernorm":
        return orc.residual_layernorm(x, r, ref_eps())
    if op == "layernorm_affine":
        return orc.layernorm_affine(x, g, b, r=r, eps=ref_eps())
    if op == "rmsnorm_weighted":
        return orc.rmsnorm_weighted(x, g, eps=ref_eps())
    return orc.run(op, x, eps=ref_eps())


@pytest.mark.parametrize("dtype", ["f32", "bf16", "f16"])
@pytest.mark.parametrize("op", OPS)
@pytest.mark.parametrize("pid", STAGED)
def test_staged_plan(pid, op, dtype):
    info = tile.tile_plan_info_ex(pid, 0, dtype, 1, 8)
    if info is None:                      # R-row plan not built for this type
        assert tile.tile_plan_info(pid, 0, 1, 8)["path"] == 3
        return
    assert info["path"] in (2, 3)
    ev = info["vec"]
    cap = info["max_width"]
    tdt = {"f32": torch.float32, "bf16": torch.bfloat16, "f16": torch.float16}[dtype]
    for width in sorted({ev, 256, cap // 2, cap}):
        rows = 20001 if width <= 512 else 3001      # odd: an R-row CTA replays a row
        x = torch.from_numpy(synth.rows_of(3, rows, width, which="x")).to(tdt)
        r = torch.from_numpy(synth.rows_of(3, rows, width, which="r")).to(tdt)
        xf, rf = x.float().numpy(), r.float().numpy()
        g = synth.uniform_pm1(3001, width) * np.float32(2.0)
        b = synth.uniform_pm1(3002, width)
        with_res = op in ("residual_layernorm", "layernorm_affine")
        out = torch.full((rows, width), float("nan"), dtype=tdt, device="cuda")
        tile.tile_run_plan_args_f32(
            op, pid, x.cuda(), out, residual=r.cuda() if with_res else None,
            gamma=torch.from_numpy(g).cuda() if op in ("layernorm_affine", "rmsnorm_weighted")
            else None,
            beta=torch.from_numpy(b).cuda() if op == "layernorm_affine" else None, eps=EPS)
        ref = _reference(op, xf, rf if with_res else None, g, b)
        got = out.float().cpu().numpy().astype(np.float64)
        atol = 1e-5 if op == "layernorm_affine" else ATOL
        rtol = RTOL + HALF_ULP_REL[dtype]
        err = np.abs(got - ref)
        bad = ~(err <= atol + rtol * np.abs(ref))
        assert not bad.any(), (f"staged plan {pid} {op} {dtype} {rows}x{width}: "
                               f"{int(bad.sum())} beyond the bound, max err {np.nanmax(err):.3e}")
    assert tile.tile_check_device_status() == 0


def test_staged_plans_reject_unaligned_rows_and_partial_vectors():
    pid = STAGED[0]
    x = torch.zeros(4 * 256 + 8, device="cuda")
    out = torch.zeros(4 * 256 + 8, device="cuda")
    with pytest.raises(tile.TileError) as e:            # rows not 16-byte aligned
        tile.tile_run_plan_args_f32("rmsnorm", pid, x[1:1 + 1024].view(4, 256),
                                    out[1:1 + 1024].view(4, 256))
    assert e.value.status == -8
    with pytest.raises(tile.TileError) as e:            # width not whole vectors
        tile.tile_run_plan_args_f32("rmsnorm", pid, x[:4 * 254].view(4, 254),
                                    out[:4 * 254].view(4, 254))
    assert e.value.status == -8
    assert tile.tile_plan_info(pid, "rmsnorm", 4, 254) is None


def test_staged_results_are_deterministic():
    pid = STAGED[-1]
    x = torch.from_numpy(synth.rows_of(3, 5000, 1024, which="x")).cuda()
    a = torch.empty_like(x)
    b = torch.empty_like(x)
    tile.tile_run_plan_args_f32("layernorm", pid, x, a, eps=EPS)
    tile.tile_run_plan_args_f32("layernorm", pid, x, b, eps=EPS)
    assert torch.equal(a, b)


@pytest.mark.parametrize("op,dtype,pid", [("layernorm", "bf16", 45),
                                          ("residual_layernorm", "f32", 41)])
def test_staged_wait_runs_out_and_the_next_call_is_correct(op, dtype, pid):
    """The bounded wait made to run out, with no fault: through the test
    entry point no CTA issues the copy of its first row, and waits give up
    after 4096 polls.  Every CTA (4096 rows: several rows, and so several
    copies in flight, per CTA) times out on its first row, stops copying,
    drains the copies it did issue and returns.  The device status word then
    reports the error once (read and cleared by tile_check_device_status),
    and a normal call of the same plan on the same buffers is correct."""
    import time
    rows, width = 4096, 4096
    tdt = {"f32": torch.float32, "bf16": torch.bfloat16}[dtype]
    x = torch.from_numpy(synth.rows_of(3, rows, width, which="x")).to(tdt)
    r = torch.from_numpy(synth.rows_of(3, rows, width, which="r")).to(tdt)
    xf, rf = x.float().numpy(), r.float().numpy()
    with_res = op == "residual_layernorm"
    xd, rd = x.cuda(), (r.cuda() if with_res else None)
    out = torch.full((rows, width), float("nan"), dtype=tdt, device="cuda")
    assert tile.tile_check_device_status() == 0
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    tile.tile_test_staged_wait_timeout(op, pid, xd, out, 4096, residual=rd, eps=EPS)
    torch.cuda.synchronize()
    assert time.perf_counter() - t0 < 30.0
    assert tile.tile_check_device_status() == -9          # TILE_ERR_DEVICE, then cleared
    assert tile.tile_check_device_status() == 0
    out.fill_(float("nan"))
    tile.tile_run_plan_args_f32(op, pid, xd, out, residual=rd, eps=EPS)
    ref = _reference(op, xf, rf if with_res else None, None, None)
    got = out.float().cpu().numpy().astype(np.float64)
    err = np.abs(got - ref)
    bad = ~(err <= ATOL + (RTOL + HALF_ULP_REL[dtype]) * np.abs(ref))
    assert not bad.any(), f"{int(bad.sum())} beyond the bound after the timed-out launch"
    assert tile.tile_check_device_status() == 0


def test_staged_wait_hook_rejects_register_plans():
    x = torch.zeros(4, 256, device="cuda")
    out = torch.zeros(4, 256, device="cuda")
    with pytest.raises(tile.TileError) as e:
        tile.tile_test_staged_wait_timeout("rmsnorm", 7, x, out, 16)
    assert e.value.status == -8


def _register_twin(pid):
    """The register plan with the same warps and vectors per row as R-row
    plan `pid` (one CTA or program per row), or None."""
    info = tile.tile_plan_info(pid, 0, 1, 8)
    for q in range(tile.tile_plan_count()):
        other = tile.tile_plan_info(q, 0, 1, 8)
        if (other is not None and other["path"] == 0 and other["vec"] == 4
                and other["warps_per_program"] == info["warps_per_program"]
                and other["chunks"] == info["chunks"]):
            return q
    return None


# R-row plans that have a register plan with the same warps and vectors
# per row (all but S = 16, K = 1)
ROWS_PLANS = [pid for pid in STAGED if tile.tile_plan_info(pid, 0, 1, 8)["path"] == 3
              and _register_twin(pid) is not None]


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("pid", ROWS_PLANS)
def test_rows_plan_is_bitwise_its_register_twin(pid, dtype):
    twin = _register_twin(pid)
    assert tile.tile_plan_info_ex(pid, 0, dtype, 1, 8) is not None
    assert tile.tile_plan_info_ex(twin, 0, dtype, 1, 8) is not None
    tdt = {"f32": torch.float32, "bf16": torch.bfloat16}[dtype]
    cap = min(tile.tile_plan_info_ex(pid, 0, dtype, 1, 8)["max_width"],
              tile.tile_plan_info_ex(twin, 0, dtype, 1, 8)["max_width"] // 8 * 8)
    rows, width = 999, cap
    x = torch.from_numpy(synth.rows_of(3, rows, width, which="x")).to(tdt).cuda()
    r = torch.from_numpy(synth.rows_of(3, rows, width, which="r")).to(tdt).cuda()
    g = torch.from_numpy(synth.uniform_pm1(3001, width) * np.float32(2.0)).cuda()
    b = torch.from_numpy(synth.uniform_pm1(3002, width)).cuda()
    for op in OPS:
        outs = []
        for plan in (pid, twin):
            out = torch.full((rows, width), float("nan"), dtype=tdt, device="cuda")
            tile.tile_run_plan_args_f32(
                op, plan, x, out,
                residual=r if op in ("residual_layernorm", "layernorm_affine") else None,
                gamma=g if op in ("layernorm_affine", "rmsnorm_weighted") else None,
                beta=b if op == "layernorm_affine" else None, eps=EPS)
            outs.append(out)
        assert torch.equal(outs[0], outs[1]), f"plan {pid} vs {twin}: {op} {dtype}"
    assert tile.tile_check_device_status() == 0


@pytest.mark.parametrize("rows", [1, 2, 3, 5])
@pytest.mark.parametrize("pid", [p for p in STAGED if tile.tile_plan_info(p, 0, 1, 8)["path"] == 3])
def test_rows_plan_with_fewer_rows_than_a_cta_holds(pid, rows):
    """R-row plans on row counts below and just above R: the replayed rows
    write nothing (sentinels past the output stay), the real rows match the
    oracle."""
    width = 256
    x = synth.rows_of(3, rows, width, which="x")
    buf = torch.full(((rows + 4) * width,), 7.0, device="cuda")
    out = buf[:rows * width].view(rows, width)
    tile.tile_run_plan_args_f32("layernorm", pid, torch.from_numpy(x).cuda(), out, eps=EPS)
    ref = oracle.get().layernorm(x, ref_eps())
    got = out.cpu().numpy().astype(np.float64)
    assert np.all(np.abs(got - ref) <= ATOL + RTOL * np.abs(ref))
    assert bool((buf[rows * width:] == 7.0).all())
    assert tile.tile_check_device_status() == 0
