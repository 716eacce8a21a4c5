"""GPU parity of the FP16 (IEEE binary16) row operations against the FP64
oracle.

Inputs are the seeded FP32 workloads rounded to FP16; the oracle receives
those FP16 values exactly (widened to FP32).  The kernels compute in FP32 and
round each output to nearest-even FP16, so the bound is the FP32 one plus
half an FP16 ulp (at most 2^-11 |ref|):

    |y - ref| <= 2e-6 + (2e-5 + 2^-11) |ref|

and, sharper, every output with |ref| > 1e-2 is round_f16(ref) except where
ref lies within the FP32 tolerance (2e-6 + 2e-5 |ref|) of the rounding
boundary between two FP16 neighbours: only there can an FP32 result inside
its tolerance round either way, and the output must then be one of those
two neighbours."""

from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
import synth
import tile_compiler_row_gb300 as tile
from parity import ATOL, EPS, RTOL, ref_eps, expects_staged

pytestmark = pytest.mark.gpu

F16_HALF_ULP_REL = 2.0 ** -11


@pytest.fixture(scope="module", autouse=True)
def device():
    from tile_compiler_row_gb300 import _build
    _build.build()
    torch.cuda.set_device(0)
    yield
    assert tile.tile_check_device_status() == 0


def _f16_rows(cfg, rows, width, which="x"):
    """(f16 CUDA tensor, its exact FP32 values on the host)."""
    t = torch.from_numpy(synth.rows_of(cfg, rows, width, which=which)).to(torch.float16)
    return t, t.float().numpy()


def _placed(t, offset=0):
    buf = torch.empty(t.numel() + 16, dtype=t.dtype, device="cuda")
    view = buf[offset:offset + t.numel()].view(t.shape)
    view.copy_(t)
    return view


def _round_f16(ref):
    """Round-to-nearest-even FP16 of FP64 values (numpy's binary16)."""
    return np.asarray(ref, np.float64).astype(np.float16).astype(np.float64)


def check_f16(got_t, ref, atol=ATOL, what=""):
    got = got_t.float().cpu().numpy().astype(np.float64)
    assert got.shape == ref.shape, what
    assert np.all(np.isfinite(got)), what
    err = np.abs(got - ref)
    bound = atol + (RTOL + F16_HALF_ULP_REL) * np.abs(ref)
    assert np.all(err <= bound), f"{what}: max err {err.max():.3e}"
    # Rounding checks where the FP16 spacing dwarfs the FP32 error (|ref| >
    # 1e-2: half an FP16 ulp is >= 3.8e-6 there, the FP32 error about 1e-8);
    # for smaller outputs the FP32 error can reach an FP16 ulp of the output.
    big = np.abs(ref) > 1e-2
    rn = _round_f16(ref[big])
    ulp = 2.0 ** (np.floor(np.log2(np.abs(rn))) - 10)
    assert np.all(np.abs(got[big] - rn) <= ulp), \
        f"{what}: an output is more than one FP16 ulp from the rounded reference"
    mis = got[big] != rn
    if mis.any():
        g, rr, rf = got[big][mis], rn[mis], ref[big][mis]
        boundary = (g + rr) / 2          # neighbours: their midpoint is the tie
        assert np.all(np.abs(rf - boundary) <= ATOL + RTOL * np.abs(rf)), \
            f"{what}: an output rounds away from round_f16(ref) far from a rounding boundary"


SHAPES = [(1, 127), (17, 257), (7, 1537), (64, 4096), (1024, 4096), (128, 8192), (32, 65536)]


@pytest.mark.parametrize("rows,width", SHAPES)
@pytest.mark.parametrize("op", ["residual_layernorm", "layernorm", "rmsnorm", "softmax"])
def test_f16_ops(op, rows, width):
    cfg = 4 if width in (8192, 65536) and op != "residual_layernorm" else 3
    x, xf = _f16_rows(cfg, rows, width)
    r, rf = _f16_rows(cfg, rows, width, "r")
    out = torch.empty(rows, width, dtype=torch.float16, device="cuda")
    tx = _placed(x)
    if op == "residual_layernorm":
        tile.tile_residual_layernorm_f16(tx, _placed(r), out, EPS)
        ref = oracle.get().residual_layernorm(xf, rf, ref_eps())
    else:
        getattr(tile, f"tile_{op}_f16")(tx, out, EPS)
        ref = oracle.get().run(op, xf, eps=ref_eps())
    check_f16(out, ref, what=f"f16 {op} {rows}x{width}")


@pytest.mark.parametrize("offset", [1, 3, 5, 7])
@pytest.mark.parametrize("op", ["residual_layernorm", "layernorm", "rmsnorm", "softmax"])
def test_f16_unaligned_rows(op, offset):
    for rows, width in [(5, 127), (3, 1537), (2, 4099)]:
        x, xf = _f16_rows(3, rows, width)
        r, rf = _f16_rows(3, rows, width, "r")
        buf = torch.empty(rows * width + 16, dtype=torch.float16, device="cuda")
        out = buf[offset:offset + rows * width].view(rows, width)
        if op == "residual_layernorm":
            tile.tile_residual_layernorm_f16(_placed(x, offset), _placed(r, offset), out, EPS)
            ref = oracle.get().residual_layernorm(xf, rf, ref_eps())
        else:
            getattr(tile, f"tile_{op}_f16")(_placed(x, offset), out, EPS)
            ref = oracle.get().run(op, xf, eps=ref_eps())
        check_f16(out, ref, what=f"f16 {op} offset {offset} {rows}x{width}")
        # different phases for input and output: the scalar plans
        out2 = torch.empty(rows, width, dtype=torch.float16, device="cuda")
        if op == "residual_layernorm":
            tile.tile_residual_layernorm_f16(_placed(x, offset), _placed(r, offset), out2, EPS)
        else:
            getattr(tile, f"tile_{op}_f16")(_placed(x, offset), out2, EPS)
        check_f16(out2, ref, what=f"f16 {op} mixed phases {rows}x{width}")


@pytest.mark.parametrize("rows,width", [(7, 1537), (64, 4096), (128, 8192)])
def test_f16_affine_and_weighted(rows, width):
    x, xf = _f16_rows(3, rows, width)
    r, rf = _f16_rows(3, rows, width, "r")
    g = synth.uniform_pm1(3001, width) * np.float32(2.0)
    b = synth.uniform_pm1(3002, width)
    tg, tb = torch.from_numpy(g).cuda(), torch.from_numpy(b).cuda()
    out = torch.empty(rows, width, dtype=torch.float16, device="cuda")
    tile.tile_layernorm_affine_f16(_placed(x), _placed(r), tg, tb, out, EPS)
    ref = oracle.get().layernorm_affine(xf, g, b, r=rf, eps=ref_eps())
    check_f16(out, ref, atol=1e-5, what=f"f16 affine {rows}x{width}")
    tile.tile_rmsnorm_weighted_f16(_placed(x), tg, out, EPS)
    ref = oracle.get().rmsnorm_weighted(xf, g, eps=ref_eps())
    check_f16(out, ref, what=f"f16 weighted {rows}x{width}")


@pytest.mark.parametrize("rows,width", [(17, 257), (64, 4096), (32, 65536), (1000, 1)])
def test_f16_row_sum_and_minmax(rows, width):
    x, xf = _f16_rows(3, rows, width)
    sums = torch.empty(rows, device="cuda")
    tile.tile_row_sum_f16(_placed(x, 1), sums)
    ref = oracle.get().row_sum(xf)
    got = sums.cpu().numpy().astype(np.float64)
    assert np.all(np.abs(got - ref) <= ATOL + RTOL * np.abs(ref))
    mins, maxs = torch.empty(rows, device="cuda"), torch.empty(rows, device="cuda")
    tile.tile_row_minmax_f16(_placed(x, 3), mins, maxs)
    mn, mx = oracle.get().row_minmax(xf)
    assert np.array_equal(mins.cpu().numpy().astype(np.float64), mn)
    assert np.array_equal(maxs.cpu().numpy().astype(np.float64), mx)


def _f16_plan_cases():
    from tile_compiler_row_gb300 import _build
    _build.build()
    out = []
    for pid in range(tile.tile_plan_count()):
        info = tile.tile_plan_info_ex(pid, 0, "f16", 1, 1)
        if info is None:
            continue
        maxw = info["max_width"]
        rows = 3 if maxw > 16384 else 2 * info["programs_per_cta"] + 1
        for op in ("residual_layernorm", "layernorm", "rmsnorm", "softmax"):
            out.append((pid, op, rows, sorted({1, 9, min(maxw, 77), maxw})))
    return out


@pytest.mark.parametrize("pid,op,rows,widths", _f16_plan_cases(),
                         ids=lambda v: str(v) if not isinstance(v, list) else "w")
def test_every_f16_plan(pid, op, rows, widths):
    for w in widths:
        x, xf = _f16_rows(3, rows, w)
        r, rf = _f16_rows(3, rows, w, "r")
        for off in (0, 3):
            out = _placed(torch.zeros(rows, w, dtype=torch.float16), off)
            tile.tile_run_plan_args_f32(op, pid, _placed(x, off), out,
                                        residual=_placed(r, off) if op == "residual_layernorm"
                                        else None, eps=EPS)
            ref = (oracle.get().residual_layernorm(xf, rf, ref_eps()) if op == "residual_layernorm"
                   else oracle.get().run(op, xf, eps=ref_eps()))
            check_f16(out, ref, what=f"f16 plan {pid} {op} w={w} off={off}")


@pytest.mark.parametrize("op", ["residual_layernorm", "layernorm", "rmsnorm", "softmax"])
@pytest.mark.parametrize("rows,width", [(2048, 4096), (1024, 8192), (1024, 12288),
                                        (512, 16384)])
def test_f16_selected_staged_plans(op, rows, width):
    """Large FP16 rows of whole vectors select a shared-memory-staged plan
    where it measured faster; the same rows one element off the 16-byte phase
    fall back to a register plan.  Both must meet the bound."""
    x, xf = _f16_rows(3, rows, width)
    r, rf = _f16_rows(3, rows, width, "r")
    ref = (oracle.get().residual_layernorm(xf, rf, ref_eps()) if op == "residual_layernorm"
           else oracle.get().run(op, xf, eps=ref_eps()))
    for off in (0, 1):
        buf = torch.empty(rows * width + 16, dtype=torch.float16, device="cuda")
        out = buf[off:off + rows * width].view(rows, width)
        if op == "residual_layernorm":
            tile.tile_residual_layernorm_f16(_placed(x, off), _placed(r, off), out, EPS)
        else:
            getattr(tile, f"tile_{op}_f16")(_placed(x, off), out, EPS)
        check_f16(out, ref, what=f"f16 {op} {rows}x{width} offset {off}")
    # the staged kernel exactly where the measured table takes it
    staged = expects_staged(op, rows, width)
    assert (tile.tile_describe_plan_ex(op, "f16", rows, width)["path"] == 2) == staged


@pytest.mark.parametrize("op", ["layernorm", "residual_layernorm"])
@pytest.mark.parametrize("rows,width", [(4, 257), (2048, 4096), (512, 16384)])
def test_f16_constant_rows_normalise_to_zero(op, rows, width):
    """Constant rows (the closed form gives LayerNorm output 0) on register
    and staged plans: every output within the absolute bound of 0."""
    vals = torch.tensor([0.1, 3.140625, -7.5, 1000.0, -20000.0], dtype=torch.float32)
    x = vals[torch.arange(rows) % len(vals)][:, None].expand(rows, width).contiguous()
    x = x.to(torch.float16).cuda()
    y = torch.full_like(x, float("nan"))
    if op == "residual_layernorm":
        r = torch.zeros_like(x)
        tile.tile_residual_layernorm_f16(x, r, y, EPS)
    else:
        tile.tile_layernorm_f16(x, y, EPS)
    torch.cuda.synchronize()
    got = y.float().cpu().numpy()
    assert np.all(np.abs(got) <= ATOL), f"{op} {rows}x{width}: max |y| {np.abs(got).max():.3e}"
