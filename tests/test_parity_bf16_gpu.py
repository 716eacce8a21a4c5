"""GPU parity of the BF16 row operations against the FP64 oracle.

Inputs are the seeded FP32 workloads rounded to BF16; the oracle receives
those BF16 values exactly (widened to FP32).  The kernels compute in FP32 and
round each output to nearest-even BF16, so the bound is the FP32 one plus
half a BF16 ulp (at most 2^-8 |ref|):

    |y - ref| <= 2e-6 + (2e-5 + 2^-8) |ref|

and, sharper, every output with |ref| > 1e-2 is within one BF16 ulp of
round_bf16(ref) and at least 99.9 % of them equal it (there the FP32 error is
far below the BF16 spacing, so only outputs next to a rounding boundary may
differ)."""

from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
import synth
import tile_compiler_row_gb300 as tile
from parity import ATOL, EPS, RTOL, oracle_blocks, ref_eps, expects_staged

pytestmark = pytest.mark.gpu

BF16_HALF_ULP_REL = 2.0 ** -8


@pytest.fixture(scope="module", autouse=True)
def device():
    from tile_compiler_row_gb300 import _build
    _build.build()
    torch.cuda.set_device(0)
    yield
    assert tile.tile_check_device_status() == 0


def _bf16_rows(cfg, rows, width, which="x"):
    """(bf16 CUDA tensor, its exact FP32 values on the host)."""
    t = torch.from_numpy(synth.rows_of(cfg, rows, width, which=which)).to(torch.bfloat16)
    return t, t.float().numpy()


def _placed(t, offset=0):
    buf = torch.empty(t.numel() + 16, dtype=t.dtype, device="cuda")
    view = buf[offset:offset + t.numel()].view(t.shape)
    view.copy_(t)
    return view


def _round_bf16(ref):
    """Round-to-nearest-even BF16 of FP64 values (through FP32)."""
    b = np.asarray(ref, np.float32).view(np.uint32).astype(np.uint64)
    b = (b + 0x7FFF + ((b >> 16) & 1)) >> 16
    return (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def check_bf16(got_t, ref, atol=ATOL, what=""):
    got = got_t.float().cpu().numpy().astype(np.float64)
    assert got.shape == ref.shape, what
    assert np.all(np.isfinite(got)), what
    err = np.abs(got - ref)
    bound = atol + (RTOL + BF16_HALF_ULP_REL) * np.abs(ref)
    assert np.all(err <= bound), f"{what}: max err {err.max():.3e}"
    # Rounding checks where the BF16 spacing dwarfs the FP32 error (|ref| >
    # 1e-2: half a BF16 ulp is >= 2e-5 there, the FP32 error about 2e-7);
    # for smaller outputs the FP32 error can reach a BF16 ulp of the output.
    big = np.abs(ref) > 1e-2
    rn = _round_bf16(ref[big])
    ulp = 2.0 ** (np.floor(np.log2(np.abs(rn))) - 7)
    assert np.all(np.abs(got[big] - rn) <= ulp), \
        f"{what}: an output is more than one BF16 ulp from the rounded reference"
    if big.any():
        rate = float(np.mean(got[big] == rn))
        assert rate >= 0.999, f"{what}: only {rate:.4f} correctly rounded"


SHAPES = [(1, 127), (17, 257), (7, 1537), (64, 4096), (1024, 4096), (128, 8192), (32, 65536)]


@pytest.mark.parametrize("rows,width", SHAPES)
@pytest.mark.parametrize("op", ["residual_layernorm", "layernorm", "rmsnorm", "softmax"])
def test_bf16_ops(op, rows, width):
    cfg = 4 if width in (8192, 65536) and op != "residual_layernorm" else 3
    x, xf = _bf16_rows(cfg, rows, width)
    r, rf = _bf16_rows(cfg, rows, width, "r")
    out = torch.empty(rows, width, dtype=torch.bfloat16, device="cuda")
    tx = _placed(x)
    if op == "residual_layernorm":
        tile.tile_residual_layernorm_bf16(tx, _placed(r), out, EPS)
        ref = oracle.get().residual_layernorm(xf, rf, ref_eps())
    else:
        getattr(tile, f"tile_{op}_bf16")(tx, out, EPS)
        ref = oracle.get().run(op, xf, eps=ref_eps())
    check_bf16(out, ref, what=f"bf16 {op} {rows}x{width}")


@pytest.mark.parametrize("offset", [1, 3, 5, 7])
@pytest.mark.parametrize("op", ["residual_layernorm", "layernorm", "rmsnorm", "softmax"])
def test_bf16_unaligned_rows(op, offset):
    for rows, width in [(5, 127), (3, 1537), (2, 4099)]:
        x, xf = _bf16_rows(3, rows, width)
        r, rf = _bf16_rows(3, rows, width, "r")
        buf = torch.empty(rows * width + 16, dtype=torch.bfloat16, device="cuda")
        out = buf[offset:offset + rows * width].view(rows, width)
        if op == "residual_layernorm":
            tile.tile_residual_layernorm_bf16(_placed(x, offset), _placed(r, offset), out, EPS)
            ref = oracle.get().residual_layernorm(xf, rf, ref_eps())
        else:
            getattr(tile, f"tile_{op}_bf16")(_placed(x, offset), out, EPS)
            ref = oracle.get().run(op, xf, eps=ref_eps())
        check_bf16(out, ref, what=f"bf16 {op} offset {offset} {rows}x{width}")
        # different phases for input and output: the scalar plans
        out2 = torch.empty(rows, width, dtype=torch.bfloat16, device="cuda")
        if op == "residual_layernorm":
            tile.tile_residual_layernorm_bf16(_placed(x, offset), _placed(r, offset), out2, EPS)
        else:
            getattr(tile, f"tile_{op}_bf16")(_placed(x, offset), out2, EPS)
        check_bf16(out2, ref, what=f"bf16 {op} mixed phases {rows}x{width}")


@pytest.mark.parametrize("rows,width", [(7, 1537), (64, 4096), (128, 8192)])
def test_bf16_affine_and_weighted(rows, width):
    x, xf = _bf16_rows(3, rows, width)
    r, rf = _bf16_rows(3, rows, width, "r")
    g = synth.uniform_pm1(3001, width) * np.float32(2.0)
    b = synth.uniform_pm1(3002, width)
    tg, tb = torch.from_numpy(g).cuda(), torch.from_numpy(b).cuda()
    out = torch.empty(rows, width, dtype=torch.bfloat16, device="cuda")
    tile.tile_layernorm_affine_bf16(_placed(x), _placed(r), tg, tb, out, EPS)
    ref = oracle.get().layernorm_affine(xf, g, b, r=rf, eps=ref_eps())
    check_bf16(out, ref, atol=1e-5, what=f"bf16 affine {rows}x{width}")
    tile.tile_rmsnorm_weighted_bf16(_placed(x), tg, out, EPS)
    ref = oracle.get().rmsnorm_weighted(xf, g, eps=ref_eps())
    check_bf16(out, ref, what=f"bf16 weighted {rows}x{width}")


@pytest.mark.parametrize("rows,width", [(17, 257), (64, 4096), (32, 65536), (1000, 1)])
def test_bf16_row_sum_and_minmax(rows, width):
    x, xf = _bf16_rows(3, rows, width)
    sums = torch.empty(rows, device="cuda")
    tile.tile_row_sum_bf16(_placed(x, 1), sums)
    ref = oracle.get().row_sum(xf)
    got = sums.cpu().numpy().astype(np.float64)
    assert np.all(np.abs(got - ref) <= ATOL + RTOL * np.abs(ref))
    mins, maxs = torch.empty(rows, device="cuda"), torch.empty(rows, device="cuda")
    tile.tile_row_minmax_bf16(_placed(x, 3), mins, maxs)
    mn, mx = oracle.get().row_minmax(xf)
    assert np.array_equal(mins.cpu().numpy().astype(np.float64), mn)
    assert np.array_equal(maxs.cpu().numpy().astype(np.float64), mx)


def _bf16_plan_cases():
    from tile_compiler_row_gb300 import _build
    _build.build()
    out = []
    for pid in range(tile.tile_plan_count()):
        info = tile.tile_plan_info_ex(pid, 0, "bf16", 1, 1)
        if info is None:
            continue
        maxw = info["max_width"]
        rows = 3 if maxw > 16384 else 2 * info["programs_per_cta"] + 1
        for op in ("residual_layernorm", "layernorm", "rmsnorm", "softmax"):
            out.append((pid, op, rows, sorted({1, 9, min(maxw, 77), maxw})))
    return out


@pytest.mark.parametrize("pid,op,rows,widths", _bf16_plan_cases(),
                         ids=lambda v: str(v) if not isinstance(v, list) else "w")
def test_every_bf16_plan(pid, op, rows, widths):
    for w in widths:
        x, xf = _bf16_rows(3, rows, w)
        r, rf = _bf16_rows(3, rows, w, "r")
        for off in (0, 3):
            out = _placed(torch.zeros(rows, w, dtype=torch.bfloat16), off)
            tile.tile_run_plan_args_f32(op, pid, _placed(x, off), out,
                                        residual=_placed(r, off) if op == "residual_layernorm"
                                        else None, eps=EPS)
            ref = (oracle.get().residual_layernorm(xf, rf, ref_eps()) if op == "residual_layernorm"
                   else oracle.get().run(op, xf, eps=ref_eps()))
            check_bf16(out, ref, what=f"bf16 plan {pid} {op} w={w} off={off}")


@pytest.mark.parametrize("op", ["residual_layernorm", "layernorm", "rmsnorm", "softmax"])
@pytest.mark.parametrize("rows,width", [(2048, 4096), (1024, 8192), (1024, 12288),
                                        (512, 16384)])
def test_bf16_selected_staged_plans(op, rows, width):
    """Large BF16 rows of whole vectors select a shared-memory-staged plan
    where it measured faster; the same rows one element off the 16-byte phase
    fall back to a register plan.  Both must meet the bound."""
    x, xf = _bf16_rows(3, rows, width)
    r, rf = _bf16_rows(3, rows, width, "r")
    ref = (oracle.get().residual_layernorm(xf, rf, ref_eps()) if op == "residual_layernorm"
           else oracle.get().run(op, xf, eps=ref_eps()))
    for off in (0, 1):
        buf = torch.empty(rows * width + 16, dtype=torch.bfloat16, device="cuda")
        out = buf[off:off + rows * width].view(rows, width)
        if op == "residual_layernorm":
            tile.tile_residual_layernorm_bf16(_placed(x, off), _placed(r, off), out, EPS)
        else:
            getattr(tile, f"tile_{op}_bf16")(_placed(x, off), out, EPS)
        check_bf16(out, ref, what=f"bf16 {op} {rows}x{width} offset {off}")
    # the staged kernel exactly where the measured table takes it
    staged = expects_staged(op, rows, width)
    assert (tile.tile_describe_plan_ex(op, "bf16", rows, width)["path"] == 2) == staged


@pytest.mark.parametrize("op", ["layernorm", "residual_layernorm"])
@pytest.mark.parametrize("rows,width", [(4, 257), (2048, 4096), (512, 16384)])
def test_bf16_constant_rows_normalise_to_zero(op, rows, width):
    """Constant rows (the closed form gives LayerNorm output 0) on register
    and staged plans: every output within the absolute bound of 0."""
    vals = torch.tensor([0.1, 3.140625, -7.5, 1000.0, -20000.0], dtype=torch.float32)
    x = vals[torch.arange(rows) % len(vals)][:, None].expand(rows, width).contiguous()
    x = x.to(torch.bfloat16).cuda()
    y = torch.full_like(x, float("nan"))
    if op == "residual_layernorm":
        r = torch.zeros_like(x)
        tile.tile_residual_layernorm_bf16(x, r, y, EPS)
    else:
        tile.tile_layernorm_bf16(x, y, EPS)
    torch.cuda.synchronize()
    got = y.float().cpu().numpy()
    assert np.all(np.abs(got) <= ATOL), f"{op} {rows}x{width}: max |y| {np.abs(got).max():.3e}"


def test_bf16_residual_layernorm_65536x4096():
    """The BF16 residual LayerNorm launch that bench.py times (65536 x 4096,
    512 MiB per tensor, the shared-memory-staged plan): every output against
    the oracle, block by block on every host core, under the BF16 bound; the
    correctly-rounded rate is taken over the whole output."""
    rows, width = 65536, 4096
    x, xf = _bf16_rows(5, rows, width)
    r, rf = _bf16_rows(5, rows, width, "r")
    info = tile.tile_describe_plan_ex("residual_layernorm", "bf16", rows, width)
    assert info["path"] == 2, info
    tx, tr = x.cuda(), r.cuda()
    y = torch.full_like(tx, float("nan"))
    tile.tile_residual_layernorm_bf16(tx, tr, y, EPS)
    torch.cuda.synchronize()
    got_all = y.float().cpu().numpy()
    del tx, tr, y
    big_n, equal_n = 0, 0
    for a, b, ref in oracle_blocks("residual_layernorm", xf, rf):
        what = f"bf16 residual_layernorm 65536x4096 rows {a}..{b - 1}"
        got = got_all[a:b].astype(np.float64)
        assert np.all(np.isfinite(got)), what
        err = np.abs(got - ref)
        bound = ATOL + (RTOL + BF16_HALF_ULP_REL) * np.abs(ref)
        assert np.all(err <= bound), f"{what}: max err {err.max():.3e}"
        big = np.abs(ref) > 1e-2
        rn = _round_bf16(ref[big])
        ulp = 2.0 ** (np.floor(np.log2(np.abs(rn))) - 7)
        assert np.all(np.abs(got[big] - rn) <= ulp), \
            f"{what}: an output is more than one BF16 ulp from the rounded reference"
        big_n += int(big.sum())
        equal_n += int(np.count_nonzero(got[big] == rn))
    assert big_n > 0 and equal_n / big_n >= 0.999, f"only {equal_n / big_n:.5f} correctly rounded"


@pytest.mark.parametrize("rows,width", [(400, 12288), (512, 16384)])
def test_bf16_residual_affine_and_weighted_on_staged_plans(rows, width):
    """2-byte affine LayerNorm with a residual takes the shared-memory-staged
    plan at these widths (weighted RMSNorm at 12288), gamma and beta applied
    in the staged kernel: both against the oracle."""
    x, xf = _bf16_rows(3, rows, width)
    r, rf = _bf16_rows(3, rows, width, "r")
    g = synth.uniform_pm1(3001, width) * np.float32(2.0)
    b = synth.uniform_pm1(3002, width)
    tg, tb = torch.from_numpy(g).cuda(), torch.from_numpy(b).cuda()
    out = torch.empty(rows, width, dtype=torch.bfloat16, device="cuda")
    tile.tile_layernorm_affine_bf16(x.cuda(), r.cuda(), tg, tb, out, EPS)
    ref = oracle.get().layernorm_affine(xf, g, b, r=rf, eps=ref_eps())
    check_bf16(out, ref, atol=1e-5, what=f"bf16 residual affine {rows}x{width}")
    tile.tile_rmsnorm_weighted_bf16(x.cuda(), tg, out, EPS)
    ref = oracle.get().rmsnorm_weighted(xf, g, eps=ref_eps())
    check_bf16(out, ref, what=f"bf16 weighted {rows}x{width}")
    staged = tile.tile_describe_plan_ex("rmsnorm_weighted", "bf16", rows, width)["path"] == 2
    assert staged == expects_staged("rmsnorm_weighted", rows, width)
