"""GPU parity: the CUDA library (through its C ABI) against the FP64 oracle.

Every element must satisfy |y - ref| <= 2e-6 + 2e-5*|ref|.  Covered: the five
workloads (the 65536x4096 one on every element, plus whole-output properties),
every built plan, ragged widths, nonzero row origins, pointers with
different 16-byte phases, rows fewer than the programs of a CTA, width 1, the
maximum width, sentinel guards after three dispatches, determinism, row
independence and argument errors on real device buffers."""

from __future__ import annotations

import numpy as np
import pytest
import torch

import synth
import tile_compiler_row_gb300 as tile
from parity import ATOL, EPS, RTOL, compare, compare_full, oracle_of

pytestmark = pytest.mark.gpu

OPS = ("residual_layernorm", "layernorm", "rmsnorm", "softmax")


@pytest.fixture(scope="module", autouse=True)
def device():
    from tile_compiler_row_gb300 import _build
    _build.build()
    tile.load()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    torch.cuda.set_device(0)
    yield torch.device("cuda:0")
    assert tile.tile_check_device_status() == 0


def _dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def gpu_run(op, x, r=None, eps=EPS, plan=None, offset=0, out_offset=None):
    """Run ``op`` on host arrays; ``offset`` (floats) shifts every buffer's
    start so rows begin at a non-16-byte-aligned address."""
    rows, width = x.shape
    out_offset = offset if out_offset is None else out_offset
    n = rows * width

    def place(a, off):
        buf = torch.empty(n + 8, dtype=torch.float32, device="cuda")
        view = buf[off:off + n].view(rows, width)
        if a is not None:
            view.copy_(torch.from_numpy(np.ascontiguousarray(a)))
        return view

    tx = place(x, offset)
    tr = place(r, offset) if r is not None else None
    out = place(None, out_offset)
    out.fill_(float("nan"))
    if plan is None:
        tile.run(op, tx, tr, out, eps)
    else:
        tile.tile_run_plan_f32(op, plan, tx, tr, out, eps)
    torch.cuda.synchronize()
    return out.cpu().numpy()


def inputs(cfg, rows, width, op):
    x = synth.rows_of(cfg, rows, width, which="x")
    r = synth.rows_of(cfg, rows, width, which="r") if op == "residual_layernorm" else None
    return x, r


def check(op, x, r=None, **kw):
    got = gpu_run(op, x, r, **kw)
    return compare(got, oracle_of(op, x, r), f"{op} {x.shape} {kw}")


# ---------------------------------------------------------------------------
# the workloads
# ---------------------------------------------------------------------------

def test_residual_layernorm_17x257():
    x, r = inputs(1, 17, 257, "residual_layernorm")
    check("residual_layernorm", x, r)


@pytest.mark.parametrize("op", ["softmax", "rmsnorm", "layernorm"])
def test_1024x4096(op):
    x, r = inputs(2, 1024, 4096, op)
    check(op, x, r)


@pytest.mark.parametrize("shape", [(1, 127), (7, 1537), (17, 257), (64, 4096)])
@pytest.mark.parametrize("op", ["residual_layernorm", "rmsnorm", "softmax"])
def test_ragged_sweep(op, shape):
    x, r = inputs(3, *shape, op)
    check(op, x, r)


@pytest.mark.parametrize("shape", [(128, 8192), (32, 65536)])
@pytest.mark.parametrize("op", ["softmax", "rmsnorm", "layernorm"])
def test_wide_rows(op, shape):
    rows, width = shape
    x, r = inputs(4, rows, width, op)
    got = gpu_run(op, x, r)
    compare(got, oracle_of(op, x, r), f"{op} {shape}")
    # row 0 is constant: LayerNorm gives 0, softmax gives 1/width
    if op == "layernorm":
        assert np.all(np.abs(got[0]) <= ATOL)
    if op == "softmax":
        assert np.all(np.abs(got[0] - 1.0 / width) <= ATOL + RTOL / width)
        # the +40 outlier takes almost all the mass of row 1
        assert got[1, synth.outlier_column(width)] > 0.999


# ---------------------------------------------------------------------------
# 65536 x 4096 (1 GiB per tensor): every element against the oracle, and
# properties of the whole output
# ---------------------------------------------------------------------------

ROWS5, WIDTH5 = 65536, 4096


@pytest.fixture(scope="module")
def big_inputs():
    x = synth.rows_of(5, ROWS5, WIDTH5, which="x")
    r = synth.rows_of(5, ROWS5, WIDTH5, which="r")
    return x, r, _dev(x), _dev(r)


@pytest.mark.parametrize("op", ["residual_layernorm", "rmsnorm", "softmax"])
def test_65536x4096(op, big_inputs):
    """The launch bench.py times (the selector's plan on allocator-aligned
    tensors): all 268,435,456 outputs against the oracle, computed in row
    blocks on every host core."""
    x, r, tx, tr = big_inputs
    out = torch.full_like(tx, float("nan"))
    tile.run(op, tx, tr if op == "residual_layernorm" else None, out, EPS)
    torch.cuda.synchronize()
    got = out.cpu().numpy()
    rr = r if op == "residual_layernorm" else None
    compare_full(got, op, x, rr, what=f"{op} 65536x4096")
    # whole-output properties implied by the element bound
    y = out.double()
    n = WIDTH5
    if op == "softmax":
        dev = (y.sum(dim=1) - 1.0).abs().max().item()
        assert dev <= n * ATOL + RTOL
    else:
        c = tx.double() + (tr.double() if op == "residual_layernorm" else 0.0)
        if op == "residual_layernorm":
            v = c.var(dim=1, unbiased=False)
            assert y.mean(dim=1).abs().max().item() <= ATOL + RTOL
        else:
            v = (c * c).mean(dim=1)
        want = v / (v + np.float32(EPS))
        assert ((y * y).mean(dim=1) - want).abs().max().item() <= 4 * (ATOL + RTOL)
    del out, y


# ---------------------------------------------------------------------------
# every built plan
# ---------------------------------------------------------------------------

def _plan_cases():
    cases = []
    for pid in range(tile.tile_plan_count()):
        info = tile.tile_plan_info(pid, 0, 1, 1)
        if info is None:          # staged plans: tests/test_staged_gpu.py
            continue
        maxw = info["max_width"]
        widths = sorted({1, 3, min(maxw, 37), max(1, maxw // 2 - 1), maxw})
        rows = 2 * info["programs_per_cta"] + 1          # a packed tail
        if maxw > 16384:
            rows = 3
        for op in OPS:
            cases.append((pid, op, rows, widths))
    return cases


@pytest.mark.parametrize("pid,op,rows,widths", _plan_cases(),
                         ids=lambda v: str(v) if not isinstance(v, list) else "w")
def test_every_plan(pid, op, rows, widths):
    info = tile.tile_plan_info(pid, op, rows, 1)
    for w in widths:
        x, r = inputs(3, rows, w, op)
        check(op, x, r, plan=pid)
        if info["vec"] == 4:
            check(op, x, r, plan=pid, offset=1)          # head/tail scalars
        else:
            check(op, x, r, plan=pid, offset=1, out_offset=2)


# ---------------------------------------------------------------------------
# edge cases
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("op", OPS)
def test_width_one(op):
    x, r = inputs(3, 9, 1, op)
    got = gpu_run(op, x, r)
    compare(got, oracle_of(op, x, r), op)
    if op in ("layernorm", "residual_layernorm"):
        assert np.all(got == 0.0)
    if op == "softmax":
        assert np.all(got == 1.0)


@pytest.mark.parametrize("offset", [1, 2, 3])
@pytest.mark.parametrize("op", OPS)
def test_nonzero_row_origin(op, offset):
    for rows, width in [(5, 127), (3, 1537), (2, 4099)]:
        x, r = inputs(3, rows, width, op)
        check(op, x, r, offset=offset)


@pytest.mark.parametrize("op", OPS)
def test_pointers_with_different_phases(op):
    for rows, width in [(4, 255), (3, 4096), (2, 20000)]:
        x, r = inputs(3, rows, width, op)
        check(op, x, r, offset=0, out_offset=1)


@pytest.mark.parametrize("op", OPS)
def test_rows_fewer_than_programs(op):
    for rows in (1, 2, 3):
        x, r = inputs(3, rows, 64, op)               # plan packs 8 rows per CTA
        check(op, x, r)


@pytest.mark.parametrize("op", OPS)
def test_max_width(op):
    w = tile.tile_max_width()
    x, r = inputs(3, 2, w, op)
    check(op, x, r)
    x, r = inputs(3, 2, w - 1, op)
    check(op, x, r, offset=1)


def test_rows_zero_leaves_output_untouched():
    out = torch.full((0, 16), 7.0, device="cuda")
    tile.tile_softmax_f32(torch.empty(0, 16, device="cuda"), out)
    sentinel = torch.full((4, 16), 7.0, device="cuda")
    st = tile.load().tile_rmsnorm_f32(sentinel.data_ptr(), sentinel.data_ptr() + 1024, 0, 16,
                                      1e-5, None)
    assert st == 0
    torch.cuda.synchronize()
    assert bool((sentinel == 7.0).all())


@pytest.mark.parametrize("op", OPS)
def test_sentinels_and_three_dispatches(op):
    """Guard rows before and after the output keep their canary after three
    dispatches; the inputs are unmodified; the three results are bitwise equal."""
    rows, width = 37, 1537
    x, r = inputs(3, rows, width, op)
    tx, tr = _dev(x), (_dev(r) if r is not None else None)
    guard = 3 * width + 5
    canary = -12345.678
    buf = torch.full((guard + rows * width + guard,), canary, device="cuda")
    out = buf[guard:guard + rows * width].view(rows, width)
    results = []
    for _ in range(3):
        tile.run(op, tx, tr, out, EPS)
        torch.cuda.synchronize()
        results.append(out.cpu().numpy().copy())
    assert bool((buf[:guard] == canary).all()) and bool((buf[-guard:] == canary).all())
    assert np.array_equal(tx.cpu().numpy(), x)
    if r is not None:
        assert np.array_equal(tr.cpu().numpy(), r)
    assert np.array_equal(results[0], results[1]) and np.array_equal(results[1], results[2])
    compare(results[0], oracle_of(op, x, r), op)


@pytest.mark.parametrize("op", OPS)
def test_row_independence(op):
    rows, width = 33, 4096
    x, r = inputs(3, rows, width, op)
    a = gpu_run(op, x, r)
    x2 = x.copy()
    x2[7] = x2[7][::-1] * np.float32(2.0)
    b = gpu_run(op, x2, r)
    keep = [i for i in range(rows) if i != 7]
    assert np.array_equal(a[keep], b[keep])


@pytest.mark.parametrize("op", OPS)
def test_non_default_stream(op):
    x, r = inputs(3, 64, 4096, op)
    tx, tr = _dev(x), (_dev(r) if r is not None else None)
    out = torch.empty_like(tx)
    s = torch.cuda.Stream()
    torch.cuda.synchronize()
    with torch.cuda.stream(s):
        tile.run(op, tx, tr, out, EPS)
    s.synchronize()
    compare(out.cpu().numpy(), oracle_of(op, x, r), op)


def test_alias_rejected_on_device_buffers():
    t = torch.zeros(4, 64, device="cuda")
    with pytest.raises(tile.TileError) as e:
        tile.tile_layernorm_f32(t, t)
    assert e.value.status == -3
    with pytest.raises(tile.TileError) as e:
        tile.tile_residual_layernorm_f32(t, torch.zeros_like(t), t)
    assert e.value.status == -3


def test_device_status_is_clean():
    assert tile.tile_check_device_status() == 0
