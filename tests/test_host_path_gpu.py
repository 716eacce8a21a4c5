"""GPU tests of the end-to-end entry point on host buffers: results match the
oracle and the device entry point, for chunkings from one row per chunk to
the whole matrix, with pinned and pageable host memory."""

import numpy as np
import pytest
import torch

import synth
import tile_compiler_row_gb300 as tile
from parity import EPS, compare, oracle_of

pytestmark = pytest.mark.gpu

OPS = ("residual_layernorm", "layernorm", "rmsnorm", "softmax")


@pytest.fixture(scope="module", autouse=True)
def device():
    from tile_compiler_row_gb300 import _build
    _build.build()
    torch.cuda.set_device(0)
    yield
    assert tile.tile_check_device_status() == 0


def _host(a, pinned):
    t = torch.from_numpy(np.ascontiguousarray(a))
    return t.pin_memory() if pinned else t.clone()


def _run_host(op, x, r, chunk_rows, pinned=True, stream=None, pinned_out=None):
    """pinned: inputs (and, unless pinned_out says otherwise, the output) in
    pinned memory.  All pinned: one kernel on the host buffers; pageable
    inputs with a pinned output: the copy pipeline with direct output
    stores; all pageable: the pipeline with copies out."""
    rows, width = x.shape
    ws_bytes = tile.tile_host_workspace_bytes(op, width, chunk_rows)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device="cuda")
    hx = _host(x, pinned)
    hr = _host(r, pinned) if r is not None else None
    out = torch.full(x.shape, float("nan"))
    out = out.pin_memory() if (pinned if pinned_out is None else pinned_out) else out
    tile.tile_run_host_f32(op, hx, hr, out, ws, EPS, stream)
    (stream or torch.cuda.current_stream()).synchronize()
    return out.numpy().copy()


def _run_device(op, x, r):
    tx = torch.from_numpy(x).cuda()
    tr = torch.from_numpy(r).cuda() if r is not None else None
    y = torch.empty_like(tx)
    tile.run(op, tx, tr, y, EPS)
    torch.cuda.synchronize()
    return y.cpu().numpy()


@pytest.mark.parametrize("op", OPS)
@pytest.mark.parametrize("rows,width,chunk", [(37, 1537, 1), (37, 1537, 7), (1000, 4096, 125),
                                              (1000, 4096, 300), (5, 131072, 2), (3, 127, 64)])
@pytest.mark.parametrize("mode", ["in_place", "pipeline"])
def test_host_path_matches_oracle_and_device_path(op, rows, width, chunk, mode):
    """in_place: every buffer pinned, one kernel on the host buffers;
    pipeline: pageable inputs, pinned output (chunked copies in, direct
    stores out)."""
    x = synth.rows_of(3, rows, width, which="x")
    r = synth.rows_of(3, rows, width, which="r") if op == "residual_layernorm" else None
    got = _run_host(op, x, r, chunk, pinned=mode == "in_place", pinned_out=True)
    compare(got, oracle_of(op, x, r), f"host {op} {rows}x{width} chunk {chunk}")
    # Every chunk runs the whole matrix's plan, so the results are bitwise
    # those of the device call wherever every row start has the same 16-byte
    # phase in both (chunks start 256-byte aligned in the workspace; rows of
    # the full tensor do only when width is a multiple of 4).
    if width % 4 == 0:
        assert np.array_equal(got, _run_device(op, x, r))


@pytest.mark.parametrize("op", OPS)
@pytest.mark.parametrize("rows,width", [(20000, 257), (9001, 1024), (8192, 4096)])
@pytest.mark.parametrize("pinned", [True, False])
def test_host_path_ring_of_four_slots(op, rows, width, pinned):
    # pageable inputs, so the copy pipeline runs; pinned: direct output stores
    """Workspace for the whole matrix: about 16 chunks cycle through a ring
    of four slots (each slot reused four times), with results stored
    directly (pinned) or copied out (pageable); bitwise those of the device
    call where the rows keep their 16-byte phase."""
    ws = tile.tile_host_workspace_bytes(op, width, rows)
    chunk, slots = tile.tile_host_schedule(op, rows, width, ws, direct_output=pinned)
    assert slots == 4 and -(-rows // chunk) >= 12
    x = synth.rows_of(3, rows, width, which="x")
    r = synth.rows_of(3, rows, width, which="r") if op == "residual_layernorm" else None
    got = _run_host(op, x, r, rows, pinned=False, pinned_out=pinned)
    compare(got, oracle_of(op, x, r), f"ring {op} {rows}x{width} pinned={pinned}")
    # (8192 x 4096: quarter-size first and last chunks of 128 rows)
    if width % 4 == 0:
        assert np.array_equal(got, _run_device(op, x, r))


@pytest.mark.parametrize("op", ["residual_layernorm", "softmax"])
def test_host_path_pageable_memory_and_side_stream(op):
    x = synth.rows_of(3, 64, 4096, which="x")
    r = synth.rows_of(3, 64, 4096, which="r") if op == "residual_layernorm" else None
    s = torch.cuda.Stream()
    got = _run_host(op, x, r, 9, pinned=False, stream=s)
    compare(got, oracle_of(op, x, r), f"pageable {op}")


@pytest.mark.parametrize("pinned_out", [True, False])
def test_host_path_back_to_back_calls_share_the_workspace(pinned_out):
    """Two calls in a row on one stream through one workspace (pageable
    inputs, so the copy pipeline runs): the second must not overwrite the
    first call's chunks before they are consumed or copied out."""
    op = "residual_layernorm"
    rows, width = 300, 2048
    x = synth.rows_of(3, rows, width, which="x")
    r = synth.rows_of(3, rows, width, which="r")
    x2 = (x[::-1] * np.float32(0.5)).copy()
    ws = torch.empty(tile.tile_host_workspace_bytes(op, width, 16), dtype=torch.uint8,
                     device="cuda")
    outs = []
    for xi in (x, x2):
        o = torch.empty(rows, width)
        o = o.pin_memory() if pinned_out else o
        tile.tile_run_host_f32(op, _host(xi, False), _host(r, False), o, ws, EPS)
        outs.append(o)
    torch.cuda.synchronize()
    compare(outs[0].numpy(), oracle_of(op, x, r), "first call")
    compare(outs[1].numpy(), oracle_of(op, x2, r), "second call")


def test_host_path_workspace_too_small_raises():
    x = torch.zeros(4, 4096).pin_memory()
    ws = torch.empty(1024, dtype=torch.uint8, device="cuda")
    with pytest.raises(tile.TileError) as e:
        tile.tile_run_host_f32("layernorm", x, None, torch.zeros(4, 4096), ws)
    assert e.value.status == -10


def _pinned_off(a):
    """A pinned host view of `a` starting one float into its allocation:
    device-addressable but not 16-byte aligned."""
    buf = torch.empty(a.size + 1).pin_memory()
    v = buf[1:1 + a.size].view(a.shape)
    v.copy_(torch.from_numpy(np.ascontiguousarray(a)))
    return v


@pytest.mark.parametrize("op", OPS)
@pytest.mark.parametrize("rows,width", [(33, 1029), (1, 4096), (5, 4100)])
def test_host_path_in_place_on_unaligned_pinned_buffers(op, rows, width):
    """Pinned buffers that start off the 16-byte phase run in place on the
    scalar plans; a single row too."""
    x = synth.rows_of(3, rows, width, which="x")
    r = synth.rows_of(3, rows, width, which="r") if op == "residual_layernorm" else None
    hx = _pinned_off(x)
    hr = _pinned_off(r) if r is not None else None
    out = _pinned_off(np.full((rows, width), np.nan, np.float32))
    ws = torch.empty(tile.tile_host_workspace_bytes(op, width, max(1, rows // 2)),
                     dtype=torch.uint8, device="cuda")
    tile.tile_run_host_f32(op, hx, hr, out, ws, EPS)
    torch.cuda.current_stream().synchronize()
    compare(out.numpy(), oracle_of(op, x, r), f"in place unaligned {op} {rows}x{width}")
