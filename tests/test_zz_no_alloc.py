"""The host-buffer entry point that allocates nothing.

tile_run_host_static_f32 is for callers that cannot allocate device memory
where they run: code running after an application has fixed its device
memory budget, plugin code inside a framework that owns the device
allocator, or latency-critical code that must not call cudaMalloc.  It
stages rows through a static device array inside the library instead of a
workspace the caller allocates.

Each case calls it twice in a row through the C ABI (the second call is
enqueued before the first has finished, with different inputs, so stale
contents of the shared array or an overlap between the calls would show)
and checks both results against tile_run_host_f32 with a caller workspace,
within the tolerance of the other parity tests: with pageable inputs (the
rows stage through the array) and with every buffer pinned (in place).  This file is collected last
and depends on nothing that earlier tests set up.
"""

import numpy as np
import pytest
import torch

import synth
import tile_compiler_row_gb300 as tile
from parity import ATOL, EPS, RTOL

pytestmark = pytest.mark.gpu

# (op, rows, width): several chunks through the 64 MiB area in each case.
CASES = [("residual_layernorm", 3000, 4096), ("softmax", 40, 131072), ("layernorm", 257, 1537)]


@pytest.fixture(scope="module", autouse=True)
def device():
    from tile_compiler_row_gb300 import _build
    _build.build()
    tile.load()
    torch.cuda.set_device(0)


def _pinned(a):
    return torch.from_numpy(np.ascontiguousarray(a)).pin_memory()


def _inputs(op, rows, width, scale, pinned=True):
    x = synth.rows_of(3, rows, width, which="x") * np.float32(scale)
    r = synth.rows_of(3, rows, width, which="r") if op == "residual_layernorm" else None
    host = _pinned if pinned else (lambda a: torch.from_numpy(np.ascontiguousarray(a)).clone())
    return host(x), (host(r) if r is not None else None)


def _with_workspace(op, x, r):
    rows, width = x.shape
    ws = torch.empty(tile.tile_host_workspace_bytes(op, width, max(1, rows // 5)),
                     dtype=torch.uint8, device="cuda")
    out = torch.empty(rows, width).pin_memory()
    tile.tile_run_host_f32(op, x, r, out, ws, EPS)
    torch.cuda.synchronize()
    return out.numpy().copy()


# staged: pageable inputs go through the static array (with the output
# pinned, stored directly; or pageable, copied out); in_place: every buffer
# pinned, one kernel on the host buffers and no staging
MODES = {"staged_direct_out": (False, True), "staged_copy_out": (False, False),
         "in_place": (True, True)}


@pytest.mark.parametrize("mode", list(MODES))
@pytest.mark.parametrize("op,rows,width", CASES)
def test_static_staging_matches_workspace_entry_point_on_two_calls(op, rows, width, mode):
    lib = tile.load()
    stream = torch.cuda.current_stream().cuda_stream
    pin_in, pin_out = MODES[mode]
    calls = [_inputs(op, rows, width, 1.0, pin_in), _inputs(op, rows, width, -2.5, pin_in)]
    outs = []
    for x, r in calls:                       # two calls in a row, no sync between
        out = torch.full((rows, width), float("nan"))
        out = out.pin_memory() if pin_out else out
        st = lib.tile_run_host_static_f32(tile.OPS[op], x.data_ptr(),
                                          r.data_ptr() if r is not None else None,
                                          out.data_ptr(), rows, width, EPS, stream)
        assert st == 0, tile.tile_status_string(st)
        outs.append(out)
    torch.cuda.synchronize()
    for (x, r), out in zip(calls, outs):
        got = out.numpy()
        want = _with_workspace(op, x, r)
        assert np.all(np.isfinite(got))
        assert np.all(np.abs(got - want) <= ATOL + RTOL * np.abs(want))


def test_static_staging_rejects_a_width_beyond_the_maximum():
    x = torch.zeros(2, 8).pin_memory()
    lib = tile.load()
    st = lib.tile_run_host_static_f32(1, x.data_ptr(), None, x.data_ptr() + 4096, 2,
                                      tile.tile_max_width() + 1, EPS, None)
    assert st == -2
