"""The host-buffer entry point that allocates nothing.

tile_run_host_static_f32 is for callers that cannot allocate device memory
where they run: code running after an application has fixed its device
memory budget, plugin code inside a framework that owns the device
allocator, or latency-critical code that must not call cudaMalloc.  It
stages rows through a static device array inside the library instead of a
workspace the caller allocates.

Each case calls it twice in a row through the C ABI with different inputs
(the second call is enqueued before the first has finished, so stale
contents of the shared array or an overlap between the calls would show)
and checks both results against the FP64 oracle under the acceptance bound
of the other parity tests, and against tile_run_host_f32 with a caller
workspace: bit for bit where rows are whole 16-byte vectors (both entry
points then run the same plan on rows of the same alignment), within the
bound otherwise.  Modes: pageable inputs (the rows stage through the array)
with the output pinned or pageable, and every buffer pinned (in place).
One more case issues the two calls on two different streams with no
synchronisation between them: only the library's ordering of calls on the
shared array keeps them apart there; another makes the first call fail
part-way (a launch failure injected on the host) before the second.  This file is collected last and
depends on nothing that earlier tests set up.
"""

import numpy as np
import pytest
import torch

import synth
import tile_compiler_row_gb300 as tile
from parity import ATOL, EPS, RTOL, compare, oracle_of

pytestmark = pytest.mark.gpu

# (op, rows, width): several chunks through the 64 MiB area in each case.
CASES = [("residual_layernorm", 3000, 4096), ("softmax", 40, 131072), ("layernorm", 257, 1537)]


@pytest.fixture(scope="module", autouse=True)
def device():
    from tile_compiler_row_gb300 import _build
    _build.build()
    tile.load()
    torch.cuda.set_device(0)


def _host(a, pinned):
    t = torch.from_numpy(np.ascontiguousarray(a))
    return t.pin_memory() if pinned else t.clone()


def _inputs(op, rows, width, scale, pinned=True):
    """(x, r) host tensors and the FP32 arrays they hold: workload-3 rows,
    x scaled by `scale` in FP32 (the oracle gets the same rounded values)."""
    x = synth.rows_of(3, rows, width, which="x") * np.float32(scale)
    r = synth.rows_of(3, rows, width, which="r") if op == "residual_layernorm" else None
    return (_host(x, pinned), _host(r, pinned) if r is not None else None), (x, r)


def _with_workspace(op, x, r):
    rows, width = x.shape
    ws = torch.empty(tile.tile_host_workspace_bytes(op, width, max(1, rows // 5)),
                     dtype=torch.uint8, device="cuda")
    out = torch.empty(rows, width).pin_memory()
    tile.tile_run_host_f32(op, x, r, out, ws, EPS)
    torch.cuda.synchronize()
    return out.numpy().copy()


def _call_static(op, x, r, out, stream):
    lib = tile.load()
    rows, width = x.shape
    st = lib.tile_run_host_static_f32(tile.OPS[op], x.data_ptr(),
                                      r.data_ptr() if r is not None else None,
                                      out.data_ptr(), rows, width, EPS, stream)
    assert st == 0, tile.tile_status_string(st)


def _check(op, got, host_in, values, what):
    x, r = values
    compare(got, oracle_of(op, x, r), f"{what}: against the oracle")
    want = _with_workspace(op, *host_in)
    if x.shape[1] % 4 == 0:
        assert np.array_equal(got, want), f"{what}: differs from tile_run_host_f32"
    else:
        assert np.all(np.abs(got - want) <= ATOL + RTOL * np.abs(want)), what


# staged: pageable inputs go through the static array (with the output
# pinned, stored directly; or pageable, copied out); in_place: every buffer
# pinned, one kernel on the host buffers and no staging
MODES = {"staged_direct_out": (False, True), "staged_copy_out": (False, False),
         "in_place": (True, True)}


@pytest.mark.parametrize("mode", list(MODES))
@pytest.mark.parametrize("op,rows,width", CASES)
def test_static_staging_matches_oracle_on_two_calls(op, rows, width, mode):
    stream = torch.cuda.current_stream().cuda_stream
    pin_in, pin_out = MODES[mode]
    calls = [_inputs(op, rows, width, 1.0, pin_in), _inputs(op, rows, width, -2.5, pin_in)]
    outs = []
    for (x, r), _ in calls:                  # two calls in a row, no sync between
        out = torch.full((rows, width), float("nan"))
        out = out.pin_memory() if pin_out else out
        _call_static(op, x, r, out, stream)
        outs.append(out)
    torch.cuda.synchronize()
    for k, ((host_in, values), out) in enumerate(zip(calls, outs)):
        _check(op, out.numpy(), host_in, values, f"{op} {rows}x{width} {mode} call {k}")


@pytest.mark.parametrize("op,rows,width", CASES)
def test_static_staging_calls_on_two_streams(op, rows, width):
    """Two calls on two different streams, enqueued back to back with no
    synchronisation: pageable inputs stage through the shared array and the
    results go straight into pinned outputs, so nothing on the host orders
    the two calls and only the library's ordering on the GPU keeps the
    second call's copies from overwriting rows the first call's kernels
    have not read yet."""
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    calls = [_inputs(op, rows, width, 1.0, False), _inputs(op, rows, width, -2.5, False)]
    outs = []
    for ((x, r), _), s in zip(calls, streams):
        out = torch.full((rows, width), float("nan")).pin_memory()
        _call_static(op, x, r, out, s.cuda_stream)
        outs.append(out)
    torch.cuda.synchronize()
    for k, ((host_in, values), out) in enumerate(zip(calls, outs)):
        _check(op, out.numpy(), host_in, values, f"{op} {rows}x{width} stream {k}")


def test_static_staging_stays_ordered_after_a_failed_call():
    """A call that fails part-way (a kernel launch failure injected on the
    host after two chunks were launched, with their copies and the next
    chunk's copies already enqueued) returns TILE_ERR_CUDA; the next call,
    on another stream with no synchronisation, must still wait for
    everything the failed call enqueued on the shared array: its results
    match the oracle."""
    op, rows, width = "residual_layernorm", 3000, 4096
    lib = tile.load()
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    (x0, r0), _ = _inputs(op, rows, width, 1.0, False)
    (x1, r1), values = _inputs(op, rows, width, -2.5, False)
    out0 = torch.full((rows, width), float("nan")).pin_memory()
    out1 = torch.full((rows, width), float("nan")).pin_memory()
    try:
        assert lib.tile_inject_launch_failure(719, 2, 1) == 0
        st = lib.tile_run_host_static_f32(tile.OPS[op], x0.data_ptr(), r0.data_ptr(),
                                          out0.data_ptr(), rows, width, EPS,
                                          streams[0].cuda_stream)
        assert st == -5 and lib.tile_last_cuda_error() == 719
    finally:
        assert lib.tile_inject_launch_failure(0, 0, 0) == 0
    _call_static(op, x1, r1, out1, streams[1].cuda_stream)
    torch.cuda.synchronize()
    _check(op, out1.numpy(), (x1, r1), values, f"{op} {rows}x{width} after a failed call")
    assert tile.tile_check_device_status() == 0


def test_static_staging_rejects_a_width_beyond_the_maximum():
    x = torch.zeros(2, 8).pin_memory()
    lib = tile.load()
    st = lib.tile_run_host_static_f32(1, x.data_ptr(), None, x.data_ptr() + 4096, 2,
                                      tile.tile_max_width() + 1, EPS, None)
    assert st == -2
