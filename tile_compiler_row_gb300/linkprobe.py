"""Host link and end-to-end path of residual LayerNorm FP32 (the figures of
``profiles/host_link_e2e_65536x4096.md``).

    python -m tile_compiler_row_gb300.linkprobe [--rows 65536] [--width 4096]

Prints one JSON object: the host->device and device->host copy rates of one
input tensor from pinned memory (one stream; several streams at once; both
directions at once), ``tile_run_host_f32`` on pageable inputs at several
chunk counts (the copy pipeline, direct stores into the pinned output) and
on all-pinned buffers (one kernel on the host buffers), and the device entry
point run on the pinned host pointers themselves (the kernel reads and
writes host memory over the link; its output bitwise that of the
device-resident call).  CUDA events,
one warm-up and ``--iters`` timed calls each; medians.
"""

from __future__ import annotations

import argparse
import json
import statistics
import sys


def main(argv=None) -> int:
    ap = argparse.ArgumentParser()
    ap.add_argument("--rows", type=int, default=65536)
    ap.add_argument("--width", type=int, default=4096)
    ap.add_argument("--iters", type=int, default=5)
    args = ap.parse_args(argv)

    import torch

    import synth
    import tile_compiler_row_gb300 as tile
    from tile_compiler_row_gb300 import _build
    _build.build()
    lib = tile.load()
    torch.cuda.set_device(0)
    rows, width, iters = args.rows, args.width, args.iters
    nbytes = rows * width * 4
    x_h = synth.rows_of(5, rows, width, which="x")
    r_h = synth.rows_of(5, rows, width, which="r")
    xp = torch.from_numpy(x_h).pin_memory()
    rp = torch.from_numpy(r_h).pin_memory()
    yp = torch.empty_like(xp).pin_memory()
    x, r = xp.cuda(), rp.cuda()
    y, yd = torch.empty_like(x), torch.empty_like(x)
    s = torch.cuda.current_stream()

    def timed(fn, streams=(None,)):
        """Median ms of fn over iters, events around all given streams."""
        fn()
        torch.cuda.synchronize()
        out = []
        for _ in range(iters):
            a = torch.cuda.Event(enable_timing=True)
            b = torch.cuda.Event(enable_timing=True)
            a.record(s)
            for st in streams:
                if st is not None:
                    st.wait_event(a)
            fn()
            for st in streams:
                if st is not None:
                    e = torch.cuda.Event()
                    e.record(st)
                    s.wait_event(e)
            b.record(s)
            torch.cuda.synchronize()
            out.append(a.elapsed_time(b))
        return statistics.median(out)

    res = {"rows": rows, "width": width, "tensor_bytes": nbytes}
    gbs = lambda b, ms: round(b / (ms * 1e-3) / 1e9, 1)

    ms = timed(lambda: x.copy_(xp, non_blocking=True))
    res["h2d"] = {"ms": round(ms, 3), "gbs": gbs(nbytes, ms)}
    ms = timed(lambda: yp.copy_(x, non_blocking=True))
    res["d2h"] = {"ms": round(ms, 3), "gbs": gbs(nbytes, ms)}
    side = torch.cuda.Stream()

    def both():
        x.copy_(xp, non_blocking=True)
        with torch.cuda.stream(side):
            yp.copy_(r, non_blocking=True)

    ms = timed(both, streams=(side,))
    res["both_directions"] = {"ms": round(ms, 3), "aggregate_gbs": gbs(2 * nbytes, ms)}
    for n in (2, 4):
        sts = [torch.cuda.Stream() for _ in range(n)]
        part = rows // n

        def split(sts=sts, part=part):
            for k, st in enumerate(sts):
                with torch.cuda.stream(st):
                    x[k * part:(k + 1) * part].copy_(xp[k * part:(k + 1) * part],
                                                     non_blocking=True)

        ms = timed(split, streams=tuple(sts))
        res[f"h2d_{n}_streams"] = {"ms": round(ms, 3), "gbs": gbs(nbytes, ms)}

    # tile_run_host_f32 at several chunk counts (workspace sized for the
    # chunk), on pageable inputs and the pinned output: the copy pipeline with
    # direct output stores (all-pinned buffers take the one-kernel path)
    code = tile.OPS["residual_layernorm"]
    xq = torch.from_numpy(x_h)
    rq = torch.from_numpy(r_h)
    res["host_pipeline_pageable_inputs"] = []
    for chunks in (16, 32, 64, 128):
        chunk_rows = max(1, rows // chunks)
        ws_bytes = tile.tile_host_workspace_bytes("residual_layernorm", width, chunk_rows)
        ws = torch.empty(ws_bytes, dtype=torch.uint8, device="cuda")
        used, slots = tile.tile_host_schedule("residual_layernorm", rows, width, ws_bytes,
                                              direct_output=True)

        def host(ws=ws):
            st = lib.tile_run_host_f32(code, xq.data_ptr(), rq.data_ptr(), yp.data_ptr(), rows,
                                       width, 1e-5, ws.data_ptr(), ws.numel(), s.cuda_stream)
            if st != 0:
                raise tile.TileError(st, "tile_run_host_f32")

        ms = timed(host)
        res["host_pipeline_pageable_inputs"].append(
            {"chunk_rows": used, "slots": slots, "ms": round(ms, 3), "gbs": gbs(3 * nbytes, ms)})
        del ws

    # tile_run_host_f32 on the all-pinned buffers (the one-kernel path; the
    # workspace is a real one of its stated size, though this path leaves it
    # untouched)
    ws = torch.empty(tile.tile_host_workspace_bytes("residual_layernorm", width,
                                                    max(1, rows // 16)),
                     dtype=torch.uint8, device="cuda")

    def host_pinned():
        st = lib.tile_run_host_f32(code, xp.data_ptr(), rp.data_ptr(), yp.data_ptr(), rows, width,
                                   1e-5, ws.data_ptr(), ws.numel(), s.cuda_stream)
        if st != 0:
            raise tile.TileError(st, "tile_run_host_f32")

    ms = timed(host_pinned)
    res["host_call_all_pinned"] = {"ms": round(ms, 3), "gbs": gbs(3 * nbytes, ms)}

    # the device entry point on the pinned host pointers (unified addresses)
    def direct(out):
        st = lib.tile_residual_layernorm_f32(xp.data_ptr(), rp.data_ptr(), out, rows, width,
                                             1e-5, s.cuda_stream)
        if st != 0:
            raise tile.TileError(st, "tile_residual_layernorm_f32")

    ms = timed(lambda: direct(yp.data_ptr()))
    res["kernel_on_host_memory"] = {"ms": round(ms, 3), "gbs": gbs(3 * nbytes, ms)}
    ms = timed(lambda: direct(yd.data_ptr()))
    res["kernel_reads_host_writes_device"] = {"ms": round(ms, 3),
                                              "input_gbs": gbs(2 * nbytes, ms)}
    tile.residual_layernorm(x, r, y)
    torch.cuda.synchronize()
    res["direct_output_bitwise_equal"] = bool(torch.equal(yp.cuda(), y))
    print(json.dumps(res), flush=True)
    return 0


if __name__ == "__main__":
    sys.exit(main())
