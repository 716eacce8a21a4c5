"""Measured plan sweep: time every built plan that covers a shape.

The width->plan selector of the library is a table frozen from this sweep
(measurement picks the mapping, not an analytic score).  For each
(op, rows, width) every covering float4 plan is timed with CUDA events on
the current stream: ``--warmup`` calls, then ``--iters`` calls, median of
the per-call times.  The two fastest plans are then timed again in
alternating order (A B B A); the spread of A's two runs is the A/A noise
floor that B's margin over A is read against (``confirm`` in each entry).  Inputs are uniform random device tensors; only timing
is recorded here (parity of every plan is covered by the GPU tests).

    python -m tile_compiler_row_gb300.sweep --out sweep.json [--quick]
"""

from __future__ import annotations

import argparse
import json
import statistics
import sys

OPS = ("residual_layernorm", "layernorm", "rmsnorm", "softmax")
MORE_OPS = ("row_sum", "row_minmax", "layernorm_affine", "rmsnorm_weighted")
#: algorithmic bytes per element (row outputs and gamma/beta are negligible)
BYTES = {"residual_layernorm": 12, "layernorm": 8, "rmsnorm": 8, "softmax": 8, "row_sum": 4,
         "row_minmax": 4, "layernorm_affine": 8, "rmsnorm_weighted": 8,
         "layernorm_affine+residual": 12}

#: widths of the sweep ladder; ``rows`` fills about 2**26 elements per tensor
#: (256 MiB, well above L2) so the large-row regime is HBM bound.
LADDER = (64, 127, 257, 512, 1024, 1537, 2048, 3072, 4096, 6144, 8192, 12288, 16384,
          32768, 65536, 131072)
#: the small shapes of the workloads (L2 resident).
SMALL = ((1, 127), (17, 257), (7, 1537), (64, 4096), (1024, 4096), (128, 8192),
         (32, 65536))


def shapes(quick=False, elems_log2=26):
    """The ladder at about 2**elems_log2 elements per tensor (256 MiB of FP32
    at 26, of BF16 at 27: twice the 129 MB L2), then the small shapes."""
    out = []
    ladder = LADDER if not quick else (257, 1024, 4096, 8192, 65536)
    for w in ladder:
        out.append((max(16, (1 << elems_log2) // w), w))
    out.extend(SMALL)
    return out


def time_call(call, warmup, iters, stream, graph=False, cutoff=None):
    """Median microseconds per call of ``call(s)`` (s: the raw CUDA stream
    to launch on).  With ``cutoff`` (µs), a call whose first timing after
    one warm-up already takes longer is not timed further: that single
    call's time is returned."""
    import torch

    s = stream.cuda_stream
    if cutoff is not None and not graph:
        call(s)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        call(s)
        e1.record(stream)
        torch.cuda.synchronize()
        first = e0.elapsed_time(e1) * 1e3
        if first > cutoff:
            return first
    for _ in range(warmup):
        call(s)
    if graph:
        # ``iters`` calls captured in one CUDA graph and replayed: the time per
        # call without host launch overhead (what back-to-back device work sees)
        cap = torch.cuda.Stream()
        torch.cuda.synchronize()
        cg = torch.cuda.CUDAGraph()
        with torch.cuda.graph(cg, stream=cap):
            for _ in range(iters):
                call(cap.cuda_stream)
        cg.replay()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(3):
            cg.replay()
        e1.record(stream)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) * 1e3 / (3 * iters)
    evs = [torch.cuda.Event(enable_timing=True) for _ in range(iters + 1)]
    evs[0].record(stream)
    for i in range(iters):
        call(s)
        evs[i + 1].record(stream)
    torch.cuda.synchronize()
    per = [evs[i].elapsed_time(evs[i + 1]) * 1e3 for i in range(iters)]
    return statistics.median(per)


def time_plan(lib, op_code, plan, x, r, y, rows, width, warmup, iters, stream, g=None, y2=None,
              graph=False, cutoff=None, b=None):
    """Median microseconds per call of forward plan ``plan`` (time_call)."""
    import ctypes

    import torch

    import tile_compiler_row_gb300 as tile
    a = tile.TileRowArgs()
    a.in_, a.out = x.data_ptr(), y.data_ptr()
    a.residual = r.data_ptr() if r is not None else None
    a.gamma = g.data_ptr() if g is not None else None
    a.beta = b.data_ptr() if b is not None else None
    a.out2 = y2.data_ptr() if y2 is not None else None
    a.rows, a.width, a.eps = rows, width, 1e-5
    a.dtype = {torch.bfloat16: 1, torch.float16: 2}.get(x.dtype, 0)
    ref = ctypes.byref(a)

    def call(s):
        st = lib.tile_run_plan_args_f32(op_code, plan, ref, s)
        if st != 0:
            raise RuntimeError(f"plan {plan}: status {st}")

    return time_call(call, warmup, iters, stream, graph, cutoff)


#: ops whose calls take the residual in a sweep: residual LayerNorm always;
#: affine LayerNorm is timed without one (tile_describe_plan_ex describes
#: that call).
USES_RESIDUAL = ("residual_layernorm",)


def make_tensors(rows, width, dtype):
    """Uniform random device inputs of one sweep shape, seeded by the shape."""
    import torch
    gen = torch.Generator(device="cuda").manual_seed(rows * 131 + width)
    x = torch.rand(rows, width, device="cuda", generator=gen) * 2 - 1
    r = torch.rand(rows, width, device="cuda", generator=gen) * 2 - 1
    if dtype != "f32":
        t = torch.bfloat16 if dtype == "bf16" else torch.float16
        x, r = x.to(t), r.to(t)
    return {"x": x, "r": r, "y": torch.empty_like(x),
            "g": torch.rand(width, device="cuda", generator=gen) + 0.5,
            "b": torch.rand(width, device="cuda", generator=gen) - 0.5,
            "y2": torch.empty(rows, device="cuda")}


def sweep_entry(lib, op, dtype, rows, width, t, warmup, iters, stream, graph=False,
                only=None, beta=False):
    """Every covering 16-byte-vector plan of ``op`` at one shape, timed (µs,
    median); then the two fastest again in alternating order A B B A: the two
    runs of A give the A/A noise floor that B's margin is read against.
    ``beta``: affine LayerNorm called with a beta vector as well (the tables
    are swept without one)."""
    import tile_compiler_row_gb300 as tile
    base = op.split("+")[0]          # "layernorm_affine+residual": with a residual
    code = tile.OPS[base]
    r = t["r"] if (op in USES_RESIDUAL or op.endswith("+residual")) else None
    # the selector's choice, where tile_describe_plan_ex can describe the call
    chosen = tile.tile_describe_plan_ex(base, dtype, rows, width)["id"] if base == op else None
    bvec = t["b"] if beta and base == "layernorm_affine" else None
    entry = {"op": op, "rows": rows, "width": width, "selected": chosen, "plans": {},
             "dtype": dtype, "beta": bvec is not None,
             "timing": "cuda graph replay" if graph else "back-to-back launches"}
    for pid in range(tile.tile_plan_count()):
        info = tile.tile_plan_info_ex(pid, base, dtype, rows, width)
        if info is None or info["vec"] == 1 or info["grid"] > 0x7FFFFFFF:
            continue
        if only is not None and pid not in only:
            continue
        best_so_far = min(entry["plans"].values(), default=None)
        us = time_plan(lib, code, pid, t["x"], r, t["y"], rows, width, warmup, iters, stream,
                       g=t["g"], y2=t["y2"], graph=graph,
                       cutoff=None if best_so_far is None else 3.0 * best_so_far, b=bvec)
        entry["plans"][pid] = round(us, 3)
    best = min(entry["plans"], key=entry["plans"].get)
    ranked = sorted(entry["plans"], key=entry["plans"].get)
    if len(ranked) >= 2:
        a, b = ranked[0], ranked[1]
        rerun = {a: [], b: []}
        for pid in (a, b, b, a):
            rerun[pid].append(round(time_plan(lib, code, pid, t["x"], r, t["y"], rows, width,
                                              warmup, iters, stream, g=t["g"], y2=t["y2"],
                                              graph=graph, b=bvec), 3))
        entry["confirm"] = {
            "order": [a, b, b, a], "us": {str(a): rerun[a], str(b): rerun[b]},
            "aa_noise": round(abs(rerun[a][0] - rerun[a][1]) / min(rerun[a]), 4),
            "margin": round(min(rerun[b]) / min(rerun[a]) - 1.0, 4)}
    entry["best"] = best
    scale = 0.5 if dtype != "f32" else 1.0      # 2-byte elements
    entry["best_gbs"] = round(scale * BYTES[op] * rows * width / (entry["plans"][best] * 1e-6)
                              / 1e9, 1)
    entry["selected_over_best"] = (round(entry["plans"][chosen] / entry["plans"][best], 4)
                                   if chosen is not None and chosen in entry["plans"] else None)
    return entry


#: backward ops of the sweeps (the library's op name + "_backward")
BWD_OPS = ("layernorm_backward", "rmsnorm_backward", "softmax_backward")


def sweep_backward_entry(lib, op, dtype, rows, width, t, warmup, iters, stream):
    """Every covering 16-byte-vector register plan of backward ``op`` at one
    shape (LayerNorm and RMSNorm with gamma and row statistics; softmax on
    the tensors as given), timed and rerun as ``sweep_entry`` does."""
    import torch

    import tile_compiler_row_gb300 as tile
    base = op[:-len("_backward")]
    code = tile.OPS[base]
    dcode = {"f32": 0, "bf16": 1, "f16": 2}[dtype]
    chosen = tile.tile_describe_backward_plan(base, dtype, rows, width)["id"]
    norm = base != "softmax"
    stats = torch.empty(2 * rows, device="cuda") if norm else None
    x, dy, dx = t["x"], t["r"], t["y"]
    g = t["g"] if norm else None

    def caller(pid):
        def call(s):
            st = lib.tile_run_backward_plan_ex(
                code, pid, dcode, x.data_ptr(), g.data_ptr() if g is not None else None,
                dy.data_ptr(), dx.data_ptr(), stats.data_ptr() if stats is not None else None,
                rows, width, 1e-5, s)
            if st != 0:
                raise RuntimeError(f"backward plan {pid}: status {st}")
        return call

    entry = {"op": op, "rows": rows, "width": width, "selected": chosen, "plans": {},
             "dtype": dtype, "timing": "back-to-back launches"}
    for pid in range(tile.tile_plan_count()):
        info = tile.tile_plan_info_ex(pid, base, dtype, rows, width)
        if info is None or info["vec"] == 1 or info["path"] in (2, 3) \
                or info["grid"] > 0x7FFFFFFF:
            continue
        # a register plan the backward kernels do not build returns TILE_ERR_PLAN
        # before launching anything
        st = lib.tile_run_backward_plan_ex(code, pid, dcode, None, None, None, None, None,
                                           0, width, 1e-5, None)
        if st != 0:
            continue
        best_so_far = min(entry["plans"].values(), default=None)
        entry["plans"][pid] = round(time_call(
            caller(pid), warmup, iters, stream,
            cutoff=None if best_so_far is None else 3.0 * best_so_far), 3)
    ranked = sorted(entry["plans"], key=entry["plans"].get)
    if len(ranked) >= 2:
        a, b = ranked[0], ranked[1]
        rerun = {a: [], b: []}
        for pid in (a, b, b, a):
            rerun[pid].append(round(time_call(caller(pid), warmup, iters, stream), 3))
        entry["confirm"] = {
            "order": [a, b, b, a], "us": {str(a): rerun[a], str(b): rerun[b]},
            "aa_noise": round(abs(rerun[a][0] - rerun[a][1]) / min(rerun[a]), 4),
            "margin": round(min(rerun[b]) / min(rerun[a]) - 1.0, 4)}
    entry["best"] = ranked[0]
    entry["selected_over_best"] = (round(entry["plans"][chosen] / entry["plans"][ranked[0]], 4)
                                   if chosen in entry["plans"] else None)
    return entry


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--out", default=None)
    ap.add_argument("--quick", action="store_true")
    ap.add_argument("--ops", default=",".join(OPS))
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--iters", type=int, default=30)
    ap.add_argument("--shapes", default=None, help="comma list of ROWSxWIDTH (default: ladder)")
    ap.add_argument("--graph", action="store_true",
                    help="time calls replayed from a CUDA graph (no host launch overhead)")
    ap.add_argument("--small", action="store_true", help="only the small workload shapes")
    ap.add_argument("--dtype", default="f32", choices=("f32", "bf16", "f16"))
    ap.add_argument("--beta", action="store_true",
                    help="call affine LayerNorm with a beta vector too")
    ap.add_argument("--plans", default=None,
                    help="comma list of plan ids to time (default: every covering plan)")
    args = ap.parse_args(argv)
    only = None if args.plans is None else {int(p) for p in args.plans.split(",")}

    import torch

    import tile_compiler_row_gb300 as tile
    from tile_compiler_row_gb300 import _build
    _build.build()
    lib = tile.load()
    torch.cuda.set_device(0)
    stream = torch.cuda.current_stream()
    results = []
    todo = shapes(args.quick, 26 if args.dtype == "f32" else 27) if args.shapes is None else \
        [tuple(int(v) for v in sh.split("x")) for sh in args.shapes.split(",")]
    if args.small:
        todo = list(SMALL)
    for rows, width in todo:
        t = make_tensors(rows, width, args.dtype)
        for op in args.ops.split(","):
            entry = sweep_entry(lib, op, args.dtype, rows, width, t, args.warmup, args.iters,
                                stream, graph=args.graph, only=only, beta=args.beta)
            results.append(entry)
            print(json.dumps(entry), flush=True)
        del t
    assert tile.tile_check_device_status() == 0
    if args.out:
        with open(args.out, "w") as fh:
            json.dump(results, fh, indent=1)
    return results


if __name__ == "__main__":
    sys.exit(0 if main() is not None else 1)
