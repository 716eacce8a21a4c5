"""Evidence for the width->plan selector: a measured sweep of every bucket
of the selector's tables, and its summary.

The selector maps (op, element type, rows, width) to a plan through tables
frozen from measured sweeps (measurement, not an analytic score, picks the
mapping).  This module reads the buckets back from the library itself
(``tile_describe_plan_ex`` over every width of whole 16-byte vectors: 4
FP32 or 8 BF16/FP16 elements), picks one representative width per bucket
(a width of the sweep ladder inside it when there is one, else the
bucket's widest), and times every covering plan there with
``sweep.sweep_entry``: CUDA events, median of back-to-back calls on about
2**26 FP32 (2**27 2-byte) elements per tensor, then the two fastest again
in the order A B B A for the A/A noise floor and the runner-up's margin.
The small, L2-resident workload shapes are timed the same way from CUDA
graph replays.  ``summary`` writes the table that
``tests/test_selector_evidence.py`` checks the selector against.

    python -m tile_compiler_row_gb300.selector_evidence sweep --out ev.json
    python -m tile_compiler_row_gb300.selector_evidence summary ev.json > profiles/selector_sweep.md
"""

from __future__ import annotations

import argparse
import json
import sys

#: ops the selector has tables for (names of the library's op codes)
OPS = ("residual_layernorm", "layernorm", "rmsnorm", "softmax", "row_sum", "row_minmax",
       "layernorm_affine", "rmsnorm_weighted")
DTYPES = ("f32", "bf16", "f16")
#: backward ops of the selector's backward tables
BWD_OPS = ("layernorm_backward", "rmsnorm_backward", "softmax_backward")
#: widths preferred as a bucket's representative (whole 16-byte vectors)
LADDER = (64, 128, 256, 512, 1024, 1536, 2048, 3072, 4096, 6144, 8192, 12288, 16384, 32768,
          65536, 131072)
#: rows of the scan of the large-problem tables (rows * width above 2**22)
SCAN_ROWS = 1 << 24
#: the small, L2-resident workload shapes (FP32 only has small-problem tables)
SMALL = ((1, 128), (17, 256), (7, 1536), (64, 4096), (1024, 4096), (128, 8192), (32, 65536))


def vec(dtype):
    return 4 if dtype == "f32" else 8


def describe(op, dtype, rows, width):
    """The plan the library takes for a call (backward ops through
    tile_describe_backward_plan)."""
    import tile_compiler_row_gb300 as tile
    if op in BWD_OPS:
        return tile.tile_describe_backward_plan(op[:-len("_backward")], dtype, rows, width)
    return tile.tile_describe_plan_ex(op, dtype, rows, width)


def buckets(op, dtype):
    """[(lo, hi, plan)]: the plan the library describes for widths of whole
    16-byte vectors, in runs of equal plans.  Host only."""
    import tile_compiler_row_gb300 as tile
    out = []
    ev = vec(dtype)
    for w in range(ev, tile.tile_max_width() + 1, ev):
        pid = describe(op, dtype, SCAN_ROWS, w)["id"]
        if out and out[-1][2] == pid:
            out[-1][1] = w
        else:
            out.append([w, w, pid])
    return [tuple(b) for b in out]


def representative(lo, hi):
    inside = [w for w in LADDER if lo <= w <= hi]
    return max(inside) if inside else hi


def sweep_rows(dtype, width):
    return max(16, (1 << (26 if dtype == "f32" else 27)) // width)


def plan_cases():
    """{(dtype, width): [(op, lo, hi, plan)]}: the representative shape of
    every bucket, grouped so each shape's tensors are made once."""
    todo = {}
    for dtype in DTYPES:
        for op in OPS + BWD_OPS:
            for lo, hi, pid in buckets(op, dtype):
                todo.setdefault((dtype, representative(lo, hi)), []).append((op, lo, hi, pid))
    return todo


def run_sweep(out, warmup=5, iters=30):
    import torch

    import tile_compiler_row_gb300 as tile
    from tile_compiler_row_gb300 import _build
    from tile_compiler_row_gb300.sweep import make_tensors, sweep_backward_entry, sweep_entry
    _build.build()
    lib = tile.load()
    torch.cuda.set_device(0)
    stream = torch.cuda.current_stream()
    records = []
    for (dtype, width), cases in sorted(plan_cases().items()):
        rows = sweep_rows(dtype, width)
        t = make_tensors(rows, width, dtype)
        for op, lo, hi, pid in cases:
            if op in BWD_OPS:
                e = sweep_backward_entry(lib, op, dtype, rows, width, t, warmup, iters, stream)
            else:
                e = sweep_entry(lib, op, dtype, rows, width, t, warmup, iters, stream)
            e.update({"regime": "large", "bucket": [lo, hi]})
            assert e["selected"] == pid
            records.append(e)
            print(json.dumps(e), flush=True)
        del t
    for rows, width in SMALL:
        t = make_tensors(rows, width, "f32")
        for op in OPS:
            e = sweep_entry(lib, op, "f32", rows, width, t, warmup, 200, stream, graph=True)
            e.update({"regime": "small"})
            records.append(e)
            print(json.dumps(e), flush=True)
        del t
    assert tile.tile_check_device_status() == 0
    with open(out, "w") as fh:
        json.dump(records, fh, indent=1)


def _cell(e):
    c = e.get("confirm")
    ranked = sorted(e["plans"], key=e["plans"].get)
    second = ranked[1] if len(ranked) > 1 else None
    sel = str(e["selected"])
    return {
        "selected": e["selected"], "sel_us": e["plans"][sel],
        "best": e["best"], "best_us": e["plans"][str(e["best"])],
        "second": second if second is None else int(second),
        "second_us": e["plans"][second] if second is not None else None,
        "aa": c["aa_noise"] if c else None, "margin": c["margin"] if c else None,
        "ratio": e["selected_over_best"],
    }


def summary(paths):
    records = []
    for p in paths:
        with open(p) as fh:
            records.extend(json.load(fh))
    lines = [
        "# Selector evidence: every bucket of the width->plan tables, measured",
        "",
        "The selector's tables map (op, element type, width) to a built plan. Each",
        "row below is one bucket as the library reports it (`tile_describe_plan_ex`",
        "over widths of whole 16-byte vectors; `rows * width` above 2^22, the large-",
        "problem tables), timed at one representative width: every covering plan,",
        "CUDA events, median of 30 back-to-back calls after 5 warm-up calls, about",
        "2^26 FP32 (2^27 BF16/FP16) elements per tensor (inputs larger than L2).",
        "`best` and `2nd` are the two fastest plans; they were timed again in the",
        "order A B B A: `A/A` is the spread of the best plan's two reruns, `margin`",
        "the runner-up's excess over the best. `sel/best` is the selected plan's",
        "time over the best plan's (1 = the selector picked the fastest).",
        "Affine LayerNorm is timed without a residual (the call",
        "`tile_describe_plan_ex` describes); BF16/FP16 rows of whole vectors on",
        "16-byte aligned pointers may take the shared-memory-staged plans (40-52).",
        "The second table is the small, L2-resident workload shapes (FP32), timed",
        "from CUDA graph replays of 200 calls.",
        "",
        "Over all rows: {n} buckets and shapes, selected/best mean {mean:.4f},",
        "maximum {worst:.4f}; {over3} rows above 1.03.",
        "",
        "Command (one GB300):",
        "",
        "    python -m tile_compiler_row_gb300.selector_evidence sweep --out ev.json",
        "    python -m tile_compiler_row_gb300.selector_evidence summary ev.json",
        "",
        "The selector's tables were generated from other sweeps",
        "(`tile_compiler_row_gb300/selector_tables.py`); this one is an independent",
        "run on another GB300 lease. tests/test_selector_evidence.py parses the",
        "tables: the library must still select the recorded plan at every row's",
        "shape, and every selected plan must be within 5 % of the fastest.",
        "",
        "## Large problems",
        "",
        "| op | dtype | widths | width | rows | selected | µs | best | µs | 2nd | µs | A/A | margin | sel/best |",
        "|---|---|---|---:|---:|---:|---:|---:|---:|---:|---:|---:|---:|---:|",
    ]

    ratios = [e["selected_over_best"] for e in records]
    lines = [ln.format(n=len(ratios), mean=sum(ratios) / len(ratios), worst=max(ratios),
                       over3=sum(r > 1.03 for r in ratios)) if "{" in ln else ln
             for ln in lines]

    def fmt(v, nd=3):
        return "—" if v is None else (f"{v:.{nd}f}" if isinstance(v, float) else str(v))

    for e in records:
        if e.get("regime") != "large" or e["op"] in BWD_OPS:
            continue
        c = _cell(e)
        lo, hi = e["bucket"]
        lines.append(
            f"| {e['op']} | {e['dtype']} | {lo}-{hi} | {e['width']} | {e['rows']} | "
            f"{c['selected']} | {fmt(c['sel_us'], 2)} | {c['best']} | {fmt(c['best_us'], 2)} | "
            f"{fmt(c['second'])} | {fmt(c['second_us'], 2)} | {fmt(c['aa'], 4)} | "
            f"{fmt(c['margin'], 4)} | {c['ratio']:.4f} |")
    lines += ["", "## Backward", "",
              "LayerNorm and RMSNorm backward with gamma and row statistics, softmax",
              "backward; every covering register plan the backward kernels build, timed",
              "as above (`tile_describe_backward_plan` gives the selected plan).", "",
              "| op | dtype | widths | width | rows | selected | µs | best | µs | 2nd | µs | A/A | margin | sel/best |",
              "|---|---|---|---:|---:|---:|---:|---:|---:|---:|---:|---:|---:|---:|"]
    for e in records:
        if e.get("regime") != "large" or e["op"] not in BWD_OPS:
            continue
        c = _cell(e)
        lo, hi = e["bucket"]
        lines.append(
            f"| {e['op']} | {e['dtype']} | {lo}-{hi} | {e['width']} | {e['rows']} | "
            f"{c['selected']} | {fmt(c['sel_us'], 2)} | {c['best']} | {fmt(c['best_us'], 2)} | "
            f"{fmt(c['second'])} | {fmt(c['second_us'], 2)} | {fmt(c['aa'], 4)} | "
            f"{fmt(c['margin'], 4)} | {c['ratio']:.4f} |")
    lines += ["", "## Small problems (L2-resident, CUDA graph replay)", "",
              "| op | dtype | shape | selected | µs | best | µs | 2nd | µs | A/A | margin | sel/best |",
              "|---|---|---|---:|---:|---:|---:|---:|---:|---:|---:|---:|"]
    for e in records:
        if e.get("regime") != "small":
            continue
        c = _cell(e)
        lines.append(
            f"| {e['op']} | {e['dtype']} | {e['rows']}x{e['width']} | {c['selected']} | "
            f"{fmt(c['sel_us'], 3)} | {c['best']} | {fmt(c['best_us'], 3)} | "
            f"{fmt(c['second'])} | {fmt(c['second_us'], 3)} | {fmt(c['aa'], 4)} | "
            f"{fmt(c['margin'], 4)} | {c['ratio']:.4f} |")
    return "\n".join(lines) + "\n"


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__,
                                 formatter_class=argparse.RawDescriptionHelpFormatter)
    sub = ap.add_subparsers(dest="cmd", required=True)
    sw = sub.add_parser("sweep")
    sw.add_argument("--out", required=True)
    sm = sub.add_parser("summary")
    sm.add_argument("paths", nargs="+")
    args = ap.parse_args(argv)
    if args.cmd == "sweep":
        run_sweep(args.out)
    else:
        sys.stdout.write(summary(args.paths))
    return 0


if __name__ == "__main__":
    sys.exit(main())
