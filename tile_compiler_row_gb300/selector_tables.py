"""Generate the selector's width->plan tables from a measured plan sweep.

Measurement, not an analytic score, picks each mapping.  ``sweep`` times
every built plan that covers a width of the ladder below, for every table
op and both element families (FP32; BF16, whose tables FP16 rows share),
on about 2**26 FP32 (2**27 2-byte) elements per tensor, plus the small,
L2-resident workload shapes (FP32, CUDA graph replay).  ``emit`` turns the
sweep into ``csrc/selector_tables.h``:

* one register-plan table per (family, op): the bucket of ladder width w
  holds the widths (previous ladder width, w + tail], with tail = one
  16-byte vector less one element (3 FP32, 7 BF16), and takes the fastest
  register plan measured at w, or the plan built before if that one is
  within 0.5 % of the fastest (measurement noise does not flip a choice);
* one whole-vector-plan table per (family, op): the fastest plan among
  those that need 16-byte aligned rows of whole vectors (the shared-memory-
  staged plans and the R-rows-per-CTA plans) at w where it beat the fastest
  register plan by more than 1 % (-1 elsewhere); calls take it only on such
  rows;
* one register-plan table per (family, backward op) for LayerNorm, RMSNorm
  and softmax backward (with gamma and row statistics), chosen as the
  forward register tables are;
* two small-problem tables per op (FP32, L2-resident): "tiny" for
  rows * width <= 2**19, "small" up to 2**22.  At the ladder bucket of each
  small workload width of the tier, the plan fastest over that width's
  workloads when it beats the large-problem choice there by more than 1 %
  (-1 elsewhere: the large-problem table).

Several sweeps may be given: each plan's time at a shape is then the mean
of the runs that timed it (plans built after an older sweep count from the
newer ones only), and FP16 runs count for the 2-byte tables with the BF16
ones (the two types share the tables).

    python -m tile_compiler_row_gb300.selector_tables sweep --out tables.json   (GPU)
    python -m tile_compiler_row_gb300.selector_tables sweep --family bf16 --out b16.json
    python -m tile_compiler_row_gb300.selector_tables sweep --family f16 --out f16.json
    python -m tile_compiler_row_gb300.selector_tables emit tables.json          (writes the header)

``sweeps/selector_sweeps.json.gz`` holds the sweeps the committed header was
generated from; ``emit`` with no file regenerates it from them.
"""

from __future__ import annotations

import argparse
import json
import os
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
HEADER = os.path.join(HERE, "csrc", "selector_tables.h")
#: the committed sweeps the header was generated from
SWEEPS = os.path.join(HERE, "sweeps", "selector_sweeps.json.gz")

#: ops with their own tables.  "layernorm_affine+residual" is affine
#: LayerNorm called with a residual (a different stream count).
TABLE_OPS = ("residual_layernorm", "layernorm", "rmsnorm", "softmax", "row_sum", "row_minmax",
             "layernorm_affine", "rmsnorm_weighted", "layernorm_affine+residual")
#: C++ name stem of each table op
STEM = {"residual_layernorm": "ResidualLN", "layernorm": "LN", "rmsnorm": "RMS",
        "softmax": "Softmax", "row_sum": "RowSum", "row_minmax": "RowMinmax",
        "layernorm_affine": "Affine", "rmsnorm_weighted": "Weighted",
        "layernorm_affine+residual": "ResidualAffine"}
#: backward ops with their own register-plan tables (no whole-vector plans)
BWD_OPS = ("layernorm_backward", "rmsnorm_backward", "softmax_backward")
STEM.update({"layernorm_backward": "BwdLN", "rmsnorm_backward": "BwdRMS",
             "softmax_backward": "BwdSoftmax"})
FAMILIES = {"f32": "F32", "bf16": "B16"}
LADDER = {"f32": (128, 256, 512, 1024, 1536, 2048, 3072, 3584, 4096, 6144, 8192, 12288, 16384,
                  32768, 65536, 131072),
          "bf16": (128, 256, 512, 1024, 1536, 2048, 3072, 4096, 6144, 8192, 12288, 16384, 32768,
                   65536, 131072)}
TAIL = {"f32": 3, "bf16": 7}
MAX_WIDTH = 131072
#: the small, L2-resident workload shapes (rows, width)
SMALL = ((1, 127), (17, 257), (7, 1537), (64, 4096), (1024, 4096), (128, 8192), (32, 65536))
KEEP = 0.005       # keep the previous plan within 0.5 % of the fastest
STAGED_WIN = 0.01  # a staged plan must win by more than 1 %
SMALL_WIN = 0.01
FIRST_STAGED = 40  # ids of the whole-vector plans (staged, then R rows per CTA) start here


def sweep_rows(dtype, width):
    return max(16, (1 << (26 if dtype == "f32" else 27)) // width)


def run_sweep(out, warmup=5, iters=30, forward=True, backward=True, families=tuple(FAMILIES)):
    import torch

    import tile_compiler_row_gb300 as tile
    from tile_compiler_row_gb300 import _build
    from tile_compiler_row_gb300.sweep import make_tensors, sweep_backward_entry, sweep_entry
    _build.build()
    lib = tile.load()
    torch.cuda.set_device(0)
    stream = torch.cuda.current_stream()
    records = []
    for dtype in families:
        for width in LADDER[family(dtype)]:
            rows = sweep_rows(dtype, width)
            t = make_tensors(rows, width, dtype)
            for op in (TABLE_OPS if forward else ()) + (BWD_OPS if backward else ()):
                if op in BWD_OPS:
                    e = sweep_backward_entry(lib, op, dtype, rows, width, t, warmup, iters, stream)
                else:
                    e = sweep_entry(lib, op, dtype, rows, width, t, warmup, iters, stream)
                e["regime"] = "large"
                records.append(e)
                print(json.dumps(e), flush=True)
            del t
    for rows, width in (SMALL if forward and "f32" in families else ()):
        t = make_tensors(rows, width, "f32")
        for op in TABLE_OPS:
            e = sweep_entry(lib, op, "f32", rows, width, t, warmup, 200, stream, graph=True)
            e["regime"] = "small"
            records.append(e)
            print(json.dumps(e), flush=True)
        del t
    assert tile.tile_check_device_status() == 0
    with open(out, "w") as fh:
        json.dump(records, fh, indent=1)


def _fastest(plans, pred):
    cand = {int(k): v for k, v in plans.items() if pred(int(k))}
    if not cand:
        return None, None
    pid = min(cand, key=lambda q: (cand[q], q))      # equal times: the lower id
    return pid, cand[pid]


def _bound(dtype, width):
    return MAX_WIDTH if width == LADDER[dtype][-1] else width + TAIL[dtype]


TINY_ELEMS = 1 << 19


def family(dtype):
    return "f32" if dtype == "f32" else "bf16"


def tier(rows, width):
    return "tiny" if rows * width <= TINY_ELEMS else "small"


def merged(entries):
    """One entry whose plan times are the means over the ``entries`` that
    timed each plan (a plan built after an older sweep counts from the
    newer ones only); "selected" is the first entry's."""
    plans = sorted(set().union(*(set(e["plans"]) for e in entries)), key=int)
    e = dict(entries[0])
    e["plans"] = {}
    for p in plans:
        times = [x["plans"][p] for x in entries if p in x["plans"]]
        e["plans"][p] = sum(times) / len(times)
    return e


def tables(records):
    """{(family, op): {"reg": [(max_width, plan)], "staged": [...]}} and
    {(tier, op): [(max_width, plan)]} for the small problems."""
    groups = {}
    for e in records:
        if e["regime"] == "large" and e["width"] in LADDER[family(e["dtype"])]:
            groups.setdefault((family(e["dtype"]), e["op"], e["width"]), []).append(e)
    large = {k: merged(v) for k, v in groups.items()}
    out = {}
    for dtype in FAMILIES:
        for op in TABLE_OPS:
            reg, stg = [], []
            for w in LADDER[dtype]:
                e = large[(dtype, op, w)]
                rid, rt = _fastest(e["plans"], lambda p: p < FIRST_STAGED)
                prev = e.get("selected")
                if prev is not None and prev < FIRST_STAGED and str(prev) in e["plans"] \
                        and e["plans"][str(prev)] <= rt * (1 + KEEP):
                    rid = prev
                sid, st = _fastest(e["plans"], lambda p: p >= FIRST_STAGED)
                reg.append((_bound(dtype, w), rid))
                stg.append((_bound(dtype, w),
                            sid if sid is not None and st < rt * (1 - STAGED_WIN) else -1))
            out[(dtype, op)] = {"reg": reg, "staged": stg}
        for op in BWD_OPS:
            if not any((dtype, op, w) in large for w in LADDER[dtype]):
                continue
            reg = []
            for w in LADDER[dtype]:
                e = large[(dtype, op, w)]
                rid, rt = _fastest(e["plans"], lambda p: p < FIRST_STAGED)
                prev = e.get("selected")
                if prev is not None and str(prev) in e["plans"] \
                        and e["plans"][str(prev)] <= rt * (1 + KEEP):
                    rid = prev
                reg.append((_bound(dtype, w), rid))
            out[(dtype, op)] = {"reg": reg, "staged": None}
    small = {}
    by_shape = {}
    for e in records:
        if e["regime"] == "small" and (e["rows"], e["width"]) in SMALL:
            by_shape.setdefault((e["op"], e["rows"], e["width"]), []).append(e)
    by_op = {}
    for (op, rows, width), v in by_shape.items():
        by_op.setdefault((tier(rows, width), op), []).append(merged(v))
    for (tr, op), entries in by_op.items():
        reg = out[("f32", op)]["reg"]
        pick = {}
        for w in sorted({e["width"] for e in entries}):
            group = [e for e in entries if e["width"] == w]
            bound, large_pick = next((b, p) for b, p in reg if w <= b)
            plans = set.intersection(*(set(e["plans"]) for e in group))
            plans = {p for p in plans if int(p) < FIRST_STAGED}

            def worst(p):
                return max(e["plans"][p] / min(v for k, v in e["plans"].items()
                                                if int(k) < FIRST_STAGED) for e in group)
            best = min(sorted(plans, key=int), key=lambda p: (worst(p), int(p)))
            base = worst(str(large_pick)) if str(large_pick) in plans else float("inf")
            if worst(best) * (1 + SMALL_WIN) < base:
                pick[bound] = int(best)
        # every bucket of the large table, -1 (use the large table) where no
        # small workload was measured or the large choice held
        small[(tr, op)] = [(b, pick.get(b, -1)) for b, _ in reg]
    return out, small


def committed_records(path=SWEEPS):
    """The sweep records the committed header was generated from."""
    import gzip
    with gzip.open(path, "rt") as fh:
        data = json.load(fh)
    return [e for run in data["runs"] for e in run]


def render(records):
    """The text of csrc/selector_tables.h for these sweep records."""
    big, small = tables(records)

    def arr(name, rows, comment=None):
        cells = ", ".join(f"{{{b}, {p}}}" for b, p in rows)
        return (f"// {comment}\n" if comment else "") + f"constexpr Bucket {name}[] = {{{cells}}};\n"

    parts = ["// Width->plan tables of the selector, generated by",
             "// tile_compiler_row_gb300/selector_tables.py from a measured plan sweep on GB300",
             "// (every built plan timed at each width of the ladder, CUDA events).  Do not edit:",
             "// re-run the sweep and the generator.  Bucket = {widest width, plan}; -1 = none.",
             "#pragma once", ""]
    for dtype, fam in FAMILIES.items():
        for op in TABLE_OPS:
            t = big[(dtype, op)]
            parts.append(arr(f"k{fam}Reg{STEM[op]}", t["reg"]))
            parts.append(arr(f"k{fam}Staged{STEM[op]}", t["staged"]))
        for op in BWD_OPS:
            if (dtype, op) in big:
                parts.append(arr(f"k{fam}Reg{STEM[op]}", big[(dtype, op)]["reg"]))
    for tr, name in (("tiny", "Tiny"), ("small", "Small")):
        for op in TABLE_OPS:
            parts.append(arr(f"kF32{name}{STEM[op]}", small.get((tr, op), [(MAX_WIDTH, -1)])))
    return "\n".join(parts)


def emit(records, path=HEADER):
    with open(path, "w") as fh:
        fh.write(render(records))
    return path


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__,
                                 formatter_class=argparse.RawDescriptionHelpFormatter)
    sub = ap.add_subparsers(dest="cmd", required=True)
    sw = sub.add_parser("sweep")
    sw.add_argument("--out", required=True)
    sw.add_argument("--only", choices=("forward", "backward"), default=None)
    sw.add_argument("--family", choices=tuple(FAMILIES) + ("f16",), default=None,
                    help="sweep one element type (default: FP32 and BF16; FP16 records count "
                         "with the BF16 ones)")
    em = sub.add_parser("emit", help="sweep JSON files -> the header (default: the "
                                       "committed sweeps)")
    em.add_argument("paths", nargs="*")
    em.add_argument("--header", default=HEADER)
    args = ap.parse_args(argv)
    if args.cmd == "sweep":
        run_sweep(args.out, forward=args.only != "backward", backward=args.only != "forward",
                  families=(args.family,) if args.family else tuple(FAMILIES))
    else:
        records = []
        for p in args.paths:
            with open(p) as fh:
                records.extend(json.load(fh))
        print(emit(records or committed_records(), args.header))
    return 0


if __name__ == "__main__":
    sys.exit(main())
