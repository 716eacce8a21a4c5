"""Throughput of every operation of the library at one shape.

For each op: ``--warmup`` calls, then ``--iters`` calls timed one by one
with CUDA events on the current stream; the mean call time gives the
achieved bandwidth from the op's algorithmic bytes (each input element read
once, each output element written once), reported against the measured HBM
copy bandwidth.  Inputs are uniform random device tensors (timing only;
parity is covered by the GPU tests).  The default 65536 x 4096 shape keeps
every working set far above the 129 MB L2.

    python -m tile_compiler_row_gb300.opsbench [--rows R --width W] [--json out.json]
"""

from __future__ import annotations

import argparse
import json
import os
import statistics
import sys


def measured_hbm_gbs():
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    try:
        with open(os.path.join(root, "MEASURED_PEAKS.json")) as fh:
            return float(json.load(fh)["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return 6800.0, "fallback"


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--rows", type=int, default=65536)
    ap.add_argument("--width", type=int, default=4096)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--iters", type=int, default=50)
    ap.add_argument("--json", default=None)
    ap.add_argument("--only", default=None, help="comma list of op names")
    args = ap.parse_args(argv)

    import torch

    import tile_compiler_row_gb300 as tile
    from tile_compiler_row_gb300 import _build
    _build.build()
    tile.load()
    torch.cuda.set_device(0)
    rows, width = args.rows, args.width
    n = rows * width
    gen = torch.Generator(device="cuda").manual_seed(7)
    x = torch.rand(rows, width, device="cuda", generator=gen) * 2 - 1
    r = torch.rand(rows, width, device="cuda", generator=gen) * 2 - 1
    y = torch.empty_like(x)
    y2 = torch.empty_like(x)
    g = torch.rand(width, device="cuda", generator=gen) + 0.5
    b = torch.rand(width, device="cuda", generator=gen) - 0.5
    vec_a = torch.empty(rows, device="cuda")
    vec_b = torch.empty(rows, device="cuda")
    stats = torch.empty(2 * rows, device="cuda")
    xb, rb, yb = x.to(torch.bfloat16), r.to(torch.bfloat16), torch.empty_like(x, dtype=torch.bfloat16)
    xh, rh, yh = x.to(torch.float16), r.to(torch.float16), torch.empty_like(x, dtype=torch.float16)
    ws = torch.empty(tile.tile_norm_param_grad_workspace_bytes(rows, width), dtype=torch.uint8,
                     device="cuda")
    dg, db = torch.empty(width, device="cuda"), torch.empty(width, device="cuda")
    # softmax backward wants a softmax output
    tile.tile_softmax_f32(x, y2)
    sm = y2.clone()
    smb = sm.to(torch.bfloat16)
    smh = sm.to(torch.float16)
    tile.tile_layernorm_backward_f32(x, None, r, y, stats)

    ops = {
        # name: (callable, algorithmic bytes per element, plan description)
        "residual_layernorm": (lambda: tile.tile_residual_layernorm_f32(x, r, y), 12),
        "layernorm": (lambda: tile.tile_layernorm_f32(x, y), 8),
        "rmsnorm": (lambda: tile.tile_rmsnorm_f32(x, y), 8),
        "softmax": (lambda: tile.tile_softmax_f32(x, y), 8),
        "layernorm_affine": (lambda: tile.tile_layernorm_affine_f32(x, None, g, b, y), 8),
        "residual_layernorm_affine": (lambda: tile.tile_layernorm_affine_f32(x, r, g, b, y), 12),
        "rmsnorm_weighted": (lambda: tile.tile_rmsnorm_weighted_f32(x, g, y), 8),
        "row_sum": (lambda: tile.tile_row_sum_f32(x, vec_a), 4),
        "row_minmax": (lambda: tile.tile_row_minmax_f32(x, vec_a, vec_b), 4),
        "sigmoid_pair": (lambda: tile.tile_sigmoid_pair_f32(x, y, y2), 12),
        "gelu_tanh_pair": (lambda: tile.tile_gelu_tanh_pair_f32(x, y, y2), 12),
        "residual_layernorm_bf16": (lambda: tile.tile_residual_layernorm_bf16(xb, rb, yb), 6),
        "layernorm_bf16": (lambda: tile.tile_layernorm_bf16(xb, yb), 4),
        "rmsnorm_bf16": (lambda: tile.tile_rmsnorm_bf16(xb, yb), 4),
        "softmax_bf16": (lambda: tile.tile_softmax_bf16(xb, yb), 4),
        "layernorm_affine_bf16": (lambda: tile.tile_layernorm_affine_bf16(xb, None, g, b, yb), 4),
        "rmsnorm_weighted_bf16": (lambda: tile.tile_rmsnorm_weighted_bf16(xb, g, yb), 4),
        "residual_layernorm_f16": (lambda: tile.tile_residual_layernorm_f16(xh, rh, yh), 6),
        "layernorm_f16": (lambda: tile.tile_layernorm_f16(xh, yh), 4),
        "rmsnorm_f16": (lambda: tile.tile_rmsnorm_f16(xh, yh), 4),
        "softmax_f16": (lambda: tile.tile_softmax_f16(xh, yh), 4),
        "layernorm_affine_f16": (lambda: tile.tile_layernorm_affine_f16(xh, None, g, b, yh), 4),
        "rmsnorm_weighted_f16": (lambda: tile.tile_rmsnorm_weighted_f16(xh, g, yh), 4),
        "layernorm_backward": (lambda: tile.tile_layernorm_backward_f32(x, g, r, y, stats), 12),
        "rmsnorm_backward": (lambda: tile.tile_rmsnorm_backward_f32(x, g, r, y, stats), 12),
        "softmax_backward": (lambda: tile.tile_softmax_backward_f32(sm, r, y), 12),
        "norm_param_grad": (lambda: tile.tile_norm_param_grad_f32(x, r, stats, dg, db, ws), 8),
        "layernorm_backward_bf16": (lambda: tile.tile_layernorm_backward_bf16(xb, g, rb, yb, stats),
                                    6),
        "rmsnorm_backward_bf16": (lambda: tile.tile_rmsnorm_backward_bf16(xb, g, rb, yb, stats), 6),
        "softmax_backward_bf16": (lambda: tile.tile_softmax_backward_bf16(smb, rb, yb), 6),
        "norm_param_grad_bf16": (lambda: tile.tile_norm_param_grad_bf16(xb, rb, stats, dg, db, ws),
                                 4),
        "layernorm_backward_f16": (lambda: tile.tile_layernorm_backward_f16(xh, g, rh, yh, stats),
                                   6),
        "rmsnorm_backward_f16": (lambda: tile.tile_rmsnorm_backward_f16(xh, g, rh, yh, stats), 6),
        "softmax_backward_f16": (lambda: tile.tile_softmax_backward_f16(smh, rh, yh), 6),
        "norm_param_grad_f16": (lambda: tile.tile_norm_param_grad_f16(xh, rh, stats, dg, db, ws),
                                4),
    }
    only = set(args.only.split(",")) if args.only else None
    peak, src = measured_hbm_gbs()
    stream = torch.cuda.current_stream()
    results = []
    for name, (fn, bpe) in ops.items():
        if only and name not in only:
            continue
        for _ in range(args.warmup):
            fn()
        evs = [torch.cuda.Event(enable_timing=True) for _ in range(args.iters + 1)]
        evs[0].record(stream)
        for i in range(args.iters):
            fn()
            evs[i + 1].record(stream)
        torch.cuda.synchronize()
        per = [evs[i].elapsed_time(evs[i + 1]) for i in range(args.iters)]
        ms = statistics.mean(per)
        gbs = bpe * n / (ms * 1e-3) / 1e9
        res = {"op": name, "rows": rows, "width": width, "bytes_per_elem": bpe,
               "us_per_call": round(ms * 1e3, 2), "median_us": round(statistics.median(per) * 1e3, 2),
               "achieved_gbs": round(gbs, 1), "frac_of_copy": round(gbs / peak, 4),
               "peak": f"{peak} GB/s ({src} HBM copy)"}
        results.append(res)
        print(json.dumps(res), flush=True)
    assert tile.tile_check_device_status() == 0
    if args.json:
        with open(args.json, "w") as fh:
            json.dump(results, fh, indent=1)
    return results


if __name__ == "__main__":
    sys.exit(0 if main() is not None else 1)
