#!/usr/bin/env python3
"""Benchmark of the fused FP32 row-normalisation library on one GB300.

One step = one call of ``tile_residual_layernorm_f32`` on a 65536x4096 FP32
matrix (x and residual read once, y written once: 12 bytes per element,
3 GiB per step).  Inputs are seeded synthetic uniform[-1, 1) values, resident
in HBM before the timed region; the 3 GiB working set is far larger than the
129 MB L2, so no flush is needed between steps.

Printed: one JSON line with the device-timed throughput (algorithmic GB/s),
the end-to-end throughput through the C ABI with host buffers (the inputs
cross the host link and the result comes back inside the timed region), the roofline of the kernel against the measured HBM copy
bandwidth, the SM clocks seen during the run, and the FP64 CPU oracle timed
on this host as a baseline.

  python bench.py [--gpus N --steps K --warmup W]        our CUDA library
  python bench.py --impl reference ...                    the CPU oracle

Under torchrun (N > 1) every rank runs the same workload on its own GPU
(independent replicas, no collective on the data path); the timed region is
bracketed by barriers and the maximum time over ranks is used.
"""

from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time
from concurrent.futures import ThreadPoolExecutor

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "HBM GB/s (% of GB300 peak) and µs/call, residual LayerNorm FP32 65536×4096"
UNIT = "GB/s"
FALLBACK_HBM_GBS = 6800.0
BYTES_PER_ELEM = {"residual_layernorm": 12, "layernorm": 8, "rmsnorm": 8, "softmax": 8}
EPS = 1e-5
SEED_CFG = 5
L2_BYTES = 129 * 10**6      # GB300 L2


def parse_args():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--rows", type=int, default=65536, help="rows (profiling runs use fewer)")
    ap.add_argument("--width", type=int, default=4096)
    ap.add_argument("--op", default="residual_layernorm", choices=sorted(BYTES_PER_ELEM))
    ap.add_argument("--no-extra", action="store_true", help="skip the RMSNorm/softmax lines")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu", action="store_true", help="skip the CPU oracle baseline")
    ap.add_argument("--plan", type=int, default=None, help="force a built plan (sweeps)")
    return ap.parse_args()


# ---------------------------------------------------------------------------
# distributed plumbing (replicas only)
# ---------------------------------------------------------------------------

class Dist:
    def __init__(self, gpus):
        self.world = int(os.environ.get("WORLD_SIZE", "1"))
        self.rank = int(os.environ.get("RANK", "0"))
        self.local_rank = int(os.environ.get("LOCAL_RANK", "0"))
        self.pg = None
        if gpus != self.world and self.world > 1:
            raise SystemExit(f"--gpus {gpus} but WORLD_SIZE={self.world}")

    def init(self, backend="nccl"):
        self.backend = backend
        if self.world > 1:
            import torch.distributed as dist
            dist.init_process_group(backend=backend)
            self.pg = dist

    def barrier(self):
        if self.pg is not None:
            if self.backend == "nccl":
                import torch
                self.pg.barrier(device_ids=[torch.cuda.current_device()])
            else:
                self.pg.barrier()

    def max(self, value):
        """Maximum of ``value`` over ranks (the timed region's slowest rank)."""
        if self.pg is None:
            return value
        import torch
        dev = "cuda" if self.backend == "nccl" else "cpu"
        t = torch.tensor([value], dtype=torch.float64, device=dev)
        self.pg.all_reduce(t, op=self.pg.ReduceOp.MAX)
        return float(t.item())

    def close(self):
        if self.pg is not None:
            self.pg.destroy_process_group()


# ---------------------------------------------------------------------------
# clocks during the timed region
# ---------------------------------------------------------------------------

CLOCK_FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
                "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
                "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")


class ClockSampler:
    """nvidia-smi sampling every 50 ms while the GPU is under load."""

    def __init__(self, gpu_selector):
        self.samples = []
        self.proc = None
        self.thread = None
        self.selector = gpu_selector

    def start(self):
        cmd = ["nvidia-smi", f"--query-gpu={CLOCK_FIELDS}", "--format=csv,noheader,nounits", "-lms", "50"]
        if self.selector:
            cmd += ["-i", self.selector]
        try:
            self.proc = subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()
        time.sleep(0.3)       # let the first samples arrive

    def _read(self):
        for line in self.proc.stdout:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                self.samples.append({
                    "t": time.perf_counter(), "sm": float(parts[1]), "sm_max": float(parts[2]),
                    "power": float(parts[3]) if parts[3] not in ("[N/A]", "N/A") else None,
                    "hw_slowdown": parts[5], "hw_thermal": parts[6], "sw_thermal": parts[7],
                    "sw_power_cap": parts[8]})
            except ValueError:
                continue

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        if self.thread is not None:
            self.thread.join(timeout=5)

    def summary(self, t0, t1):
        inside = [s for s in self.samples if t0 <= s["t"] <= t1]
        use = inside if inside else self.samples
        if not use:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0,
                    "note": "nvidia-smi gave no samples"}
        reasons = set()
        for s in use:
            for key, name in (("hw_slowdown", "hw_slowdown"), ("hw_thermal", "hw_thermal_slowdown"),
                              ("sw_thermal", "sw_thermal_slowdown"), ("sw_power_cap", "sw_power_cap")):
                if s[key].lower().startswith("active"):
                    reasons.add(name)
        return {"sm_mhz": statistics.median(s["sm"] for s in use),
                "sm_max_mhz": max(s["sm_max"] for s in use),
                "reasons": sorted(reasons), "samples": len(use),
                "window": "timed region" if inside else "warm-up and timed region"}


def gpu_selector():
    try:
        import torch
        uuid = str(torch.cuda.get_device_properties(torch.cuda.current_device()).uuid)
        return uuid if uuid.startswith("GPU-") else f"GPU-{uuid}"
    except Exception:
        return None


# ---------------------------------------------------------------------------
# helpers
# ---------------------------------------------------------------------------

def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as fh:
            mp = json.load(fh)
        return float(mp["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback"


def profile_traffic(op, rows, width, plan_id):
    """DRAM bytes per launch from the committed ncu summary, if it was taken on
    the kernel source that is built now and on the same plan (else None)."""
    from tile_compiler_row_gb300 import _build
    path = os.path.join(ROOT, "profiles", f"{op}_{rows}x{width}.md")
    try:
        text = open(path).read()
    except OSError:
        return None
    fields = {}
    for line in text.splitlines():
        line = line.strip().lstrip("-* ").strip()
        if ":" in line:
            k, v = line.split(":", 1)
            fields[k.strip().strip("`")] = v.strip().strip("`")
    if fields.get("kernel_sha256") != _build.kernel_hash():
        return None
    if fields.get("plan_id") != str(plan_id):
        return None
    try:
        return int(float(fields["dram_bytes_per_launch"]))
    except (KeyError, ValueError):
        return None


def metric_of(op, rows, width):
    """The metric name of a run: the headline's for its workload, else the
    same measure named for the workload that ran."""
    if (op, rows, width) == ("residual_layernorm", 65536, 4096):
        return METRIC
    return f"HBM GB/s and µs/call, {op} FP32 {rows}×{width}"


def workload_config(op, rows, width, world):
    """The ``config`` object of the JSON line: the workload alone, the same
    in both arms (plan and host-thread details go in their own keys)."""
    elems = rows * width
    nin = 2 if op == "residual_layernorm" else 1
    return {"workload": f"{op.replace('_', ' ')} FP32 {rows}x{width}", "rows": rows,
            "width": width, "eps": EPS,
            "l2": (f"inputs larger than L2: {(nin + 1) * elems * 4 / 2**30:.2f} GiB working set, "
                   "no flush") if (nin + 1) * elems * 4 > L2_BYTES else
                  f"L2-resident: {(nin + 1) * elems * 4 / 2**20:.1f} MiB working set, no flush",
            "parallelism": f"replicas x{world}"}


def provenance():
    """What the line was measured on: the git commit when the tree has one,
    the SHA-256 of the kernel sources and of the loaded library, the GPU."""
    from tile_compiler_row_gb300 import _build
    try:
        head = subprocess.run(["git", "rev-parse", "HEAD"], cwd=ROOT, capture_output=True,
                              text=True, timeout=10)
        git = head.stdout.strip() if head.returncode == 0 and head.stdout.strip() else None
    except (OSError, subprocess.SubprocessError):
        git = None
    h = hashlib.sha256()
    with open(_build.LIBRARY, "rb") as fh:
        for block in iter(lambda: fh.read(1 << 20), b""):
            h.update(block)
    out = {"git": git, "source_sha256": _build.source_hash(), "so_sha256": h.hexdigest()}
    try:
        import torch
        out["gpu_name"] = torch.cuda.get_device_name(torch.cuda.current_device())
    except Exception:
        out["gpu_name"] = None
    return out


def job_throughput(world, bytes_per_step, steps, max_ms):
    """Whole-job GB/s: every rank moves ``bytes_per_step`` per step (weak
    scaling), divided by the slowest rank's time."""
    return world * bytes_per_step * steps / (max_ms / 1e3) / 1e9


def time_calls(fn, steps, stream):
    """Per-call CUDA-event durations (ms) of ``steps`` back-to-back calls on
    ``stream``, plus the total elapsed (ms) between the first and last event."""
    import torch
    evs = [torch.cuda.Event(enable_timing=True) for _ in range(steps + 1)]
    evs[0].record(stream)
    for i in range(steps):
        fn()
        evs[i + 1].record(stream)
    torch.cuda.synchronize()
    per = [evs[i].elapsed_time(evs[i + 1]) for i in range(steps)]
    return per, evs[0].elapsed_time(evs[-1])


# ---------------------------------------------------------------------------
# our CUDA library
# ---------------------------------------------------------------------------

def run_ours(args, dist):
    import numpy as np
    import torch

    import synth
    import tile_compiler_row_gb300 as tile
    from tile_compiler_row_gb300 import _build

    _build.build()
    lib = tile.load()
    torch.cuda.set_device(dist.local_rank)
    dist.init("nccl")
    stream = torch.cuda.current_stream()
    rows, width, op = args.rows, args.width, args.op
    elems = rows * width
    nbytes = BYTES_PER_ELEM[op] * elems

    x_h = synth.rows_of(SEED_CFG, rows, width, which="x")
    r_h = synth.rows_of(SEED_CFG, rows, width, which="r")
    x = torch.from_numpy(x_h).cuda()
    r = torch.from_numpy(r_h).cuda()
    y = torch.empty_like(x)
    s = stream.cuda_stream

    def call_op(name, out, plan=None):
        px, pr, po = x.data_ptr(), r.data_ptr(), out.data_ptr()
        if plan is not None:
            st = lib.tile_run_plan_f32(tile.OPS[name], plan, px, pr, po, rows, width, EPS, s)
        elif name == "residual_layernorm":
            st = lib.tile_residual_layernorm_f32(px, pr, po, rows, width, EPS, s)
        else:
            st = getattr(lib, f"tile_{name}_f32")(px, po, rows, width, EPS, s)
        if st != 0:
            raise tile.TileError(st, name)

    plan = tile.tile_describe_plan(op, rows, width) if args.plan is None else \
        tile.tile_plan_info(args.plan, op, rows, width)
    sampler = ClockSampler(gpu_selector())
    sampler.start()

    step = lambda: call_op(op, y, args.plan)       # noqa: E731
    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    dist.barrier()
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    per, total_ms = time_calls(step, args.steps, stream)
    torch.cuda.synchronize()
    dist.barrier()
    t1 = time.perf_counter()
    total_ms = dist.max(total_ms)
    sampler.stop()
    clocks = sampler.summary(t0, t1)
    if tile.tile_check_device_status() != 0:
        raise SystemExit("device status word set after the timed region")
    # the timed call's output, for the oracle comparison after the CPU baseline
    check = not args.no_cpu and dist.world == 1 and dist.rank == 0
    timed_out = y.cpu().numpy() if check else None

    ms_per_step = total_ms / args.steps
    value = job_throughput(dist.world, nbytes, args.steps, total_ms)
    kernel_ms = statistics.mean(per)
    peak, peak_src = measured_peaks()
    achieved = nbytes / (kernel_ms / 1e3) / 1e9
    traffic = profile_traffic(op, rows, width, plan["id"])
    line = {
        "metric": metric_of(op, rows, width),
        "value": round(value, 2), "unit": UNIT, "n_gpus": dist.world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_per_step, 6),
        "us_per_call": round(ms_per_step * 1e3, 3),
        "pct_of_peak": round(100.0 * achieved / peak, 2),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": f"synthetic: SplitMix64 uniform[-1,1), seeds {synth.x_seed(SEED_CFG)}/"
                f"{synth.r_seed(SEED_CFG)}",
        "config": workload_config(op, rows, width, dist.world),
        "plan": {k: plan[k] for k in ("id", "path", "vec", "warps_per_program",
                                      "programs_per_cta", "chunks", "cluster", "threads",
                                      "grid")},
        "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak,
                     "unit": "GB/s", "frac": round(achieved / peak, 4), "traffic": traffic,
                     "peak_source": f"{peak_src} HBM copy bandwidth",
                     "algorithmic_bytes_per_launch": nbytes,
                     "kernel_ms_mean": round(kernel_ms, 6),
                     "kernel_ms_median": round(statistics.median(per), 6),
                     "kernel_ms_min": round(min(per), 6),
                     "kernel_ms_p90": round(sorted(per)[(9 * len(per)) // 10], 6),
                     "frac_of_8TBps_nominal": round(achieved / 8000.0, 4)},
        "clocks": clocks,
        "gpu_launches": args.steps,
        "per_call_ms": [round(v, 5) for v in per],
        "provenance": provenance(),
    }

    # --- the other two large-shape ops (same inputs; one launch per call) ---
    if not args.no_extra and (rows, width) == (65536, 4096) and args.plan is None:
        extra = {}
        for name in ("rmsnorm", "softmax"):
            if name == op:
                continue
            f = lambda name=name: call_op(name, y)      # noqa: E731
            for _ in range(max(3, args.warmup)):
                f()
            per_x, tot_x = time_calls(f, max(20, min(args.steps, 200)), stream)
            k_ms = statistics.mean(per_x)
            b = BYTES_PER_ELEM[name] * elems
            extra[name] = {"us_per_call": round(k_ms * 1e3, 3),
                           "achieved_gbs": round(b / (k_ms / 1e3) / 1e9, 1),
                           "frac": round(b / (k_ms / 1e3) / 1e9 / peak, 4),
                           "plan_id": tile.tile_describe_plan(name, rows, width)["id"]}
        # the same residual LayerNorm on BF16 rows (6 bytes per element)
        xb, rb = x.to(torch.bfloat16), r.to(torch.bfloat16)
        yb = torch.empty_like(xb)

        def f_bf16():
            st = lib.tile_residual_layernorm_bf16(xb.data_ptr(), rb.data_ptr(), yb.data_ptr(),
                                                  rows, width, EPS, s)
            if st != 0:
                raise tile.TileError(st, "tile_residual_layernorm_bf16")

        for _ in range(max(3, args.warmup)):
            f_bf16()
        per_x, _ = time_calls(f_bf16, max(20, min(args.steps, 200)), stream)
        k_ms = statistics.mean(per_x)
        b = 6 * elems
        extra["residual_layernorm_bf16"] = {
            "us_per_call": round(k_ms * 1e3, 3), "achieved_gbs": round(b / (k_ms / 1e3) / 1e9, 1),
            "frac": round(b / (k_ms / 1e3) / 1e9 / peak, 4),
            "plan_id": tile.tile_describe_plan_ex("residual_layernorm", "bf16", rows, width)["id"]}
        del xb, rb, yb
        line["other_ops"] = extra
        with_cpu = not args.no_cpu and dist.world == 1 and dist.rank == 0
        line["small_shapes"] = small_shapes(tile, cpu=with_cpu)
        line["single_call"] = single_call(tile, lib, x, r, y, stream)

    # --- end to end through the C ABI with pinned host buffers -------------
    if not args.no_e2e:
        xp = torch.from_numpy(x_h).pin_memory()
        rp = torch.from_numpy(r_h).pin_memory()
        yp = torch.empty_like(xp).pin_memory()
        ws_bytes = tile.tile_host_workspace_bytes(op, width, max(1, -(-rows // 8)))
        ws = torch.empty(ws_bytes, dtype=torch.uint8, device="cuda")
        code = tile.OPS[op]
        chunk, slots = tile.tile_host_schedule(op, rows, width, ws_bytes, direct_output=True)

        def e2e_step():
            st = lib.tile_run_host_f32(code, xp.data_ptr(), rp.data_ptr(), yp.data_ptr(), rows,
                                       width, EPS, ws.data_ptr(), ws.numel(), s)
            if st != 0:
                raise tile.TileError(st, "tile_run_host_f32")

        for _ in range(2):
            e2e_step()
        torch.cuda.synchronize()
        n_e2e = max(3, min(args.steps, 10))
        # Nine rounds of n_e2e steps (about 0.1 s each); the median round is
        # reported (the host side of the link is shared with other jobs on the
        # machine: runs have seen two and three of five rounds at about twice
        # the time of the others, so five rounds were not enough).
        rounds = []
        for _ in range(9):
            dist.barrier()
            _, ms = time_calls(e2e_step, n_e2e, stream)
            rounds.append(dist.max(ms))
        e2e_ms = sorted(rounds)[len(rounds) // 2]
        h2d = (2 if op == "residual_layernorm" else 1) * elems * 4
        line["e2e"] = {"value": round(job_throughput(dist.world, nbytes, n_e2e, e2e_ms), 2),
                       "unit": UNIT, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": elems * 4,
                       "steps": n_e2e, "ms_per_step": round(e2e_ms / n_e2e, 4),
                       "rounds_ms_per_step": [round(r / n_e2e, 4) for r in rounds],
                       "path": "tile_run_host_f32 on pinned, device-addressable host "
                               "buffers: one kernel reads x and r and writes y over the host "
                               "link (no staging copies; pageable buffers would take the "
                               f"copy pipeline of {chunk}-row chunks in {slots} slots)"}
        ref = torch.empty_like(x)
        call_op(op, ref, args.plan)
        torch.cuda.synchronize()
        # rows spread over the matrix (both ends of every pipeline-sized
        # chunk), bit for bit
        pick = sorted({i for c in range(0, rows, chunk) for i in (c, min(rows, c + chunk) - 1)}
                      | {rows // 2 + 1})
        idx = torch.tensor(pick)
        if not torch.equal(yp[idx].cuda(), ref[idx.cuda()]):
            raise SystemExit("e2e output differs from the device path")
        # The link alone on this machine, for context (these overwrite ref and
        # yp): a plain host->device copy of one pinned input tensor (the
        # call's floor is its host->device bytes at this rate), the
        # device->host copy, and kernel stores into the pinned output (the
        # call's way out).
        for _ in range(2):
            ref.copy_(xp, non_blocking=True)
        _, link_ms = time_calls(lambda: ref.copy_(xp, non_blocking=True), 5, stream)
        link_gbs = elems * 4 * 5 / (link_ms * 1e-3) / 1e9
        line["e2e"]["link_h2d_gbs"] = round(link_gbs, 1)
        line["e2e"]["link_floor_ms"] = round(h2d / (link_gbs * 1e9) * 1e3, 3)
        _, d2h_ms = time_calls(lambda: yp.copy_(ref, non_blocking=True), 5, stream)
        line["e2e"]["link_d2h_gbs"] = round(elems * 4 * 5 / (d2h_ms * 1e-3) / 1e9, 1)

        def store_to_host():
            st = lib.tile_rmsnorm_f32(x.data_ptr(), yp.data_ptr(), rows, width, EPS, s)
            if st != 0:
                raise tile.TileError(st, "tile_rmsnorm_f32")

        store_to_host()
        _, st_ms = time_calls(store_to_host, 5, stream)
        line["e2e"]["kernel_store_to_host_gbs"] = round(elems * 4 * 5 / (st_ms * 1e-3) / 1e9, 1)

    # --- the FP64 CPU oracle on this host (rank 0, N = 1 only); its output
    # also checks every element of the timed call's output (untimed) --------
    if check:
        line["cpu_baseline"], line["parity"] = cpu_baseline(
            op, x_h, r_h if op == "residual_layernorm" else None, got=timed_out)

    dist.close()
    if dist.rank == 0:
        print(json.dumps(line), flush=True)


def host_cores():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def oracle_rows(orc, op, x_h, r_h, eps, threads):
    """The oracle over disjoint contiguous row blocks, one per thread.  The
    C oracle runs with the GIL released, so the blocks run in parallel; each
    block's result is exactly what one call over all rows gives for it.
    Returns the blocks' results in row order."""
    rows = x_h.shape[0]
    if threads <= 1 or rows < 2:
        return [orc.run(op, x_h, r_h, eps)]
    bounds = [rows * i // threads for i in range(threads + 1)]
    blocks = [(a, b) for a, b in zip(bounds[:-1], bounds[1:]) if b > a]
    with ThreadPoolExecutor(max_workers=len(blocks)) as ex:
        return list(ex.map(lambda ab: orc.run(op, x_h[ab[0]:ab[1]],
                                              None if r_h is None else r_h[ab[0]:ab[1]], eps),
                           blocks))


# The small workloads (the L2-resident configurations): (workload number,
# op, rows, width).  Workload 4 is N(0, 3^2) with a constant row and a +40
# outlier; the others are uniform[-1, 1).
SMALL_SHAPES = (
    (1, "residual_layernorm", 17, 257),
    (2, "softmax", 1024, 4096), (2, "rmsnorm", 1024, 4096), (2, "layernorm", 1024, 4096),
    (3, "residual_layernorm", 1, 127), (3, "residual_layernorm", 7, 1537),
    (3, "residual_layernorm", 64, 4096), (3, "rmsnorm", 1, 127), (3, "rmsnorm", 7, 1537),
    (3, "rmsnorm", 17, 257), (3, "rmsnorm", 64, 4096), (3, "softmax", 1, 127),
    (3, "softmax", 7, 1537), (3, "softmax", 17, 257), (3, "softmax", 64, 4096),
    (4, "softmax", 128, 8192), (4, "rmsnorm", 128, 8192), (4, "layernorm", 128, 8192),
    (4, "softmax", 32, 65536), (4, "rmsnorm", 32, 65536), (4, "layernorm", 32, 65536),
)


def small_shapes(tile, calls=200, cpu=False):
    """Device time per call of the small workloads: `calls` back-to-back calls
    captured in one CUDA graph and replayed (so host launch overhead is not
    counted).  Their working sets sit in the L2, so the GB/s are labelled
    effective (L2), not HBM.  With ``cpu``, each entry also carries the FP64
    oracle timed on the same inputs, on one core and on every host core."""
    import torch

    import synth
    out = []
    cap = torch.cuda.Stream()
    for cfg, op, rows, width in SMALL_SHAPES:
        x_h = synth.rows_of(cfg, rows, width, which="x")
        r_h = synth.rows_of(cfg, rows, width, which="r") if op == "residual_layernorm" else None
        x = torch.from_numpy(x_h).cuda()
        r = torch.from_numpy(r_h).cuda() if r_h is not None else None
        y = torch.empty_like(x)
        tile.run(op, x, r, y, EPS)                   # first call: lazy set-up
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=cap):
            for _ in range(calls):
                tile.run(op, x, r, y, EPS)
        g.replay()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(5):
            g.replay()
        e1.record()
        torch.cuda.synchronize()
        us = e0.elapsed_time(e1) * 1e3 / (5 * calls)
        b = BYTES_PER_ELEM[op] * rows * width
        entry = {"workload": cfg, "op": op, "shape": f"{rows}x{width}",
                 "us_per_call": round(us, 3), "rows_per_s": round(rows / (us * 1e-6)),
                 "gbs_effective_l2": round(b / (us * 1e-6) / 1e9, 1)}
        if cpu:
            entry["cpu_baseline"] = oracle_per_call(op, x_h, r_h)
        out.append(entry)
        del g, x, r, y
    return out


def oracle_per_call(op, x_h, r_h, min_seconds=0.05):
    """The FP64 oracle on one workload, as it stands: repeated until at least
    ``min_seconds`` have passed, on one core and on every host core (row
    blocks, at most one per row).  µs per call, rows/s and GB/s of FP32
    input and output moved."""
    import oracle
    orc = oracle.get()
    eps = oracle.kernel_eps(EPS)
    rows, width = x_h.shape
    b = BYTES_PER_ELEM[op] * rows * width
    res = {}
    for name, threads in (("single_core", 1), ("all_cores", min(host_cores(), rows))):
        n, t0 = 0, time.perf_counter()
        while True:
            oracle_rows(orc, op, x_h, r_h, eps, threads)
            n += 1
            dt = time.perf_counter() - t0
            if dt >= min_seconds:
                break
        sec = dt / n
        res[name] = {"us_per_call": round(sec * 1e6, 2), "rows_per_s": round(rows / sec),
                     "gbs": round(b / sec / 1e9, 4), "cores": threads, "calls": n}
    return res


def single_call(tile, lib, x_big, r_big, y_big, stream, samples=60):
    """Latency of one call on its own, as a caller sees it, in two separate
    phases per workload: (1) GPU time, CUDA events around one call with the
    device idle before it; (2) host wall, from the C-ABI call (through
    ctypes) to the return of cudaStreamSynchronize on the call's stream.
    ``samples`` of each, after 5 warm-up calls; p50, minimum and p90 in µs.
    Workloads: the 1024x4096 softmax, RMSNorm and LayerNorm and the
    65536x4096 residual LayerNorm."""
    import torch

    import synth
    x2 = torch.from_numpy(synth.rows_of(2, 1024, 4096, which="x")).cuda()
    y2 = torch.empty_like(x2)
    s = stream.cuda_stream
    cases = [("softmax", x2, None, y2), ("rmsnorm", x2, None, y2), ("layernorm", x2, None, y2),
             ("residual_layernorm", x_big, r_big, y_big)]

    def stats(v):
        v = sorted(v)
        return {"p50": round(statistics.median(v), 3), "min": round(v[0], 3),
                "p90": round(v[(9 * len(v)) // 10], 3)}

    out = []
    for op, x, r, y in cases:
        rows, width = x.shape
        fn = getattr(lib, f"tile_{op}_f32")
        args = ((x.data_ptr(), r.data_ptr(), y.data_ptr()) if r is not None
                else (x.data_ptr(), y.data_ptr())) + (rows, width, EPS, s)

        def call():
            st = fn(*args)
            if st != 0:
                raise tile.TileError(st, op)

        for _ in range(5):
            call()
        torch.cuda.synchronize()
        gpu = []
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        for _ in range(samples):
            e0.record(stream)
            call()
            e1.record(stream)
            stream.synchronize()
            gpu.append(e0.elapsed_time(e1) * 1e3)
        wall = []
        for _ in range(samples):
            torch.cuda.synchronize()
            t0 = time.perf_counter_ns()
            call()
            stream.synchronize()
            wall.append((time.perf_counter_ns() - t0) / 1e3)
        out.append({"op": op, "shape": f"{rows}x{width}", "samples": samples,
                    "gpu_us": stats(gpu), "host_wall_us": stats(wall)})
    del x2, y2
    return out


ATOL, RTOL = 2e-6, 2e-5      # the acceptance bound |y - ref| <= ATOL + RTOL*|ref|


def cpu_baseline(op, x_h, r_h, got=None):
    """The FP64 oracle over the whole workload on this host: once on every
    host core (row blocks in parallel, the reported value) and once on one
    core.  With ``got`` (the timed call's output, on the host), the
    all-core pass's result also checks every element of it, after the
    timing: returns (baseline, parity)."""
    import numpy as np

    import oracle
    orc = oracle.get()
    rows, width = x_h.shape
    eps = oracle.kernel_eps(EPS)
    b = BYTES_PER_ELEM[op] * rows * width
    cores = host_cores()
    t = time.perf_counter()
    blocks = oracle_rows(orc, op, x_h, r_h, eps, cores)
    dt_all = time.perf_counter() - t
    parity = None
    if got is not None:
        worst_abs, worst_rel, worst_ratio, bad, row0 = 0.0, 0.0, 0.0, 0, 0
        for ref in blocks:
            g = got[row0:row0 + ref.shape[0]].astype(np.float64)
            row0 += ref.shape[0]
            err = np.abs(g - ref)
            mag = np.abs(ref)
            worst_abs = max(worst_abs, float(err.max()))
            big = mag > 1e-6
            if big.any():
                worst_rel = max(worst_rel, float((err[big] / mag[big]).max()))
            ratio = err / (ATOL + RTOL * mag)
            worst_ratio = max(worst_ratio, float(ratio.max()))
            bad += int(np.count_nonzero(~(ratio <= 1.0)))
        parity = {"against": "FP64 oracle, every element", "elements": int(got.size),
                  "max_abs_err": worst_abs, "max_rel_err": worst_rel,
                  "max_err_over_bound": round(worst_ratio, 4),
                  "bound": f"{ATOL} + {RTOL}*|ref|", "beyond_bound": bad}
        if bad:
            print(f"warning: {bad} outputs beyond the bound", file=sys.stderr)
    del blocks
    t = time.perf_counter()
    orc.run(op, x_h, r_h, eps)
    dt_one = time.perf_counter() - t
    base = {"value": round(b / dt_all / 1e9, 4), "unit": UNIT, "cores": cores, "kind": "oracle",
            "sample": f"all {rows} rows x {width}, one pass, FP64 C, row blocks on {cores} "
                      "threads",
            "seconds": round(dt_all, 3),
            "single_core": {"value": round(b / dt_one / 1e9, 4), "unit": UNIT, "cores": 1,
                            "seconds": round(dt_one, 3)}}
    return base, parity


# ---------------------------------------------------------------------------
# reference arm: the FP64 CPU oracle as it stands, on host cores
# ---------------------------------------------------------------------------

def run_reference(args, dist):
    if dist.rank != 0:
        return                               # rank 0 alone runs and prints
    import oracle
    import synth

    rows, width, op = args.rows, args.width, args.op
    cores = host_cores()
    n = rows                                 # every step: the whole workload
    x_h = synth.rows_of(SEED_CFG, rows, width, which="x")
    r_h = synth.rows_of(SEED_CFG, rows, width, which="r") if op == "residual_layernorm" else None
    orc = oracle.get()
    eps = oracle.kernel_eps(EPS)
    for _ in range(args.warmup):
        oracle_rows(orc, op, x_h, r_h, eps, cores)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle_rows(orc, op, x_h, r_h, eps, cores)
    total = time.perf_counter() - t0
    b = BYTES_PER_ELEM[op] * n * width
    value = b * args.steps / total / 1e9
    sample = f"all {n} rows x {width} per step, FP64 C, row blocks on {cores} threads"
    line = {
        "impl": "reference",
        "metric": metric_of(op, rows, width),
        "value": round(value, 4), "unit": UNIT,
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(total / args.steps * 1e3, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": f"synthetic: SplitMix64 uniform[-1,1), seeds {synth.x_seed(SEED_CFG)}/"
                f"{synth.r_seed(SEED_CFG)}",
        "config": workload_config(op, rows, width, dist.world),
        "host_threads": cores,
        "cpu_baseline": {"value": round(value, 4), "unit": UNIT, "cores": cores,
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": round(value, 4), "unit": UNIT, "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }
    print(json.dumps(line), flush=True)


def main():
    args = parse_args()
    dist = Dist(args.gpus)
    if args.impl == "reference":
        run_reference(args, dist)
        return
    run_ours(args, dist)


if __name__ == "__main__":
    main()
