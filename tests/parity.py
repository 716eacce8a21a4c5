"""Shared helpers of the GPU parity tests: run an op through the C ABI and
compare with the FP64 oracle under the acceptance bound
|y - ref| <= ATOL + RTOL*|ref| (from the pages' runner tolerance, atol 2e-6
and rtol 2e-5)."""

from __future__ import annotations

import numpy as np

import oracle

ATOL = 2e-6
RTOL = 2e-5
EPS = 1e-5


def ref_eps(eps=EPS):
    """The oracle gets the FP32 eps the kernel receives, widened to FP64."""
    return oracle.kernel_eps(eps)


def compare(got, ref, what=""):
    """Assert the bound element by element; return (max abs err, max rel err)."""
    got = np.asarray(got, dtype=np.float64)
    assert got.shape == ref.shape, f"{what}: shape {got.shape} != {ref.shape}"
    assert np.all(np.isfinite(got)), f"{what}: non-finite output"
    err = np.abs(got - ref)
    bound = ATOL + RTOL * np.abs(ref)
    bad = err > bound
    if bad.any():
        idx = np.argwhere(bad)[:5]
        detail = ", ".join(f"{tuple(i)}: got {got[tuple(i)]:.9g} ref {ref[tuple(i)]:.9g}"
                           for i in idx)
        raise AssertionError(f"{what}: {int(bad.sum())} elements beyond tolerance "
                             f"(max abs err {err.max():.3e}); {detail}")
    big = np.abs(ref) > 1e-6
    rel = float((err[big] / np.abs(ref[big])).max()) if big.any() else 0.0
    return float(err.max()), rel


def oracle_of(op, x, r=None, eps=EPS):
    return oracle.get().run(op, x, r, ref_eps(eps))


def host_threads():
    """Host cores this process may run on."""
    import os
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def oracle_blocks(op, x, r=None, eps=EPS, block_rows=1024, threads=None):
    """The oracle over a large matrix in contiguous row blocks, computed on
    every host core (the C oracle runs with the GIL released) a wave of
    blocks at a time, so at most ``threads`` FP64 blocks are held at once.
    Yields ``(row0, row1, ref)`` in row order; each block is exactly what one
    call over all rows gives for those rows (rows are independent)."""
    from concurrent.futures import ThreadPoolExecutor
    rows = x.shape[0]
    threads = threads or host_threads()
    orc = oracle.get()
    e = ref_eps(eps)
    spans = [(a, min(rows, a + block_rows)) for a in range(0, rows, block_rows)]

    def one(ab):
        a, b = ab
        return orc.run(op, x[a:b], None if r is None else r[a:b], e)

    with ThreadPoolExecutor(max_workers=threads) as ex:
        for w in range(0, len(spans), threads):
            wave = spans[w:w + threads]
            for (a, b), ref in zip(wave, ex.map(one, wave)):
                yield a, b, ref


def compare_full(got, op, x, r=None, eps=EPS, what="", block_rows=1024):
    """``compare`` over every element of a whole [rows, width] output, block
    by block against ``oracle_blocks``.  Returns (max abs err, max rel err)
    over the whole output."""
    assert got.shape == x.shape, f"{what}: shape {got.shape} != {x.shape}"
    worst_abs, worst_rel = 0.0, 0.0
    for a, b, ref in oracle_blocks(op, x, r, eps, block_rows):
        ea, er = compare(got[a:b], ref, f"{what} rows {a}..{b - 1}")
        worst_abs, worst_rel = max(worst_abs, ea), max(worst_rel, er)
    return worst_abs, worst_rel


def staged_table(op):
    """The 2-byte selector's measured staged-plan table for `op` (a table op
    name of the selector generator, e.g. "layernorm_affine+residual"), read
    from the generated header: [(widest width, plan or -1)]."""
    import re
    from tile_compiler_row_gb300 import selector_tables
    text = open(selector_tables.HEADER).read()
    m = re.search(r"kB16Staged%s\[\] = \{(.*?)\};" % selector_tables.STEM[op], text)
    return [(int(a), int(b)) for a, b in re.findall(r"\{(\d+), (-?\d+)\}", m.group(1))]


def expects_staged(op, rows, width):
    """Whether the selector should take a staged plan for 2-byte rows of
    whole 16-byte vectors on aligned pointers (large problems only)."""
    if rows * width <= (1 << 22) or width % 8:
        return False
    return next(p for w, p in staged_table(op) if width <= w) >= 0
