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
