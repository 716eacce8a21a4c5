"""The FP64 oracle against hand-worked cases, closed forms, invariants and
torch's FP64 functional ops (see ``oracle_pins.py``)."""

import os

import numpy as np
import pytest

import oracle
from oracle_pins import check_all, golden_cases, _run_golden


@pytest.fixture(scope="module")
def orc():
    return oracle.get()


@pytest.mark.parametrize("path", golden_cases(), ids=os.path.basename)
def test_golden(orc, path):
    assert _run_golden(orc, path) is None


def test_all_pins(orc):
    assert check_all(orc) == []


def test_empty_inputs(orc):
    for op in ("layernorm", "rmsnorm", "softmax"):
        assert orc.run(op, np.zeros((0, 7), np.float32)).shape == (0, 7)
    z = np.zeros((0, 5), np.float32)
    assert orc.residual_layernorm(z, z).shape == (0, 5)


def test_kernel_eps_is_fp32_rounding():
    assert oracle.kernel_eps(1e-5) == float(np.float32(1e-5))
    assert abs(oracle.kernel_eps(1e-5) - 1e-5) < 1e-12
