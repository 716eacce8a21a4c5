"""The seeded input generator: published SplitMix64 outputs, determinism,
counter-based slicing and the workload recipes."""

import numpy as np

import synth


def test_splitmix64_published_sequence():
    # First outputs of SplitMix64 started from state 0 (Steele, Lea and Flood,
    # OOPSLA 2014; the reference Java/C implementation).
    h = synth.splitmix64(0, 0, 3)
    assert [int(v) for v in h] == [0xE220A8397B1DCDAF, 0x6E789E6AA1B965F4, 0x06C45D188009454F]


def test_counter_based_slices_agree():
    full = synth.uniform_pm1(1234, 10000)
    assert np.array_equal(full[3000:3100], synth.uniform_pm1(1234, 100, start=3000))
    nfull = synth.normal(77, 5000, 3.0)
    assert np.array_equal(nfull[1234:1300], synth.normal(77, 66, 3.0, start=1234))


def test_uniform_range_and_exactness():
    u = synth.uniform_pm1(1005, 1 << 20)
    assert u.dtype == np.float32
    assert u.min() >= -1.0 and u.max() < 1.0
    # every value is a multiple of 2^-23
    assert np.all((u.astype(np.float64) * 2.0 ** 23) % 1.0 == 0.0)
    assert abs(float(u.mean())) < 5e-3
    assert abs(float(u.var()) - 1.0 / 3.0) < 5e-3


def test_normal_moments():
    n = synth.normal(1004, 1 << 18, 3.0)
    assert abs(float(n.mean())) < 0.05
    assert abs(float(n.std()) - 3.0) < 0.05


def test_wide_row_recipe():
    x = synth.rows_of(4, 128, 8192)
    assert np.all(x[0] == x[0, 0])                       # constant row
    assert x[1, synth.outlier_column(8192)] == 40.0      # +40 outlier
    assert x[1].max() == 40.0
    sub = synth.rows_of(4, 128, 8192, row_ids=[5, 0, 1, 127])
    assert np.array_equal(sub, x[[5, 0, 1, 127]])


def test_seeds_differ():
    assert not np.array_equal(synth.rows_of(5, 4, 64, which="x"), synth.rows_of(5, 4, 64, which="r"))
