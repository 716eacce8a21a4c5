"""The generated selector tables, checked on the CPU: for every op, element
type and row-count regime (tiny and small L2-resident problems, large
problems) and a dense set of widths, the plan the library describes exists
for that element type and covers the row (its workers own every element),
and a plan that needs rows of whole 16-byte vectors is only described for
such rows; the backward selector's plans are built for the backward kernels
and cover every width."""

import random

import pytest

import tile_compiler_row_gb300 as tile
from tile_compiler_row_gb300 import _build

OPS = ("residual_layernorm", "layernorm", "rmsnorm", "softmax", "row_sum", "row_minmax",
       "layernorm_affine", "rmsnorm_weighted")
ROWS = (1, 7, 64, 1024, 16384, 1 << 20)          # tiny, small and large regimes


@pytest.fixture(scope="module", autouse=True)
def lib():
    _build.build()
    return tile.load()


def _widths():
    rng = random.Random(11)
    ws = set(range(1, 300)) | {w + d for w in (512, 1024, 1536, 2048, 3072, 3584, 4096, 6144,
                                               8192, 12288, 16384, 32768, 65536)
                               for d in (-8, -1, 0, 1, 3, 4, 7, 8)}
    ws |= {rng.randint(1, tile.tile_max_width()) for _ in range(300)}
    ws.add(tile.tile_max_width())
    return sorted(w for w in ws if 1 <= w <= tile.tile_max_width())


WIDTHS = _widths()


@pytest.mark.parametrize("dtype", ["f32", "bf16", "f16"])
@pytest.mark.parametrize("op", OPS)
def test_every_described_plan_is_built_and_covers_the_row(op, dtype):
    ev = 4 if dtype == "f32" else 8
    for rows in ROWS:
        for w in WIDTHS:
            p = tile.tile_describe_plan_ex(op, dtype, rows, w)
            what = f"{op} {dtype} {rows}x{w}: plan {p['id']}"
            assert p["max_width"] >= w, what
            assert tile.tile_plan_info_ex(p["id"], op, dtype, rows, w) is not None, what
            cap = p["chunks"] * p["workers"] * p["cluster"]
            assert (w // ev if p["vec"] > 1 else w) <= cap, what
            if p["path"] in (2, 3):           # staged, R rows per CTA: whole vectors only
                assert w % ev == 0 and rows * w > (1 << 22), what


@pytest.mark.parametrize("dtype", ["f32", "bf16", "f16"])
@pytest.mark.parametrize("op", ["layernorm", "rmsnorm", "softmax"])
def test_every_described_backward_plan_is_built_and_covers_the_row(lib, op, dtype):
    """The backward selector's plans: built for the backward kernels of the
    element type (a forced run of the plan on zero rows is accepted) and
    covering every width."""
    code = tile.OPS[op]
    dcode = {"f32": 0, "bf16": 1, "f16": 2}[dtype]
    for w in WIDTHS:
        p = tile.tile_describe_backward_plan(op, dtype, 1024, w)
        what = f"{op} backward {dtype} w={w}: plan {p['id']}"
        assert p["max_width"] >= w and p["path"] in (0, 1), what
        assert lib.tile_run_backward_plan_ex(code, p["id"], dcode, None, None, None, None, None,
                                             0, w, 1e-5, None) == 0, what
