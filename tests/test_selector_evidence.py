"""The width->plan selector against its committed evidence (CPU only).

profiles/selector_sweep.md records, for every bucket of the selector's
tables, the plans timed on a GB300 at one representative shape: the plan
the selector chose, the fastest plan, the runner-up and the A/A noise.
These tests parse that summary and check, without a GPU, that the library
still selects the recorded plan at every recorded shape (so the tables in
the source and the evidence cannot drift apart), that the evidence covers
every bucket the library reports today, and that every selected plan was
within 5 % of the fastest plan measured there (the generated tables take
the fastest plan of the sweeps they were made from, or the previous plan
within 0.5 % of it; 5 % allows for run-to-run and GPU-to-GPU differences
between those sweeps and this independent one)."""

import os
import re

import pytest

import tile_compiler_row_gb300 as tile
from tile_compiler_row_gb300 import _build, selector_evidence

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SUMMARY = os.path.join(ROOT, "profiles", "selector_sweep.md")
WITHIN = 1.05


def _rows(section):
    text = open(SUMMARY).read()
    part = text.split(section, 1)[1].split("\n## ", 1)[0]
    out = []
    for line in part.splitlines():
        cells = [c.strip() for c in line.strip().strip("|").split("|")]
        if len(cells) < 8 or not re.fullmatch(r"[a-z_]+", cells[0]) or cells[0] == "op":
            continue
        out.append(cells)
    return out


@pytest.fixture(scope="module", autouse=True)
def lib():
    _build.build()
    return tile.load()


def large():
    return [dict(op=c[0], dtype=c[1], lo=int(c[2].split("-")[0]), hi=int(c[2].split("-")[1]),
                 width=int(c[3]), rows=int(c[4]), selected=int(c[5]), best=int(c[7]),
                 ratio=float(c[13])) for c in _rows("## Large problems")]


def backward():
    return [dict(op=c[0], dtype=c[1], lo=int(c[2].split("-")[0]), hi=int(c[2].split("-")[1]),
                 width=int(c[3]), rows=int(c[4]), selected=int(c[5]), best=int(c[7]),
                 ratio=float(c[13])) for c in _rows("## Backward")]


def small():
    return [dict(op=c[0], dtype=c[1], rows=int(c[2].split("x")[0]), width=int(c[2].split("x")[1]),
                 selected=int(c[3]), best=int(c[5]), ratio=float(c[11]))
            for c in _rows("## Small problems")]


def test_summary_is_committed_and_parses():
    assert os.path.exists(SUMMARY)
    assert len(large()) > 200 and len(small()) >= 50 and len(backward()) > 50


def test_every_recorded_shape_still_selects_the_recorded_plan():
    for e in large() + small() + backward():
        got = selector_evidence.describe(e["op"], e["dtype"], e["rows"], e["width"])["id"]
        assert got == e["selected"], f"{e}: the library now selects plan {got}"


def test_every_bucket_of_the_selector_has_a_line_of_evidence():
    have = {(e["op"], e["dtype"], e["lo"], e["hi"]) for e in large() + backward()}
    for dtype in selector_evidence.DTYPES:
        for op in selector_evidence.OPS + selector_evidence.BWD_OPS:
            for lo, hi, pid in selector_evidence.buckets(op, dtype):
                assert (op, dtype, lo, hi) in have, f"no evidence for {op} {dtype} {lo}-{hi} (plan {pid})"


def test_every_selected_plan_was_within_5_percent_of_the_fastest():
    slow = [e for e in large() + small() + backward() if e["ratio"] > WITHIN]
    assert not slow, f"selected plans slower than {WITHIN} x the fastest: {slow}"


def test_the_committed_tables_are_what_the_committed_sweeps_generate():
    """csrc/selector_tables.h is generated, not edited: regenerating it from
    the committed sweep records gives the same text."""
    from tile_compiler_row_gb300 import selector_tables
    text = selector_tables.render(selector_tables.committed_records())
    assert text == open(selector_tables.HEADER).read()
