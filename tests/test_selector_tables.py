"""The rules of the selector-table generator (selector_tables.tables), on
synthetic sweep records (CPU only): the fastest register plan is taken, the
plan selected when the sweep ran is kept while it is within 0.5 % of the
fastest, a whole-vector plan enters its table only when it beats the best
register plan by more than 1 %, equal times go to the lower plan id, and
FP16 records are averaged with the BF16 ones (the two types share the
2-byte tables)."""

import pytest

from tile_compiler_row_gb300 import selector_tables as st


def _base_records():
    """One large-problem record per (family, op, ladder width), every one
    won by register plan 2 with no whole-vector plan timed."""
    recs = []
    for dtype in st.FAMILIES:
        for op in st.TABLE_OPS:
            for w in st.LADDER[dtype]:
                recs.append({"op": op, "dtype": dtype, "width": w, "rows": 1 << 14,
                             "regime": "large", "selected": None,
                             "plans": {"2": 100.0, "3": 120.0}})
    return recs


def _with(recs, dtype, op, width, plans, selected=None, extra=()):
    out = [r for r in recs if not (r["dtype"] == dtype and r["op"] == op and r["width"] == width)]
    out.append({"op": op, "dtype": dtype, "width": width, "rows": 1 << 14, "regime": "large",
                "selected": selected, "plans": plans})
    out.extend(extra)
    return out


def _pick(records, family, op, width, table="reg"):
    big, _ = st.tables(records)
    bound = width + st.TAIL[family] if width != st.LADDER[family][-1] else st.MAX_WIDTH
    rows = big[(family, op)][table]
    return dict(rows)[bound]


def test_every_bucket_takes_the_fastest_register_plan():
    big, _ = st.tables(_base_records())
    for (family, op), t in big.items():
        assert all(p == 2 for _, p in t["reg"]), (family, op)
        assert all(p == -1 for _, p in t["staged"]), (family, op)


def test_the_fastest_register_plan_replaces_a_slower_selected_one():
    recs = _with(_base_records(), "bf16", "layernorm", 4096,
                 {"6": 100.0, "5": 90.0, "44": 80.0}, selected=6)
    assert _pick(recs, "bf16", "layernorm", 4096) == 5
    assert _pick(recs, "bf16", "layernorm", 4096, "staged") == 44


def test_the_selected_plan_is_kept_within_half_a_percent():
    recs = _with(_base_records(), "f32", "softmax", 2048, {"6": 100.4, "5": 100.0}, selected=6)
    assert _pick(recs, "f32", "softmax", 2048) == 6
    recs = _with(_base_records(), "f32", "softmax", 2048, {"6": 100.6, "5": 100.0}, selected=6)
    assert _pick(recs, "f32", "softmax", 2048) == 5


@pytest.mark.parametrize("staged_us,expect", [(99.4, -1), (98.9, 44)])
def test_a_whole_vector_plan_must_win_by_more_than_one_percent(staged_us, expect):
    recs = _with(_base_records(), "bf16", "rmsnorm", 8192, {"5": 100.0, "44": staged_us})
    assert _pick(recs, "bf16", "rmsnorm", 8192, "staged") == expect
    assert _pick(recs, "bf16", "rmsnorm", 8192) == 5


def test_equal_times_go_to_the_lower_plan_id():
    recs = _with(_base_records(), "f32", "layernorm", 1024, {"7": 100.0, "5": 100.0})
    assert _pick(recs, "f32", "layernorm", 1024) == 5


def test_fp16_records_are_averaged_with_the_bf16_ones():
    recs = _with(_base_records(), "bf16", "softmax", 6144, {"8": 93.0, "7": 93.5})
    assert _pick(recs, "bf16", "softmax", 6144) == 8
    f16 = {"op": "softmax", "dtype": "f16", "width": 6144, "rows": 1 << 14, "regime": "large",
           "selected": None, "plans": {"8": 93.1, "7": 81.9}}
    assert _pick(recs + [f16], "bf16", "softmax", 6144) == 7    # means 93.05 against 87.7


def test_a_plan_timed_only_by_a_newer_sweep_counts_from_that_sweep():
    old = _with(_base_records(), "f32", "rmsnorm", 4096, {"5": 100.0, "6": 102.0})
    new = {"op": "rmsnorm", "dtype": "f32", "width": 4096, "rows": 1 << 14, "regime": "large",
           "selected": None, "plans": {"5": 100.0, "6": 102.0, "39": 95.0}}
    assert _pick(old + [new], "f32", "rmsnorm", 4096) == 39
