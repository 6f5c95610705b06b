"""Host logic of bench.py's shape-table arm (no GPU): the shapes it asks the sweep
for and the with/without report it builds from the two timings."""
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
import gemv_dg_bf16_gb300 as dg  # noqa: E402


def test_table_shapes_cover_every_timed_decode_shape():
    sh = bench._table_shapes(dg)
    assert len(sh) == len(set(sh))
    gemv = {(M, N, K) for (op, M, N, K, _, _) in sh if op == dg.DG_OP_GEMV_BF16}
    assert {(M, N, K) for (N, K) in bench.SWEEP_NK for M in bench.SWEEP_M} <= gemv
    assert (1, 2048, 1024) in gemv
    assert {M for (op, M, *_r) in sh if op == dg.DG_OP_GATE_UP_SILU} == set(bench.GATE_UP_M)
    assert {M for (op, M, *_r) in sh if op == dg.DG_OP_HEAD_FP8_ARGMAX} == set(bench.HEAD_M)
    for op, n, k in ((dg.DG_OP_MOE_W1, bench.MOE_I, bench.MOE_K), (dg.DG_OP_MOE_W2, bench.MOE_K, bench.MOE_I)):
        rows = [s for s in sh if s[0] == op]
        assert {s[1] for s in rows} == set(bench.MOE_M)
        assert all(s[2:] == (n, k, bench.MOE_TOPK, bench.MOE_E) for s in rows)
    # every row count is one of the selector's buckets, so no two requests share a key
    assert all(s[1] in dg.ROWS_BUCKETS for s in sh)


def test_table_report_compares_the_same_shapes():
    pick = {"variant": 4, "params": [2, 8, 0, 4, 0, 0]}
    default = {"variant": 4, "params": [0, 0, 0, 0, 0, 0]}
    table = {"identity": {"build": "abc", "arch": "sm_103"},
             "entries": [{"op": "gemv_bf16", "M": 2, "N": 4096, "K": 4096, "pick": pick, "pick_us": 9.0,
                          "default": default, "default_us": 10.0},
                         {"op": "gemv_bf16", "M": 1, "N": 4096, "K": 4096, "pick": default, "pick_us": 7.0,
                          "default": default, "default_us": 7.0}]}
    sweep = [{"M": 1, "N": 4096, "K": 4096, "us": 7.0, "weight_bytes": 7000},
             {"M": 2, "N": 4096, "K": 4096, "us": 9.0, "weight_bytes": 9000}]
    defaults = [{"M": 2, "N": 4096, "K": 4096, "us": 10.0, "weight_bytes": 9000},
                {"M": 1, "N": 4096, "K": 4096, "us": 7.0, "weight_bytes": 7000}]

    class FakeDg:
        @staticmethod
        def dg_table_entries():
            return 2

    r = bench._table_report(table, "/x/y/table.json", FakeDg, defaults, sweep, peak=1.0)
    assert r["path"] == "table.json" and r["identity"]["build"] == "abc"
    assert r["entries"] == 2 and r["entries_not_default"] == 1
    assert r["changed"][0]["M"] == 2 and r["changed"][0]["pick"] == pick
    # 16000 bytes in 17 us with the defaults
    assert r["defaults_value"] == pytest.approx(16000 / 17e-6 / 1e9, abs=0.05)
    assert [(s["M"], s["us_table"], s["us_default"]) for s in r["shapes"]] == [(1, 7.0, 7.0), (2, 9.0, 10.0)]


@pytest.mark.parametrize("wb_mb", [4.2, 16.8, 33.6, 67.1, 100.7, 201.3, 1017.1])
def test_weight_copies_defeat_l2_across_consecutive_graphs(wb_mb):
    """A graph of R calls rotates over the copies; the next graph over the same copies
    (the next row count) starts again at copy 0.  With at most R copies every call's copy
    was last used at least 3x L2 of other weights earlier, inside a graph and across the
    seam; with more copies than calls (matrices under 3x L2 / R) a graph uses its first R
    copies, all distinct."""
    l2, R = 126 * 2 ** 20, 16
    wb = int(wb_mb * 1e6)
    n = bench._copies_for(wb, l2)
    assert n >= 2 and n * wb >= 3 * l2
    seq = [i % n for i in range(R)] * 3                      # three graphs back to back
    used = min(R, n)
    for pos, c in enumerate(seq):
        prev = [p for p in range(pos) if seq[p] == c]
        if prev:
            gap = pos - prev[-1] - 1                         # other calls in between
            assert gap * wb >= min(3 * l2, (used - 1) * wb), (n, pos, c, gap)
    if n <= R:
        assert R % n == 0                                    # whole rotations per graph
