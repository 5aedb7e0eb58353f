"""Pins of visibility programs and tile classes (M5.4 §0x04-§0x05, M4.5 §0x05C, §0x08)."""

import numpy as np
import pytest

from oracle import masks
from tests.conftest import golden


def test_sliding_window_trace():
    g = golden("retention_fixture.json")["window"]
    for F, want in g["cases"]:
        assert masks.sliding_window(F, g["W"]).tolist() == want


def test_sink_recent_trace_and_counts():
    g = golden("retention_fixture.json")["sink_recent"]
    K_s, W = g["K_s"], g["W"]
    for F, want in g["sets"]:
        assert masks.sink_recent(F, K_s, W).tolist() == want
    counts = [len(masks.sink_recent(F, K_s, W)) for F in range(0, 12)]
    assert max(counts) == g["max_rows"]
    assert counts.index(g["max_rows"]) == g["first_full_F"]
    # first irrecoverable middle omission: some position < F - W that is not a sink
    first_omission = next(F for F in range(20)
                          if set(range(F)) - set(masks.sink_recent(F, K_s, W).tolist()))
    assert first_omission == g["first_omission_F"]


@pytest.mark.parametrize("K_s,W", [(0, 5), (2, 3), (4, 4096), (64, 512), (7, 1)])
def test_sink_recent_closed_form_matches_set(K_s, W):
    for F in list(range(0, 40)) + [4099, 4100, 4101, 32768]:
        assert masks.sink_recent_count(F, K_s, W) == len(masks.sink_recent(F, K_s, W))


def test_sink_window_covers_everything_when_frontier_within_window():
    for F in range(0, 50):
        assert masks.visible_positions("sink_window", F, 1, 0, n_sink=4, window=64).tolist() == \
            list(range(F))


def test_causal_bottom_right_rows():
    g = golden("phase_fixture.json")["append_rows"]
    T, C = g["T"], g["C"]
    for i, (a, e) in enumerate(g["visible"]):
        assert masks.causal_visible(T + C, C, i).tolist() == list(range(a, e))


def test_short_request_rows_are_all_masked():
    """A request holding one row with four verify queries: rows 0..2 see nothing."""
    vis = [masks.causal_visible(1, 4, i).tolist() for i in range(4)]
    assert vis == [[], [], [], [0]]


def test_phase_cells_and_mixed_batch():
    g = golden("phase_fixture.json")
    for (T, C), want in g["cases"]:
        assert list(masks.phase_cells(T, C)) == want
        # closed forms of §0x08B
        assert want[1] == C * T + C * (C + 1) // 2 and want[2] == C * (C - 1) // 2
    m = g["mixed"]
    qo, vis, rect = masks.mixed_batch(m["TC"])
    assert qo == m["qo_indptr"] and vis == m["visible"] and rect == m["rect"]
    n = len(m["TC"])
    max_c = max(c for _, c in m["TC"])
    max_kv = max(t + c for t, c in m["TC"])
    assert n * max_c * max_kv == m["envelope_cells"]
    assert m["envelope_cells"] - rect == m["beyond_rectangles"]


def test_tile_class_against_dense_matrix():
    rng = np.random.default_rng(5)
    for _ in range(200):
        rows = rng.integers(1, 5)
        n = 24
        sets = [np.flatnonzero(rng.random(n) < rng.random()) for _ in range(rows)]
        dense = masks.dense_mask(sets, n)
        k0 = rng.integers(0, n - 1)
        k1 = rng.integers(k0 + 1, n + 1)
        tile = dense[:, k0:k1]
        want = "SKIP" if not tile.any() else ("FULL" if tile.all() else "PARTIAL")
        assert masks.tile_class(sets, k0, k1) == want


def test_index_list_rows_respect_causal_prefix():
    lst = [0, 3, 5, 9, 10]
    assert masks.visible_positions("index_list", 11, 1, 0, index_list=lst).tolist() == lst
    assert masks.visible_positions("index_list", 11, 3, 0, index_list=lst).tolist() == [0, 3, 5]
