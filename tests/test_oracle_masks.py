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


# ---- FlashMask two-interval columns (M4.5 §0x06A-§0x06D) -------------------------------

def _fm_golden():
    import json
    import os
    with open(os.path.join(os.path.dirname(__file__), "golden", "flashmask_column.json")) as f:
        return json.load(f)


def test_flashmask_worked_column_half_open():
    g = _fm_golden()
    iv = np.zeros((g["column"] + 1, 4), np.int64)
    iv[g["column"]] = [g["UT"][0], g["UT"][1], g["LT"][0], g["LT"][1]]
    masked = [i for i in range(16) if masks.flashmask_masked(iv, i)[g["column"]]]
    assert masked == g["masked_rows"]
    for i in g["visible_rows_between"] + [g["first_row_after_LT"]]:
        assert g["column"] in masks.visible_positions("flashmask", g["column"] + 1, 16, i, intervals=iv)


def _random_intervals(rng, n, S_q):
    a = rng.integers(0, S_q + 1, size=(n, 2))
    b = rng.integers(0, S_q + 1, size=(n, 2))
    iv = np.concatenate([np.sort(a, axis=1), np.sort(b, axis=1)], axis=1)
    full = rng.random(n) < 0.15                       # some columns masked for every row
    iv[full] = [0, S_q, 0, 0]
    empty = rng.random(n) < 0.3                       # and some visible to every row
    iv[empty] = [0, 0, 0, 0]
    return iv


@pytest.mark.parametrize("seed", range(6))
def test_flashmask_tile_class_is_conservative_and_exact_on_uniform_blocks(seed):
    """The eight-summary classifier never calls a tile SKIP when a cell is visible nor FULL
    when a cell is hidden (brute force over the dense mask); on blocks whose columns share
    one interval pair it is exact."""
    rng = np.random.default_rng(seed)
    S_q, n, Bc = 12, 96, 16
    iv = _random_intervals(rng, n, S_q)
    dense_masked = np.stack([masks.flashmask_masked(iv, i) for i in range(S_q)])      # [rows, keys]
    for k0 in range(0, n, Bc):
        summ = masks.flashmask_summaries(iv, k0, k0 + Bc)
        for q0 in range(S_q):
            for q1 in range(q0 + 1, S_q + 1):
                cls = masks.flashmask_tile_class(q0, q1, summ)
                cells = dense_masked[q0:q1, k0:k0 + Bc]
                if cls == "SKIP":
                    assert cells.all()
                if cls == "FULL":
                    assert not cells.any()
    # uniform blocks: the summary is exact
    for trial in range(50):
        row = _random_intervals(rng, 1, S_q)[0]
        ivu = np.tile(row, (Bc, 1))
        summ = masks.flashmask_summaries(ivu, 0, Bc)
        q0 = int(rng.integers(0, S_q))
        q1 = int(rng.integers(q0 + 1, S_q + 1))
        vis = [masks.visible_positions("flashmask", Bc, S_q, i, intervals=ivu) for i in range(q0, q1)]
        exact = masks.tile_class(vis, 0, Bc)
        got = masks.flashmask_tile_class(q0, q1, summ)
        if exact != "PARTIAL":
            assert got in (exact, "PARTIAL")
        if got != "PARTIAL":
            assert got == exact


def _dfs_tree(rng, n):
    parent = [-1] + [int(rng.integers(0, j)) for j in range(1, n)]   # parent index < child index
    children = [[] for _ in range(n)]
    for j in range(1, n):
        children[parent[j]].append(j)
    order, span = [], {}

    def visit(u):
        start = len(order)
        order.append(u)
        for c in children[u]:
            visit(c)
        span[u] = (start, len(order))
    visit(0)
    return parent, order, span


@pytest.mark.parametrize("seed", range(4))
def test_flashmask_encodes_a_dfs_ordered_speculation_tree(seed):
    """Draft tokens in DFS order: row r (node order[r]) sees node u iff u is an ancestor of
    (or is) order[r]; the rows that see u are its subtree, one contiguous range [s, e), so
    U = [0, s) and L = [e, S_q) encode the column exactly (prefix columns: no interval)."""
    rng = np.random.default_rng(seed)
    S_q, T0 = 10, 7
    parent, order, span = _dfs_tree(rng, S_q)
    pos = {u: r for r, u in enumerate(order)}
    iv = np.zeros((T0 + S_q, 4), np.int64)
    for r, u in enumerate(order):
        s, e = span[u]
        iv[T0 + r] = [0, s, e, S_q]
    for r, u in enumerate(order):
        anc = set()
        x = u
        while x != -1:
            anc.add(x)
            x = parent[x]
        expect = list(range(T0)) + sorted(T0 + pos[a] for a in anc)
        got = masks.visible_positions("flashmask", T0 + S_q, S_q, r, intervals=iv).tolist()
        assert got == expect


def test_flashmask_reproduces_bottom_right_causal():
    """Causal rows of a verify call written as upper intervals: column j hides rows
    i < j - (T - S_q); the visible sets equal the causal ones."""
    for T, S_q in ((10, 4), (3, 5), (64, 1), (1, 3)):
        iv = np.zeros((T, 4), np.int64)
        for j in range(T):
            iv[j] = [0, max(0, min(S_q, j - (T - S_q))), 0, 0]
        for i in range(S_q):
            assert np.array_equal(masks.visible_positions("flashmask", T, S_q, i, intervals=iv),
                                  masks.causal_visible(T, S_q, i))
