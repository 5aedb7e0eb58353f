"""Visibility programs and exact tile classes.

Test infrastructure only (see ``oracle/__init__.py``).

Follows:

* "M4.5 Decode Attention Kernels, Mask Programs, and Backend Boundaries"
  §0x05A (visibility predicate V(b, h, q, k)), §0x05C (SKIP / FULL / PARTIAL
  from set relations), §0x08B (bottom-right causal alignment p_i = T + i,
  A_i = [0, T + i + 1)), §0x08C (phase cell counts), §0x08F (mixed batch).
* "M5.4 Long-Context KV Policies: Retention, Compression, Budget Allocation"
  §0x04 (sliding window V_win(F; W)) and §0x05 (sink + recent union).
* M4.5 §0x06A-§0x06D FlashMask: per key column j two half-open masked
  query-row intervals U_j = [UTS_j, UTE_j), L_j = [LTS_j, LTE_j); eight
  min/max summaries per key block; the conservative three-way tile class.
  Reading for a decode or verify call: the masked "query rows" are the call's
  rows i in [0, S_q), the columns the request's stored keys j in [0, T_b),
  and the intervals alone decide visibility (no implicit causal limit).

Reading taken for a request whose stored length T_b already holds its S_q new
rows: the committed length before the call is T = T_b - S_q, so query row i
sits at p_i = T_b - S_q + i and its frontier is F_i = p_i + 1.  A negative p_i
(a request shorter than its query rows) leaves that row with no visible key.
"""

from __future__ import annotations

import numpy as np

MASK_CAUSAL = "causal"
MASK_SINK_WINDOW = "sink_window"
MASK_INDEX_LIST = "index_list"
MASK_FLASHMASK = "flashmask"


def query_position(T_b: int, S_q: int, i: int) -> int:
    """p_i = T + i with T = T_b - S_q committed rows  (M4.5 §0x08B)."""
    return T_b - S_q + i


def causal_visible(T_b: int, S_q: int, i: int) -> np.ndarray:
    """A_i = [0, p_i + 1), clipped to the stored rows  (M4.5 §0x08B)."""
    p = query_position(T_b, S_q, i)
    return np.arange(0, max(0, min(T_b, p + 1)), dtype=np.int64)


def sliding_window(F: int, W: int) -> np.ndarray:
    """V_win(F; W) = {max(0, F - W), ..., F - 1}  (M5.4 §0x04)."""
    return np.arange(max(0, F - W), F, dtype=np.int64)


def sink_recent(F: int, K_s: int, W: int) -> np.ndarray:
    """S_sink(F; K_s) union S_recent(F; W), never double counted  (M5.4 §0x05)."""
    sink = np.arange(0, min(K_s, F), dtype=np.int64)
    return np.union1d(sink, sliding_window(F, W))


def sink_recent_count(F: int, K_s: int, W: int) -> int:
    """|V| = min(K_s, F) + min(W, F) - I(F)  with the overlap I(F)  (M5.4 §0x05)."""
    overlap = max(0, min(K_s, F) - max(0, F - W))
    return min(K_s, F) + min(W, F) - overlap


def flashmask_masked(intervals, i: int) -> np.ndarray:
    """Boolean per key column: is query row i inside U_j or L_j?  intervals [n, 4] =
    (UTS, UTE, LTS, LTE), half-open  (M4.5 §0x06A)."""
    iv = np.asarray(intervals, dtype=np.int64).reshape(-1, 4)
    in_u = (iv[:, 0] <= i) & (i < iv[:, 1])
    in_l = (iv[:, 2] <= i) & (i < iv[:, 3])
    return in_u | in_l


def flashmask_summaries(intervals, k0: int, k1: int) -> dict:
    """The eight min/max values of the four endpoint vectors over key block [k0, k1)  (§0x06C)."""
    iv = np.asarray(intervals, dtype=np.int64).reshape(-1, 4)[k0:k1]
    out = {}
    for c, name in enumerate(("UTS", "UTE", "LTS", "LTE")):
        out[name + "_min"] = int(iv[:, c].min())
        out[name + "_max"] = int(iv[:, c].max())
    return out


def _family_relation(q0: int, q1: int, s_min: int, s_max: int, e_min: int, e_max: int) -> str:
    """Tile rows [q0, q1) against one interval family [s_j, e_j) over the block  (§0x06D)."""
    if q0 >= s_max and q1 <= e_min:
        return "COVERS"                   # every row inside every column's interval
    if q1 > s_min and q0 < e_max:
        return "MAY_OVERLAP"
    return "DISJOINT"


def flashmask_tile_class(q0: int, q1: int, summary: dict) -> str:
    """SKIP / FULL / PARTIAL of rows [q0, q1) x one key block from its eight summaries (§0x06D):
    SKIP when either family covers the tile, FULL when both are disjoint from it."""
    up = _family_relation(q0, q1, summary["UTS_min"], summary["UTS_max"], summary["UTE_min"], summary["UTE_max"])
    lo = _family_relation(q0, q1, summary["LTS_min"], summary["LTS_max"], summary["LTE_min"], summary["LTE_max"])
    if up == "COVERS" or lo == "COVERS":
        return "SKIP"
    if up == "DISJOINT" and lo == "DISJOINT":
        return "FULL"
    return "PARTIAL"


def visible_positions(mask: str, T_b: int, S_q: int, i: int, *, n_sink: int = 0,
                      window: int = 0, index_list=None, intervals=None) -> np.ndarray:
    """Sorted logical key positions visible to query row i of a request.

    * ``causal``: A_i of M4.5 §0x08B (for S_q = 1 every stored row).
    * ``sink_window``: the M5.4 §0x05 union evaluated at the row's frontier
      F_i = p_i + 1 (the window moves with the query position).
    * ``index_list``: a per-(request, kv-head) retained set (M5.4 §0x06E
      heavy + recent shape), intersected with the row's causal prefix.
    * ``flashmask``: the request's keys j in [0, T_b) whose two intervals
      (``intervals`` [T_b, 4]) do not hold row i (M4.5 §0x06A).
    """
    if mask == MASK_FLASHMASK:
        iv = np.asarray(intervals, dtype=np.int64).reshape(-1, 4)[:T_b]
        return np.nonzero(~flashmask_masked(iv, i))[0].astype(np.int64)
    p = query_position(T_b, S_q, i)
    F = max(0, min(T_b, p + 1))
    if mask == MASK_CAUSAL:
        return causal_visible(T_b, S_q, i)
    if mask == MASK_SINK_WINDOW:
        return sink_recent(F, n_sink, window)
    if mask == MASK_INDEX_LIST:
        lst = np.asarray(index_list, dtype=np.int64)
        return lst[lst < F]
    raise ValueError(mask)


def dense_mask(visible_sets, n_keys: int) -> np.ndarray:
    """Boolean [rows, n_keys] matrix, True where the key is visible (M4.5 §0x05A)."""
    out = np.zeros((len(visible_sets), n_keys), dtype=bool)
    for r, vs in enumerate(visible_sets):
        out[r, np.asarray(vs, dtype=np.int64)] = True
    return out


def tile_class(visible_sets, k0: int, k1: int) -> str:
    """Exact class of the tile (all rows) x [k0, k1)  (M4.5 §0x05C).

    SKIP if every score coordinate is masked, FULL if none is, PARTIAL otherwise.
    """
    n_cells = len(visible_sets) * (k1 - k0)
    n_visible = sum(int(np.count_nonzero((np.asarray(v) >= k0) & (np.asarray(v) < k1)))
                    for v in visible_sets)
    if n_visible == 0:
        return "SKIP"
    if n_visible == n_cells:
        return "FULL"
    return "PARTIAL"


def phase_cells(T: int, C: int):
    """(rectangle, visible, causally masked) cells of C new rows after T old ones (M4.5 §0x08B).

    Counted cell by cell from A_i = [0, T + i + 1) rather than from the closed form.
    """
    rect = C * (T + C)
    visible = sum(len(range(0, T + i + 1)) for i in range(C))
    return rect, visible, rect - visible


def mixed_batch(TC):
    """qo_indptr and the visible / rectangle totals of a mixed batch  (M4.5 §0x08F)."""
    qo = [0]
    vis = rect = 0
    for T, C in TC:
        qo.append(qo[-1] + C)
        r, v, _ = phase_cells(T, C)
        vis += v
        rect += r
    return qo, vis, rect
