"""Decode attention by its definition, per query row, in float64.

Test infrastructure only (see ``oracle/__init__.py``).

"M4.5 Decode Attention Kernels, Mask Programs, and Backend Boundaries":

* §0x01   s_t = q K^T / sqrt(d_h),  o_t = softmax(s_t) V;
* §0x02B  O = u / l, LSE = m + ln l (natural log);
* §0x02C  a row with no visible key gives O = 0, LSE = -inf;
* §0x02E  the result is independent of any disjoint exact partition, which
          ``decode_rows_split`` exercises through ``oracle.split_state``;
* §0x03A  query head h_q reads kv head floor(h_q / g).

Query row r of request b is (b, i, h_q) with the query tensor laid out as
[B, S_q, H_q, d] bf16; the visible set comes from ``oracle.masks`` and the
rows from ``oracle.cache.read_rows`` (the oracle's own page walk).

A mixed batch (§0x08F) carries ``qo_indptr`` [B+1] in the problem: request b
has C_b = qo_indptr[b+1] - qo_indptr[b] query rows, packed as rows
qo_indptr[b] + i of a [qo_indptr[B], H_q, d] query, each at position
T_b - C_b + i of its request's T_b stored rows (§0x08B bottom-right).
"""

from __future__ import annotations

import math

import numpy as np

from . import address, cache as cache_mod, masks, quant, split_state


def attend(q, K, V, scale: float):
    """(O, LSE) of one query row over the given visible rows (§0x01, §0x02B-C)."""
    q = np.asarray(q, dtype=np.float64)
    if K.shape[0] == 0:
        return np.zeros(V.shape[1]), -math.inf
    s = (K @ q) * scale
    m = s.max()
    w = np.exp(s - m)
    l = w.sum()
    return (w @ V) / l, m + math.log(l)


def query_count(problem: dict, b: int) -> int:
    """C_b: query rows of request b (S_q unless the batch is mixed, §0x08F)."""
    qo = problem.get("qo_indptr")
    return problem["S_q"] if qo is None else int(qo[b + 1] - qo[b])


def query_offset(problem: dict, b: int) -> int:
    """qo_indptr[b]: request b's first packed query row (b S_q when uniform)."""
    qo = problem.get("qo_indptr")
    return b * problem["S_q"] if qo is None else int(qo[b])


def visible_for(problem: dict, T_b: int, i: int, index_list=None, b: int = 0):
    intervals = None
    if problem.get("mask") == masks.MASK_FLASHMASK:      # packed ragged [sum T_b, 4], fm_indptr [B+1]
        ip = problem["fm_indptr"]
        intervals = np.asarray(problem["fm_intervals"]).reshape(-1, 4)[ip[b]:ip[b + 1]]
    return masks.visible_positions(problem.get("mask", masks.MASK_CAUSAL), T_b, query_count(problem, b), i,
                                   n_sink=problem.get("n_sink", 0), window=problem.get("window", 0),
                                   index_list=index_list, intervals=intervals)


def index_list_of(problem: dict, b: int, h_kv: int):
    if problem.get("mask") != masks.MASK_INDEX_LIST:
        return None
    ip = problem["index_indptr"]
    k = b * problem["H_kv"] + h_kv
    return problem["index_list"][ip[k]:ip[k + 1]]


def decode_rows(problem: dict, cache, q_bits, rows=None):
    """O [n, d] and LSE [n] for query rows ``rows`` = [(b, i, h_q), ...] (all when None).

    ``problem`` holds B, S_q, H_q, H_kv, d, sm_scale (0 -> 1/sqrt(d)), mask and
    its parameters; ``q_bits`` is the bf16 query [B, S_q, H_q, d] as uint16
    ([qo_indptr[B], H_q, d] for a mixed batch).
    """
    B, H_q, H_kv, d = (problem[k] for k in ("B", "H_q", "H_kv", "d"))
    scale = problem.get("sm_scale") or 1.0 / math.sqrt(d)
    if rows is None:
        rows = [(b, i, h) for b in range(B) for i in range(query_count(problem, b)) for h in range(H_q)]
    q = quant.bf16_bits_to_f64(q_bits).reshape(-1, H_q, d)
    O = np.zeros((len(rows), d))
    LSE = np.zeros(len(rows))
    cached = {}
    for n, (b, i, h_q) in enumerate(rows):
        h_kv = address.kv_head(h_q, H_q, H_kv)
        key = (b, i, h_kv)
        if key not in cached:
            vis = visible_for(problem, int(cache.kv_len[b]), i, index_list_of(problem, b, h_kv), b)
            cached = {key: cache_mod.read_rows(cache, b, h_kv, vis)}
        K, V = cached[key]
        O[n], LSE[n] = attend(q[query_offset(problem, b) + i, h_q], K, V, scale)
    return O, LSE


def decode_rows_split(problem: dict, cache, q_bits, rows, n_splits: int, order=None, tree=False):
    """Same rows computed as n_splits balanced partial states merged afterwards (§0x02E, §0x03B).

    Splits partition the row's visible list; ``order`` permutes the fold and
    ``tree`` uses a balanced reduction instead of a left fold.
    """
    H_q, H_kv, d = problem["H_q"], problem["H_kv"], problem["d"]
    scale = problem.get("sm_scale") or 1.0 / math.sqrt(d)
    q = quant.bf16_bits_to_f64(q_bits).reshape(-1, H_q, d)
    O = np.zeros((len(rows), d))
    LSE = np.zeros(len(rows))
    for n, (b, i, h_q) in enumerate(rows):
        h_kv = address.kv_head(h_q, H_q, H_kv)
        vis = visible_for(problem, int(cache.kv_len[b]), i, index_list_of(problem, b, h_kv), b)
        K, V = cache_mod.read_rows(cache, b, h_kv, vis)
        s = (K @ q[query_offset(problem, b) + i, h_q]) * scale
        states = []
        for a, e in split_state.balanced_split_bounds(len(vis), n_splits):
            states.append(split_state.summarize(s[a:e], V[a:e], np.ones(e - a, bool)))
        st = split_state.merge_balanced(states) if tree else split_state.merge_all(states, order)
        O[n], LSE[n] = split_state.finalize(st)
    return O, LSE
