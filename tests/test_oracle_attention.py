"""Pins of the oracle's decode attention (M4.5 §0x01, §0x02B-§0x02E, §0x08B; M5.4 §0x05)."""

import math

import numpy as np
import pytest
from scipy.special import logsumexp

from oracle import attention, masks
from oracle import cache as cm
from oracle import quant
from tests.conftest import golden


def _bf16(rng, shape, scale=1.0):
    x = (rng.standard_normal(shape) * scale).astype(np.float32)
    u = x.view(np.uint32).astype(np.uint64)
    return ((u + 0x7FFF + ((u >> 16) & 1)) >> 16).astype(np.uint16)


def _paged_case(rng, lens, H_kv, d, P, extra_pages=5):
    """Logical K/V [B][T][H][d] plus a permuted paged copy written by the oracle writer."""
    n_pages = [-(-T // P) for T in lens]
    pool = sum(n_pages) + extra_pages
    perm = rng.permutation(pool)
    indptr = np.concatenate([[0], np.cumsum(n_pages)]).astype(np.int64)
    indices = perm[:indptr[-1]]
    rows_indptr = np.concatenate([[0], np.cumsum(lens)]).astype(np.int64)
    k = _bf16(rng, (rows_indptr[-1], H_kv, d))
    v = _bf16(rng, (rows_indptr[-1], H_kv, d))
    c = cm.empty_paged("bf16", pool, H_kv, P, d, len(lens))
    c.k[:] = 0x7FC0          # poison: unreferenced pages and tails hold NaN
    c.v[:] = 0x7FC0
    cm.write_history(c, indptr, indices, rows_indptr, k, v)
    return c, k, v, rows_indptr


def _brute(problem, k, v, rows_indptr, q, b, i, h_q, index_list=None):
    """Dense-matrix attention on the logical tensors with a library softmax."""
    H_q, H_kv, d, S_q = problem["H_q"], problem["H_kv"], problem["d"], problem["S_q"]
    T = rows_indptr[b + 1] - rows_indptr[b]
    h = h_q // (H_q // H_kv)
    K = quant.bf16_bits_to_f64(k[rows_indptr[b]:rows_indptr[b + 1], h])
    V = quant.bf16_bits_to_f64(v[rows_indptr[b]:rows_indptr[b + 1], h])
    s = K @ quant.bf16_bits_to_f64(q[b, i, h_q]) / math.sqrt(d)
    vis = masks.visible_positions(problem.get("mask", "causal"), T, S_q, i,
                                  n_sink=problem.get("n_sink", 0), window=problem.get("window", 0),
                                  index_list=index_list)
    allowed = masks.dense_mask([vis], T)[0]
    if not allowed.any():
        return np.zeros(d), -math.inf
    s = np.where(allowed, s, -np.inf)
    lse = logsumexp(s)
    return np.exp(s - lse) @ V, lse


@pytest.mark.parametrize("mask,S_q", [("causal", 1), ("causal", 3), ("sink_window", 1),
                                      ("sink_window", 2), ("index_list", 1)])
def test_decode_rows_match_brute_force(mask, S_q):
    rng = np.random.default_rng(11)
    lens = [37, 1, 64, 50]
    B, H_q, H_kv, d, P = len(lens), 8, 2, 16, 16
    c, k, v, ri = _paged_case(rng, lens, H_kv, d, P)
    q = _bf16(rng, (B, S_q, H_q, d))
    problem = dict(B=B, S_q=S_q, H_q=H_q, H_kv=H_kv, d=d, mask=mask, n_sink=3, window=9)
    if mask == "index_list":
        lists, ptr = [], [0]
        for b, T in enumerate(lens):
            for h in range(H_kv):
                lst = np.sort(rng.choice(T, size=max(1, T // 3), replace=False))
                lists.append(lst)
                ptr.append(ptr[-1] + len(lst))
        problem["index_indptr"] = np.array(ptr)
        problem["index_list"] = np.concatenate(lists)
    O, LSE = attention.decode_rows(problem, c, q)
    n = 0
    for b in range(B):
        for i in range(S_q):
            for h in range(H_q):
                il = attention.index_list_of(problem, b, h // (H_q // H_kv))
                o, lse = _brute(problem, k, v, ri, q, b, i, h, il)
                if lse == -math.inf:
                    assert LSE[n] == -math.inf and not O[n].any()
                else:
                    np.testing.assert_allclose(O[n], o, rtol=1e-12, atol=1e-13)
                    assert LSE[n] == pytest.approx(lse, rel=1e-13)
                n += 1
    assert np.isfinite(O).all()


@pytest.mark.parametrize("n_splits", [1, 2, 3, 4, 7, 16, 64])
def test_split_count_invariance(n_splits):
    rng = np.random.default_rng(12)
    lens = [100, 3, 0, 64]
    c, k, v, ri = _paged_case(rng, lens, 2, 32, 16)
    problem = dict(B=4, S_q=1, H_q=4, H_kv=2, d=32)
    q = _bf16(rng, (4, 1, 4, 32))
    rows = [(b, 0, h) for b in range(4) for h in range(4)]
    O, LSE = attention.decode_rows(problem, c, q, rows)
    for tree in (False, True):
        O2, LSE2 = attention.decode_rows_split(problem, c, q, rows, n_splits, tree=tree)
        np.testing.assert_allclose(O2, O, rtol=1e-12, atol=1e-14)
        fin = np.isfinite(LSE)
        np.testing.assert_allclose(LSE2[fin], LSE[fin], rtol=1e-12)
        assert np.array_equal(LSE2[~fin], LSE[~fin])


def test_single_visible_key_and_equal_keys():
    rng = np.random.default_rng(13)
    d = 8
    q = rng.normal(size=d)
    K = rng.normal(size=(1, d))
    V = rng.normal(size=(1, d))
    o, lse = attention.attend(q, K, V, 0.5)
    assert np.array_equal(o, V[0]) and lse == pytest.approx(0.5 * float(K[0] @ q), rel=1e-15)
    K = np.repeat(rng.normal(size=(1, d)), 6, axis=0)
    V = rng.normal(size=(6, d))
    o, lse = attention.attend(q, K, V, 0.5)
    np.testing.assert_allclose(o, V.mean(axis=0), rtol=1e-14)
    assert lse == pytest.approx(0.5 * float(K[0] @ q) + math.log(6), rel=1e-14)


def test_all_masked_rows_give_zero_and_minus_inf():
    rng = np.random.default_rng(14)
    c, k, v, ri = _paged_case(rng, [1], 1, 8, 4)
    q = _bf16(rng, (1, 4, 2, 8))
    O, LSE = attention.decode_rows(dict(B=1, S_q=4, H_q=2, H_kv=1, d=8), c, q)
    assert np.all(LSE[:6] == -math.inf) and not O[:6].any()
    assert np.isfinite(LSE[6:]).all()
    np.testing.assert_array_equal(O[6], quant.bf16_bits_to_f64(v[0, 0]))


def test_sink_window_within_window_equals_full_attention():
    rng = np.random.default_rng(15)
    lens = [20, 33]
    c, k, v, ri = _paged_case(rng, lens, 2, 16, 8)
    q = _bf16(rng, (2, 1, 4, 16))
    full = attention.decode_rows(dict(B=2, S_q=1, H_q=4, H_kv=2, d=16), c, q)
    sw = attention.decode_rows(dict(B=2, S_q=1, H_q=4, H_kv=2, d=16, mask="sink_window",
                                    n_sink=4, window=40), c, q)
    assert np.array_equal(full[0], sw[0]) and np.array_equal(full[1], sw[1])


def test_symbolic_gather_through_index_lists():
    """Payload ids K[l,h,t,c] = 1000 l + 100 h + 10 t + c gathered through the page walk."""
    g = golden("retention_fixture.json")["gather"]
    L, H, T, d, P = g["L"], g["H_kv"], g["T"], g["d_h"], 4
    n_pages = L * (T // P)
    perm = np.random.default_rng(16).permutation(n_pages)
    indptr = np.arange(0, n_pages + 1, T // P)
    kpool = np.zeros((n_pages, H, P, d), np.int64)
    vpool = np.zeros_like(kpool)
    c = cm.Cache("paged", "bf16", H, d, P=P, page_indptr=indptr, page_indices=perm,
                 kv_len=np.full(L, T))
    for l in range(L):
        pages, rows = cm._pages_and_rows(c, l, np.arange(T))
        for h in range(H):
            for t in range(T):
                kpool[pages[t], h, rows[t]] = [1000 * l + 100 * h + 10 * t + x for x in range(d)]
                vpool[pages[t], h, rows[t]] = [5000 + 1000 * l + 100 * h + 10 * t + x for x in range(d)]
    pr = g["probe"]
    lst = np.array(g["positions"][pr["layer"]][pr["h_kv"]])
    pages, rows = cm._pages_and_rows(c, pr["layer"], lst)
    assert lst[pr["packed_row"]] == pr["position"]
    assert kpool[pages, pr["h_kv"], rows][pr["packed_row"]].tolist() == pr["K"]
    assert vpool[pages, pr["h_kv"], rows][pr["packed_row"]].tolist() == pr["V"]


def test_mixed_batch_rows_follow_their_own_request():
    """§0x08F mixed batch: packed query rows, C_b per request, bottom-right positions.

    The phase fixture's three requests (prefill (0,4), append (6,2), decode (9,1))
    after their rows are staged: T_b + C_b stored rows, qo_indptr [0, 4, 6, 7].
    Each packed row is checked against a dense softmax over keys [0, T_b + i + 1)
    written out here, and the visible cells against the fixture's total.
    """
    g = golden("phase_fixture.json")["mixed"]
    TC = g["TC"]
    lens = [T + C for T, C in TC]
    qo = np.array(g["qo_indptr"])
    rng = np.random.default_rng(16)
    B, H_q, H_kv, d, P = len(TC), 4, 2, 16, 4
    c, k, v, ri = _paged_case(rng, lens, H_kv, d, P)
    S_q = max(C for _, C in TC)
    q = _bf16(rng, (int(qo[-1]), H_q, d))
    problem = dict(B=B, S_q=S_q, H_q=H_q, H_kv=H_kv, d=d, qo_indptr=qo)
    cells = sum(len(attention.visible_for(problem, lens[b], i, None, b)) for b in range(B)
                for i in range(TC[b][1]))
    assert cells == g["visible"]
    O, LSE = attention.decode_rows(problem, c, q)
    assert len(O) == qo[-1] * H_q
    n = 0
    for b, (T, C) in enumerate(TC):
        for i in range(C):
            for h in range(H_q):
                hk = h // (H_q // H_kv)
                K = quant.bf16_bits_to_f64(k[ri[b]:ri[b] + T + i + 1, hk])
                V = quant.bf16_bits_to_f64(v[ri[b]:ri[b] + T + i + 1, hk])
                s = K @ quant.bf16_bits_to_f64(q[qo[b] + i, h]) / math.sqrt(d)
                lse = logsumexp(s)
                np.testing.assert_allclose(O[n], np.exp(s - lse) @ V, rtol=1e-12, atol=1e-13)
                assert LSE[n] == pytest.approx(lse, rel=1e-13)
                n += 1
    # a request alone, as a uniform batch of S_q = C_b rows, gives the same rows
    n = 0
    for b, (T, C) in enumerate(TC):
        one = cm.empty_paged("bf16", c.k.shape[0], H_kv, P, d, 1)
        one.k, one.v = c.k, c.v
        one.page_indptr = np.array([0, c.page_indptr[b + 1] - c.page_indptr[b]])
        one.page_indices = c.page_indices[c.page_indptr[b]:c.page_indptr[b + 1]]
        one.kv_len = np.array([lens[b]])
        O1, L1 = attention.decode_rows(dict(B=1, S_q=C, H_q=H_q, H_kv=H_kv, d=d), one,
                                       q[qo[b]:qo[b + 1]].reshape(1, C, H_q, d))
        np.testing.assert_array_equal(O1, O[n:n + C * H_q])
        np.testing.assert_array_equal(L1, LSE[n:n + C * H_q])
        n += C * H_q
