"""Pins of the oracle's split-state algebra (M4.5 §0x02A-§0x02H)."""

import math

import numpy as np
import pytest
from scipy.special import logsumexp

from oracle import split_state as ss
from tests.conftest import golden


def _worked():
    g = golden("worked_empty_middle.json")
    states = []
    for sc, vals in zip(g["scores"], g["values"]):
        allowed = [x is not None for x in sc]
        scores = [x if x is not None else 0.0 for x in sc]
        states.append(ss.summarize(scores, vals, allowed))
    return g, states


def test_worked_three_split_trace_states():
    g, (s0, s1, s2) = _worked()
    assert s0.valid and s0.m == g["split0"]["m"]
    assert s0.l == pytest.approx(g["split0"]["l"], rel=1e-15, abs=0)
    np.testing.assert_allclose(s0.u, g["split0"]["u"], rtol=1e-15, atol=1e-17)
    assert not s1.valid and s1.m == -math.inf and s1.l == 0 and not s1.u.any()
    assert s2.m == g["split2"]["m"]
    assert s2.l == pytest.approx(g["split2"]["l"], rel=1e-15)
    np.testing.assert_allclose(s2.u, g["split2"]["u"], rtol=1e-15)


def test_worked_three_split_trace_merge_and_outputs():
    g, states = _worked()
    seq = ss.merge_all(states)
    assert seq.m == g["merged"]["m"]
    assert seq.l == pytest.approx(g["merged"]["l"], rel=1e-15)
    np.testing.assert_allclose(seq.u, g["merged"]["u"], rtol=1e-15)
    o, lse = ss.finalize(seq)
    np.testing.assert_allclose(o, g["O"], rtol=1e-15)
    assert lse == pytest.approx(g["LSE"], rel=1e-15)
    # sequential, balanced and permuted trees agree to the printed bound
    for other in (ss.merge_balanced(states), ss.merge_all(states, order=[2, 0, 1]),
                  ss.merge_all(states, order=[1, 2, 0])):
        o2, lse2 = ss.finalize(other)
        assert np.max(np.abs(o2 - o)) <= g["tree_agreement_max"]
        assert abs(lse2 - lse) <= g["tree_agreement_max"] * 16


def test_worked_trace_equals_unsplit_dense_softmax():
    """Library softmax over the visible scores (no split algebra involved)."""
    g, _ = _worked()
    s = np.array([4, -1, 3, -2, 1], float)
    v = np.array([[1, 0], [0, 2], [2, 3], [-1, 4], [4, -2]], float)
    lse = logsumexp(s)
    o = np.exp(s - lse) @ v
    np.testing.assert_allclose(o, g["O"], rtol=1e-14)
    assert lse == pytest.approx(g["LSE"], rel=1e-15)


def test_empty_identity_laws():
    rng = np.random.default_rng(0)
    a = ss.summarize(rng.normal(size=5), rng.normal(size=(5, 3)), np.ones(5, bool))
    e = ss.empty_state(3)
    for x in (ss.merge(e, a), ss.merge(a, e)):
        assert x.valid and x.m == a.m and x.l == a.l and np.array_equal(x.u, a.u)
    ee = ss.merge(e, e)
    assert not ee.valid and ee.m == -math.inf and ee.l == 0
    o, lse = ss.finalize(ee)
    assert lse == -math.inf and not o.any() and not np.isnan(o).any()


def test_merge_equals_summary_of_union_commutative_associative():
    rng = np.random.default_rng(1)
    s = rng.normal(scale=4, size=30)
    v = rng.normal(size=(30, 4))
    allowed = rng.random(30) < 0.7
    parts = [(0, 7), (7, 19), (19, 30)]
    st = [ss.summarize(s[a:e], v[a:e], allowed[a:e]) for a, e in parts]
    whole = ss.summarize(s, v, allowed)
    ab = ss.merge(st[0], st[1])
    ba = ss.merge(st[1], st[0])
    assert ab.m == ba.m
    np.testing.assert_allclose(ab.u, ba.u, rtol=1e-14)
    left = ss.merge(ab, st[2])
    right = ss.merge(st[0], ss.merge(st[1], st[2]))
    for x in (left, right):
        assert x.m == whole.m
        assert x.l == pytest.approx(whole.l, rel=1e-14)
        np.testing.assert_allclose(x.u, whole.u, rtol=1e-13)


@pytest.mark.parametrize("n_splits", [1, 2, 3, 5, 8, 16, 33, 64])
def test_partition_invariance_balanced_bounds(n_splits):
    rng = np.random.default_rng(n_splits)
    T = 200
    s = rng.normal(scale=3, size=T)
    v = rng.normal(size=(T, 5))
    allowed = rng.random(T) < 0.5
    whole = ss.finalize(ss.summarize(s, v, allowed))
    states = [ss.summarize(s[a:e], v[a:e], allowed[a:e])
              for a, e in ss.balanced_split_bounds(T, n_splits)]
    for st in (ss.merge_all(states), ss.merge_balanced(states),
               ss.merge_all(states, order=rng.permutation(n_splits))):
        o, lse = ss.finalize(st)
        np.testing.assert_allclose(o, whole[0], rtol=1e-12, atol=1e-14)
        assert lse == pytest.approx(whole[1], rel=1e-12)


def test_all_masked_row_policy():
    st = ss.summarize([1.0, 2.0], [[5.0], [6.0]], [False, False])
    o, lse = ss.finalize(st)
    assert lse == -math.inf and o.tolist() == [0.0]


def test_lse_o_form_matches_mlu_form():
    """Normalised (LSE, O) merge of §0x02F is a second, independent path."""
    g, states = _worked()
    outs = [ss.to_out_state(x) for x in states]
    acc = outs[0]
    for x in outs[1:]:
        acc = ss.merge_out(acc, x)
    np.testing.assert_allclose(acc.o, g["O"], rtol=1e-14)
    assert acc.lse == pytest.approx(g["LSE"], rel=1e-15)


def test_averaging_counterexample():
    g = golden("averaging_counterexample.json")
    a = ss.summarize(g["split_a"]["scores"], np.array(g["split_a"]["values"], float)[:, None], [True, True])
    b = ss.summarize(g["split_b"]["scores"], np.array(g["split_b"]["values"], float)[:, None], [True, True])
    oa, ob = ss.to_out_state(a), ss.to_out_state(b)
    assert oa.o[0] == g["O_a"] and ob.o[0] == g["O_b"]
    assert ss.naive_average([oa, ob])[0] == g["naive_average"]
    o, _ = ss.finalize(ss.merge(a, b))
    assert round(o[0], 10) == g["O_exact_10dp"]
    assert ss.merge_out(oa, ob).o[0] == pytest.approx(o[0], rel=1e-15)


def test_fp16_order_sensitivity_and_fp64_exactness():
    g = golden("fp16_order.json")
    vals = g["equal_scores_values"]
    h = np.float16

    def seq(xs):
        acc = h(0)
        for x in xs:
            acc = h(acc + h(x))
        return acc

    def bal(xs):
        return h(h(h(xs[0]) + h(xs[1])) + h(h(xs[2]) + h(xs[3])))

    n = len(vals)
    assert float(seq(vals)) / n == g["fp16_sequential"]
    assert float(bal(vals)) / n == g["fp16_balanced"]
    assert float(seq([vals[0], vals[2], vals[1], vals[3]])) / n == g["fp16_permuted"]
    # the float64 oracle returns the exact output for equal scores
    st = ss.summarize(np.zeros(n), np.array(vals, float)[:, None], np.ones(n, bool))
    assert ss.finalize(st)[0][0] == g["exact_output"]


# ---- shared-shift partials with a range guard (M4.5 §0x09C) --------------------

def test_shared_shift_gives_the_exact_softmax_for_any_frame():
    """A common shift phi leaves the softmax ratio unchanged; partitions need no rescaling."""
    rng = np.random.default_rng(60)
    s = rng.normal(size=200) * 2.0
    v = rng.normal(size=(200, 8))
    allowed = rng.random(200) < 0.8
    exact = np.exp(s[allowed] - s[allowed].max()) @ v[allowed] / np.exp(s[allowed] - s[allowed].max()).sum()
    bounds = ss.balanced_split_bounds(200, 7)
    for phi in (0.0, 2.5, s[allowed].max(), -1.0):
        o, fell_back = ss.shared_shift_attention(s, v, allowed, bounds, phi, -40.0, 40.0)
        assert not fell_back
        np.testing.assert_allclose(o, exact, rtol=1e-12, atol=1e-12)


def test_shared_shift_guard_boundaries_and_fallback():
    s = np.array([0.0, 1.0, 2.9, -2.9])
    v = np.eye(4)
    allowed = np.ones(4, bool)
    n, l = ss.shared_shift_partial(s, v, allowed, 0.0, -3.0, 3.0)
    assert l == pytest.approx(1 + math.e + math.exp(2.9) + math.exp(-2.9))
    # the guard is exclusive at both ends (the pages' delta <= lower / delta >= upper)
    assert ss.shared_shift_partial(np.array([3.0]), v[:1], allowed[:1], 0.0, -3.0, 3.0) is ss.FALLBACK
    assert ss.shared_shift_partial(np.array([-3.0]), v[:1], allowed[:1], 0.0, -3.0, 3.0) is ss.FALLBACK
    # a masked key outside the range does not trip the guard
    assert ss.shared_shift_partial(np.array([0.0, 9.0]), v[:2], np.array([True, False]), 0.0, -3.0, 3.0) \
        is not ss.FALLBACK
    # one failing partition sends the whole row to synchronized partial softmax: still exact
    s2 = np.array([0.0, 0.5, 6.0, 1.0])
    o, fell_back = ss.shared_shift_attention(s2, v, allowed, [(0, 2), (2, 4)], 0.0, -3.0, 3.0)
    assert fell_back
    w = np.exp(s2 - s2.max())
    np.testing.assert_allclose(o, w / w.sum(), rtol=1e-12)
    # an all-masked row has no partial to guard and gives zeros
    o, fell_back = ss.shared_shift_attention(s2, v, np.zeros(4, bool), [(0, 4)], 0.0, -3.0, 3.0)
    assert not fell_back and not o.any()
