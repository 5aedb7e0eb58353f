"""Split-state algebra and split/workspace ledgers, in float64.

Test infrastructure only (see ``oracle/__init__.py``).

Follows "M4.5 Decode Attention Kernels, Mask Programs, and Backend
Boundaries":

* §0x02A  canonical summary of one allowed set: (valid, m, l, u);
* §0x02B  binary merge through the common frame m = max(m_A, m_B);
* §0x02C  empty identity and the all-masked output policy (O = 0, LSE = -inf);
* §0x02F  the equivalent normalised (LSE, O) merge;
* §0x03B  balanced quotient/remainder split bounds and fixed-width chunks;
* §0x03C  producer / reducer owner counts;
* §0x03E  workspace byte formulas;
* §0x03F  reduction-path bytes and the K/V unique vs per-q-head ledgers;
* §0x03G  capacity-envelope tail and head-width padding.
"""

from __future__ import annotations

import math
from dataclasses import dataclass

import numpy as np


@dataclass(frozen=True)
class State:
    """Canonical split summary Sigma(A) = (valid, m, l, u)  (§0x02A).

    ``u`` is the unnormalised value accumulator of width d_v; it is not yet
    divided by ``l``.
    """

    valid: bool
    m: float
    l: float
    u: np.ndarray


def empty_state(d_v: int) -> State:
    """The empty identity e = (false, -inf, 0, 0)  (§0x02C)."""
    return State(False, -math.inf, 0.0, np.zeros(d_v, dtype=np.float64))


def summarize(scores, values, allowed) -> State:
    """Summary of the allowed positions of one split  (§0x02A).

    ``scores`` [n], ``values`` [n, d_v], ``allowed`` [n] bool.  The validity
    branch is taken before any max or exponential (§0x03I pseudocode).
    """
    scores = np.asarray(scores, dtype=np.float64)
    values = np.asarray(values, dtype=np.float64)
    allowed = np.asarray(allowed, dtype=bool)
    d_v = values.shape[1]
    if not allowed.any():
        return empty_state(d_v)
    s = scores[allowed]
    v = values[allowed]
    m = float(s.max())
    w = np.exp(s - m)
    return State(True, m, float(w.sum()), w @ v)


def merge(a: State, b: State) -> State:
    """Binary merge with validity branches before exp  (§0x02B, §0x02C)."""
    if not a.valid:
        return b
    if not b.valid:
        return a
    m = max(a.m, b.m)
    alpha = math.exp(a.m - m)
    beta = math.exp(b.m - m)
    return State(True, m, alpha * a.l + beta * b.l, alpha * a.u + beta * b.u)


def merge_all(states, order=None) -> State:
    """Left fold of ``merge`` over ``states`` (optionally permuted)."""
    states = list(states)
    if order is not None:
        states = [states[i] for i in order]
    acc = empty_state(len(states[0].u)) if states else None
    for s in states:
        acc = merge(acc, s)
    return acc


def merge_balanced(states) -> State:
    """Balanced binary-tree reduction of ``states`` (§0x02E, §0x02G)."""
    level = list(states)
    while len(level) > 1:
        nxt = [merge(level[i], level[i + 1]) for i in range(0, len(level) - 1, 2)]
        if len(level) % 2:
            nxt.append(level[-1])
        level = nxt
    return level[0]


def finalize(st: State):
    """O = u / l and LSE = m + ln l; all-masked rows give (0, -inf)  (§0x02B-C)."""
    if not st.valid:
        return np.zeros_like(st.u), -math.inf
    return st.u / st.l, st.m + math.log(st.l)


# ---- normalised (LSE, O) form, §0x02F ---------------------------------------

@dataclass(frozen=True)
class OutState:
    valid: bool
    lse: float
    o: np.ndarray


def to_out_state(st: State) -> OutState:
    """O_A = u_A / l_A and L_A = m_A + ln l_A  (§0x02F)."""
    o, lse = finalize(st)
    return OutState(st.valid, lse, o)


def merge_out(a: OutState, b: OutState) -> OutState:
    """(LSE, O) merge through the pivot p = max(L_A, L_B)  (§0x02F)."""
    if not a.valid:
        return b
    if not b.valid:
        return a
    p = max(a.lse, b.lse)
    lse = p + math.log(math.exp(a.lse - p) + math.exp(b.lse - p))
    return OutState(True, lse, math.exp(a.lse - lse) * a.o + math.exp(b.lse - lse) * b.o)


def naive_average(outs) -> np.ndarray:
    """The incorrect average of normalised split outputs (§0x02F counterexample)."""
    return sum(o.o for o in outs) / len(outs)


# ---- split bounds, §0x03B ---------------------------------------------------

# ---- shared-shift partials with a range guard (M4.5 §0x09C) --------------------

FALLBACK = None


def shared_shift_partial(scores, values, allowed, phi: float, lower: float, upper: float):
    """One partition's numerator and denominator in the common frame phi:
    n = sum e^{s - phi} v, l = sum e^{s - phi} over the allowed keys, or FALLBACK when
    some allowed key has s - phi <= lower or >= upper (the range guard)."""
    s = np.asarray(scores, dtype=np.float64)
    a = np.asarray(allowed, dtype=bool)
    delta = s[a] - phi
    if np.any(delta <= lower) or np.any(delta >= upper):
        return FALLBACK
    w = np.exp(delta)
    return w @ np.asarray(values, dtype=np.float64)[a], float(w.sum())


def shared_shift_attention(scores, values, allowed, bounds, phi: float, lower: float, upper: float):
    """Partitions [a, e) of one row with a shared shift; no cross-partition rescaling.  If any
    partition's guard fails the row is recomputed with synchronized partial softmax states
    (summarize + merge).  Returns (O, used_fallback)."""
    parts = [shared_shift_partial(scores[a:e], values[a:e], allowed[a:e], phi, lower, upper) for a, e in bounds]
    if any(x is FALLBACK for x in parts):
        st = merge_all([summarize(scores[a:e], values[a:e], allowed[a:e]) for a, e in bounds])
        return finalize(st)[0], True
    n = sum(x[0] for x in parts)
    l = sum(x[1] for x in parts)
    return (n / l if l > 0 else np.zeros(np.asarray(values).shape[-1])), False


def balanced_split_bounds(T: int, S: int):
    """Half-open [start, end) of each of S splits of [0, T)  (§0x03B).

    q = floor(T / S), r = T mod S, n_s = q + [s < r], start_s = s q + min(s, r).
    """
    q, r = divmod(T, S)
    out = []
    for s in range(S):
        start = s * q + min(s, r)
        out.append((start, start + q + (1 if s < r else 0)))
    return out


def fixed_chunk_bounds(T: int, C: int):
    """Fixed chunk width C gives ceil(T / C) chunks, the last one shorter  (§0x03B table)."""
    return [(a, min(a + C, T)) for a in range(0, T, C)]


# ---- owners and tails, §0x03C and §0x03G ------------------------------------

def owner_counts(B: int, H_q: int, S_cap: int, S: int | None = None):
    """Producer grid B*H_q*S_cap, reducer grid B*H_q, non-empty merges B*H_q*(S-1)  (§0x03C)."""
    S = S_cap if S is None else S
    return {
        "producers": B * H_q * S_cap,
        "reducers": B * H_q,
        "binary_merges": B * H_q * (S - 1),
    }


def capacity_envelope(T_list, S: int, S_cap: int, H_q: int):
    """Counts of the fixed-capacity fixture: active vs identity producer slots  (§0x03G).

    A slot (b, h_q, s) is active when s < S and its balanced split is non-empty.
    """
    producers = len(T_list) * H_q * S_cap
    active = 0
    per_request = []
    for T in T_list:
        lens = [e - a for a, e in balanced_split_bounds(T, S)]
        per_request.append(lens + [None] * (S_cap - S))
        active += H_q * sum(1 for n in lens if n > 0)
    return {
        "producers": producers,
        "active": active,
        "identity": producers - active,
        "reducers": len(T_list) * H_q,
        "split_lengths": per_request,
    }


def padded_width(d_v: int, align: int) -> int:
    """d_v_padded = round_up(d_v, vector_alignment_elements)  (§0x03D)."""
    return -(-d_v // align) * align


# ---- workspace and traffic ledgers, §0x03E-F --------------------------------

def workspace_mlu_bytes(n_states: int, d_v: int, b_u: int = 4, b_state: int = 4, b_valid: int = 1) -> int:
    """M_mlu = N (d_v b_u + 2 b_state + b_valid)  (§0x03E)."""
    return n_states * (d_v * b_u + 2 * b_state + b_valid)


def workspace_lse_o_bytes(n_states: int, d_v: int, b_o: int = 2, b_state: int = 4, b_valid: int = 1) -> int:
    """M_lse,o = N (d_v b_O + b_state + b_valid)  (§0x03E)."""
    return n_states * (d_v * b_o + b_state + b_valid)


def reduction_path_bytes(m_partial: int, B: int, H_q: int, d_v: int, b_o: int = 2,
                         b_state: int = 4, write_lse: bool = True) -> int:
    """2 M_partial + B H_q d_v b_O + [write LSE] B H_q b_state  (§0x03F)."""
    return 2 * m_partial + B * H_q * d_v * b_o + (B * H_q * b_state if write_lse else 0)


def kv_unique_bytes(T_list, H_kv: int, d_h: int, d_v: int, b_cache: int) -> int:
    """Sum_b T_b H_kv (d_h + d_v) b_cache  (§0x03F)."""
    return sum(T_list) * H_kv * (d_h + d_v) * b_cache


def kv_qhead_demand_bytes(T_list, H_q: int, d_h: int, d_v: int, b_cache: int) -> int:
    """Sum_b T_b H_q (d_h + d_v) b_cache  (§0x03F)."""
    return sum(T_list) * H_q * (d_h + d_v) * b_cache
