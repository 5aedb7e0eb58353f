"""GPU parity of the shared-shift partials (FlashDecoding++, "M4.5 Decode Attention Kernels,
Mask Programs, and Backend Boundaries" §0x09C) against the fp64 oracle, through dattn_run_ex.

With the guard holding, the partials live in the common frame phi and need no rescaling, so the
result is the exact softmax up to rounding; when the guard fails somewhere the kernel moves to
synchronized states, and the result is the same.  The oracle's shared_shift_attention decides,
per row, whether the guard holds: where it holds for every row the kernel must count no fallback,
where it fails for every row the kernel must count some.
"""

import math

import numpy as np
import pytest
import torch

import split_kv_decode_flash_gb300 as dattn
import workloads as W
from oracle import address, attention, quant, split_state
from oracle import cache as ocache
from tests import gpu_helpers as H

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    dattn.load()


def run_shift(w, shift, *, num_sms=None, chunk_tokens=0, fused_merge=False):
    p = w.problem
    B, S_q, H_q, d = p["B"], p["S_q"], p["H_q"], p["d"]
    plan = dattn.dattn_plan(p, w.kv_len, page_indptr=w.page_indptr, index_indptr=w.index_indptr,
                            index_list=w.index_list, num_sms=num_sms, chunk_tokens=chunk_tokens,
                            fused_merge=fused_merge, qo_indptr=w.qo_indptr)
    n_rows = B * S_q if w.qo_indptr is None else int(w.qo_indptr[-1])
    o = torch.full((n_rows, H_q, d), float("nan"), dtype=torch.bfloat16, device="cuda")
    lse = torch.full((n_rows, H_q), float("nan"), dtype=torch.float32, device="cuda")
    ws = torch.empty(max(256, plan.workspace_bytes), dtype=torch.uint8, device="cuda")
    dattn.dattn_run_ex(plan, p, dattn.tensors_from(**H.device_tensors(w, o, lse)), ws, shared_shift=shift)
    torch.cuda.synchronize()
    flags = dattn.dattn_device_status(ws)
    fallbacks = dattn.dattn_shift_fallbacks(ws)
    if w.qo_indptr is None:
        o, lse = o.view(B, S_q, H_q, d), lse.view(B, S_q, H_q)
    return o.float().cpu(), lse.cpu(), flags, fallbacks


def oracle_guard(w, rows, shift):
    """Per row: does the oracle's shared-shift reading fall back (one partition per row)?"""
    phi, lo, hi = shift
    p = H.oracle_problem(w)
    cache = H.oracle_cache(w)
    H_q, H_kv, d = p["H_q"], p["H_kv"], p["d"]
    q = quant.bf16_bits_to_f64(H.bits(w.q)).reshape(-1, H_q, d)
    scale = p.get("sm_scale") or 1.0 / math.sqrt(d)
    out = []
    for b, i, h in rows:
        h_kv = address.kv_head(h, H_q, H_kv)
        vis = attention.visible_for(p, int(cache.kv_len[b]), i, attention.index_list_of(p, b, h_kv), b)
        K, V = ocache.read_rows(cache, b, h_kv, vis)
        s = (K @ q[attention.query_offset(p, b) + i, h]) * scale
        _, fell = split_state.shared_shift_attention(s, V, np.ones(len(s), bool), [(0, len(s))], phi, lo, hi)
        out.append(fell)
    return np.array(out)


def small():
    return W.paged_ragged_gqa("cuda", B=5, lo=1, hi=700, pool_pages=400)


def test_guard_holds_exact_and_no_fallback():
    w = small()
    shift = (0.0, -20.0, 20.0)
    O, L, flags, fb = run_shift(w, shift, num_sms=7, chunk_tokens=128)
    assert flags == 0
    H.compare(O, L, w)
    rows = H.sample_rows(H.oracle_problem(w), 40, seed=3)
    assert not oracle_guard(w, rows, shift).any()
    assert fb == 0


@pytest.mark.parametrize("shift", [(60.0, -20.0, 20.0), (-45.0, -20.0, 20.0), (0.0, -80.0, -10.0)])
def test_guard_fails_everywhere_still_exact(shift):
    w = small()
    O, L, flags, fb = run_shift(w, shift, num_sms=7, chunk_tokens=128)
    assert flags == 0
    H.compare(O, L, w)
    rows = H.sample_rows(H.oracle_problem(w), 40, seed=4)
    assert oracle_guard(w, rows, shift).all()
    assert fb > 0


def test_guard_fails_midway_still_exact():
    # a narrow guard: some 32-key tiles pass, later ones fail and move the accepted keys
    w = small()
    O, L, flags, fb = run_shift(w, (0.0, -0.5, 0.5), num_sms=7, chunk_tokens=128)
    assert flags == 0 and fb > 0
    H.compare(O, L, w)


@pytest.mark.parametrize("mask,S_q,extra", [("causal", 4, {}), ("sink_window", 1, dict(n_sink=4, window=300))])
def test_masks_and_query_rows(mask, S_q, extra):
    w = W.paged_bf16("shift-mask", B=3, S_q=S_q, H_q=8, H_kv=2, d=128, lens=[700, 5, 260], P=16, seed=21,
                     device="cuda", pool_pages=70, mask=mask, **extra)
    O, L, flags, fb = run_shift(w, (0.0, -30.0, 30.0), num_sms=5, chunk_tokens=64)
    assert flags == 0 and fb == 0
    H.compare(O, L, w)


def test_fused_merge_and_width_64():
    w = W.paged_bf16("shift-d64", B=3, S_q=1, H_q=16, H_kv=4, d=64, lens=[300, 77, 1], P=16, seed=22,
                     device="cuda", pool_pages=60)
    O, L, flags, fb = run_shift(w, (1.0, -30.0, 30.0), num_sms=4, chunk_tokens=64, fused_merge=True)
    assert flags == 0 and fb == 0
    H.compare(O, L, w)


def test_full_size_sampled_rows():
    w = W.paged_ragged_gqa("cuda")
    O, L, flags, fb = run_shift(w, (0.0, -30.0, 30.0))
    assert flags == 0 and fb == 0
    H.finite_or_masked(O, L)
    H.compare(O, L, w, H.sample_rows(w.problem, 64, seed=5, must=[(0, 0, 0), (15, 0, 31)]))


@pytest.mark.parametrize("shift", [(float("nan"), -1.0, 1.0), (0.0, 1.0, 1.0), (0.0, -90.0, 1.0), (0.0, -1.0, 50.0)])
def test_invalid_guard_rejected(shift):
    w = small()
    with pytest.raises(dattn.DattnError, match="EINVAL"):
        run_shift(w, shift)


def test_quantized_formats_rejected():
    w = small()
    w.problem = dict(w.problem, fmt="int8")
    with pytest.raises(dattn.DattnError, match="EUNSUPPORTED"):
        run_shift(w, (0.0, -20.0, 20.0))
