"""Shared helpers of the GPU parity tests: run the CUDA path through the C ABI,
build the oracle's view of the same inputs, compare within the tolerance.

Tolerance (bf16 output, fp32 LSE), fixed by the decode contract:
  |O - O_ref| <= 4e-3 + 1e-2 |O_ref|  elementwise;
  |LSE - LSE_ref| <= 1e-4 max(1, |LSE_ref|);
  rows without a visible key: O exactly 0 and LSE exactly -inf on both sides.
"""

from __future__ import annotations

import math

import numpy as np
import torch

import split_kv_decode_flash_gb300 as dattn
from oracle import attention
from oracle import cache as ocache

O_ATOL, O_RTOL, LSE_RTOL = 4e-3, 1e-2, 1e-4


def bits(t: torch.Tensor) -> np.ndarray:
    """bf16 tensor -> uint16 bit patterns on the host."""
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def oracle_cache(w) -> ocache.Cache:
    p = w.problem
    if p["layout"] == "packed":
        return ocache.Cache("packed", "bf16", p["H_kv"], p["d"], k=bits(w.k), v=bits(w.v),
                            kv_len=w.kv_len.numpy().astype(np.int64),
                            extra={"row_offsets": w.index_indptr.numpy().astype(np.int64),
                                   "position_map": w.index_list.numpy().astype(np.int64)})
    if p["layout"] == "contig":
        c = ocache.Cache("contig", "bf16", p["H_kv"], p["d"], T_c=p["T_cap"], k=bits(w.k), v=bits(w.v),
                         kv_len=w.kv_len.numpy().astype(np.int64))
        if w.cache_batch_idx is not None:
            c.cache_batch_idx = w.cache_batch_idx.numpy()
        return c
    return ocache.Cache("paged", "bf16", p["H_kv"], p["d"], P=p["P"], k=bits(w.k), v=bits(w.v),
                        page_indptr=w.page_indptr.numpy().astype(np.int64),
                        page_indices=w.page_indices.numpy().astype(np.int64),
                        kv_len=w.kv_len.numpy().astype(np.int64))


def oracle_problem(w) -> dict:
    p = dict(w.problem)
    if w.index_list is not None:
        p["index_indptr"] = w.index_indptr.numpy()
        p["index_list"] = w.index_list.numpy()
    if w.fm_intervals is not None:
        p["fm_intervals"] = w.fm_intervals.numpy()
        p["fm_indptr"] = np.concatenate([[0], np.cumsum(w.kv_len.numpy().astype(np.int64))])
    if w.qo_indptr is not None:
        p["qo_indptr"] = w.qo_indptr.numpy().astype(np.int64)
    return p


def query_rows(w, b):
    """(first packed query row, C_b) of request b."""
    if w.qo_indptr is None:
        return b * w.problem["S_q"], w.problem["S_q"]
    a, e = int(w.qo_indptr[b]), int(w.qo_indptr[b + 1])
    return a, e - a


def device_tensors(w, o, lse, dev="cuda"):
    kw = dict(q=w.q.to(dev), k=w.k.to(dev), v=w.v.to(dev), o=o, lse=lse)
    if w.page_indptr is not None:
        kw["page_indptr"] = w.page_indptr.to(dev)
        kw["page_indices"] = w.page_indices.to(dev)
    if w.cache_batch_idx is not None:
        kw["cache_batch_idx"] = w.cache_batch_idx.to(dev)
    if w.index_list is not None:
        kw["index_indptr"] = w.index_indptr.to(dev)
        kw["index_list"] = w.index_list.to(dev)
    if w.fm_intervals is not None:
        kw["fm_intervals"] = w.fm_intervals.to(dev).contiguous()
    return kw


def run_gpu(w, *, num_sms=None, ctas_per_sm=0, chunk_tokens=0, problem=None, keep=None, fused_merge=False,
            merge_tags=0):
    """One dattn_run over workload ``w``; returns (O fp32 cpu, LSE cpu, plan info, status flags)."""
    p = problem or w.problem
    B, S_q, H_q, d = p["B"], p["S_q"], p["H_q"], p["d"]
    plan = dattn.dattn_plan(p, w.kv_len, page_indptr=w.page_indptr, index_indptr=w.index_indptr,
                            index_list=w.index_list, num_sms=num_sms, ctas_per_sm=ctas_per_sm,
                            chunk_tokens=chunk_tokens, fused_merge=fused_merge, qo_indptr=w.qo_indptr,
                            merge_tags=merge_tags)
    n_rows = B * S_q if w.qo_indptr is None else int(w.qo_indptr[-1])
    o = torch.full((n_rows, H_q, d), float("nan"), dtype=torch.bfloat16, device="cuda")
    lse = torch.full((n_rows, H_q), float("nan"), dtype=torch.float32, device="cuda")
    ws = torch.empty(max(256, plan.workspace_bytes), dtype=torch.uint8, device="cuda")
    kw = device_tensors(w, o, lse)
    dattn.dattn_run(plan, p, dattn.tensors_from(**kw), ws)
    torch.cuda.synchronize()
    flags = dattn.dattn_device_status(ws)
    if keep is not None:
        keep.update(plan=plan, ws=ws, kw=kw)
    if w.qo_indptr is None:
        o, lse = o.view(B, S_q, H_q, d), lse.view(B, S_q, H_q)
    return o.float().cpu(), lse.cpu(), plan.info, flags


def all_rows(p):
    """Every (b, i, h_q) query row; i < C_b for a mixed batch."""
    qo = p.get("qo_indptr")
    return [(b, i, h) for b in range(p["B"])
            for i in range(p["S_q"] if qo is None else int(qo[b + 1] - qo[b])) for h in range(p["H_q"])]


def gpu_row(O, w, b, i, h):
    """Row (b, i, h_q) of a GPU result in [B, S_q, H_q, ...] or packed [sum C_b, H_q, ...] form."""
    if w.qo_indptr is None:
        return O[b, i, h]
    return O[int(w.qo_indptr[b]) + i, h]


def cache_arrays(w):
    """(spec, arrays) of a bf16 workload's cache for ``oracle_pool.decode_rows_parallel``."""
    p = w.problem
    spec = dict(kind="cache", layout=p["layout"], H_kv=p["H_kv"], d=p["d"], P=p.get("P", 0), T_cap=p.get("T_cap", 0))
    i64 = lambda t: None if t is None else t.numpy().astype(np.int64)
    arrays = dict(k=bits(w.k), v=bits(w.v), kv_len=i64(w.kv_len), page_indptr=i64(w.page_indptr),
                  page_indices=i64(w.page_indices), cache_batch_idx=i64(w.cache_batch_idx))
    if p["layout"] == "packed":
        arrays.update(row_offsets=i64(w.index_indptr), position_map=i64(w.index_list))
    return spec, arrays


def compare(O, LSE, w, rows=None, cache=None, ref=None):
    """Element-by-element comparison of the GPU rows against the oracle; returns max errors.

    ``ref`` = (O_ref, LSE_ref) of ``rows`` computed beforehand (e.g. in parallel)."""
    p = oracle_problem(w)
    rows = rows or all_rows(p)
    if ref is None:
        cache = cache or oracle_cache(w)
        Oref, Lref = attention.decode_rows(p, cache, bits(w.q), rows)
    else:
        Oref, Lref = ref
    og = np.stack([gpu_row(O, w, b, i, h).numpy() for b, i, h in rows]).astype(np.float64)
    lg = np.array([gpu_row(LSE, w, b, i, h).item() for b, i, h in rows], dtype=np.float64)
    masked = np.isneginf(Lref)
    assert np.array_equal(np.isneginf(lg), masked), "all-masked rows differ"
    assert not og[masked].any(), "masked rows must give exactly zero output"
    assert np.isfinite(og).all(), "non-finite output"
    err = np.abs(og - Oref)
    bound = O_ATOL + O_RTOL * np.abs(Oref)
    worst = np.unravel_index(np.argmax(err - bound), err.shape)
    assert (err <= bound).all(), f"O error {err[worst]:.3g} > {bound[worst]:.3g} at row {rows[worst[0]]}"
    fin = ~masked
    lerr = np.abs(lg[fin] - Lref[fin])
    assert (lerr <= LSE_RTOL * np.maximum(1.0, np.abs(Lref[fin]))).all(), f"LSE error {lerr.max():.3g}"
    return {"max_abs_O": float(err.max()), "max_abs_LSE": float(lerr.max()) if lerr.size else 0.0,
            "rows": len(rows)}


def compare_all_rows(O, LSE, w):
    """Every query row of a bf16 workload against the oracle, the oracle run over worker
    processes (full-size workloads)."""
    from tests import oracle_pool
    p = oracle_problem(w)
    rows = all_rows(p)
    spec, arrays = cache_arrays(w)
    ref = oracle_pool.decode_rows_parallel(p, spec, arrays, bits(w.q), rows)
    return compare(O, LSE, w, rows, ref=ref)


def sample_rows(p, n, seed=0, must=()):
    rng = np.random.default_rng(seed)
    rows = set(must)
    allr = all_rows(p)
    for k in rng.choice(len(allr), size=min(n, len(allr)), replace=False):
        rows.add(allr[k])
    return sorted(rows)


def finite_or_masked(O, LSE):
    o = O.numpy()
    assert np.isfinite(o).all()
    assert not np.isnan(LSE.numpy()).any()
    return True


def inf():
    return math.inf
