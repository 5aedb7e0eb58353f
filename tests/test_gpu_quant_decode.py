"""GPU parity of decode over INT8, per-head INT4, FP8 and KIVI-INT4 caches (M8.6 §0x03, §0x05B,
§0x06B-C, §0x09C, §0x0A).

The GPU cache is written by kv_append; the oracle writes its own cache from
the same bf16 history with its own quantiser and dequantises it in float64.
(The two sets of codes are bit-identical by test_gpu_append, but nothing here
relies on it: the comparison is between two independent pipelines.)
"""

import numpy as np
import pytest
import torch

import split_kv_decode_flash_gb300 as dattn
import workloads as W
from oracle import attention
from oracle import cache as ocache
from tests import gpu_helpers as H
from tests.test_gpu_append import append_history, fp8_scales

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    dattn.load()


def _oracle_cache(w, fmt, requests=None):
    """Oracle cache for ``requests`` (all when None); other requests stay empty."""
    p = w.problem
    ks, vs = fp8_scales(w)
    c = ocache.empty_paged(fmt, p["num_pages"], p["H_kv"], p["P"], p["d"], p["B"], G=p["kivi_group"],
                           Gv=p["kivi_v_group"], R=p["kivi_residual"], k_scale=ks, v_scale=vs)
    ri = w.rows_indptr.numpy().astype(np.int64)
    lens = w.kv_len.numpy().astype(np.int64)
    if requests is None:
        return ocache.write_history(c, w.page_indptr.numpy(), w.page_indices.numpy(), ri,
                                    H.bits(w.k_rows), H.bits(w.v_rows))
    keep = np.zeros(p["B"], bool)
    keep[list(requests)] = True
    sub_len = np.where(keep, lens, 0)
    sub_ptr = np.concatenate([[0], np.cumsum(sub_len)])
    rows = np.concatenate([np.arange(ri[b], ri[b + 1]) for b in range(p["B"]) if keep[b]])
    k = H.bits(w.k_rows[torch.as_tensor(rows, device=w.k_rows.device)])
    v = H.bits(w.v_rows[torch.as_tensor(rows, device=w.v_rows.device)])
    ocache.write_history(c, w.page_indptr.numpy(), w.page_indices.numpy(), sub_ptr, k, v)
    c.kv_len = lens
    return c


def _run(w, fmt, p, cache, **plan_kw):
    B, S_q, H_q, d = p["B"], p["S_q"], p["H_q"], p["d"]
    plan = dattn.dattn_plan(p, w.kv_len, page_indptr=w.page_indptr, **plan_kw)
    o = torch.full((B, S_q, H_q, d), float("nan"), dtype=torch.bfloat16, device="cuda")
    lse = torch.full((B, S_q, H_q), float("nan"), dtype=torch.float32, device="cuda")
    ws = torch.empty(plan.workspace_bytes, dtype=torch.uint8, device="cuda")
    t = dattn.tensors_from(q=w.q.cuda(), o=o, lse=lse, **cache)
    dattn.dattn_run(plan, p, t, ws)
    torch.cuda.synchronize()
    assert dattn.dattn_device_status(ws) == 0
    return o.float().cpu(), lse.cpu(), plan.info


def _compare(O, L, w, p, cache_ref, rows):
    w2 = W.Workload(w.name, p, w.q, w.kv_len)
    return H.compare(O, L, w2, rows, cache=cache_ref)


@pytest.mark.parametrize("fmt", ["int8", "int4_head", "int4_kivi", "fp8_e4m3", "fp8_e5m2"])
@pytest.mark.parametrize("chunk,num_sms", [(0, 152), (64, 5)])
def test_quantized_decode_small_all_rows(fmt, chunk, num_sms):
    lens = [700, 129, 128, 161, 40, 1]
    w = W.quantized_history("q", B=len(lens), S_q=1, H_q=32, H_kv=8, d=128, lens=lens, P=16, seed=21,
                            device="cuda", fmt=fmt, pool_pages=sum(-(-t // 16) for t in lens) + 2)
    p, cache = append_history(w, fmt, [[] for _ in lens])
    O, L, info, = _run(w, fmt, p, cache, chunk_tokens=chunk, num_sms=num_sms)[:3]
    ref = _oracle_cache(w, fmt)
    _compare(O, L, w, p, ref, H.all_rows(p))


@pytest.mark.parametrize("fmt", ["int8", "int4_head", "int4_kivi", "fp8_e4m3", "fp8_e5m2"])
def test_quantized_decode_d64_multi_row_sink_window(fmt):
    lens = [500, 90]
    w = W.quantized_history("q64", B=2, S_q=2, H_q=8, H_kv=2, d=64, lens=lens, P=16, seed=22, device="cuda",
                            fmt=fmt, pool_pages=40)
    p = dict(w.problem, mask="sink_window", n_sink=3, window=200, kivi_v_group=16)
    w.problem = p
    p, cache = append_history(w, fmt, [[100, 300], [60]])
    O, L, info = _run(w, fmt, p, cache, chunk_tokens=64, num_sms=3)
    _compare(O, L, w, p, _oracle_cache(w, fmt), H.all_rows(p))


def test_int4_kivi_verify_rows_cross_the_residual_boundary():
    lens = [300, 4]
    w = W.quantized_history("q4", B=2, S_q=4, H_q=16, H_kv=2, d=128, lens=lens, P=16, seed=23, device="cuda",
                            fmt="int4_kivi", pool_pages=25)
    p, cache = append_history(w, "int4_kivi", [[150], [2]])
    O, L, info = _run(w, "int4_kivi", p, cache, chunk_tokens=64, num_sms=2)
    _compare(O, L, w, p, _oracle_cache(w, "int4_kivi"), H.all_rows(p))


@pytest.mark.parametrize("fmt", ["int8", "int4_head", "int4_kivi", "fp8_e4m3", "fp8_e5m2"])
def test_quantized_full_size_all_rows(fmt):
    """B=32, T ~ U[2048, 32768], K outlier channels: the full quantized workload, every
    query row against the oracle's own cache (written by the oracle's quantiser in worker
    processes, see ``tests.oracle_pool``)."""
    from tests import oracle_pool
    w = W.quantized("cuda", fmt=fmt)
    p, cache = append_history(w, fmt, [[] for _ in range(w.problem["B"])])
    if fmt == "int4_kivi":      # the 128 most recent tokens of every request stay bf16
        assert p["kivi_residual"] == 160
    O, L, info = _run(w, fmt, p, cache)
    rows = H.all_rows(p)
    ks, vs = fp8_scales(w)
    spec = dict(kind="history", fmt=fmt, H_kv=p["H_kv"], d=p["d"], P=p["P"], G=p["kivi_group"],
                Gv=p["kivi_v_group"], R=p["kivi_residual"], k_scale=ks, v_scale=vs)
    i64 = lambda t: t.numpy().astype(np.int64)
    arrays = dict(k_rows=H.bits(w.k_rows), v_rows=H.bits(w.v_rows), rows_indptr=i64(w.rows_indptr),
                  page_indptr=i64(w.page_indptr), page_indices=i64(w.page_indices), kv_len=i64(w.kv_len))
    ref = oracle_pool.decode_rows_parallel(dict(p), spec, arrays, H.bits(w.q), rows)
    w2 = W.Workload(w.name, p, w.q, w.kv_len)
    assert H.compare(O, L, w2, rows, ref=ref)["rows"] == 32 * 32


@pytest.mark.parametrize("S_q,H_q,H_kv,mask,chunk,num_sms,R", [
    (1, 64, 8, "causal", 0, 152, 160),         # 8 rows per kv head
    (2, 8, 2, "sink_window", 0, 152, 160),     # 8 rows, two-run stages, causal verify rows
    (2, 8, 2, "sink_window", 50, 4, 160),      # chunks that start inside K groups
    (1, 16, 8, "sink_window", 64, 3, 160),     # 2 rows
    (1, 64, 8, "causal", 64, 7, 64),           # a power-of-two residual ring
    (2, 8, 2, "sink_window", 0, 152, 96),      # a residual ring of three groups
    (4, 32, 8, "causal", 0, 152, 160),         # 16 rows: two row blocks share a stage's keys
    (3, 32, 8, "sink_window", 50, 4, 96),      # 12 rows: a ragged second row block
    (4, 64, 8, "sink_window", 0, 152, 160),    # 32 rows: four row blocks, a warp per stage
    (5, 32, 8, "causal", 64, 7, 160),          # 20 rows: four blocks, the last nearly empty
])
def test_int4_kivi_tensor_core_rows_and_windows(S_q, H_q, H_kv, mask, chunk, num_sms, R):
    """d = 128, Gv = 32, 1 to 32 rows (one to four row blocks of 8): K groups
    that straddle 16-key blocks (window starts off the group grid), stages of
    two runs touching up to ten groups, residual-only and just-closed-group
    requests, residual rings of several lengths R."""
    lens = [2000, 1999, 1777, 300, 129, 7]
    w = W.quantized_history("q4t", B=len(lens), S_q=S_q, H_q=H_q, H_kv=H_kv, d=128, lens=lens, P=16, seed=26,
                            device="cuda", fmt="int4_kivi", pool_pages=sum(-(-t // 16) for t in lens) + 3)
    w.problem = dict(w.problem, mask=mask, n_sink=34, window=1000, kivi_residual=R)
    p, cache = append_history(w, "int4_kivi", [[900, 1500], [], [1000], [160], [], []])
    O, L, info = _run(w, "int4_kivi", p, cache, chunk_tokens=chunk, num_sms=num_sms)
    assert info["rows"] == S_q * H_q // H_kv
    _compare(O, L, w, p, _oracle_cache(w, "int4_kivi"), H.all_rows(p))


@pytest.mark.parametrize("d,Gv,P,S_q,H_q,H_kv,mask", [
    (128, 16, 16, 1, 32, 8, "causal"),         # Gv = 16: two channel groups per 32-channel chunk
    (128, 16, 16, 3, 32, 8, "sink_window"),    # Gv = 16, 12 rows
    (64, 16, 16, 1, 32, 8, "sink_window"),     # d = 64 (Gv <= d / 4), 4 rows
    (64, 16, 16, 4, 32, 8, "causal"),          # d = 64, 16 rows
    (64, 16, 32, 4, 64, 8, "sink_window"),     # d = 64, 32 rows, a page per K group
    (128, 32, 64, 1, 32, 8, "sink_window"),    # two K groups per page
    (128, 32, 8, 2, 32, 8, "causal"),          # four pages per K group
    (128, 32, 96, 1, 32, 8, "sink_window"),    # P = 96, not a power of two: byte-format kernel
    (64, 16, 96, 4, 16, 2, "causal"),          # the same at d = 64 with 32 rows
])
def test_int4_kivi_head_dims_groups_and_pages(d, Gv, P, S_q, H_q, H_kv, mask):
    """KIVI shapes beyond d = 128 / Gv = 32 / P = 16: head dimension 64, V channel
    groups of 16, K groups that span several pages or share one, and page sizes
    that are not a power of two; every query row against the oracle."""
    lens = [1500, 777, 160, 33, 2]
    w = W.quantized_history("q4s", B=len(lens), S_q=S_q, H_q=H_q, H_kv=H_kv, d=d, lens=lens, P=P, seed=27,
                            device="cuda", fmt="int4_kivi", pool_pages=sum(-(-t // P) for t in lens) + 3)
    w.problem = dict(w.problem, mask=mask, n_sink=34, window=600, kivi_v_group=Gv)
    p, cache = append_history(w, "int4_kivi", [[700], [400, 500], [], [32], []])
    O, L, info = _run(w, "int4_kivi", p, cache, chunk_tokens=0, num_sms=152)
    assert info["rows"] == S_q * H_q // H_kv
    _compare(O, L, w, p, _oracle_cache(w, "int4_kivi"), H.all_rows(p))


@pytest.mark.parametrize("fmt,qmul,kmul", [
    ("int4_kivi", 600.0, 40.0),    # 16 q s_g beyond 2^15 (and |q| > 2^10): the rescaled Q' split
    ("int4_head", 20000.0, 1.0),   # |q| beyond 2^14: the query divided by a power of two
    ("int8", 20000.0, 1.0),        # the same on the INT8 kernels (f16 queries)
])
@pytest.mark.parametrize("S_q,H_q,H_kv", [(1, 32, 8), (4, 16, 2)])
def test_quantized_large_magnitudes_take_the_scaled_paths(fmt, qmul, kmul, S_q, H_q, H_kv):
    """Queries and keys far outside the unit range, with sm_scale small enough to keep the
    scores moderate: the kernels' power-of-two rescaling of f16 query operands (and KIVI's
    f32 redo of the Q' split) must give the oracle's rows."""
    lens = [700, 233, 90]
    w = W.quantized_history("big", B=len(lens), S_q=S_q, H_q=H_q, H_kv=H_kv, d=128, lens=lens, P=16, seed=29,
                            device="cuda", fmt=fmt, pool_pages=sum(-(-t // 16) for t in lens) + 2)
    w.q = (w.q.float() * qmul).to(torch.bfloat16)
    w.k_rows = (w.k_rows.float() * kmul).to(torch.bfloat16)
    w.problem = dict(w.problem, sm_scale=2e-5)
    p, cache = append_history(w, fmt, [[300], [], []])
    O, L, info = _run(w, fmt, p, cache, chunk_tokens=128, num_sms=5)
    assert torch.isfinite(L).all()
    _compare(O, L, w, p, _oracle_cache(w, fmt), H.all_rows(p))


@pytest.mark.parametrize("P", [4, 64])
def test_int8_decode_page_sizes(P):
    lens = [300, 70, 5]
    w = W.quantized_history("q8", B=3, S_q=1, H_q=16, H_kv=4, d=128, lens=lens, P=P, seed=24, device="cuda",
                            fmt="int8", pool_pages=sum(-(-t // P) for t in lens) + 2)
    p, cache = append_history(w, "int8", [[64, 200], [], []])
    O, L, info = _run(w, "int8", p, cache, chunk_tokens=128, num_sms=3)
    _compare(O, L, w, p, _oracle_cache(w, "int8"), H.all_rows(p))


@pytest.mark.parametrize("fmt", ["int8", "int4_head", "fp8_e4m3", "fp8_e5m2"])
@pytest.mark.parametrize("S_q,H_q,H_kv,d", [(3, 16, 4, 128), (4, 16, 2, 128), (4, 16, 2, 64)])
def test_byte_codes_decode_more_than_eight_rows(fmt, S_q, H_q, H_kv, d):
    """12 and 32 query rows per kv head (row tiles of 16 on the mma M side), causal verify rows."""
    lens = [420, 37, 3]
    w = W.quantized_history("q8r", B=3, S_q=S_q, H_q=H_q, H_kv=H_kv, d=d, lens=lens, P=16, seed=25,
                            device="cuda", fmt=fmt, pool_pages=sum(-(-t // 16) for t in lens) + 3)
    p, cache = append_history(w, fmt, [[200], [], []])
    O, L, info = _run(w, fmt, p, cache, chunk_tokens=128, num_sms=3)
    assert info["rows"] == S_q * H_q // H_kv
    _compare(O, L, w, p, _oracle_cache(w, fmt), H.all_rows(p))


@pytest.mark.parametrize("fmt", ["fp8_e4m3", "fp8_e5m2"])
def test_fp8_decode_without_scales_and_with_saturation(fmt):
    """FP8 with no scales (1) and with scales that saturate part of the range."""
    lens = [300, 65, 8]
    for mode in ("none", "tight"):
        w = W.quantized_history("f8s", B=3, S_q=1, H_q=16, H_kv=4, d=128, lens=lens, P=16, seed=26,
                                device="cuda", fmt=fmt, pool_pages=sum(-(-t // 16) for t in lens) + 2)
        if mode == "none":
            del w.meta["k_scale"], w.meta["v_scale"]
        else:
            w.meta["k_scale"] = w.meta["k_scale"] / 8
            w.meta["v_scale"] = w.meta["v_scale"] / 8
        p, cache = append_history(w, fmt, [[] for _ in lens])
        O, L, info = _run(w, fmt, p, cache, chunk_tokens=64, num_sms=4)
        _compare(O, L, w, p, _oracle_cache(w, fmt), H.all_rows(p))


@pytest.mark.parametrize("S_q,H_q,H_kv,d,mask", [
    (1, 32, 8, 128, "index_list"),   # 4 rows: one row block
    (2, 32, 8, 64, "causal"),        # 8 rows
    (5, 12, 4, 128, "sink_window"),  # 15 rows: two row blocks, the last one short
    (3, 64, 8, 128, "causal"),       # 24 rows: four row blocks
])
def test_int4_head_rows_masks_and_widths(S_q, H_q, H_kv, d, mask):
    """Per-head INT4: 8-row blocks on the mma N side (1, 2 and 4 blocks), every visibility
    program, partial stages and requests shorter than their query rows."""
    lens = [1300, 257, 256, 17, 2]
    w = W.quantized_history("q4h", B=len(lens), S_q=S_q, H_q=H_q, H_kv=H_kv, d=d, lens=lens, P=16, seed=27,
                            device="cuda", fmt="int4_head", pool_pages=sum(-(-t // 16) for t in lens) + 3)
    if mask == "sink_window":
        w.problem = dict(w.problem, mask=mask, n_sink=5, window=300)
    elif mask == "index_list":
        gen = torch.Generator().manual_seed(3)
        lists = [sorted(torch.randperm(T, generator=gen)[:max(1, T // 3)].tolist()) for T in lens for _ in range(H_kv)]
        w.index_indptr = torch.tensor(np.concatenate([[0], np.cumsum([len(x) for x in lists])]), dtype=torch.int32)
        w.index_list = torch.tensor(np.concatenate(lists), dtype=torch.int32)
        w.problem = dict(w.problem, mask=mask)
    p, cache = append_history(w, "int4_head", [[600], [], [100], [], []])
    plan_kw = dict(chunk_tokens=128, num_sms=5)
    if mask == "index_list":
        cache.update(index_indptr=w.index_indptr.cuda(), index_list=w.index_list.cuda())
        plan_kw.update(index_indptr=w.index_indptr, index_list=w.index_list)
    O, L, info = _run(w, "int4_head", p, cache, **plan_kw)
    assert info["rows"] == S_q * H_q // H_kv
    w2 = W.Workload(w.name, p, w.q, w.kv_len, index_indptr=w.index_indptr, index_list=w.index_list)
    H.compare(O, L, w2, H.all_rows(p), cache=_oracle_cache(w, "int4_head"))


@pytest.mark.parametrize("fmt", ["int8", "int4_head"])
def test_quantized_bounds_check_flags_out_of_pool_page(fmt):
    """A page id past the pool in the run's page list is caught before any address is formed;
    the other request still matches the oracle."""
    lens = [300, 200]
    w = W.quantized_history("oob", B=2, S_q=1, H_q=8, H_kv=2, d=128, lens=lens, P=16, seed=28, device="cuda",
                            fmt=fmt, pool_pages=sum(-(-t // 16) for t in lens) + 1)
    p, cache = append_history(w, fmt, [[] for _ in lens])
    bad = cache["page_indices"].clone()
    bad[3] = p["num_pages"]                 # request 0, logical block 3
    cache["page_indices"] = bad
    plan = dattn.dattn_plan(p, w.kv_len, page_indptr=w.page_indptr, num_sms=4)
    o = torch.zeros((2, 1, 8, 128), dtype=torch.bfloat16, device="cuda")
    lse = torch.zeros((2, 1, 8), dtype=torch.float32, device="cuda")
    ws = torch.empty(plan.workspace_bytes, dtype=torch.uint8, device="cuda")
    dattn.dattn_run(plan, p, dattn.tensors_from(q=w.q.cuda(), o=o, lse=lse, **cache), ws)
    torch.cuda.synchronize()
    assert dattn.dattn_device_status(ws) & 1            # kStPageRange
    _compare(o.float().cpu(), lse.cpu(), w, p, _oracle_cache(w, fmt), [(1, 0, h) for h in range(8)])


# ---- mixed batches and FlashMask columns on the quantized formats (M4.5 §0x08F, §0x06A-§0x06D) ----

def _packed_run(w, fmt, p, cache, qo_indptr=None, **plan_kw):
    """dattn_run with the query, O and LSE packed by qo_indptr (uniform when None)."""
    H_q, d = p["H_q"], p["d"]
    n_rows = p["B"] * p["S_q"] if qo_indptr is None else int(qo_indptr[-1])
    plan = dattn.dattn_plan(p, w.kv_len, page_indptr=w.page_indptr, qo_indptr=qo_indptr, **plan_kw)
    o = torch.full((n_rows, H_q, d), float("nan"), dtype=torch.bfloat16, device="cuda")
    lse = torch.full((n_rows, H_q), float("nan"), dtype=torch.float32, device="cuda")
    ws = torch.empty(max(256, plan.workspace_bytes), dtype=torch.uint8, device="cuda")
    dattn.dattn_run(plan, p, dattn.tensors_from(q=w.q.cuda().reshape(n_rows, H_q, d), o=o, lse=lse, **cache), ws)
    torch.cuda.synchronize()
    assert dattn.dattn_device_status(ws) == 0
    if qo_indptr is None:
        return o.float().cpu().reshape(p["B"], p["S_q"], H_q, d), lse.cpu().reshape(p["B"], p["S_q"], H_q)
    return o.float().cpu(), lse.cpu()


@pytest.mark.parametrize("fmt", ["int8", "fp8_e4m3", "fp8_e5m2", "int4_head", "int4_kivi"])
@pytest.mark.parametrize("H_q,H_kv,chunk,num_sms", [(32, 8, 64, 7), (32, 8, 0, 152), (8, 8, 64, 5)])
def test_byte_codes_mixed_batch_all_rows(fmt, H_q, H_kv, chunk, num_sms):
    """Prefill, append, decode and idle requests in one launch over INT8 / FP8 / INT4 codes:
    32 rows per kv head for the widest request (two 16-row tiles, or four row blocks of 8 on
    the INT4 kernels) and 8 (keys on the mma M side)."""
    TC = [(0, 8), (130, 1), (0, 1), (65, 3), (7, 0), (300, 8), (1, 2), (64, 5), (200, 1)]
    lens = [t + c for t, c in TC]
    w = W.quantized_history("mixq", B=len(TC), S_q=8, H_q=H_q, H_kv=H_kv, d=128, lens=lens, P=16, seed=51,
                            device="cuda", fmt=fmt, pool_pages=sum(-(-t // 16) for t in lens) + 2)
    qo = np.concatenate([[0], np.cumsum([c for _, c in TC])]).astype(np.int32)
    gen = torch.Generator(device="cuda").manual_seed(52)
    w.q = torch.randn((int(qo[-1]), H_q, 128), generator=gen, device="cuda").to(torch.bfloat16)
    p, cache = append_history(w, fmt, [[] for _ in TC])
    O, L = _packed_run(w, fmt, p, cache, qo_indptr=qo, chunk_tokens=chunk, num_sms=num_sms)
    w2 = W.Workload(w.name, p, w.q, w.kv_len, qo_indptr=torch.tensor(qo))
    assert H.compare(O, L, w2, cache=_oracle_cache(w, fmt))["rows"] == int(qo[-1]) * H_q


@pytest.mark.parametrize("fmt", ["int8", "fp8_e4m3", "fp8_e5m2", "int4_head", "int4_kivi"])
@pytest.mark.parametrize("S_q,H_q,H_kv", [(4, 16, 2), (3, 16, 4), (8, 8, 8), (2, 8, 2)])
def test_byte_codes_flashmask_random_intervals(fmt, S_q, H_q, H_kv):
    """FlashMask two-interval columns over INT8 / FP8 / INT4 codes: columns hidden from every
    row, columns every row sees, and a request whose only key is hidden; 32, 12 and 8 rows."""
    from tests.test_gpu_decode import _random_fm_intervals
    lens = [300, 65, 1, 0, 130]
    w = W.quantized_history("fmq", B=len(lens), S_q=S_q, H_q=H_q, H_kv=H_kv, d=128, lens=lens, P=16, seed=53,
                            device="cuda", fmt=fmt, pool_pages=sum(-(-t // 16) for t in lens) + 2)
    rng = np.random.default_rng(54 + S_q)
    iv = _random_fm_intervals(rng, lens, S_q)
    iv[sum(lens[:2])] = [0, S_q, 0, 0]                     # request 2: its only key hidden from all rows
    w.problem = dict(w.problem, mask="flashmask")
    fm = torch.tensor(iv, dtype=torch.int32)
    p, cache = append_history(w, fmt, [[] for _ in lens])
    cache["fm_intervals"] = fm.cuda().contiguous()
    O, L = _packed_run(w, fmt, p, cache, chunk_tokens=64, num_sms=7)
    assert torch.isinf(L[2]).all() and (L[2] < 0).all()
    w2 = W.Workload(w.name, p, w.q, w.kv_len, fm_intervals=fm)
    H.compare(O, L, w2, cache=_oracle_cache(w, fmt))


@pytest.mark.parametrize("fmt", ["int8", "fp8_e4m3", "int4_head", "int4_kivi"])
def test_byte_codes_tree_verify_full_size_all_rows(fmt):
    """The speculative-tree verify workload (B=16, prefixes U[1024, 8192], 8 DFS-ordered draft
    rows, FlashMask intervals) over INT8 / FP8 / INT4 codes, every row."""
    from tests import oracle_pool
    t = W.tree_verify("cpu")
    w = W.quantized_history("treeq", B=16, S_q=8, H_q=32, H_kv=8, d=128, lens=t.kv_len.tolist(), P=16, seed=55,
                            device="cuda", fmt=fmt)
    w.problem = dict(w.problem, mask="flashmask")
    p, cache = append_history(w, fmt, [[] for _ in range(16)])
    cache["fm_intervals"] = t.fm_intervals.cuda().contiguous()
    O, L = _packed_run(w, fmt, p, cache)
    w2 = W.Workload(w.name, p, w.q, w.kv_len, fm_intervals=t.fm_intervals)
    prob = H.oracle_problem(w2)
    rows = H.all_rows(prob)
    ks, vs = fp8_scales(w)
    spec = dict(kind="history", fmt=fmt, H_kv=p["H_kv"], d=p["d"], P=p["P"], G=p["kivi_group"],
                Gv=p["kivi_v_group"], R=p["kivi_residual"], k_scale=ks, v_scale=vs)
    i64 = lambda x: x.numpy().astype(np.int64)
    arrays = dict(k_rows=H.bits(w.k_rows), v_rows=H.bits(w.v_rows), rows_indptr=i64(w.rows_indptr),
                  page_indptr=i64(w.page_indptr), page_indices=i64(w.page_indices), kv_len=i64(w.kv_len))
    ref = oracle_pool.decode_rows_parallel(prob, spec, arrays, H.bits(w.q), rows)
    assert H.compare(O, L, w2, rows, ref=ref)["rows"] == 16 * 8 * 32
