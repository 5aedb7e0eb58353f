"""GPU parity of the decode path (bf16 K/V) against the fp64 oracle, through the C ABI.

Every output row is compared, element by element: small cases that span
several tiles and ragged tails, and the full-size workloads in the launch
configuration the benchmark times (the oracle then runs over worker
processes, see ``tests.oracle_pool``).
"""

import numpy as np
import pytest
import torch

import split_kv_decode_flash_gb300 as dattn
import workloads as W
from oracle import address, masks
from oracle import cache as ocache
from tests import gpu_helpers as H

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    dattn.load()


def test_tiny_contiguous_four_fixed_splits():
    w = W.tiny_contiguous("cuda")
    O, L, info, flags = H.run_gpu(w)
    assert flags == 0
    assert info["n_items"] == 2 * 4 and info["n_merge_groups"] == 2 and info["max_splits"] == 4
    H.compare(O, L, w)


@pytest.mark.parametrize("chunk,num_sms", [(0, 152), (64, 7), (128, 3), (192, 152), (100000, 152)])
def test_paged_ragged_small_all_rows(chunk, num_sms):
    w = W.paged_ragged_gqa("cuda", B=5, lo=1, hi=700, pool_pages=400)
    O, L, info, flags = H.run_gpu(w, chunk_tokens=chunk, num_sms=num_sms)
    assert flags == 0
    H.compare(O, L, w)


def test_paged_ragged_full_size_all_rows():
    w = W.paged_ragged_gqa("cuda")
    O, L, info, flags = H.run_gpu(w)
    assert flags == 0 and info["n_merge_groups"] > 0
    assert H.compare_all_rows(O, L, w)["rows"] == 16 * 32


@pytest.mark.parametrize("lens,P,fixed", [([0, 1, 2, 17], 16, 0), ([0, 3, 5], 16, 8), ([33, 1, 64], 1, 0),
                                          ([200, 129, 64], 64, 3), ([1000], 16, 64), ([70, 3, 64], 2, 0),
                                          ([130, 33], 4, 0), ([500, 65, 31], 32, 0)])
def test_edge_lengths_pages_and_splits(lens, P, fixed):
    pool = sum(-(-t // P) for t in lens) + 3
    w = W.paged_bf16("edge", B=len(lens), S_q=1, H_q=8, H_kv=2, d=128, lens=lens, P=P, seed=9, device="cuda",
                     pool_pages=pool, fixed_splits=fixed)
    O, L, info, flags = H.run_gpu(w, num_sms=5, chunk_tokens=64)
    assert flags == 0
    H.compare(O, L, w)


def test_head_width_64_paged():
    w = W.paged_bf16("d64", B=3, S_q=1, H_q=16, H_kv=4, d=64, lens=[300, 77, 1], P=16, seed=5, device="cuda",
                     pool_pages=60)
    O, L, info, flags = H.run_gpu(w, num_sms=4, chunk_tokens=128)
    assert flags == 0
    H.compare(O, L, w)


def test_contiguous_cache_row_remap_and_capacity_tail():
    w = W.contiguous_bf16("remap", B=3, S_q=1, H_q=8, H_kv=2, d=64, lens=[100, 7, 64], T_cap=128, seed=6,
                          device="cuda", B_cache=5, cache_batch_idx=[4, 0, 2])
    O, L, info, flags = H.run_gpu(w, num_sms=3, chunk_tokens=64)
    assert flags == 0
    H.compare(O, L, w)


@pytest.mark.parametrize("S_q,lens", [(4, [1, 2, 3, 4, 70]), (2, [1, 65]), (3, [130, 5])])
def test_causal_verify_rows_small(S_q, lens):
    w = W.paged_bf16("verify", B=len(lens), S_q=S_q, H_q=16, H_kv=2, d=128, lens=lens, P=16, seed=7,
                     device="cuda", pool_pages=sum(-(-t // 16) for t in lens) + 2)
    O, L, info, flags = H.run_gpu(w, num_sms=4, chunk_tokens=64)
    assert flags == 0
    H.compare(O, L, w)


@pytest.mark.parametrize("S_q", [1, 4])
def test_long_context_full_size_all_rows(S_q):
    w = W.long_context("cuda", S_q=S_q)
    O, L, info, flags = H.run_gpu(w)
    assert flags == 0
    assert H.compare_all_rows(O, L, w)["rows"] == 4 * S_q * 64
    if S_q == 4:      # request of length 1: rows 0..2 see nothing
        assert np.isneginf(L[3, :3].numpy()).all() and not O[3, :3].any()


@pytest.mark.parametrize("n_sink,window,lens", [(4, 64, [5, 60, 64, 65, 300]), (0, 16, [40, 1]),
                                                (3, 100, [1000, 99])])
def test_sink_window_small(n_sink, window, lens):
    w = W.paged_bf16("sw", B=len(lens), S_q=1, H_q=8, H_kv=2, d=128, lens=lens, P=16, seed=8, device="cuda",
                     pool_pages=sum(-(-t // 16) for t in lens) + 2, mask="sink_window", n_sink=n_sink,
                     window=window)
    O, L, info, flags = H.run_gpu(w, num_sms=3, chunk_tokens=64)
    assert flags == 0
    H.compare(O, L, w)


def test_sink_window_multi_row():
    w = W.paged_bf16("sw4", B=2, S_q=4, H_q=8, H_kv=2, d=128, lens=[90, 6], P=16, seed=10, device="cuda",
                     pool_pages=12, mask="sink_window", n_sink=2, window=9)
    O, L, info, flags = H.run_gpu(w, num_sms=2, chunk_tokens=64)
    assert flags == 0
    H.compare(O, L, w)


def test_retention_sink_window_full_size_all_rows():
    w = W.retention("cuda", "sink_window")
    O, L, info, flags = H.run_gpu(w)
    assert flags == 0 and info["stream_keys"] == 8 * 8 * 4100
    assert H.compare_all_rows(O, L, w)["rows"] == 8 * 32


def test_index_lists_small():
    w = W.retention("cuda", "index_list", B=3, T=3000)
    O, L, info, flags = H.run_gpu(w, num_sms=5, chunk_tokens=128)
    assert flags == 0
    H.compare(O, L, w)


def test_index_list_bounds_that_disagree_with_the_plan_drop_the_group():
    """A device index_indptr that disagrees with the planned one for group (0, 1): its keys
    are dropped (every slot masked), the status word gets the list bit (4), its rows come out
    all-masked (O = 0, LSE = -inf) and every other row still matches the oracle."""
    w = W.retention("cuda", "index_list", B=3, T=3000)
    p = w.problem
    plan = dattn.dattn_plan(p, w.kv_len, page_indptr=w.page_indptr, index_indptr=w.index_indptr,
                            index_list=w.index_list, num_sms=5, chunk_tokens=128)
    o = torch.full((3, 1, 32, 128), float("nan"), dtype=torch.bfloat16, device="cuda")
    lse = torch.full((3, 1, 32), float("nan"), dtype=torch.float32, device="cuda")
    kw = H.device_tensors(w, o, lse)
    bad = kw["index_indptr"].clone()
    bad[1] += 1                                  # group 1 = (request 0, kv head 1) starts one entry late
    kw["index_indptr"] = bad
    ws = torch.empty(plan.workspace_bytes, dtype=torch.uint8, device="cuda")
    dattn.dattn_run(plan, p, dattn.tensors_from(**kw), ws)
    torch.cuda.synchronize()
    assert dattn.dattn_device_status(ws) & 4
    O, L = o.float().cpu(), lse.cpu()
    assert torch.isinf(L[0, 0, 4:8]).all() and (L[0, 0, 4:8] < 0).all() and not O[0, 0, 4:8].any()
    rows = [(b, 0, h) for b in range(3) for h in range(32) if not (b == 0 and 4 <= h < 8)]
    H.compare(O, L, w, rows)


def test_index_lists_full_size_all_rows():
    w = W.retention("cuda", "index_list")
    O, L, info, flags = H.run_gpu(w)
    assert flags == 0 and info["stream_keys"] == 8 * 8 * 2048
    assert H.compare_all_rows(O, L, w)["rows"] == 8 * 32


# ---- fail-closed bounded waits (M4.5 §0x07B) ----------------------------------------------

@pytest.mark.parametrize("fused,S_q", [(False, 1), (True, 1), (False, 4)])
def test_bounded_wait_gives_up_and_the_step_fails_closed(fused, S_q):
    """The test hook withholds the completion of CTA 0's first ring stage: its consumers'
    wait runs out after 1 ms, the CTA stops and the status word gets the timeout bit (16).
    No output row may come from the states it left unwritten: its warps mark their state
    slots unwritten (merge kernel) or count none of their items (fused merge), so the rows
    of every group CTA 0 took part in stay unwritten, and every other row is exact.  With
    S_q = 4 (16 rows per kv head) the merge waits for each state's tag rather than for the
    whole grid (merge_tags), and the marked states come tagged.  The context stays usable: the next
    step on the same workspace gives every row exactly."""
    if S_q == 1:
        w = W.paged_ragged_gqa("cuda", B=4, lo=300, hi=900, pool_pages=300)
    else:
        w = W.paged_bf16("verify", B=4, S_q=S_q, H_q=32, H_kv=8, d=128, lens=[900, 310, 640, 505], P=16,
                         seed=9, device="cuda", pool_pages=300)
    p = w.problem
    plan = dattn.dattn_plan(p, w.kv_len, page_indptr=w.page_indptr, num_sms=6, fused_merge=fused,
                            merge_tags=1 if S_q > 1 else -1)
    assert plan.info["n_merge_groups"] > 0 and bool(plan.info["fused_merge"]) == fused
    assert plan.info["merge_tags"] == (1 if S_q > 1 else 0)
    o = torch.full((p["B"], S_q, p["H_q"], p["d"]), float("nan"), dtype=torch.bfloat16, device="cuda")
    lse = torch.full((p["B"], S_q, p["H_q"]), float("nan"), dtype=torch.float32, device="cuda")
    ws = torch.empty(plan.workspace_bytes, dtype=torch.uint8, device="cuda")
    t = dattn.tensors_from(**H.device_tensors(w, o, lse))
    dattn.dattn_run_ex(plan, p, t, ws, wait_limit_us=1000, test_skip_arrival=True)
    torch.cuda.synchronize()
    assert dattn.dattn_device_status(ws) & 16
    O, L = o.float().cpu(), lse.cpu()
    written = ~torch.isnan(L)
    assert torch.equal(written, ~torch.isnan(O).all(dim=-1)), "rows written in part"
    cta0 = {(it["b"], it["h_kv"]) for it in plan.items() if it["cta"] == 0}
    assert cta0
    g = p["H_q"] // p["H_kv"]
    for b, h in cta0:          # groups that CTA 0 took part in: never written
        assert not written[b, :, h * g:(h + 1) * g].any()
    rows = [(b, i, h) for b in range(p["B"]) for i in range(S_q) for h in range(p["H_q"]) if written[b, i, h]]
    assert rows
    H.compare(O, L, w, rows)
    dattn.dattn_run(plan, p, t, ws)         # uploads the plan again (fresh counters and status)
    torch.cuda.synchronize()
    assert dattn.dattn_device_status(ws) == 0
    H.compare(o.float().cpu(), lse.cpu(), w)


@pytest.mark.parametrize("S_q", [1, 4])
def test_timeline_trace_is_ordered_and_leaves_the_outputs_unchanged(S_q):
    """dattn_run_options.trace: per CTA the stamps come in pipeline order, every merge block
    finds its states ready after the partial kernel began (with merge tags the merge of a
    group starts once its states carry the run's tag, possibly before the last partial CTA
    ends; without, it waits for the whole grid), and the traced step gives the same bits."""
    if S_q == 1:
        w = W.paged_ragged_gqa("cuda", B=6, lo=200, hi=2000, pool_pages=800)
    else:
        w = W.paged_bf16("verify", B=6, S_q=S_q, H_q=32, H_kv=8, d=128, lens=[1900, 240, 1333, 777, 2000, 450],
                         P=16, seed=10, device="cuda", pool_pages=800)
    keep = {}
    O, L, info, flags = H.run_gpu(w, num_sms=16, keep=keep, merge_tags=1 if S_q > 1 else -1)
    assert flags == 0 and info["n_merge_groups"] > 0 and info["merge_tags"] == (1 if S_q > 1 else 0)
    n = info["n_ctas"]
    buf = torch.zeros(16 * n + 2 * info["n_merge_groups"] * info["rows"], dtype=torch.int64, device="cuda")
    keep["kw"]["o"].fill_(float("nan"))
    dattn.dattn_run_ex(keep["plan"], w.problem, dattn.tensors_from(**keep["kw"]), keep["ws"], trace=buf)
    torch.cuda.synchronize()
    assert torch.equal(keep["kw"]["o"].float().cpu().reshape(O.shape), O)
    t = buf.cpu().numpy()
    P = t[:16 * n].reshape(n, 16)
    assert (P[:, 0] > 0).all() and (P[:, 1] >= P[:, 0]).all()
    # (the first stage can land, L2-resident, before producer warp 0 stamps its own first copy)
    assert (P[:, 2] >= P[:, 1]).all() and (P[:, 3] >= P[:, 2]).all() and (P[:, 4] >= P[:, 2]).all()
    assert (P[:, 8:16] >= P[:, 4:5]).all()
    M = t[16 * n:].reshape(-1, 2)
    M = M[M[:, 0] > 0]
    assert len(M) and (M[:, 0] >= P[:, 0].min()).all() and (M[:, 1] >= M[:, 0]).all()
    if S_q == 1:      # no tags: every merge block waits for the whole partial grid
        assert (M[:, 0] >= P[:, 8:16].max()).all()


def test_wait_limit_options_are_checked():
    w = W.paged_ragged_gqa("cuda", B=2, lo=10, hi=40, pool_pages=10)
    p = w.problem
    plan = dattn.dattn_plan(p, w.kv_len, page_indptr=w.page_indptr, num_sms=2)
    o = torch.zeros((2, 1, p["H_q"], p["d"]), dtype=torch.bfloat16, device="cuda")
    ws = torch.empty(plan.workspace_bytes, dtype=torch.uint8, device="cuda")
    t = dattn.tensors_from(**H.device_tensors(w, o, None))
    for limit in (0, 200000):
        with pytest.raises(dattn.DattnError, match="wait limit"):
            dattn.dattn_run_ex(plan, p, t, ws, wait_limit_us=limit, test_skip_arrival=True)


@pytest.mark.parametrize("kind", ["decode", "verify", "mixed"])
def test_merge_tags_give_the_rows_of_the_whole_grid_wait(kind):
    """merge_tags = 1 (the merge folds each group once its states carry the run's tag) and
    -1 (it waits for the whole partial grid) give the same bits on every row, equal to the
    oracle's: 4 rows per kv head, 16 (S_q = 4) and a mixed batch of up to 32."""
    if kind == "decode":
        w = W.paged_ragged_gqa("cuda", B=5, lo=300, hi=3000, pool_pages=1000)
    elif kind == "verify":
        w = W.paged_bf16("verify", B=5, S_q=4, H_q=32, H_kv=8, d=128, lens=[2900, 40, 1500, 801, 3000],
                         P=16, seed=11, device="cuda", pool_pages=1000)
    else:
        w = W.mixed_batch("cuda", B=8, lo=200, hi=2500)
    outs = {}
    for tags in (1, -1):
        O, L, info, flags = H.run_gpu(w, num_sms=24, merge_tags=tags)
        assert flags == 0 and info["n_merge_groups"] > 0 and info["merge_tags"] == (tags > 0)
        outs[tags] = (O, L)
    assert torch.equal(outs[1][0], outs[-1][0]) and torch.equal(outs[1][1], outs[-1][1])
    H.compare_all_rows(outs[1][0], outs[1][1], w)


# ---- bit-exact debug hooks --------------------------------------------------------------

def test_debug_translate_matches_oracle_offsets():
    w = W.paged_ragged_gqa("cuda", B=3, lo=1, hi=90, pool_pages=40)
    p = w.problem
    rng = np.random.default_rng(0)
    coords = []
    for _ in range(3000):
        b = int(rng.integers(0, p["B"]))
        coords.append([b, int(rng.integers(-2, int(w.kv_len[b]) + 3)), int(rng.integers(0, p["H_q"])),
                       int(rng.integers(0, p["d"]))])
    c = torch.tensor(coords, dtype=torch.int32, device="cuda")
    out = torch.empty(len(coords), dtype=torch.int64, device="cuda")
    t = dattn.tensors_from(**H.device_tensors(w, None, None))
    kv_len = w.kv_len.cuda()
    dattn.dattn_debug_translate(p, t, kv_len, c, out)
    got = out.cpu().numpy()
    ind, ptr = w.page_indices.numpy(), w.page_indptr.numpy()
    for (b, tt, hq, x), g in zip(coords, got):
        if 0 <= tt < int(w.kv_len[b]):
            pi = address.page_csr(ptr, ind, b, tt // p["P"])
            want = address.offset_paged_hnd(pi, tt % p["P"], address.kv_head(hq, p["H_q"], p["H_kv"]), x,
                                            p["P"], p["H_kv"], p["d"])
        else:
            want = -1
        assert g == want


def test_debug_translate_contiguous_remap():
    w = W.contiguous_bf16("remap", B=2, S_q=1, H_q=4, H_kv=2, d=64, lens=[12, 5], T_cap=12, seed=1,
                          device="cuda", B_cache=4, cache_batch_idx=[2, 0])
    p = w.problem
    coords = [[0, 3, 3, 2], [1, 4, 0, 63], [1, 5, 0, 0]]
    out = torch.empty(3, dtype=torch.int64, device="cuda")
    t = dattn.tensors_from(**H.device_tensors(w, None, None))
    kv_len = w.kv_len.cuda()
    cd = torch.tensor(coords, dtype=torch.int32, device="cuda")
    dattn.dattn_debug_translate(p, t, kv_len, cd, out)
    got = out.cpu().tolist()
    assert got[0] == address.offset_contig_nhd(2, 3, 1, 2, 12, 2, 64)
    assert got[1] == address.offset_contig_nhd(0, 4, 0, 63, 12, 2, 64)
    assert got[2] == -1


@pytest.mark.parametrize("mask,S_q,extra", [("causal", 4, {}), ("sink_window", 1, dict(n_sink=4, window=4096)),
                                            ("sink_window", 3, dict(n_sink=5, window=20)),
                                            ("index_list", 1, {}), ("index_list", 2, {})])
def test_debug_classify_matches_oracle_tile_classes(mask, S_q, extra):
    lens = [5000, 17, 0, 4100]
    w = W.paged_bf16("cls", B=4, S_q=S_q, H_q=8, H_kv=2, d=128, lens=lens, P=16, seed=2, device="cuda",
                     pool_pages=sum(-(-t // 16) for t in lens), mask=mask, **extra)
    if mask == "index_list":
        meta = torch.Generator().manual_seed(5)
        w.index_indptr, w.index_list = W.h2o_index_lists(lens, 2, 300, 8, 40, meta)
    p = H.oracle_problem(w)
    tiles, want = [], []
    for b, T in enumerate(lens):
        for h in range(2):
            lst = None
            if mask == "index_list":
                k = b * 2 + h
                lst = p["index_list"][p["index_indptr"][k]:p["index_indptr"][k + 1]]
            sets = [masks.visible_positions(mask, T, S_q, i, n_sink=extra.get("n_sink", 0),
                                            window=extra.get("window", 0), index_list=lst) for i in range(S_q)]
            for j in range(0, T // 16 + 2):
                tiles.append([b, h, j])
                want.append(masks.tile_class(sets, 16 * j, 16 * (j + 1)))
    out = torch.empty(len(tiles), dtype=torch.int32, device="cuda")
    t = dattn.tensors_from(**H.device_tensors(w, None, None))
    kv_len = w.kv_len.cuda()
    td = torch.tensor(tiles, dtype=torch.int32, device="cuda")
    dattn.dattn_debug_classify(w.problem, t, kv_len, td, out)
    got = [dattn.TILE_CLASSES[x] for x in out.cpu().tolist()]
    assert got == want


@pytest.mark.parametrize("mask", ["causal", "sink_window", "index_list"])
def test_debug_gather_equals_visible_union(mask):
    lens = [3000, 5, 4200]
    extra = dict(n_sink=4, window=1000) if mask == "sink_window" else {}
    w = W.paged_bf16("gather", B=3, S_q=2, H_q=8, H_kv=2, d=128, lens=lens, P=16, seed=3, device="cuda",
                     pool_pages=sum(-(-t // 16) for t in lens), mask=mask, **extra)
    if mask == "index_list":
        w.index_indptr, w.index_list = W.h2o_index_lists(lens, 2, 500, 8, 64, torch.Generator().manual_seed(6))
    keep = {}
    H.run_gpu(w, num_sms=3, chunk_tokens=256, keep=keep)
    p = H.oracle_problem(w)
    out = torch.empty(5000, dtype=torch.int32, device="cuda")
    for b, T in enumerate(lens):
        for h in range(2):
            n = dattn.dattn_debug_gather(keep["plan"], w.problem, dattn.tensors_from(**keep["kw"]), keep["ws"], b, h,
                                         out)
            got = out[:n].cpu().numpy()
            lst = None
            if mask == "index_list":
                k = b * 2 + h
                lst = p["index_list"][p["index_indptr"][k]:p["index_indptr"][k + 1]]
            want = np.unique(np.concatenate([masks.visible_positions(mask, T, 2, i, n_sink=extra.get("n_sink", 0),
                                                                     window=extra.get("window", 0), index_list=lst)
                                             for i in range(2)]))
            assert np.array_equal(got, want)


def test_device_bounds_check_flags_out_of_pool_page_without_reading_it():
    """A page id >= num_pages is caught by the kernel's own check before any address is formed."""
    w = W.paged_bf16("oob", B=2, S_q=1, H_q=8, H_kv=2, d=128, lens=[40, 40], P=16, seed=4, device="cuda",
                     pool_pages=6)
    w.page_indices = w.page_indices.clone()
    w.page_indices[1] = 6          # one past the pool: request 0, logical block 1
    O, L, info, flags = H.run_gpu(w, num_sms=2)
    assert flags & 1               # kStPageRange
    # request 1 is untouched by the bad entry and still matches the oracle
    H.compare(O, L, w, [(1, 0, h) for h in range(8)])


@pytest.mark.parametrize("chunk,num_sms,S_q", [(0, 152, 1), (64, 7, 1), (0, 152, 4), (64, 7, 2)])
def test_fused_merge_matches_and_counters_reset_for_reused_uploads(chunk, num_sms, S_q):
    """With fused_merge, bf16 groups are merged inside the partial kernel by the CTA that
    completes them (4 to 32 rows); the per-group counters must come back to zero, so runs
    that reuse the uploaded work list give bit-identical outputs."""
    w = W.paged_ragged_gqa("cuda", B=6, lo=1, hi=900, pool_pages=500)
    if S_q > 1:
        w = W.paged_bf16("fused", B=5, S_q=S_q, H_q=32, H_kv=4, d=128, lens=[700, 5, 300, 64, 1], P=16,
                         seed=31, device="cuda")
    keep = {}
    O, L, info, flags = H.run_gpu(w, chunk_tokens=chunk, num_sms=num_sms, keep=keep, fused_merge=True)
    assert flags == 0 and info["n_merge_groups"] > 0 and info["fused_merge"] == 1
    H.compare(O, L, w)
    t = dattn.tensors_from(**keep["kw"])
    for _ in range(3):
        keep["kw"]["o"].fill_(float("nan"))
        dattn.dattn_run_ex(keep["plan"], w.problem, t, keep["ws"], reuse_upload=True)
        torch.cuda.synchronize()
        assert dattn.dattn_device_status(keep["ws"]) == 0
        assert torch.equal(keep["kw"]["o"].float().cpu().reshape(O.shape), O)
        assert torch.equal(keep["kw"]["lse"].cpu().reshape(L.shape), L)


# ---- FlashMask two-interval columns (M4.5 §0x06A-§0x06D) ---------------------------------

@pytest.mark.parametrize("chunk,num_sms", [(0, 152), (64, 5)])
def test_flashmask_speculation_tree_all_rows(chunk, num_sms):
    """8 draft rows of a DFS-ordered tree (32 query rows per kv head) over short prefixes."""
    w = W.tree_verify("cuda", B=4, S_q=8, lo=1, hi=300, seed=7)
    O, L, info, flags = H.run_gpu(w, chunk_tokens=chunk, num_sms=num_sms)
    assert flags == 0
    H.compare(O, L, w)


def _random_fm_intervals(rng, lens, S_q):
    out = []
    for T in lens:
        a = np.sort(rng.integers(0, S_q + 1, size=(T, 2)), axis=1)
        b = np.sort(rng.integers(0, S_q + 1, size=(T, 2)), axis=1)
        iv = np.concatenate([a, b], axis=1)
        iv[rng.random(T) < 0.2] = [0, S_q, 0, 0]          # columns hidden from every row
        iv[rng.random(T) < 0.3] = [0, 0, 0, 0]            # columns every row sees
        out.append(iv)
    return np.concatenate(out) if out else np.zeros((0, 4), np.int64)


@pytest.mark.parametrize("S_q,H_q,H_kv", [(4, 16, 2), (1, 8, 2), (32, 32, 32), (3, 16, 4)])
def test_flashmask_random_intervals_with_hidden_columns_and_rows(S_q, H_q, H_kv):
    lens = [300, 65, 1, 0, 130]
    w = W.paged_bf16("fm", B=len(lens), S_q=S_q, H_q=H_q, H_kv=H_kv, d=128, lens=lens, P=16, seed=32,
                     device="cuda")
    rng = np.random.default_rng(33 + S_q)
    iv = _random_fm_intervals(rng, lens, S_q)
    iv[sum(lens[:2])] = [0, S_q, 0, 0]                     # request 2: its only key hidden from all rows
    w.problem = dict(w.problem, mask="flashmask")
    w.fm_intervals = torch.tensor(iv, dtype=torch.int32)
    O, L, info, flags = H.run_gpu(w, chunk_tokens=64, num_sms=7)
    assert flags == 0
    assert torch.isinf(L[2]).all() and (L[2] < 0).all()
    H.compare(O, L, w)


def test_flashmask_causal_rewrite_agrees_with_causal():
    lens = [257, 40, 4]
    S_q = 4
    w = W.paged_bf16("fmc", B=3, S_q=S_q, H_q=16, H_kv=4, d=128, lens=lens, P=16, seed=34, device="cuda")
    O0, L0, _, _ = H.run_gpu(w, chunk_tokens=64, num_sms=5)
    H.compare(O0, L0, w)
    iv = []
    for T in lens:
        iv += [(0, max(0, min(S_q, j - (T - S_q))), 0, 0) for j in range(T)]
    w.problem = dict(w.problem, mask="flashmask")
    w.fm_intervals = torch.tensor(iv, dtype=torch.int32)
    O1, L1, _, flags = H.run_gpu(w, chunk_tokens=64, num_sms=5)
    assert flags == 0
    H.compare(O1, L1, w)
    assert torch.allclose(O0, O1, atol=1e-2, rtol=1e-2) and torch.allclose(L0, L1, atol=1e-4, rtol=1e-5)


def test_flashmask_tree_verify_full_size_all_rows():
    """The tree-verification workload: B=16, prefixes U[1024, 8192], 8 draft rows."""
    w = W.tree_verify("cuda")
    O, L, info, flags = H.run_gpu(w)
    assert flags == 0
    assert H.compare_all_rows(O, L, w)["rows"] == 16 * 8 * 32


# ---- mixed prefill / append / decode batches (per-request query rows) -------------------


@pytest.mark.parametrize("chunk,num_sms", [(0, 152), (4, 3)])
def test_mixed_batch_phase_fixture_all_rows(chunk, num_sms):
    """The three-request mix of the phase fixture: prefill (0,4), append (6,2), decode (9,1)."""
    w = W.mixed_batch("cuda", TC=[(0, 4), (6, 2), (9, 1)], seed=40)
    assert w.qo_indptr.tolist() == [0, 4, 6, 7]
    O, L, info, flags = H.run_gpu(w, chunk_tokens=chunk, num_sms=num_sms)
    assert flags == 0
    assert O.shape == (7, 32, 128)
    H.compare(O, L, w)


@pytest.mark.parametrize("chunk,num_sms,fused", [(0, 152, False), (64, 7, False), (64, 7, True),
                                                 (100000, 152, False)])
def test_mixed_batch_small_all_rows(chunk, num_sms, fused):
    """Every phase plus an idle request, histories spanning several stages and a ragged tail."""
    TC = [(0, 8), (130, 1), (0, 1), (65, 3), (7, 0), (300, 8), (1, 2), (64, 5), (0, 0), (200, 1)]
    w = W.mixed_batch("cuda", TC=TC, seed=41)
    O, L, info, flags = H.run_gpu(w, chunk_tokens=chunk, num_sms=num_sms, fused_merge=fused)
    assert flags == 0
    H.compare(O, L, w)


def test_mixed_batch_sink_window():
    TC = [(0, 8), (300, 1), (90, 4), (5, 2), (0, 3)]
    w = W.mixed_batch("cuda", TC=TC, seed=42, mask="sink_window", n_sink=4, window=64)
    O, L, info, flags = H.run_gpu(w, chunk_tokens=64, num_sms=5)
    assert flags == 0
    H.compare(O, L, w)


def test_mixed_batch_no_query_rows_at_all():
    """Every request idle: the launch writes nothing (the one-row buffers stay NaN) and raises no flag."""
    w = W.mixed_batch("cuda", TC=[(5, 0), (0, 0), (70, 0)], seed=43)
    p = w.problem
    plan = dattn.dattn_plan(p, w.kv_len, page_indptr=w.page_indptr, qo_indptr=w.qo_indptr, num_sms=8)
    assert plan.info["stream_keys"] == 0
    o = torch.full((1, 32, 128), float("nan"), dtype=torch.bfloat16, device="cuda")
    lse = torch.full((1, 32), float("nan"), dtype=torch.float32, device="cuda")
    q = torch.zeros((1, 32, 128), dtype=torch.bfloat16, device="cuda")
    ws = torch.empty(max(256, plan.workspace_bytes), dtype=torch.uint8, device="cuda")
    kw = H.device_tensors(w, o, lse)
    kw["q"] = q
    dattn.dattn_run(plan, p, dattn.tensors_from(**kw), ws)
    torch.cuda.synchronize()
    assert dattn.dattn_device_status(ws) == 0
    assert o.isnan().all() and lse.isnan().all()


def test_mixed_batch_uniform_indptr_equals_plain_batch():
    """qo_indptr = [0, S_q, 2 S_q, ...] is the plain batch: identical bits."""
    w = W.paged_bf16("u", B=3, S_q=4, H_q=16, H_kv=4, d=128, lens=[200, 17, 90], P=16, seed=44, device="cuda")
    O0, L0, _, _ = H.run_gpu(w, chunk_tokens=64, num_sms=5)
    w.qo_indptr = torch.arange(0, 13, 4, dtype=torch.int32)
    w.q = w.q.reshape(12, 16, 128)
    O1, L1, _, flags = H.run_gpu(w, chunk_tokens=64, num_sms=5)
    assert flags == 0
    assert torch.equal(O0.reshape(12, 16, 128), O1) and torch.equal(L0.reshape(12, 16), L1)


def test_mixed_batch_full_size_all_rows():
    """B=16: ten decode rows, three appends, two 8-row prefills and one idle request."""
    w = W.mixed_batch("cuda")
    O, L, info, flags = H.run_gpu(w)
    assert flags == 0
    assert H.compare_all_rows(O, L, w)["rows"] == int(w.qo_indptr[-1]) * 32


def test_mixed_batch_flashmask_trees_of_different_sizes():
    """Speculation trees of 1..8 drafts per request: FlashMask intervals in each request's C_b rows."""
    TC = [(40, 8), (7, 3), (130, 1), (0, 5), (66, 0)]
    w = W.mixed_batch("cuda", TC=TC, seed=45)
    iv = []
    gen = torch.Generator().manual_seed(46)
    for T, C in TC:
        iv += [(0, 0, 0, 0)] * T
        if C:
            iv += W._dfs_tree_intervals(C, gen)
    w.problem = dict(w.problem, mask="flashmask")
    w.fm_intervals = torch.tensor(iv, dtype=torch.int32)
    assert w.fm_intervals.shape[0] == sum(T + C for T, C in TC)
    O, L, info, flags = H.run_gpu(w, chunk_tokens=64, num_sms=5)
    assert flags == 0
    H.compare(O, L, w)


def _step_host(w, mask_args=None, num_sms=152):
    """One dattn_step_host over workload w (host q and page table in, host O and LSE out)."""
    p = dict(w.problem, **(mask_args or {}))
    B, S_q, H_q, d = p["B"], p["S_q"], p["H_q"], p["d"]
    q_host = w.q.cpu().pin_memory()
    o_host = torch.full((B, S_q, H_q, d), float("nan"), dtype=torch.bfloat16).pin_memory()
    lse_host = torch.full((B, S_q, H_q), float("nan"), dtype=torch.float32).pin_memory()
    paged = p["layout"] == "paged"
    io = dattn.host_step(q_host, w.kv_len, o_host, lse=lse_host, num_sms=num_sms,
                         page_indptr=w.page_indptr if paged else None, page_indices=w.page_indices if paged else None)
    ws_bytes, sg_bytes = dattn.dattn_step_host_sizes(p, io)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device="cuda")
    staging = torch.empty(sg_bytes, dtype=torch.uint8).pin_memory()
    cache = dattn.tensors_from(k=w.k, v=w.v, cache_batch_idx=None if w.cache_batch_idx is None else
                               w.cache_batch_idx.cuda())
    dattn.dattn_step_host(p, io, cache, staging, ws)
    assert dattn.dattn_step_host_status(p, io, ws) == 0
    return p, o_host.float(), lse_host


@pytest.mark.parametrize("copy_stream", [False, True])
def test_step_host_submit_finish_pipelined_equals_the_synchronous_step(copy_stream):
    """Four steps submitted two deep (two staging buffers and events, one stream; with
    copy_stream, the transfers on two streams of their own and one workspace per slot): each step's
    O and LSE are the synchronous dattn_step_host's bits, and the first matches the oracle
    on every row."""
    w = W.paged_ragged_gqa("cuda", B=6, lo=100, hi=3000, pool_pages=1200)
    p = w.problem
    B, H_q, d = p["B"], p["H_q"], p["d"]
    cache = dattn.tensors_from(k=w.k, v=w.v)
    qs = [(w.q.cpu().float() * f).to(torch.bfloat16).pin_memory() for f in (1.0, -1.0, 0.5, 2.0)]   # exact
    outs = [(torch.full((B, 1, H_q, d), float("nan"), dtype=torch.bfloat16).pin_memory(),
             torch.full((B, 1, H_q), float("nan"), dtype=torch.float32).pin_memory()) for _ in qs]
    ios = [dattn.host_step(q, w.kv_len, o, lse=l, page_indptr=w.page_indptr, page_indices=w.page_indices)
           for q, (o, l) in zip(qs, outs)]
    ws_bytes, sg_bytes = dattn.dattn_step_host_sizes(p, ios[0])
    wss = [torch.empty(ws_bytes, dtype=torch.uint8, device="cuda") for _ in range(2 if copy_stream else 1)]
    staging = [torch.empty(sg_bytes + 4096, dtype=torch.uint8).pin_memory() for _ in range(2)]
    events = [torch.cuda.Event(), torch.cuda.Event()]
    cs = (torch.cuda.Stream(), torch.cuda.Stream())
    side = [(torch.cuda.Event(), torch.cuda.Event()) for _ in range(2)]

    def submit(k):
        slot = k % 2
        ws = wss[slot % len(wss)]
        if copy_stream:
            dattn.dattn_step_host_submit_ex(p, ios[k], cache, staging[slot], ws, events[slot], *cs, *side[slot])
        else:
            dattn.dattn_step_host_submit(p, ios[k], cache, staging[slot], ws, events[slot])

    submit(0)
    for k in range(1, len(qs) + 1):
        if k < len(qs):
            submit(k)
        dattn.dattn_step_host_finish(p, ios[k - 1], staging[(k - 1) % 2], events[(k - 1) % 2])
    torch.cuda.synchronize()
    for i, ws in enumerate(wss):
        assert dattn.dattn_step_host_status(p, ios[i], ws) == 0
    for q, (o, l) in zip(qs, outs):
        o1 = torch.full_like(o, float("nan"))
        l1 = torch.full_like(l, float("nan"))
        io1 = dattn.host_step(q, w.kv_len, o1, lse=l1, page_indptr=w.page_indptr, page_indices=w.page_indices)
        dattn.dattn_step_host(p, io1, cache, staging[0], wss[0])
        assert torch.equal(o.view(torch.int16), o1.view(torch.int16)) and torch.equal(l, l1)
    H.compare(outs[0][0].float(), outs[0][1], w)


@pytest.mark.parametrize("case", ["paged", "contig", "sink_window_verify"])
def test_step_host_matches_oracle_and_dattn_run(case):
    """The host-memory step gives the oracle's result, and the same bits as dattn_run on
    device copies of the same inputs (same plan, same kernels)."""
    if case == "contig":
        w = W.tiny_contiguous("cuda")
        mask_args = None
    else:
        w = W.paged_ragged_gqa("cuda", B=6, lo=1, hi=900, pool_pages=500)
        mask_args = None
        if case == "sink_window_verify":
            w = W.paged_bf16("swv", B=4, S_q=3, H_q=8, H_kv=2, d=128, lens=[700, 3, 64, 1],
                             P=16, seed=9, device="cuda", pool_pages=80)
            mask_args = dict(mask="sink_window", n_sink=5, window=100)
    p, O, L = _step_host(w, mask_args)
    w.problem = p
    H.compare(O, L, w)
    O2, L2, info, flags = H.run_gpu(w, num_sms=152)
    assert flags == 0
    assert torch.equal(O, O2) and torch.equal(L, L2)


def test_step_host_full_size_all_rows_and_repeated():
    """The benchmark's workload through the host-memory step, twice in a row on one workspace."""
    w = W.paged_ragged_gqa("cuda")
    outs = [_step_host(w) for _ in range(2)]
    from tests import oracle_pool
    p = H.oracle_problem(w)
    rows = H.all_rows(p)
    spec, arrays = H.cache_arrays(w)
    ref = oracle_pool.decode_rows_parallel(p, spec, arrays, H.bits(w.q), rows)
    for _, O, L in outs:
        H.compare(O, L, w, rows, ref=ref)


def test_step_host_rejects_short_buffers_after_planning():
    """A workspace or staging buffer that holds the inputs but not the plan and outputs is
    rejected after planning, before any kernel: the outputs stay untouched."""
    w = W.paged_ragged_gqa("cuda", B=3, lo=1, hi=300, pool_pages=64)
    p = w.problem
    q_host = w.q.cpu().pin_memory()
    o_host = torch.full((3, 1, 32, 128), 7.0, dtype=torch.bfloat16)
    io = dattn.host_step(q_host, w.kv_len, o_host, page_indptr=w.page_indptr, page_indices=w.page_indices)
    ws_bytes, sg_bytes = dattn.dattn_step_host_sizes(p, io)
    cache = dattn.tensors_from(k=w.k, v=w.v)
    for ws_n, sg_n in ((ws_bytes - 256, sg_bytes), (ws_bytes, sg_bytes - 256)):
        ws = torch.empty(ws_n, dtype=torch.uint8, device="cuda")
        staging = torch.empty(sg_n, dtype=torch.uint8).pin_memory()
        with pytest.raises(dattn.DattnError, match="DATTN_EWORKSPACE"):
            dattn.dattn_step_host(p, io, cache, staging, ws)
    torch.cuda.synchronize()
    assert bool((o_host.float() == 7.0).all())


# ---- the ragged packed view of retained rows (M5.4 §0x04C) ----------------------------------

@pytest.mark.parametrize("S_q,chunk,num_sms", [(1, 128, 5), (1, 0, 152), (3, 64, 7)])
def test_packed_view_matches_oracle_and_the_index_list_gather(S_q, chunk, num_sms):
    """Decode over the compacted rows equals decode over the paged cache with the same lists,
    bit for bit (the same keys in the same order), and both match the oracle."""
    w = W.retention("cuda", "index_list", B=3, T=3000)
    if S_q > 1:
        w.problem = dict(w.problem, S_q=S_q)
        w.q = torch.randn((3, S_q, 32, 128), device="cuda").to(torch.bfloat16)
    wp = W.packed_view(w)
    O1, L1, info1, f1 = H.run_gpu(w, num_sms=num_sms, chunk_tokens=chunk)
    O2, L2, info2, f2 = H.run_gpu(wp, num_sms=num_sms, chunk_tokens=chunk)
    assert f1 == 0 and f2 == 0
    assert info1["stream_keys"] == info2["stream_keys"]
    assert torch.equal(O1, O2) and torch.equal(L1, L2)
    H.compare(O2, L2, wp)


def test_packed_view_full_size_all_rows():
    wp = W.packed_view(W.retention("cuda", "index_list"))
    O, L, info, flags = H.run_gpu(wp)
    assert flags == 0 and info["stream_keys"] == 8 * 8 * 2048
    assert wp.k.shape == (8 * 8 * 2048, 128)
    assert H.compare_all_rows(O, L, wp)["rows"] == 8 * 32


def test_debug_translate_packed_view_matches_oracle_rows():
    w = W.packed_view(W.retention("cuda", "index_list", B=2, T=500))
    p = w.problem
    rng = np.random.default_rng(9)
    coords = []
    for _ in range(300):
        coords.append((int(rng.integers(0, 2)), int(rng.integers(0, 500)), int(rng.integers(0, 32)),
                       int(rng.integers(0, 128))))
    c = H.oracle_cache(w)
    want = []
    for b, t, hq, x in coords:
        try:
            want.append(int(ocache.packed_rows(c, b, hq // 4, [t])[0]) * 128 + x)
        except IndexError:
            want.append(-1)
    c_dev = torch.tensor(coords, dtype=torch.int32, device="cuda")
    out = torch.empty(len(coords), dtype=torch.int64, device="cuda")
    dattn.dattn_debug_translate(p, dattn.tensors_from(**H.device_tensors(w, None, None)), w.kv_len.cuda(), c_dev, out)
    assert out.cpu().tolist() == want and (np.asarray(want) >= 0).sum() > 30
