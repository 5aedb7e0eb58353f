"""Host-side tests of libdattn (no GPU): exports, planner pins, call validation.

The planner is plain host code, so its split bounds, chunking, CTA
assignment and workspace sizing are checked here against the pages' printed
values (M4.5 §0x03B, §0x03E, §0x03G, §0x09G) and against the oracle's
visible sets.  Each validation gets a one-field-mutation negative test
(M4.5 §0x07A-§0x07B).
"""

import ctypes
import os
import re

import numpy as np
import pytest

import split_kv_decode_flash_gb300 as dattn
from oracle import masks
from oracle import split_state as ss
from tests.conftest import ROOT, golden

HEADER = os.path.join(ROOT, "include", "dattn.h")


def _declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b([a-z_]+)\s*\(", text)) - {"sizeof"})


def test_library_exports_every_declared_symbol():
    lib = dattn.load()
    names = _declared_functions()
    assert "dattn_plan" in names and "dattn_run" in names and "kv_append" in names
    for n in names:
        assert hasattr(lib, n), f"libdattn.so does not export {n}"
    assert dattn.dattn_version() >= 100


def _problem(**kw):
    base = dict(B=2, S_q=1, H_q=8, H_kv=2, d=128, layout="paged", fmt="bf16", P=16, num_pages=1000,
                mask="causal")
    base.update(kw)
    return base


def _coverage(items, groups, n_of):
    by = {}
    for it in items:
        by.setdefault((it["b"], it["h_kv"]), []).append((it["a"], it["e"]))
    assert set(by) == set(groups)
    for g, ranges in by.items():
        ranges.sort()
        pos = 0
        for a, e in ranges:
            assert a == pos and e >= a
            pos = e
        assert pos == n_of(g)


def test_fixed_split_bounds_match_balanced_formula():
    g = golden("split_ledgers.json")
    T = g["call"]["T"]
    plan = dattn.dattn_plan(_problem(fixed_splits=8), T, num_sms=152)
    items = plan.items()
    for b, t in enumerate(T):
        got = [(it["a"], it["e"]) for it in items if it["b"] == b and it["h_kv"] == 0]
        assert got == ss.balanced_split_bounds(t, 8)
        assert [e - a for a, e in got] == g["split_lengths"][str(t)]
    info = plan.info
    assert info["n_items"] == 2 * 2 * 8 and info["n_merge_groups"] == 4 and info["max_splits"] == 8


def test_capacity_fixture_empty_splits_are_planned_identity_items():
    g = golden("split_ledgers.json")["capacity_fixture"]
    plan = dattn.dattn_plan(_problem(B=2, H_q=4, H_kv=4, fixed_splits=g["S"]), g["T"], num_sms=8)
    items = plan.items()
    lens0 = [it["e"] - it["a"] for it in items if it["b"] == 0 and it["h_kv"] == 0]
    assert lens0 == g["request0_lengths"]
    active = sum(1 for it in items if it["e"] > it["a"])
    assert active == g["active"] // 1            # 12 = 3 non-empty splits x 4 heads
    assert all(it["slot"] >= 0 for it in items)  # every slot the reducer reads is written


def test_work_schedule_pin_least_loaded_planner():
    g = golden("work_schedule.json")
    prob = _problem(B=2, H_q=1, H_kv=1, P=1, num_pages=6000)
    plan = dattn.dattn_plan(prob, g["outputs"], num_sms=g["workers"], chunk_tokens=g["chunk_limit"])
    items = plan.items()
    assert sorted((it["e"] - it["a"] for it in items), reverse=True) == g["planned_chunks_sorted"]
    loads = [0] * g["workers"]
    for it in items:
        loads[it["cta"]] += it["e"] - it["a"]
    assert loads == g["planned_loads"]
    assert plan.info["max_cta_keys"] == max(g["planned_loads"])
    # the fixed four-way split of the same workload is unbalanced: max/mean 1.6
    fixed = dattn.dattn_plan(dict(prob, fixed_splits=g["fixed_splits"]), g["outputs"], num_sms=g["workers"])
    lens = sorted((it["e"] - it["a"] for it in fixed.items()), reverse=True)
    assert lens == g["fixed_loads"]
    assert max(lens) / (sum(lens) / g["workers"]) == g["rho"]


def test_sink_window_stream_is_the_union_of_visible_sets():
    T = [5, 6, 7, 4100, 9000, 0, 1]
    prob = _problem(B=len(T), H_q=4, H_kv=1, mask="sink_window", n_sink=4, window=4096)
    plan = dattn.dattn_plan(prob, T, num_sms=4, chunk_tokens=64)
    _coverage(plan.items(), [(b, 0) for b in range(len(T))],
              lambda g: len(masks.sink_recent(T[g[0]], 4, 4096)))
    assert plan.info["stream_keys"] == sum(len(masks.sink_recent(t, 4, 4096)) for t in T)


def test_multi_row_sink_window_stream_covers_every_row():
    T, S_q = [50, 3], 4
    prob = _problem(B=2, S_q=S_q, H_q=4, H_kv=2, mask="sink_window", n_sink=2, window=5)
    plan = dattn.dattn_plan(prob, T, num_sms=4)
    want = [len(np.unique(np.concatenate([masks.visible_positions("sink_window", t, S_q, i, n_sink=2, window=5)
                                          for i in range(S_q)]))) for t in T]
    _coverage(plan.items(), [(b, h) for b in range(2) for h in range(2)], lambda g: want[g[0]])


def test_index_list_stream_and_single_chunk_direct_write():
    T = [100, 40]
    lists = [np.arange(0, 100, 3), np.array([1, 5, 99]), np.arange(40), np.array([], np.int32)]
    indptr = np.concatenate([[0], np.cumsum([len(x) for x in lists])])
    prob = _problem(B=2, H_q=4, H_kv=2, mask="index_list")
    plan = dattn.dattn_plan(prob, T, index_indptr=indptr, index_list=np.concatenate(lists), num_sms=2,
                            chunk_tokens=64)
    items = plan.items()
    _coverage(items, [(b, h) for b in range(2) for h in range(2)], lambda g: len(lists[g[0] * 2 + g[1]]))
    rows = plan.info["rows"]
    states_per_item = 8 // (1 if rows <= 16 else 2)      # bf16: one state per consumer warp and row tile
    for it in items:
        n_items = sum(1 for x in items if (x["b"], x["h_kv"]) == (it["b"], it["h_kv"]))
        assert (it["slot"] < 0) == (n_items * states_per_item == 1)


def test_default_planner_covers_ragged_batch_and_balances():
    rng = np.random.default_rng(1)
    T = rng.integers(1024, 8193, 16).tolist()
    plan = dattn.dattn_plan(_problem(B=16, H_q=32, H_kv=8), T, num_sms=152)
    _coverage(plan.items(), [(b, h) for b in range(16) for h in range(8)], lambda g: T[g[0]])
    info = plan.info
    mean = info["stream_keys"] / info["n_ctas"]
    assert info["max_cta_keys"] <= 1.5 * mean
    assert info["n_ctas"] <= 152


def _cta_cost(items, pad_of):
    """Per-CTA keys and items of a plan."""
    keys, n = {}, {}
    for it in items:
        keys[it["cta"]] = keys.get(it["cta"], 0) + it["e"] - it["a"]
        n[it["cta"]] = n.get(it["cta"], 0) + 1
    return keys, n


def test_item_cost_keeps_tiny_groups_from_piling_onto_one_cta():
    """Two 8-key requests (16 tiny groups) inside a ragged batch: without an item cost they
    land on one CTA that streams a full share of keys on top of their overheads; with the
    default cost that CTA gets correspondingly fewer keys, and the cover stays exact."""
    rng = np.random.default_rng(1)
    T = rng.integers(1024, 8193, 16).tolist()
    T = T[:12] + [8, 8] + T[12:]
    groups = [(b, h) for b in range(18) for h in range(8)]
    plain = dattn.dattn_plan(_problem(B=18, H_q=32, H_kv=8), T, num_sms=152, item_cost_keys=-1)
    costed = dattn.dattn_plan(_problem(B=18, H_q=32, H_kv=8), T, num_sms=152)
    for plan in (plain, costed):
        _coverage(plan.items(), groups, lambda g: T[g[0]])
    for plan, crowded_share in ((plain, 0.9), (costed, 0.8)):
        keys, n = _cta_cost(plan.items(), None)
        busiest = max(n, key=lambda c: n[c])
        mean = plan.info["stream_keys"] / plan.info["n_ctas"]
        if plan is plain:
            assert n[busiest] >= 16 and keys[busiest] >= crowded_share * mean
        else:
            assert keys[busiest] <= crowded_share * mean
    # a constant cost applies to every group; a negative one turns the cost off
    const = dattn.dattn_plan(_problem(B=18, H_q=32, H_kv=8), T, num_sms=152, item_cost_keys=320)
    _coverage(const.items(), groups, lambda g: T[g[0]])
    assert [(i["a"], i["e"], i["cta"]) for i in plain.items()] != [(i["a"], i["e"], i["cta"]) for i in const.items()]


def test_workspace_bytes_follow_the_mlu_ledger():
    """Partial area = n_slots * rows * (d * 4 + 2 * 4): the (m, l, u) ABI without a validity byte."""
    T = [4096, 3587]
    plan = dattn.dattn_plan(_problem(fixed_splits=8), T, num_sms=152)
    info = plan.info
    rows = info["rows"]
    partial = info["n_slots"] * rows * (128 * 4 + 2 * 4)
    assert partial == ss.workspace_mlu_bytes(info["n_slots"] * rows, 128, b_valid=0)
    assert info["workspace_bytes"] >= info["blob_bytes"] + partial
    assert info["workspace_bytes"] - info["blob_bytes"] - partial < 2 * 256


@pytest.mark.parametrize("field,value,status,reason", [
    ("H_kv", 3, "DATTN_EINVAL", "multiple of H_kv"),
    ("S_q", 0, "DATTN_EINVAL", "S_q"),
    ("d", 80, "DATTN_EUNSUPPORTED", "d_h"),
    ("P", 0, "DATTN_EINVAL", "page_size"),
    ("num_pages", 0, "DATTN_EINVAL", "num_pages"),
    ("S_q", 16, "DATTN_EUNSUPPORTED", "<= 32"),
    ("window", 0, "DATTN_EINVAL", "window"),
    ("fixed_splits", -1, "DATTN_EINVAL", "fixed_splits"),
])
def test_plan_rejects_one_mutated_field(field, value, status, reason):
    prob = _problem(mask="sink_window", n_sink=1, window=4)
    prob[field] = value
    with pytest.raises(dattn.DattnError) as e:
        dattn.dattn_plan(prob, [10, 20], num_sms=4)
    assert dattn.STATUS[e.value.status] == status
    assert reason in str(e.value)


def test_plan_rejects_bad_lengths_pages_and_lists():
    with pytest.raises(dattn.DattnError, match="kv_len"):
        dattn.dattn_plan(_problem(), [10, -1], num_sms=4)
    with pytest.raises(dattn.DattnError, match="needs 2"):
        dattn.dattn_plan(_problem(), [10, 20], page_indptr=[0, 1, 2], num_sms=4)
    prob = _problem(B=1, H_kv=2, mask="index_list")
    with pytest.raises(dattn.DattnError, match="strictly increasing"):
        dattn.dattn_plan(prob, [10], index_indptr=[0, 2, 4], index_list=[1, 1, 2, 3], num_sms=4)
    with pytest.raises(dattn.DattnError, match="outside"):
        dattn.dattn_plan(prob, [10], index_indptr=[0, 2, 4], index_list=[1, 2, 3, 10], num_sms=4)
    with pytest.raises(dattn.DattnError, match="T_cap"):
        dattn.dattn_plan(dict(_problem(layout="contig", T_cap=8, B_cache=2)), [8, 9], num_sms=4)
    with pytest.raises(dattn.DattnError, match="paged layout"):
        dattn.dattn_plan(dict(_problem(layout="contig", fmt="int8", T_cap=8, B_cache=2)), [8, 8], num_sms=4)


def test_rejection_vector_lists_every_failed_check():
    prob = _problem(H_kv=3, d=96, P=0)
    with pytest.raises(dattn.DattnError) as e:
        dattn.dattn_plan(prob, [1, 1], num_sms=4)
    text = str(e.value)
    assert "multiple of H_kv" in text and "d_h" in text and "page_size" in text
    assert dattn.STATUS[e.value.status] == "DATTN_EINVAL"


def test_run_rejects_stale_plan_and_small_workspace_without_a_gpu():
    """Admission runs before any CUDA call, so these errors are reported on any host."""
    plan = dattn.dattn_plan(_problem(), [10, 20], num_sms=4)

    class Fake:
        def __init__(self, n):
            self._n = n
            self._buf = (ctypes.c_uint8 * (n + 256))()

        def data_ptr(self):
            return (ctypes.addressof(self._buf) + 255) // 256 * 256

        def numel(self):
            return self._n

        def element_size(self):
            return 1

    t = dattn.Tensors()
    buf = Fake(1 << 16)
    for f in ("q", "k", "v", "o", "page_indptr", "page_indices"):
        setattr(t, f, buf.data_ptr())
    with pytest.raises(dattn.DattnError) as e:
        dattn.dattn_run(plan, _problem(H_q=16), t, Fake(plan.workspace_bytes), stream=0)
    assert dattn.STATUS[e.value.status] == "DATTN_ESTALE_PLAN"
    with pytest.raises(dattn.DattnError) as e:
        dattn.dattn_run(plan, _problem(), t, Fake(plan.workspace_bytes - 256), stream=0)
    assert dattn.STATUS[e.value.status] == "DATTN_EWORKSPACE"


def test_mixed_batch_streams_follow_each_requests_query_rows():
    """§0x08F: request b's stream is the union of its own C_b rows' visible sets; C_b = 0 reads nothing."""
    TC = [(0, 4), (6, 2), (9, 1), (30, 0), (100, 3)]
    T = [t + c for t, c in TC]
    qo = np.concatenate([[0], np.cumsum([c for _, c in TC])]).astype(np.int32)
    for mask, extra in (("causal", {}), ("sink_window", dict(n_sink=2, window=5))):
        prob = _problem(B=len(TC), S_q=4, H_q=4, H_kv=2, mask=mask, **extra)
        plan = dattn.dattn_plan(prob, T, qo_indptr=qo, num_sms=3, chunk_tokens=64)

        def want(g):
            C = TC[g[0]][1]
            vis = [masks.visible_positions(mask, T[g[0]], C, i, **extra) for i in range(C)]
            return len(np.unique(np.concatenate(vis))) if C else 0
        _coverage(plan.items(), [(b, h) for b in range(len(TC)) for h in range(2)], want)


def test_equal_segments_weigh_the_keys_of_wide_bf16_requests():
    """Keys of a bf16 request with more than 16 rows (the 32-row tile) weigh 1.25 in the
    equal-segment partition: a CTA holding only such keys gets about 1/1.25 of the keys of
    one holding only 4-row keys, and every CTA's weighted load is about the same."""
    B, S_q = 6, 8
    qo = np.array([0, 1, 2, 10, 11, 18, 19], np.int32)          # C_b: 1, 1, 8, 1, 7, 1
    T = [6000, 5000, 7000, 6500, 7200, 5500]
    prob = _problem(B=B, S_q=S_q, H_q=32, H_kv=8, num_pages=20000)
    pages = [-(-t // 16) for t in T]
    indptr = np.concatenate([[0], np.cumsum(pages)]).astype(np.int32)
    plan = dattn.dattn_plan(prob, T, page_indptr=indptr, qo_indptr=qo, num_sms=40, item_cost_keys=-1)
    C = np.diff(qo)
    wide = {b for b in range(B) if 4 * C[b] > 16}
    assert wide == {2, 4}
    load, keys_only = {}, {}
    for it in plan.items():
        n = it["e"] - it["a"]
        load[it["cta"]] = load.get(it["cta"], 0) + n * (1.25 if it["b"] in wide else 1.0)
        kind = "wide" if it["b"] in wide else "narrow"
        keys_only.setdefault(it["cta"], set()).add(kind)
    v = np.array([load[c] for c in sorted(load)])
    assert v.max() - v[:-1].min() <= 16 * 1.25 + 2        # equal up to a tile and a cut (last CTA short)
    pure = {c: ks for c, ks in keys_only.items() if len(ks) == 1}
    per_kind = {}
    for it in plan.items():
        if it["cta"] in pure and it["cta"] != max(load):
            per_kind.setdefault(next(iter(pure[it["cta"]])), {}).setdefault(it["cta"], 0)
            per_kind[next(iter(pure[it["cta"]]))][it["cta"]] += it["e"] - it["a"]
    nw = np.median(list(per_kind["wide"].values()))
    nn = np.median(list(per_kind["narrow"].values()))
    assert abs(nn / nw - 1.25) < 0.05


def test_merge_tags_follow_the_plan_inputs():
    """merge_tags: 1 forces state-row tags on a bf16 plan with a merge kernel, -1 turns them
    off, 0 takes them when the merge folds at least 64 group rows; never for the other
    formats or fused merges; the blob then holds one zeroed int32 tag per state row."""
    T = [4096, 3587]
    prob = _problem(fixed_splits=8)
    base = dattn.dattn_plan(prob, T, num_sms=152, merge_tags=-1).info
    on = dattn.dattn_plan(prob, T, num_sms=152, merge_tags=1).info
    assert base["merge_tags"] == 0 and on["merge_tags"] == 1
    assert dattn.dattn_plan(prob, T, num_sms=152).info["merge_tags"] == 0      # 4 groups x 4 rows
    wide = _problem(B=16, S_q=1, H_q=32, H_kv=8, fixed_splits=4)
    assert dattn.dattn_plan(wide, [600] * 16, num_sms=152).info["merge_tags"] == 1   # 128 groups x 4 rows
    assert on["blob_bytes"] >= base["blob_bytes"] + 4 * on["n_slots"] * on["rows"]
    assert on["blob_bytes"] - base["blob_bytes"] < 4 * on["n_slots"] * on["rows"] + 256
    assert dattn.dattn_plan(prob, T, num_sms=152, merge_tags=1, fused_merge=True).info["merge_tags"] == 0
    q8 = _problem(fixed_splits=8, fmt="int8")
    assert dattn.dattn_plan(q8, T, page_indptr=np.array([0, 256, 481], np.int32), num_sms=152,
                            merge_tags=1).info["merge_tags"] == 0


def test_mixed_batch_validation():
    prob = _problem(B=3, S_q=4)
    T = [5, 6, 7]
    with pytest.raises(dattn.DattnError, match=r"qo_indptr\[0\]"):
        dattn.dattn_plan(prob, T, qo_indptr=np.array([1, 2, 3, 4], np.int32), num_sms=4)
    with pytest.raises(dattn.DattnError, match="C_b <= S_q"):
        dattn.dattn_plan(prob, T, qo_indptr=np.array([0, 5, 6, 7], np.int32), num_sms=4)
    with pytest.raises(dattn.DattnError, match="0 <= C_b"):
        dattn.dattn_plan(prob, T, qo_indptr=np.array([0, 2, 1, 3], np.int32), num_sms=4)
    # non-uniform C_b on every format; KIVI only with a power-of-two page size (the
    # byte-format kernel that serves other page sizes takes uniform batches)
    kivi = dict(kivi_group=32, kivi_v_group=32, kivi_residual=64)
    for fmt in ("int8", "fp8_e4m3", "fp8_e5m2", "int4_head", "int4_kivi"):
        dattn.dattn_plan(_problem(B=3, S_q=4, fmt=fmt, **kivi), T, page_indptr=np.array([0, 1, 2, 3], np.int32),
                         qo_indptr=np.array([0, 1, 2, 4], np.int32), num_sms=4)
    k96 = _problem(B=3, S_q=4, fmt="int4_kivi", P=96, **kivi)
    with pytest.raises(dattn.DattnError, match="power-of-two page_size") as e:
        dattn.dattn_plan(k96, T, page_indptr=np.array([0, 1, 2, 3], np.int32),
                         qo_indptr=np.array([0, 1, 2, 4], np.int32), num_sms=4)
    assert dattn.STATUS[e.value.status] == "DATTN_EUNSUPPORTED"
    # a uniform qo_indptr is the plain batch, for every format and page size
    dattn.dattn_plan(k96, T, page_indptr=np.array([0, 1, 2, 3], np.int32),
                     qo_indptr=np.array([0, 4, 8, 12], np.int32), num_sms=4)


def test_flashmask_on_every_format_kivi_needs_power_of_two_pages():
    T = [5, 6]
    kivi = dict(kivi_group=32, kivi_v_group=32, kivi_residual=64)
    for fmt in ("bf16", "int8", "fp8_e4m3", "fp8_e5m2", "int4_head", "int4_kivi"):
        dattn.dattn_plan(_problem(fmt=fmt, mask="flashmask", **kivi), T, page_indptr=np.array([0, 1, 2], np.int32),
                         num_sms=4)
    with pytest.raises(dattn.DattnError, match="flashmask on INT4 KIVI needs a power-of-two page_size") as e:
        dattn.dattn_plan(_problem(fmt="int4_kivi", mask="flashmask", P=96, **kivi), T,
                         page_indptr=np.array([0, 1, 2], np.int32), num_sms=4)
    assert dattn.STATUS[e.value.status] == "DATTN_EUNSUPPORTED"


def test_step_host_sizes_and_rejections_without_a_gpu():
    """dattn_step_host: the sizes query plans on the host; a workspace without room for the
    inputs, an index-list program and missing host arrays are rejected before any transfer."""
    rng = np.random.default_rng(3)
    T = rng.integers(1, 300, 3).tolist()
    pages = [-(-t // 16) for t in T]
    indptr = np.concatenate([[0], np.cumsum(pages)]).astype(np.int32)
    indices = rng.permutation(64)[:indptr[-1]].astype(np.int32)
    p = _problem(B=3, S_q=2, H_q=8, H_kv=2, num_pages=64)
    q = np.zeros((3, 2, 8, 128), np.uint16)
    o = np.zeros_like(q)
    io = dattn.host_step(q, T, o, page_indptr=indptr, page_indices=indices, num_sms=8)
    ws, sg = dattn.dattn_step_host_sizes(p, io)
    plan = dattn.dattn_plan(p, T, page_indptr=indptr, num_sms=8)
    rows = 3 * 2 * 8
    al = lambda x: -(-x // 256) * 256
    in_bytes = al(rows * 128 * 2) + al(4 * 4) + al(4 * int(indptr[-1]))
    assert ws == in_bytes + al(plan.workspace_bytes) + al(rows * 128 * 2) + al(rows * 4)
    assert sg == in_bytes + al(plan.info["blob_bytes"]) + al(rows * 128 * 2) + al(rows * 4)
    lib = dattn.load()
    prob = dattn.make_problem(p)
    cache = dattn.Tensors()
    fake = 1 << 20          # never dereferenced: a workspace without room for the inputs fails first
    st = lib.dattn_step_host(ctypes.byref(prob), ctypes.byref(io), ctypes.byref(cache), fake, sg, fake * 4,
                             in_bytes - 256, None)
    assert st == 3 and "workspace" in dattn.dattn_last_error()
    bad = dattn.make_problem(dict(p, mask="index_list"))
    assert lib.dattn_step_host_sizes(ctypes.byref(bad), ctypes.byref(io), ctypes.byref(ctypes.c_size_t()),
                                     ctypes.byref(ctypes.c_size_t())) == 2
    io2 = dattn.host_step(q, T, o, num_sms=8)       # paged without host page tables
    assert lib.dattn_step_host_sizes(ctypes.byref(prob), ctypes.byref(io2), ctypes.byref(ctypes.c_size_t()),
                                     ctypes.byref(ctypes.c_size_t())) == 1
    # the copy-stream submit wants its done event and every field of its copies
    cp = dattn.StepCopies(fake, fake, 0, fake)
    st = lib.dattn_step_host_submit_ex(ctypes.byref(prob), ctypes.byref(io), ctypes.byref(cache), fake, sg, fake * 4,
                                       ws, None, fake, ctypes.byref(cp))
    assert st == 1 and "copies" in dattn.dattn_last_error()
    st = lib.dattn_step_host_submit_ex(ctypes.byref(prob), ctypes.byref(io), ctypes.byref(cache), fake, sg, fake * 4,
                                       ws, None, None, None)
    assert st == 1 and "done_event" in dattn.dattn_last_error()


def test_packed_view_layout_validation():
    """The packed-row layout takes the index-list program (its position map) and bf16 rows only;
    kv_append does not write it."""
    base = _problem(B=2, H_q=8, H_kv=2, layout="packed", mask="index_list")
    T = [40, 30]
    lists = [np.arange(0, 40, 3), np.arange(1, 40, 5), np.arange(0, 30, 2), np.arange(3, 30, 7)]
    indptr = np.concatenate([[0], np.cumsum([len(x) for x in lists])]).astype(np.int32)
    lst = np.concatenate(lists).astype(np.int32)
    plan = dattn.dattn_plan(base, T, index_indptr=indptr, index_list=lst, num_sms=4)
    assert plan.info["stream_keys"] == len(lst)
    with pytest.raises(dattn.DattnError, match="index-list program"):
        dattn.dattn_plan(dict(base, mask="causal"), T, num_sms=4)
    with pytest.raises(dattn.DattnError, match="bf16 rows"):
        dattn.dattn_plan(dict(base, fmt="int8"), T, index_indptr=indptr, index_list=lst, num_sms=4)
    lib = dattn.load()
    prob = dattn.make_problem(base)
    st = lib.kv_append(ctypes.byref(prob), ctypes.byref(dattn.AppendInputs()), ctypes.byref(dattn.Tensors()),
                       None, None, None, 0, None)
    assert st != 0 and "packed view" in dattn.dattn_last_error()


@pytest.mark.parametrize("shift,status", [((float("nan"), -1.0, 1.0), "EINVAL"), ((0.0, 1.0, 1.0), "EINVAL"),
                                          ((0.0, -90.0, 1.0), "EINVAL"), ((0.0, -1.0, 50.0), "EINVAL"),
                                          ((float("inf"), -1.0, 1.0), "EINVAL")])
def test_shared_shift_guard_checked_before_any_device_work(shift, status):
    """The frame and guard fields of dattn_run_options reach the library (ctypes layout = C layout)
    and are checked before the workspace or the tensors are touched."""
    plan = dattn.dattn_plan(_problem(), [10, 20], num_sms=4)

    class Never:   # a workspace that would fault if it were ever used
        def data_ptr(self):
            return 16

        def numel(self):
            return plan.workspace_bytes

        def element_size(self):
            return 1

    with pytest.raises(dattn.DattnError, match=status):
        dattn.dattn_run_ex(plan, _problem(), dattn.Tensors(), Never(), shared_shift=shift, stream=0)


def test_shared_shift_needs_bf16_and_options_layout():
    plan = dattn.dattn_plan(_problem(), [10, 20], num_sms=4)
    ws = (ctypes.c_uint8 * 16)()

    class W:
        def data_ptr(self):
            return ctypes.addressof(ws)

        def numel(self):
            return plan.workspace_bytes

        def element_size(self):
            return 1

    with pytest.raises(dattn.DattnError, match="EUNSUPPORTED"):
        dattn.dattn_run_ex(plan, _problem(fmt="int8"), dattn.Tensors(), W(), shared_shift=(0.0, -1.0, 1.0), stream=0)
    # C layout: uint32 flags, void* events[3], float phi, lo, hi, uint32 wait_limit_us, void* trace
    assert dattn.RunOptions.shift_phi.offset == 32 and dattn.RunOptions.shift_hi.offset == 40
    assert dattn.RunOptions.wait_limit_us.offset == 44 and dattn.RunOptions.trace.offset == 48
    assert ctypes.sizeof(dattn.RunOptions) == 56
