"""dattn_run_noalloc: the decode step on the library's static scratch array.

Some callers cannot allocate device memory at step time (an engine that
reserved all of HBM for its page pool, a loop that cannot take the device
synchronisation of cudaMalloc / cudaFree).  dattn_run_noalloc serves them
from a fixed array inside the library.  It runs the same plan and the same
kernels as dattn_run, so its outputs must equal dattn_run's bit for bit; the
tests check that over consecutive calls with different plans (one with the
fused merge, whose completion counters live in the shared array), so that
each call runs on whatever the previous one left there.  They also read the
array's device status word through dattn_noalloc_status after a page id
outside the pool was planted on the host.  The file name sorts last so that
the array is first used after every other test; the tests pass alone too.
"""

import numpy as np
import pytest
import torch

import split_kv_decode_flash_gb300 as dattn
import workloads as W
from tests import gpu_helpers as H


def _outputs(w, entry, fused_merge=False):
    p = w.problem
    plan = dattn.dattn_plan(p, w.kv_len, page_indptr=w.page_indptr, index_indptr=w.index_indptr,
                            index_list=w.index_list, fused_merge=fused_merge)
    assert bool(plan.info["fused_merge"]) == fused_merge
    o = torch.full((p["B"], p["S_q"], p["H_q"], p["d"]), float("nan"), dtype=torch.bfloat16, device="cuda")
    lse = torch.full((p["B"], p["S_q"], p["H_q"]), float("nan"), dtype=torch.float32, device="cuda")
    t = dattn.tensors_from(**H.device_tensors(w, o, lse))
    if entry == "noalloc":
        assert plan.workspace_bytes <= dattn.NOALLOC_SCRATCH_BYTES
        dattn.dattn_run_noalloc(plan, p, t)
        assert dattn.dattn_noalloc_status() == 0
    else:
        ws = torch.empty(max(256, plan.workspace_bytes), dtype=torch.uint8, device="cuda")
        dattn.dattn_run(plan, p, t, ws)
        assert dattn.dattn_device_status(ws) == 0
    torch.cuda.synchronize()
    return o.view(torch.int16).cpu().numpy(), lse.cpu().numpy()


def _identical(got, want):
    (og, lg), (ow, lw) = got, want
    assert np.array_equal(og, ow), "O differs from dattn_run"
    assert np.array_equal(lg.view(np.int32), lw.view(np.int32)), "LSE differs from dattn_run"


@pytest.mark.gpu
def test_noalloc_matches_dattn_run_on_consecutive_calls():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    dattn.load()
    big = W.paged_ragged_gqa("cuda")                                   # B=16, 32/8 heads, d=128, 16-token pages
    small = W.retention("cuda", program="sink_window", B=3, T=5000)
    for w, fused in ((big, False), (small, False), (big, True), (small, True), (big, False)):
        _identical(_outputs(w, "noalloc", fused), _outputs(w, "run", fused))


@pytest.mark.gpu
def test_noalloc_status_reports_a_page_outside_the_pool():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    dattn.load()
    w = W.paged_ragged_gqa("cuda", B=3, lo=40, hi=300, pool_pages=64)
    p = w.problem
    plan = dattn.dattn_plan(p, w.kv_len, page_indptr=w.page_indptr)
    o = torch.zeros((p["B"], 1, p["H_q"], p["d"]), dtype=torch.bfloat16, device="cuda")
    lse = torch.zeros((p["B"], 1, p["H_q"]), dtype=torch.float32, device="cuda")
    kw = H.device_tensors(w, o, lse)
    bad = kw["page_indices"].clone()
    bad[1] = p["num_pages"] + 5                 # request 0's second page: outside the pool
    dattn.dattn_run_noalloc(plan, p, dattn.tensors_from(**dict(kw, page_indices=bad)))
    assert dattn.dattn_noalloc_status() & 1      # page id outside [0, num_pages)
    dattn.dattn_run_noalloc(plan, p, dattn.tensors_from(**kw))
    assert dattn.dattn_noalloc_status() == 0     # each call starts from a zeroed word


def test_noalloc_rejects_a_plan_larger_than_the_scratch_without_a_gpu():
    """The size check runs on the host before any CUDA call."""
    prob = dict(B=64, S_q=1, H_q=32, H_kv=8, d=128, layout="paged", fmt="bf16", P=16, num_pages=40000,
                mask="causal", fixed_splits=64)
    plan = dattn.dattn_plan(prob, [8192] * 64, num_sms=152)
    assert plan.workspace_bytes > dattn.NOALLOC_SCRATCH_BYTES
    with pytest.raises(dattn.DattnError) as e:
        dattn.dattn_run_noalloc(plan, prob, dattn.Tensors(), stream=0)
    assert dattn.STATUS[e.value.status] == "DATTN_EWORKSPACE"
    assert "static scratch" in str(e.value)
