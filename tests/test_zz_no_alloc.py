"""dattn_run_noalloc: the decode step on the library's static scratch array.

Its outputs are checked against dattn_run (caller-owned workspace) on the
same inputs, within the decode tolerance, over consecutive calls with
different plans, so that each call runs on whatever the previous one left in
the shared array.  The file name sorts last so that the array is first used
after every other test; the GPU test passes alone as well.
"""

import numpy as np
import pytest
import torch

import split_kv_decode_flash_gb300 as dattn
import workloads as W
from tests import gpu_helpers as H


def _outputs(w, entry):
    p = w.problem
    plan = dattn.dattn_plan(p, w.kv_len, page_indptr=w.page_indptr, index_indptr=w.index_indptr,
                            index_list=w.index_list)
    o = torch.full((p["B"], p["S_q"], p["H_q"], p["d"]), float("nan"), dtype=torch.bfloat16, device="cuda")
    lse = torch.full((p["B"], p["S_q"], p["H_q"]), float("nan"), dtype=torch.float32, device="cuda")
    t = dattn.tensors_from(**H.device_tensors(w, o, lse))
    if entry == "noalloc":
        assert plan.workspace_bytes <= dattn.NOALLOC_SCRATCH_BYTES
        dattn.dattn_run_noalloc(plan, p, t)
    else:
        ws = torch.empty(max(256, plan.workspace_bytes), dtype=torch.uint8, device="cuda")
        dattn.dattn_run(plan, p, t, ws)
    torch.cuda.synchronize()
    return o.float().cpu().numpy().astype(np.float64), lse.cpu().numpy().astype(np.float64)


def _agree(got, want):
    (og, lg), (ow, lw) = got, want
    masked = np.isneginf(lw)
    assert np.array_equal(np.isneginf(lg), masked)
    assert not og[masked].any()
    assert np.isfinite(og).all() and np.isfinite(lg[~masked]).all()
    assert (np.abs(og - ow) <= H.O_ATOL + H.O_RTOL * np.abs(ow)).all()
    fin = ~masked
    assert (np.abs(lg[fin] - lw[fin]) <= H.LSE_RTOL * np.maximum(1.0, np.abs(lw[fin]))).all()


@pytest.mark.gpu
def test_noalloc_matches_dattn_run_on_consecutive_calls():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    dattn.load()
    big = W.paged_ragged_gqa("cuda")                                   # B=16, 32/8 heads, d=128, 16-token pages
    small = W.retention("cuda", program="sink_window", B=3, T=5000)
    for w in (big, small, big):
        _agree(_outputs(w, "noalloc"), _outputs(w, "run"))


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
