"""GPU tests of kv_append against the oracle's own cache writer (M8.6 §0x05B, §0x06A-B).

Codes and qparams are compared bit for bit: both sides compute the range in
fp32 (exact), the scale with a correctly rounded fp32 divide, round to fp16
with ties to even, and encode with the re-read stored values.  The history
is appended in several uneven calls (one-row appends included) so that KIVI
groups close across call boundaries and the residual ring wraps.
"""

import numpy as np
import pytest
import torch

import split_kv_decode_flash_gb300 as dattn
import workloads as W
from oracle import cache as ocache
from oracle import quant
from tests.gpu_helpers import bits

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    dattn.load()


def _alloc(fmt, p, n_pages, B, dev="cuda", scales=None):
    H, P, d = p["H_kv"], p["P"], p["d"]
    G, Gv, R = p["kivi_group"], p["kivi_v_group"], p["kivi_residual"]
    out = {}
    if fmt == "bf16":
        out["k"] = torch.zeros((n_pages, H, P, d), dtype=torch.bfloat16, device=dev)
        out["v"] = torch.zeros_like(out["k"])
    elif fmt in ("int8", "int4_head"):
        row = d if fmt == "int8" else d // 2
        out["k"] = torch.zeros((n_pages, H, P, row), dtype=torch.uint8, device=dev)
        out["v"] = torch.zeros_like(out["k"])
        out["k_qparams"] = torch.zeros((n_pages, H, P, 2), dtype=torch.float16, device=dev)
        out["v_qparams"] = torch.zeros_like(out["k_qparams"])
    elif fmt in ("fp8_e4m3", "fp8_e5m2"):
        out["k"] = torch.zeros((n_pages, H, P, d), dtype=torch.uint8, device=dev)
        out["v"] = torch.zeros_like(out["k"])
        if scales is not None:
            out["k_qparams"] = scales[0].to(dev, torch.float32).contiguous()
            out["v_qparams"] = scales[1].to(dev, torch.float32).contiguous()
    else:
        out["k"] = torch.zeros((n_pages, H, P, d // 2), dtype=torch.uint8, device=dev)
        out["v"] = torch.zeros_like(out["k"])
        out["k_qparams"] = torch.zeros((n_pages, H, max(1, P // G), d, 2), dtype=torch.float16, device=dev)
        out["v_qparams"] = torch.zeros((n_pages, H, P, d // Gv, 2), dtype=torch.float16, device=dev)
        out["k_residual"] = torch.zeros((B, R, H, d), dtype=torch.bfloat16, device=dev)
        out["v_residual"] = torch.zeros_like(out["k_residual"])
    return out


def append_history(w, fmt, cuts_per_request):
    """kv_append the workload's packed history in pieces; returns the device cache dict."""
    p = dict(w.problem, fmt=fmt)
    B = p["B"]
    scales = (w.meta["k_scale"], w.meta["v_scale"]) if fmt.startswith("fp8") and "k_scale" in w.meta else None
    cache = _alloc(fmt, p, p["num_pages"], B, scales=scales)
    cache["page_indptr"] = w.page_indptr.cuda()
    cache["page_indices"] = w.page_indices.cuda()
    ws = torch.empty(dattn.kv_append_workspace_bytes(p), dtype=torch.uint8, device="cuda")
    lens = w.kv_len.tolist()
    ri = w.rows_indptr.tolist()
    done = [0] * B
    n_calls = max(len(c) for c in cuts_per_request)
    for c in range(n_calls + 1):
        new_idx, new_ptr = [], [0]
        for b in range(B):
            cuts = cuts_per_request[b]
            upto = cuts[c] if c < len(cuts) else lens[b]
            upto = min(max(upto, done[b]), lens[b])
            new_idx.append(torch.arange(ri[b] + done[b], ri[b] + upto))
            new_ptr.append(new_ptr[-1] + upto - done[b])
        idx = torch.cat(new_idx).long().to(w.k_rows.device)
        k_new = w.k_rows.index_select(0, idx).contiguous()
        v_new = w.v_rows.index_select(0, idx).contiguous()
        t = dattn.tensors_from(**cache)
        dattn.kv_append(p, t, k_new if k_new.numel() else None, v_new if v_new.numel() else None,
                        done, new_ptr, w.page_indptr, ws)
        for b in range(B):
            done[b] += new_ptr[b + 1] - new_ptr[b]
    torch.cuda.synchronize()
    assert done == lens
    assert int(ws[:4].view(torch.int32).item()) == 0, "kv_append device check fired"
    return p, cache


def fp8_scales(w):
    """The FP8 per-head scales the workload's cache uses (None: 1, no calibration)."""
    if "k_scale" not in w.meta:
        return None, None
    return w.meta["k_scale"].numpy(), w.meta["v_scale"].numpy()


def oracle_written(w, fmt):
    p = w.problem
    ks, vs = fp8_scales(w)
    c = ocache.empty_paged(fmt, p["num_pages"], p["H_kv"], p["P"], p["d"], p["B"], G=p["kivi_group"],
                           Gv=p["kivi_v_group"], R=p["kivi_residual"], k_scale=ks, v_scale=vs)
    ocache.write_history(c, w.page_indptr.numpy(), w.page_indices.numpy(), w.rows_indptr.numpy(),
                         bits(w.k_rows), bits(w.v_rows))
    return c


def _visible_rows(w):
    """(page, row) pairs of every stored token, per request."""
    P = w.problem["P"]
    out = []
    ind, ptr = w.page_indices.numpy(), w.page_indptr.numpy()
    for b, T in enumerate(w.kv_len.tolist()):
        t = np.arange(T)
        out.append((b, t, ind[ptr[b] + t // P], t % P))
    return out


def _cuts(lens, rng):
    cuts = []
    for T in lens:
        pts = sorted(set(rng.integers(0, T + 1, size=4).tolist()))
        if T > 130:
            pts += [128, 129, 160, 161]          # residual boundary and one-row appends
        cuts.append(sorted(set(min(x, T) for x in pts)))
    return cuts


def test_bf16_append_matches_oracle_writer():
    w = W.quantized_history("bf16", B=3, S_q=1, H_q=8, H_kv=2, d=128, lens=[300, 17, 161], P=16, seed=11,
                            device="cuda", fmt="bf16", pool_pages=60)
    p, cache = append_history(w, "bf16", _cuts(w.kv_len.tolist(), np.random.default_rng(0)))
    ref = oracle_written(w, "bf16")
    k, v = bits(cache["k"]), bits(cache["v"])
    for b, t, pg, r in _visible_rows(w):
        assert np.array_equal(k[pg, :, r], ref.k[pg, :, r]) and np.array_equal(v[pg, :, r], ref.v[pg, :, r])


@pytest.mark.parametrize("d", [128, 64])
def test_int8_append_codes_and_qparams_bit_exact(d):
    w = W.quantized_history("int8", B=3, S_q=1, H_q=8, H_kv=2, d=d, lens=[333, 1, 96], P=16, seed=12,
                            device="cuda", fmt="int8", pool_pages=40)
    p, cache = append_history(w, "int8", _cuts(w.kv_len.tolist(), np.random.default_rng(1)))
    ref = oracle_written(w, "int8")
    kc, vc = cache["k"].cpu().numpy(), cache["v"].cpu().numpy()
    kq, vq = cache["k_qparams"].cpu().numpy(), cache["v_qparams"].cpu().numpy()
    for b, t, pg, r in _visible_rows(w):
        assert np.array_equal(kq[pg, :, r], ref.k_qp[pg, :, r])
        assert np.array_equal(vq[pg, :, r], ref.v_qp[pg, :, r])
        assert np.array_equal(kc[pg, :, r], ref.k[pg, :, r])
        assert np.array_equal(vc[pg, :, r], ref.v[pg, :, r])


@pytest.mark.parametrize("d", [128, 64])
def test_int4_head_append_codes_and_qparams_bit_exact(d):
    """Per-head INT4 (M8.6 §0x09C): (s, o) and packed codes bit for bit, with heads that
    are constant, positive-only (offset below -15) and of tiny range mixed in."""
    w = W.quantized_history("int4h", B=3, S_q=1, H_q=8, H_kv=2, d=d, lens=[333, 1, 96], P=16, seed=16,
                            device="cuda", fmt="int4_head", pool_pages=40)
    k = w.k_rows.clone()
    k[5] = 0.75                                    # constant rows
    k[6] = (k[6].float().abs() * 0.05 + 3.0).to(torch.bfloat16)   # positive-only rows: offset below -15
    k[7] = (1.0 + k[7].float() * 2.0 ** -12).to(torch.bfloat16)   # range below 15 * 2^-14
    w.k_rows = k.contiguous()
    p, cache = append_history(w, "int4_head", _cuts(w.kv_len.tolist(), np.random.default_rng(4)))
    ref = oracle_written(w, "int4_head")
    kc, vc = cache["k"].cpu().numpy(), cache["v"].cpu().numpy()
    kq, vq = cache["k_qparams"].cpu().numpy(), cache["v_qparams"].cpu().numpy()
    for b, t, pg, r in _visible_rows(w):
        assert np.array_equal(kq[pg, :, r].view(np.uint16), ref.k_qp[pg, :, r].view(np.uint16))
        assert np.array_equal(vq[pg, :, r].view(np.uint16), ref.v_qp[pg, :, r].view(np.uint16))
        assert np.array_equal(kc[pg, :, r], ref.k[pg, :, r])
        assert np.array_equal(vc[pg, :, r], ref.v[pg, :, r])
    assert np.any(ref.k_qp[..., 1].astype(np.float32) < -15)


@pytest.mark.parametrize("fmt", ["fp8_e4m3", "fp8_e5m2"])
@pytest.mark.parametrize("d,scales", [(128, "calibrated"), (64, "calibrated"), (128, "none"), (128, "tight")])
def test_fp8_append_codes_bit_exact(fmt, d, scales):
    """FP8 codes of x / s_h: calibrated scales, no scales (1), and scales a quarter of the
    calibrated ones, so that a quarter of the range saturates to the largest finite value."""
    w = W.quantized_history("fp8", B=3, S_q=1, H_q=8, H_kv=2, d=d, lens=[333, 1, 96], P=16, seed=15,
                            device="cuda", fmt=fmt, pool_pages=40)
    if scales == "none":
        del w.meta["k_scale"], w.meta["v_scale"]
    elif scales == "tight":
        w.meta["k_scale"] = w.meta["k_scale"] / 4
        w.meta["v_scale"] = w.meta["v_scale"] / 4
    p, cache = append_history(w, fmt, _cuts(w.kv_len.tolist(), np.random.default_rng(3)))
    ref = oracle_written(w, fmt)
    top = 0x7E if fmt == "fp8_e4m3" else 0x7B
    kc, vc = cache["k"].cpu().numpy(), cache["v"].cpu().numpy()
    n_sat = 0
    for b, t, pg, r in _visible_rows(w):
        assert np.array_equal(kc[pg, :, r], ref.k[pg, :, r])
        assert np.array_equal(vc[pg, :, r], ref.v[pg, :, r])
        n_sat += int(np.sum((kc[pg, :, r] & 0x7F) == top))
    # calibrated: only each head's largest |x| meets 448; tight: a quarter of the range saturates
    assert n_sat >= 100 if scales == "tight" else n_sat < 20


@pytest.mark.parametrize("d,P", [(128, 16), (64, 16), (128, 64)])
def test_kivi_append_groups_residual_bit_exact(d, P):
    lens = [700, 129, 128, 161, 40]
    w = W.quantized_history("kivi", B=len(lens), S_q=1, H_q=8, H_kv=2, d=d, lens=lens, P=P, seed=13,
                            device="cuda", fmt="int4_kivi",
                            pool_pages=sum(-(-t // P) for t in lens) + 3)
    w.problem["kivi_v_group"] = min(32, d // 4)
    p, cache = append_history(w, "int4_kivi", _cuts(lens, np.random.default_rng(2)))
    ref = oracle_written(w, "int4_kivi")
    got = {n: cache[n].cpu() for n in ("k", "v", "k_qparams", "v_qparams")}
    kres, vres = bits(cache["k_residual"]), bits(cache["v_residual"])
    G, R = p["kivi_group"], p["kivi_residual"]
    assert R == 160
    for b, t, pg, r in _visible_rows(w):
        T = len(t)
        n_q = quant.kivi_quantized_prefix(T, G, R)
        old = t < n_q
        assert np.array_equal(got["k"].numpy()[pg[old], :, r[old]], ref.k[pg[old], :, r[old]])
        assert np.array_equal(got["v"].numpy()[pg[old], :, r[old]], ref.v[pg[old], :, r[old]])
        assert np.array_equal(got["v_qparams"].numpy()[pg[old], :, r[old]], ref.v_qp[pg[old], :, r[old]])
        for g0 in range(0, n_q, G):
            qpg = pg[g0]
            slot = (g0 % P) // G if P >= G else 0
            assert np.array_equal(got["k_qparams"].numpy()[qpg, :, slot], ref.k_qp[qpg, :, slot])
        new = ~old
        slots = t[new] % R
        assert np.array_equal(kres[b, slots], ref.k_res[b, slots])
        assert np.array_equal(vres[b, slots], ref.v_res[b, slots])


def test_append_rejects_capacity_overflow_before_writing():
    w = W.quantized_history("cap", B=2, S_q=1, H_q=8, H_kv=2, d=128, lens=[20, 20], P=16, seed=14,
                            device="cuda", fmt="bf16", pool_pages=4)
    p = dict(w.problem)
    cache = _alloc("bf16", p, 4, 2)
    cache["page_indptr"] = w.page_indptr.cuda()
    cache["page_indices"] = w.page_indices.cuda()
    ws = torch.empty(dattn.kv_append_workspace_bytes(p), dtype=torch.uint8, device="cuda")
    k_new = w.k_rows[:26].contiguous()
    with pytest.raises(dattn.DattnError, match="append needs 33"):
        dattn.kv_append(p, dattn.tensors_from(**cache), k_new, k_new, [20, 0], [0, 13, 26], w.page_indptr, ws)
    torch.cuda.synchronize()
    assert not cache["k"].float().abs().sum().item(), "rejected append must not write"


@pytest.mark.parametrize("fmt", ["int8", "int4_head", "int4_kivi"])
def test_full_size_quantized_append_sampled(fmt):
    """The quantized workload (B=32, T ~ U[2048, 32768]) written in one call; sampled rows checked."""
    w = W.quantized("cuda", fmt=fmt)
    p, cache = append_history(w, fmt, [[] for _ in range(w.problem["B"])])
    rng = np.random.default_rng(5)
    P, G = p["P"], 32
    ind, ptr = w.page_indices.numpy(), w.page_indptr.numpy()
    kc = cache["k"]
    for b in rng.choice(p["B"], size=6, replace=False):
        T = int(w.kv_len[b])
        row0 = int(w.rows_indptr[b])
        if fmt in ("int8", "int4_head"):
            ts = rng.choice(T, size=64, replace=False)
            x = quant.bf16_bits_to_f32(bits(w.k_rows[row0 + torch.as_tensor(ts)]))
            codes, s, z = quant.int8_token_quantize(x) if fmt == "int8" else quant.int4_head_quantize(x)
            pg = ind[ptr[b] + ts // P]
            got = kc[torch.as_tensor(pg), :, torch.as_tensor(ts % P)].cpu().numpy()
            if fmt == "int4_head":
                got = quant.unpack_int4(got)
            gq = cache["k_qparams"][torch.as_tensor(pg), :, torch.as_tensor(ts % P)].cpu().numpy()
            assert np.array_equal(got, codes)
            assert np.array_equal(gq[..., 0], s) and np.array_equal(gq[..., 1], z)
        else:
            n_q = quant.kivi_quantized_prefix(T, G, p["kivi_residual"])
            for g0 in rng.choice(np.arange(0, n_q, G), size=4, replace=False):
                x = quant.bf16_bits_to_f32(bits(w.k_rows[row0 + g0: row0 + g0 + G]))   # [G, H, d]
                codes, s, z = quant.kivi_k_group_quantize(x.transpose(1, 0, 2))
                ts = np.arange(g0, g0 + G)
                pg = ind[ptr[b] + ts // P]
                got = quant.unpack_int4(kc[torch.as_tensor(pg), :, torch.as_tensor(ts % P)].cpu().numpy())
                assert np.array_equal(got, codes.transpose(1, 0, 2))
                gq = cache["k_qparams"][int(pg[0]), :, 0].cpu().numpy()
                assert np.array_equal(gq[..., 0], s) and np.array_equal(gq[..., 1], z)
