"""Seeded synthetic inputs for split-KV decode attention.

This module only draws and lays out inputs: it holds none of the method's
arithmetic (no scores, softmax, merging, quantisation or masking).  Both the
CUDA path and the CPU oracle consume exactly the tensors it returns.

Recipe (shapes and distributions of the five workloads):

1. tiny contiguous decode (seed 0): B=1, S_q=1, H_q=8, H_kv=2, d=64, 256
   visible rows; Q, K, V ~ N(0,1) rounded to bf16; contiguous [B, T, H_kv, d]
   cache; 4 fixed splits.
2. paged ragged GQA decode (seed 1): B=16, S_q=1, H_q=32, H_kv=8, d=128;
   lengths uniform integers in [1024, 8192]; K, V ~ N(0,1) bf16 with 4
   distinct outlier channels per kv head (K only) scaled by 8; 16-token
   pages; the page list is the first sum(ceil(T_b/16)) entries of a random
   permutation of a 10,000-page pool, concatenated request by request.
3. long-context split-heavy decode (seed 2): B=4, H_q=64, H_kv=8, d=128;
   lengths {131072, 100003, 65537, 1}; 64-token pages; pool = exactly the
   pages needed, permuted; S_q = 1 or 4 (bottom-right causal rows).
4. retention programs (seed 3): B=8, S_q=1, H_q=32, H_kv=8, d=128, 32768
   stored rows each, 16-token pages.  (a) 4 sinks + 4096 recent rows.
   (b) per (request, kv head) sorted index lists of 2048 positions: sinks
   [0, 64), recent [F-512, F) and the top 1472 of [64, F-512) ranked by a
   Gumbel(0,1) draw per (request, kv head, position), G = -ln(-ln U).
5. quantized KV (seed 4): B=32, S_q=1, H_q=32, H_kv=8, d=128; lengths
   uniform in [2048, 32768]; K, V ~ N(0,1) bf16 with 4 K outlier channels
   per kv head scaled by 8; 16-token pages; the history is handed over as
   packed ragged bf16 rows for the cache writer (kv_append) to encode.
   KIVI INT4: K groups of 32 tokens, V groups of 32 channels; the residual
   length R = 160 = 128 + G of the group-closing loop keeps the residual in
   (128, 160] rows, so the 128 most recent tokens always stay bf16.

Everywhere: Q ~ N(0,1) bf16 of shape [B, S_q, H_q, d]; metadata (lengths,
permutations, outlier channels, index lists) is drawn on the CPU from
``torch.Generator`` seeded with the workload seed; K/V/Q values are drawn on
the requested device from a generator seeded with ``seed + 1000``.  Pool
pages that no request references and page rows past a request's length are
filled with NaN ("poison"), so a visibility leak shows up as NaN.
"""

from __future__ import annotations

from dataclasses import dataclass, field

import torch

NAN_BF16 = float("nan")

# KIVI residual length R of the quantized workload: the group-closing loop
# (close the oldest 32 rows while more than R are in bf16) then never leaves
# fewer than 129 bf16 rows, so the 128 most recent tokens are never quantized.
KIVI_RESIDUAL = 160


@dataclass
class Workload:
    name: str
    problem: dict
    q: torch.Tensor
    kv_len: torch.Tensor                      # int32 [B] on the CPU
    k: torch.Tensor = None                    # bf16 cache (paged pool or contiguous)
    v: torch.Tensor = None
    page_indptr: torch.Tensor = None          # int32 [B+1] CPU
    page_indices: torch.Tensor = None         # int32 CPU
    cache_batch_idx: torch.Tensor = None
    index_indptr: torch.Tensor = None         # int32 [B*H_kv+1] CPU
    index_list: torch.Tensor = None           # int32 CPU
    fm_intervals: torch.Tensor = None         # int32 [sum T_b, 4] CPU, FlashMask (UTS, UTE, LTS, LTE)
    qo_indptr: torch.Tensor = None            # int32 [B+1] CPU, mixed batch: q is [qo_indptr[B], H_q, d]
    rows_indptr: torch.Tensor = None          # packed ragged history (quantized workloads)
    k_rows: torch.Tensor = None
    v_rows: torch.Tensor = None
    meta: dict = field(default_factory=dict)


def _gens(seed: int, device):
    meta = torch.Generator().manual_seed(seed)
    vals = torch.Generator(device=device).manual_seed(seed + 1000)
    return meta, vals


def _normal_bf16(shape, gen, device, outliers=None):
    x = torch.randn(shape, generator=gen, device=device, dtype=torch.float32)
    if outliers is not None:
        # outliers: [H_kv, n] channel ids; the head axis is -3 for pools [.., H, P, d]
        # and -2 for rows [.., H, d]; callers pass ``outlier_axis``.
        head_axis, chans = outliers
        for h in range(chans.shape[0]):
            idx = [slice(None)] * x.dim()
            idx[head_axis] = h
            idx[-1] = chans[h].to(device)
            x[tuple(idx)] *= 8.0
    return x.to(torch.bfloat16)


def _outlier_channels(H_kv, d, meta):
    return torch.stack([torch.randperm(d, generator=meta)[:4] for _ in range(H_kv)])


def _page_tables(lens, P, pool_pages, meta):
    n_pages = [-(-int(T) // P) for T in lens]
    total = sum(n_pages)
    if pool_pages is None:
        pool_pages = total
    assert total <= pool_pages, "pool too small"
    perm = torch.randperm(pool_pages, generator=meta)
    indptr = torch.zeros(len(lens) + 1, dtype=torch.int32)
    indptr[1:] = torch.cumsum(torch.tensor(n_pages, dtype=torch.int64), 0).to(torch.int32)
    return indptr, perm[:total].to(torch.int32).contiguous(), pool_pages


def _poison_pool(pool, lens, indptr, indices, P):
    """NaN every unreferenced page and every row past a request's length."""
    used = torch.zeros(pool.shape[0], dtype=torch.bool)
    used[indices.long()] = True
    pool[(~used).nonzero().flatten().to(pool.device)] = NAN_BF16
    for b, T in enumerate(lens):
        T = int(T)
        n = int(indptr[b + 1] - indptr[b])
        if n and T % P:
            last = int(indices[int(indptr[b + 1]) - 1])
            pool[last, :, T % P:, :] = NAN_BF16


def paged_bf16(name, *, B, S_q, H_q, H_kv, d, lens, P, seed, device, pool_pages=None,
               outliers=False, mask="causal", **mask_args) -> Workload:
    """Paged HND bf16 pools [N_pages, H_kv, P, d] filled with N(0,1) history."""
    meta, vals = _gens(seed, device)
    lens = [int(t) for t in lens]
    indptr, indices, pool_pages = _page_tables(lens, P, pool_pages, meta)
    och = _outlier_channels(H_kv, d, meta) if outliers else None
    k = _normal_bf16((pool_pages, H_kv, P, d), vals, device, (-3, och) if outliers else None)
    v = _normal_bf16((pool_pages, H_kv, P, d), vals, device)
    q = _normal_bf16((B, S_q, H_q, d), vals, device)
    _poison_pool(k, lens, indptr, indices, P)
    _poison_pool(v, lens, indptr, indices, P)
    problem = dict(B=B, S_q=S_q, H_q=H_q, H_kv=H_kv, d=d, layout="paged", fmt="bf16", P=P,
                   num_pages=pool_pages, mask=mask, **mask_args)
    return Workload(name, problem, q, torch.tensor(lens, dtype=torch.int32), k=k, v=v,
                    page_indptr=indptr, page_indices=indices,
                    meta={"outlier_channels": och, "seed": seed})


def contiguous_bf16(name, *, B, S_q, H_q, H_kv, d, lens, T_cap, seed, device, B_cache=None,
                    cache_batch_idx=None, **extra) -> Workload:
    """Contiguous NHD cache [B_cache, T_cap, H_kv, d]; rows past each length are NaN."""
    meta, vals = _gens(seed, device)
    B_cache = B_cache or B
    k = _normal_bf16((B_cache, T_cap, H_kv, d), vals, device)
    v = _normal_bf16((B_cache, T_cap, H_kv, d), vals, device)
    q = _normal_bf16((B, S_q, H_q, d), vals, device)
    cbi = list(range(B)) if cache_batch_idx is None else list(cache_batch_idx)
    used = set()
    for b, T in enumerate(lens):
        k[cbi[b], int(T):] = NAN_BF16
        v[cbi[b], int(T):] = NAN_BF16
        used.add(cbi[b])
    for c in range(B_cache):
        if c not in used:
            k[c] = NAN_BF16
            v[c] = NAN_BF16
    problem = dict(B=B, S_q=S_q, H_q=H_q, H_kv=H_kv, d=d, layout="contig", fmt="bf16",
                   T_cap=T_cap, B_cache=B_cache, mask="causal", **extra)
    return Workload(name, problem, q, torch.tensor([int(t) for t in lens], dtype=torch.int32),
                    k=k, v=v,
                    cache_batch_idx=None if cache_batch_idx is None
                    else torch.tensor(cbi, dtype=torch.int32),
                    meta={"seed": seed})


def quantized_history(name, *, B, S_q, H_q, H_kv, d, lens, P, seed, device, fmt,
                      outliers=True, pool_pages=None) -> Workload:
    """Packed ragged bf16 history rows [sum T_b, H_kv, d] plus page tables for a cache writer."""
    meta, vals = _gens(seed, device)
    lens = [int(t) for t in lens]
    indptr, indices, pool_pages = _page_tables(lens, P, pool_pages, meta)
    och = _outlier_channels(H_kv, d, meta) if outliers else None
    n = sum(lens)
    k_rows = _normal_bf16((n, H_kv, d), vals, device, (-2, och) if outliers else None)
    v_rows = _normal_bf16((n, H_kv, d), vals, device)
    q = _normal_bf16((B, S_q, H_q, d), vals, device)
    rows_indptr = torch.zeros(B + 1, dtype=torch.int32)
    rows_indptr[1:] = torch.cumsum(torch.tensor(lens, dtype=torch.int64), 0).to(torch.int32)
    problem = dict(B=B, S_q=S_q, H_q=H_q, H_kv=H_kv, d=d, layout="paged", fmt=fmt, P=P,
                   num_pages=pool_pages, mask="causal", kivi_group=32, kivi_v_group=32,
                   kivi_residual=KIVI_RESIDUAL)
    meta_out = {"outlier_channels": och, "seed": seed}
    if fmt in ("fp8_e4m3", "fp8_e5m2"):
        # per-head scales from a calibration pass over the history: max |x| / largest finite (fp32)
        top = 448.0 if fmt == "fp8_e4m3" else 57344.0
        meta_out["k_scale"] = (k_rows.float().abs().amax(dim=(0, 2)) / top).cpu()
        meta_out["v_scale"] = (v_rows.float().abs().amax(dim=(0, 2)) / top).cpu()
    return Workload(name, problem, q, torch.tensor(lens, dtype=torch.int32),
                    page_indptr=indptr, page_indices=indices, rows_indptr=rows_indptr,
                    k_rows=k_rows, v_rows=v_rows, meta=meta_out)


def h2o_index_lists(lens, H_kv, budget, n_sink, n_recent, meta):
    """Per (request, kv head) sorted lists: sinks + recent + top-k by a Gumbel draw.

    The heavy part takes the ``budget - n_sink - n_recent`` positions of
    [n_sink, F - n_recent) with the largest G = -ln(-ln U), U ~ U(0,1) drawn per
    position (ties, of probability zero, go to the lower position).
    """
    lists, indptr = [], [0]
    for T in lens:
        T = int(T)
        for _ in range(H_kv):
            sink = torch.arange(0, min(n_sink, T))
            recent = torch.arange(max(min(n_sink, T), T - n_recent), T)
            lo, hi = min(n_sink, T), max(min(n_sink, T), T - n_recent)
            k = max(0, min(budget - len(sink) - len(recent), hi - lo))
            u = torch.rand(hi - lo, generator=meta, dtype=torch.float64).clamp_min(1e-300)
            g = -torch.log(-torch.log(u))
            heavy = lo + torch.topk(g, k, sorted=False).indices if k else torch.arange(0)
            lst = torch.sort(torch.cat([sink, heavy, recent]).unique()).values
            lists.append(lst.to(torch.int32))
            indptr.append(indptr[-1] + len(lst))
    return torch.tensor(indptr, dtype=torch.int32), torch.cat(lists).contiguous()


# ---- the five workloads ------------------------------------------------------

def tiny_contiguous(device="cpu"):
    return contiguous_bf16("tiny contiguous decode B=1 H_q=8 H_kv=2 d=64 S_k=256", B=1, S_q=1,
                           H_q=8, H_kv=2, d=64, lens=[256], T_cap=256, seed=0, device=device,
                           fixed_splits=4)


def paged_ragged_gqa(device="cpu", B=16, lo=1024, hi=8192, pool_pages=10000):
    meta = torch.Generator().manual_seed(1)
    lens = torch.randint(lo, hi + 1, (B,), generator=meta).tolist()
    return paged_bf16(f"paged ragged GQA decode B={B} H_q=32 H_kv=8 d=128 P=16 T~U[{lo},{hi}]",
                      B=B, S_q=1, H_q=32, H_kv=8, d=128, lens=lens, P=16, seed=1, device=device,
                      pool_pages=pool_pages, outliers=True)


def long_context(device="cpu", S_q=1, lens=(131072, 100003, 65537, 1)):
    return paged_bf16(f"long-context decode B=4 H_q=64 H_kv=8 d=128 P=64 S_q={S_q}", B=len(lens),
                      S_q=S_q, H_q=64, H_kv=8, d=128, lens=list(lens), P=64, seed=2, device=device)


def retention(device="cpu", program="sink_window", B=8, T=32768):
    lens = [T] * B
    if program == "sink_window":
        return paged_bf16(f"sink 4 + window 4096 B={B} T={T}", B=B, S_q=1, H_q=32, H_kv=8, d=128,
                          lens=lens, P=16, seed=3, device=device, mask="sink_window", n_sink=4,
                          window=4096)
    w = paged_bf16(f"H2O-style index lists 2048/kv-head B={B} T={T}", B=B, S_q=1, H_q=32, H_kv=8,
                   d=128, lens=lens, P=16, seed=3, device=device, mask="index_list")
    meta = torch.Generator().manual_seed(3 + 77)
    w.index_indptr, w.index_list = h2o_index_lists(lens, 8, 2048, 64, 512, meta)
    return w


def packed_view(w: Workload) -> Workload:
    """The retained rows of an index-list workload compacted into the ragged packed view
    (M5.4 §0x04C): slice b H_kv + h holds the (b, h) rows at its list positions, in list
    order, so the list doubles as the position map.  A gather of stored rows, nothing more."""
    p = w.problem
    P, H = p["P"], p["H_kv"]
    ind = w.index_indptr.long()
    pos = w.index_list.long()
    s = torch.repeat_interleave(torch.arange(len(ind) - 1), ind[1:] - ind[:-1])
    b, h = s // H, s % H
    pages = w.page_indices.long()[w.page_indptr.long()[b] + pos // P]
    dev = w.k.device
    idx = (pages.to(dev), h.to(dev), (pos % P).to(dev))
    k = w.k[idx].contiguous()
    v = w.v[idx].contiguous()
    problem = dict(p, layout="packed")
    problem.pop("num_pages", None)
    return Workload(w.name + " (packed view)", problem, w.q, w.kv_len, k=k, v=v,
                    index_indptr=w.index_indptr, index_list=w.index_list, meta=dict(w.meta))


def quantized(device="cpu", fmt="int8", B=32, lo=2048, hi=32768, S_q=1, d=128, P=16):
    """The quantized-cache workload; KIVI V channel groups are 32 wide, 16 at d = 64."""
    meta = torch.Generator().manual_seed(4)
    lens = torch.randint(lo, hi + 1, (B,), generator=meta).tolist()
    extra = (f" S_q={S_q}" if S_q != 1 else "") + (f" d={d}" if d != 128 else "") + (f" P={P}" if P != 16 else "")
    w = quantized_history(f"quantized KV ({fmt}) B={B} T~U[{lo},{hi}]{extra}", B=B, S_q=S_q, H_q=32,
                          H_kv=8, d=d, lens=lens, P=P, seed=4, device=device, fmt=fmt)
    w.problem["kivi_v_group"] = min(32, d // 4)
    return w


def _dfs_tree_intervals(S_q: int, gen) -> list:
    """A random speculation tree of S_q draft tokens in DFS order: the rows that see draft
    r form its subtree [r, e_r), so its column hides U = [0, r) and L = [e_r, S_q)."""
    parent = [-1] + [int(torch.randint(0, j, (1,), generator=gen)) for j in range(1, S_q)]
    children = [[] for _ in range(S_q)]
    for j in range(1, S_q):
        children[parent[j]].append(j)
    order, span = [], {}

    def visit(u):
        start = len(order)
        order.append(u)
        for c in children[u]:
            visit(c)
        span[u] = (start, len(order))
    visit(0)
    return [(0, span[u][0], span[u][1], S_q) for u in order]


def tree_verify(device="cpu", B=16, S_q=8, lo=1024, hi=8192, seed=5):
    """Speculative-tree verification: each request's stored keys are a prefix of lo..hi
    tokens followed by S_q draft tokens in DFS order; query row r is draft r and sees the
    whole prefix and its ancestors' drafts (FlashMask intervals, one set per request)."""
    meta = torch.Generator().manual_seed(seed)
    prefix = torch.randint(lo, hi + 1, (B,), generator=meta).tolist()
    lens = [t + S_q for t in prefix]
    w = paged_bf16(f"speculative tree verify B={B} S_q={S_q} H_q=32 H_kv=8 d=128 P=16 prefix~U[{lo},{hi}]",
                   B=B, S_q=S_q, H_q=32, H_kv=8, d=128, lens=lens, P=16, seed=seed, device=device)
    iv = []
    for b in range(B):
        iv += [(0, 0, 0, 0)] * prefix[b]
        iv += _dfs_tree_intervals(S_q, meta)
    w.problem = dict(w.problem, mask="flashmask")
    w.fm_intervals = torch.tensor(iv, dtype=torch.int32)
    return w


def mixed_batch(device="cpu", TC=None, B=16, lo=1024, hi=8192, S_q=8, seed=6, **mask_args):
    """One launch over requests in different phases: request b has T_b committed rows and
    C_b new query rows (prefill T_b = 0, append C_b > 1, decode C_b = 1, C_b = 0 idle),
    its C_b rows already staged in the cache (T_b + C_b stored rows) and its query rows
    packed at qo_indptr[b] .. qo_indptr[b+1] of a [qo_indptr[B], H_q, d] query.

    Default mix: 10 decode rows, 3 appends of 2..S_q rows, 2 prefills of S_q rows and one
    idle request, T_b ~ U[lo, hi] for the ones with history."""
    meta = torch.Generator().manual_seed(seed)
    if TC is None:
        T = torch.randint(lo, hi + 1, (B,), generator=meta).tolist()
        kinds = ["decode"] * (B - 6) + ["append"] * 3 + ["prefill"] * 2 + ["idle"]
        order = torch.randperm(B, generator=meta).tolist()
        TC = []
        for b in range(B):
            k = kinds[order[b]]
            if k == "decode":
                TC.append((T[b], 1))
            elif k == "append":
                TC.append((T[b], int(torch.randint(2, S_q + 1, (1,), generator=meta))))
            elif k == "prefill":
                TC.append((0, S_q))
            else:
                TC.append((T[b], 0))
    B = len(TC)
    S_q = max(max(C for _, C in TC), 1)
    lens = [t + c for t, c in TC]
    w = paged_bf16(f"mixed prefill/append/decode batch B={B} C_b<={S_q} H_q=32 H_kv=8 d=128 P=16",
                   B=B, S_q=S_q, H_q=32, H_kv=8, d=128, lens=lens, P=16, seed=seed, device=device,
                   **mask_args)
    qo = [0]
    for _, c in TC:
        qo.append(qo[-1] + c)
    w.qo_indptr = torch.tensor(qo, dtype=torch.int32)
    gen = torch.Generator(device=device).manual_seed(seed + 2000)
    w.q = _normal_bf16((qo[-1], 32, 128), gen, device)
    w.meta["TC"] = TC
    return w
