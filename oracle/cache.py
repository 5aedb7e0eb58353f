"""The oracle's own K/V cache writer and reader (page walk + dequantisation).

Test infrastructure only (see ``oracle/__init__.py``).

The memory layout is the documented cache ABI of the library; everything
here is re-derived from it with the formulas of "M4.5 Decode Attention
Kernels, Mask Programs, and Backend Boundaries" §0x04B-§0x04F and the formats
of ``oracle.quant``.  No code is shared with the CUDA side.

Layouts (element order, outermost first):

* contiguous NHD bf16:   K, V [B_c, T_c, H_kv, d]; request b reads cache row
  c = cache_batch_idx[b] (identity when absent)                       (§0x04B)
* paged HND bf16:        K, V [N_pages, H_kv, P, d]; request b's logical block
  j lives in page indices[indptr[b] + j]                               (§0x04D)
* paged INT8:            codes [N_pages, H_kv, P, d] uint8;
                         qparams [N_pages, H_kv, P, 2] fp16 (s, z)
* paged FP8 E4M3 / E5M2: codes [N_pages, H_kv, P, d] uint8; per-head scales
                         k_qp, v_qp [H_kv] fp32 (1 when not calibrated)
* packed rows (bf16):    K, V [R_total, d]; the retained rows of slice s = b H_kv + h
                         are rows row_offsets[s] .. row_offsets[s+1]-1, row r holding
                         the source row at original position position_map[r]
                         (M5.4 §0x04C ragged packed view: a gather, not a re-encoding)
* paged INT4 per head:   codes [N_pages, H_kv, P, d/2] uint8 (packed);
                         qparams [N_pages, H_kv, P, 2] fp16 (s, o), one per
                         (token, kv head); x_hat = (code - o) * s
* paged INT4 KIVI:       codes [N_pages, H_kv, P, d/2] uint8 (packed);
                         K qparams [N_pages, H_kv, max(1, P/G), d, 2] fp16 held
                         by the page of the group's first token;
                         V qparams [N_pages, H_kv, P, d/Gv, 2] fp16;
                         residual K, V [B, R, H_kv, d] bf16, token t in slot
                         t mod R; tokens t >= n_q(T_b) are read from it.
"""

from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

from . import address, quant


@dataclass
class Cache:
    layout: str            # "contig" | "paged" | "packed"
    fmt: str               # "bf16" | "int8" | "fp8_e4m3" | "fp8_e5m2" | "int4_head" | "int4_kivi"
    H_kv: int
    d: int
    P: int = 0
    T_c: int = 0
    k: np.ndarray = None   # bf16 bits (uint16) or codes (uint8)
    v: np.ndarray = None
    k_qp: np.ndarray = None
    v_qp: np.ndarray = None
    k_res: np.ndarray = None
    v_res: np.ndarray = None
    page_indptr: np.ndarray = None
    page_indices: np.ndarray = None
    cache_batch_idx: np.ndarray = None
    kv_len: np.ndarray = None
    G: int = 32
    Gv: int = 32
    R: int = 128
    extra: dict = field(default_factory=dict)


def _pages_and_rows(cache: Cache, b: int, positions: np.ndarray):
    """Physical page and page row of each logical position (§0x04D), checked (§0x04F, §0x04H)."""
    P = cache.P
    j = positions // P
    n_pages = cache.page_indptr[b + 1] - cache.page_indptr[b]
    if positions.size and (positions.min() < 0 or positions.max() >= cache.kv_len[b]):
        raise IndexError("visibility invariant: 0 <= t < context_length")
    if positions.size and j.max() >= n_pages:
        raise IndexError("logical block beyond the request's page list")
    pages = cache.page_indices[cache.page_indptr[b] + j]
    return pages, positions % P


def read_rows(cache: Cache, b: int, h_kv: int, positions) -> tuple[np.ndarray, np.ndarray]:
    """Dequantised K_hat, V_hat [n, d] (float64) of request b, kv head h_kv, at ``positions``."""
    pos = np.asarray(positions, dtype=np.int64)
    if cache.layout == "packed":
        r = packed_rows(cache, b, h_kv, pos)
        return quant.bf16_bits_to_f64(cache.k[r]), quant.bf16_bits_to_f64(cache.v[r])
    if cache.layout == "contig":
        c = b if cache.cache_batch_idx is None else int(cache.cache_batch_idx[b])
        if pos.size and (pos.min() < 0 or pos.max() >= cache.kv_len[b]):
            raise IndexError("visibility invariant: 0 <= t < context_length")
        k = quant.bf16_bits_to_f64(cache.k[c, pos, h_kv, :])
        v = quant.bf16_bits_to_f64(cache.v[c, pos, h_kv, :])
        return k, v
    pages, rows = _pages_and_rows(cache, b, pos)
    if cache.fmt == "bf16":
        return (quant.bf16_bits_to_f64(cache.k[pages, h_kv, rows, :]),
                quant.bf16_bits_to_f64(cache.v[pages, h_kv, rows, :]))
    if cache.fmt == "int8":
        kq = cache.k_qp[pages, h_kv, rows]          # [n, 2] fp16
        vq = cache.v_qp[pages, h_kv, rows]
        k = cache.k[pages, h_kv, rows, :].astype(np.float64) * kq[:, 0:1].astype(np.float64) \
            + kq[:, 1:2].astype(np.float64)
        v = cache.v[pages, h_kv, rows, :].astype(np.float64) * vq[:, 0:1].astype(np.float64) \
            + vq[:, 1:2].astype(np.float64)
        return k, v
    if cache.fmt == "int4_head":
        kq = cache.k_qp[pages, h_kv, rows]          # [n, 2] fp16 (s, o)
        vq = cache.v_qp[pages, h_kv, rows]
        return (quant.int4_head_decode(quant.unpack_int4(cache.k[pages, h_kv, rows, :]), kq[:, 0], kq[:, 1]),
                quant.int4_head_decode(quant.unpack_int4(cache.v[pages, h_kv, rows, :]), vq[:, 0], vq[:, 1]))
    if cache.fmt in quant.FP8_FORMATS:
        return (quant.fp8_head_decode(cache.k[pages, h_kv, rows, :], cache.k_qp[h_kv], cache.fmt),
                quant.fp8_head_decode(cache.v[pages, h_kv, rows, :], cache.v_qp[h_kv], cache.fmt))
    if cache.fmt == "int4_kivi":
        n_q = quant.kivi_quantized_prefix(int(cache.kv_len[b]), cache.G, cache.R)
        k = np.zeros((pos.size, cache.d))
        v = np.zeros((pos.size, cache.d))
        old = pos < n_q
        if old.any():
            po, ro = pages[old], rows[old]
            t = pos[old]
            kc = quant.unpack_int4(cache.k[po, h_kv, ro, :])
            vc = quant.unpack_int4(cache.v[po, h_kv, ro, :])
            # K: the group's qparams live on the page of its first token.
            g0 = (t // cache.G) * cache.G
            qpage, _ = _pages_and_rows(cache, b, g0)
            qslot = (g0 % cache.P) // cache.G if cache.P >= cache.G else np.zeros_like(g0)
            kqp = cache.k_qp[qpage, h_kv, qslot]                       # [n, d, 2]
            k[old] = kc * kqp[..., 0].astype(np.float64) + kqp[..., 1].astype(np.float64)
            vqp = cache.v_qp[po, h_kv, ro]                              # [n, d/Gv, 2]
            vs = np.repeat(vqp[..., 0].astype(np.float64), cache.Gv, axis=1)
            vz = np.repeat(vqp[..., 1].astype(np.float64), cache.Gv, axis=1)
            v[old] = vc * vs + vz
        new = ~old
        if new.any():
            slot = pos[new] % cache.R
            k[new] = quant.bf16_bits_to_f64(cache.k_res[b, slot, h_kv, :])
            v[new] = quant.bf16_bits_to_f64(cache.v_res[b, slot, h_kv, :])
        return k, v
    raise ValueError(cache.fmt)


# ---- ragged packed view (M5.4 §0x04C) -----------------------------------------

def pack_view(k_slices, v_slices, position_sets):
    """Packs the rows of each slice at its ordered position set: packed row r of slice s is
    the source row at position_map[r] (M5.4 §0x04C).  k_slices[s] / v_slices[s] are the
    slice's source rows [T_s, d] (any dtype, copied as is); position_sets[s] its positions.

    Returns packed K [R_total, d], packed V, position_map [R_total], row_offsets [S + 1]
    (independent global offsets: monotonic, the last one R_total)."""
    offsets = [0]
    pmap, ks, vs = [], [], []
    for ksrc, vsrc, pos in zip(k_slices, v_slices, position_sets):
        pos = np.asarray(pos, dtype=np.int64)
        if pos.size and (np.any(np.diff(pos) <= 0) or pos[0] < 0 or pos[-1] >= len(ksrc)):
            raise ValueError("a position set must be strictly increasing and inside its source")
        ks.append(np.asarray(ksrc)[pos])
        vs.append(np.asarray(vsrc)[pos])
        pmap.append(pos)
        offsets.append(offsets[-1] + len(pos))
    d = np.asarray(k_slices[0]).shape[-1]
    dt = np.asarray(k_slices[0]).dtype
    K = np.concatenate(ks) if ks else np.zeros((0, d), dt)
    V = np.concatenate(vs) if vs else np.zeros((0, d), dt)
    return K, V, np.concatenate(pmap).astype(np.int64), np.asarray(offsets, np.int64)


def packed_rows(cache: Cache, b: int, h_kv: int, positions) -> np.ndarray:
    """Packed rows of slice (b, h_kv) holding the given original positions (each must be one
    of the slice's retained positions; the packed row is a storage coordinate only)."""
    s = b * cache.H_kv + h_kv
    lo, hi = int(cache.extra["row_offsets"][s]), int(cache.extra["row_offsets"][s + 1])
    pm = np.asarray(cache.extra["position_map"][lo:hi], dtype=np.int64)
    pos = np.asarray(positions, dtype=np.int64)
    idx = np.searchsorted(pm, pos)
    if pos.size and (np.any(idx >= len(pm)) or np.any(pm[np.minimum(idx, len(pm) - 1)] != pos)):
        raise IndexError("position not retained in the packed slice")
    return lo + idx


# ---- writers: the oracle's own construction of a paged cache ------------------

def empty_paged(fmt: str, n_pages: int, H_kv: int, P: int, d: int, B: int,
                G: int = 32, Gv: int = 32, R: int = 128, k_scale=None, v_scale=None) -> Cache:
    """Zero-filled pools of the documented shapes (FP8: with its per-head scales, 1 when None)."""
    c = Cache("paged", fmt, H_kv, d, P=P, G=G, Gv=Gv, R=R)
    if fmt == "bf16":
        c.k = np.zeros((n_pages, H_kv, P, d), np.uint16)
        c.v = np.zeros_like(c.k)
    elif fmt == "int8":
        c.k = np.zeros((n_pages, H_kv, P, d), np.uint8)
        c.v = np.zeros_like(c.k)
        c.k_qp = np.zeros((n_pages, H_kv, P, 2), np.float16)
        c.v_qp = np.zeros_like(c.k_qp)
    elif fmt == "int4_head":
        c.k = np.zeros((n_pages, H_kv, P, d // 2), np.uint8)
        c.v = np.zeros_like(c.k)
        c.k_qp = np.zeros((n_pages, H_kv, P, 2), np.float16)
        c.v_qp = np.zeros_like(c.k_qp)
    elif fmt in quant.FP8_FORMATS:
        c.k = np.zeros((n_pages, H_kv, P, d), np.uint8)
        c.v = np.zeros_like(c.k)
        c.k_qp = np.ones(H_kv, np.float32) if k_scale is None else np.asarray(k_scale, np.float32)
        c.v_qp = np.ones(H_kv, np.float32) if v_scale is None else np.asarray(v_scale, np.float32)
    elif fmt == "int4_kivi":
        c.k = np.zeros((n_pages, H_kv, P, d // 2), np.uint8)
        c.v = np.zeros_like(c.k)
        c.k_qp = np.zeros((n_pages, H_kv, max(1, P // G), d, 2), np.float16)
        c.v_qp = np.zeros((n_pages, H_kv, P, d // Gv, 2), np.float16)
        c.k_res = np.zeros((B, R, H_kv, d), np.uint16)
        c.v_res = np.zeros_like(c.k_res)
    else:
        raise ValueError(fmt)
    return c


def write_history(cache: Cache, page_indptr, page_indices, rows_indptr, k_bits, v_bits):
    """Write each request's whole bf16 history [T_b, H_kv, d] into ``cache``.

    ``k_bits`` / ``v_bits`` are packed ragged bf16 rows [sum T_b, H_kv, d]
    (rows of request b are rows_indptr[b]:rows_indptr[b+1], §0x04C).
    INT8 and per-head INT4 rows are quantised one (token, head) at a time (M8.6
    §0x05B, §0x09C), FP8 rows
    with their head's scale (§0x0AA); KIVI
    closes K groups per channel and V rows per token for the first n_q(T_b)
    tokens and keeps the rest as bf16 residual (M8.6 §0x06B).
    """
    cache.page_indptr = np.asarray(page_indptr, np.int64)
    cache.page_indices = np.asarray(page_indices, np.int64)
    rows_indptr = np.asarray(rows_indptr, np.int64)
    B = len(rows_indptr) - 1
    cache.kv_len = np.diff(rows_indptr)
    P = cache.P
    for b in range(B):
        T = int(cache.kv_len[b])
        kb = k_bits[rows_indptr[b]:rows_indptr[b + 1]]
        vb = v_bits[rows_indptr[b]:rows_indptr[b + 1]]
        t = np.arange(T)
        if T == 0:
            continue
        pages, rows = _pages_and_rows(cache, b, t)
        if cache.fmt == "bf16":
            for h in range(cache.H_kv):
                cache.k[pages, h, rows, :] = kb[:, h, :]
                cache.v[pages, h, rows, :] = vb[:, h, :]
        elif cache.fmt == "int8":
            for src, codes_pool, qp_pool in ((kb, cache.k, cache.k_qp), (vb, cache.v, cache.v_qp)):
                codes, s, z = quant.int8_token_quantize(quant.bf16_bits_to_f32(src))  # [T, H, d]
                for h in range(cache.H_kv):
                    codes_pool[pages, h, rows] = codes[:, h]
                    qp_pool[pages, h, rows, 0] = s[:, h]
                    qp_pool[pages, h, rows, 1] = z[:, h]
        elif cache.fmt == "int4_head":
            for src, codes_pool, qp_pool in ((kb, cache.k, cache.k_qp), (vb, cache.v, cache.v_qp)):
                codes, s, o = quant.int4_head_quantize(quant.bf16_bits_to_f32(src))  # [T, H, d]
                for h in range(cache.H_kv):
                    codes_pool[pages, h, rows] = quant.pack_int4(codes[:, h])
                    qp_pool[pages, h, rows, 0] = s[:, h]
                    qp_pool[pages, h, rows, 1] = o[:, h]
        elif cache.fmt in quant.FP8_FORMATS:
            for h in range(cache.H_kv):
                cache.k[pages, h, rows] = quant.fp8_head_quantize(quant.bf16_bits_to_f32(kb[:, h]),
                                                                  cache.k_qp[h], cache.fmt)
                cache.v[pages, h, rows] = quant.fp8_head_quantize(quant.bf16_bits_to_f32(vb[:, h]),
                                                                  cache.v_qp[h], cache.fmt)
        elif cache.fmt == "int4_kivi":
            G, Gv = cache.G, cache.Gv
            n_q = quant.kivi_quantized_prefix(T, G, cache.R)
            if n_q:
                kf = quant.bf16_bits_to_f32(kb[:n_q])                   # [n_q, H, d]
                groups = kf.reshape(n_q // G, G, cache.H_kv, cache.d).transpose(0, 2, 1, 3)
                kc, ks, kz = quant.kivi_k_group_quantize(groups)        # [n_g, H, G, d], [n_g, H, d]
                vc, vs, vz = quant.kivi_v_token_quantize(quant.bf16_bits_to_f32(vb[:n_q]), Gv)
                g0 = np.arange(0, n_q, G)
                qpage = pages[g0]
                qslot = (g0 % P) // G if P >= G else np.zeros_like(g0)
                for h in range(cache.H_kv):
                    kcodes = kc[:, h].reshape(n_q, cache.d)             # token order
                    cache.k[pages[:n_q], h, rows[:n_q]] = quant.pack_int4(kcodes)
                    cache.k_qp[qpage, h, qslot, :, 0] = ks[:, h]
                    cache.k_qp[qpage, h, qslot, :, 1] = kz[:, h]
                    cache.v[pages[:n_q], h, rows[:n_q]] = quant.pack_int4(vc[:, h])
                    cache.v_qp[pages[:n_q], h, rows[:n_q], :, 0] = vs[:, h]
                    cache.v_qp[pages[:n_q], h, rows[:n_q], :, 1] = vz[:, h]
            for tt in range(n_q, T):
                cache.k_res[b, tt % cache.R] = kb[tt]
                cache.v_res[b, tt % cache.R] = vb[tt]
        else:
            raise ValueError(cache.fmt)
    return cache


def page_offset(cache: Cache, b: int, t: int, h_kv: int, x: int) -> int:
    """Element offset of (b, t, h_kv, x) in the K pool of ``cache``  (§0x04B, §0x04D)."""
    if cache.layout == "contig":
        c = b if cache.cache_batch_idx is None else int(cache.cache_batch_idx[b])
        return address.offset_contig_nhd(c, t, h_kv, x, cache.T_c, cache.H_kv, cache.d)
    pi = address.page_csr(cache.page_indptr, cache.page_indices, b, t // cache.P)
    return address.offset_paged_hnd(pi, t % cache.P, h_kv, x, cache.P, cache.H_kv, cache.d)
