"""Quantized K/V formats: INT8 per token, KIVI-style INT4, and their ledgers.

Test infrastructure only (see ``oracle/__init__.py``).

Follows "M8.6 Live-Data Quantization: Activations and KV Cache":

* §0x02A  stored-scale conventions: ties-to-even rounding, encode with the
          re-read stored qparams, a sentinel scale of one for a row with no
          range, and no subnormal stored scale;
* §0x03A-C scale placement (per-token K/V scales, per-channel K scales);
* §0x04A-B byte ledger M_served = codes + qparams + residual (+ pages);
* §0x05B  per-token scaling is append-local;
* §0x06A-B KIVI: K per channel over groups of G tokens, V per token, a
          full-precision residual whose oldest G rows close while it holds
          more than R rows; §0x06E  G = 32, R = 128;
* §0x09C  the asymmetric floating-offset ABI (an offset stored as a value,
          not clamped to the code range), used by the INT8 zero point and by
          the per-head asymmetric KV4 format.

Formats (the reading of the pages that the library documents):

* INT8: per (token, kv head), separately for K and V, over the d channels:
  mn = min, mx = max (exact in fp32); s = fp16((mx - mn) / 255) computed with
  an fp32 divide, z = fp16(mn).  mx == mn stores the sentinel s = 1; a
  stored scale below 2^-14 (zero or subnormal fp16) is raised to 2^-14.
  code = clip(rint_even((x - z) / s), 0, 255) in fp32 with the RE-READ
  stored s and z.  Decoding is x_hat = code * s + z.
* INT4 KIVI: the same quantizer with 15 levels.  K: one (s, z) per
  (G-token group, channel).  V: one (s, z) per (token, Gv-channel group).
  Two codes per byte along d, the even channel in the low nibble.
* FP8 E4M3 with a per-head scale (§0x0A-0x0AA: one scale per K/V head; no
  calibration means scale 1): code = e4m3(x / s_h), the quotient in fp32
  (one correctly rounded divide), rounded to the nearest E4M3 value with
  ties to the even code and saturated to +-448; x_hat = e4m3_value(code) s_h.
  FP8 E5M2 the same way, saturated to +-57344.
* INT4 per head (QServe-style KV4, §0x09C): one fp16 (s, o) per (token, kv
  head) with s = (max - min) / 15 and a floating offset o = -min / s that is
  not clamped; code = clip(rint_even(x / s + o), 0, 15); x_hat = (code - o) s.
"""

from __future__ import annotations

import numpy as np

F16_MIN_NORMAL = np.float16(2.0 ** -14)


# ---- bf16 / fp16 conversions -------------------------------------------------

def bf16_bits_to_f64(bits) -> np.ndarray:
    """Exact value of bf16 bit patterns (uint16) as float64."""
    b = np.asarray(bits).astype(np.uint16).astype(np.uint32) << np.uint32(16)
    return b.view(np.float32).astype(np.float64)


def bf16_bits_to_f32(bits) -> np.ndarray:
    b = np.asarray(bits).astype(np.uint16).astype(np.uint32) << np.uint32(16)
    return b.view(np.float32)


def f16_bits_to_f64(bits) -> np.ndarray:
    return np.asarray(bits).astype(np.uint16).view(np.float16).astype(np.float64)


# ---- one affine group (vectorised: one group per slice of the last axis) ------

def affine_qparams(x_f32, qmax: int):
    """Stored (s, z) float16 for each group along the last axis  (M8.6 §0x02A, §0x09C)."""
    x = np.asarray(x_f32, dtype=np.float32)
    mn = x.min(axis=-1)
    mx = x.max(axis=-1)
    s = ((mx - mn) / np.float32(qmax)).astype(np.float16)     # fp32 divide, RNE to fp16
    s = np.where(s < F16_MIN_NORMAL, F16_MIN_NORMAL, s)
    s = np.where(mx == mn, np.float16(1.0), s).astype(np.float16)
    z = mn.astype(np.float16)
    return s, z


def affine_encode(x_f32, s16, z16, qmax: int) -> np.ndarray:
    """codes = clip(rint_even((x - z) / s), 0, qmax) in fp32 with the re-read stored s, z."""
    x = np.asarray(x_f32, dtype=np.float32)
    s = np.asarray(s16, dtype=np.float16).astype(np.float32)[..., None]
    z = np.asarray(z16, dtype=np.float16).astype(np.float32)[..., None]
    r = np.rint((x - z) / s)          # each operation rounded in fp32, ties to even
    return np.clip(r, 0, qmax).astype(np.uint8)


def affine_decode(codes, s16, z16) -> np.ndarray:
    """x_hat = code * s + z in float64 (s, z broadcast over the group's last axis)."""
    s = np.asarray(s16, dtype=np.float16).astype(np.float64)[..., None]
    z = np.asarray(z16, dtype=np.float16).astype(np.float64)[..., None]
    return np.asarray(codes, dtype=np.float64) * s + z


# ---- INT8 per token ----------------------------------------------------------

def int8_token_quantize(x_f32):
    """(token, head) rows [..., d] -> codes uint8 [..., d], s, z fp16 [...]  (M8.6 §0x05B)."""
    s, z = affine_qparams(x_f32, 255)
    return affine_encode(x_f32, s, z, 255), s, z


# ---- KIVI INT4 ---------------------------------------------------------------

def kivi_k_group_quantize(k_rows_f32):
    """K group [..., G, d] -> codes [..., G, d], s [..., d], z [..., d]: one scale per channel
    over the group's G tokens  (M8.6 §0x06A)."""
    k = np.swapaxes(np.asarray(k_rows_f32, dtype=np.float32), -1, -2)   # [..., d, G]
    s, z = affine_qparams(k, 15)
    codes = affine_encode(k, s, z, 15)
    return np.swapaxes(codes, -1, -2), s, z


def kivi_v_token_quantize(v_row_f32, group: int):
    """V rows [..., d] -> codes [..., d], s [..., d/Gv], z [..., d/Gv]: per token, per Gv
    channels  (M8.6 §0x06A)."""
    v = np.asarray(v_row_f32, dtype=np.float32)
    d = v.shape[-1]
    vg = v.reshape(v.shape[:-1] + (d // group, group))
    s, z = affine_qparams(vg, 15)
    codes = affine_encode(vg, s, z, 15)
    return codes.reshape(v.shape), s, z


def kivi_quantized_prefix(T: int, G: int = 32, R: int = 128) -> int:
    """Rows already closed into INT4 groups after T appends  (M8.6 §0x06B).

    The KIVILayerState loop closes the oldest G residual rows while the
    residual holds more than R rows.  Replaying it append by append keeps the
    residual in (R - G, R] once T > R.
    """
    closed = 0
    for t in range(1, T + 1):
        while t - closed > R:
            closed += G
    return closed


def pack_int4(codes) -> np.ndarray:
    """Two codes per byte along the last axis, the even channel in the low nibble."""
    c = np.asarray(codes, dtype=np.uint8)
    return (c[..., 0::2] & 0xF) | ((c[..., 1::2] & 0xF) << 4)


def unpack_int4(packed) -> np.ndarray:
    p = np.asarray(packed, dtype=np.uint8)
    out = np.empty(p.shape[:-1] + (p.shape[-1] * 2,), dtype=np.uint8)
    out[..., 0::2] = p & 0xF
    out[..., 1::2] = p >> 4
    return out


# ---- FP8 E4M3 with a per-head scale (M8.6 §0x0A-0x0AA) -----------------------
#
# E4M3 as KV caches use it: 1 sign bit, 4 exponent bits with bias 7, 3 mantissa
# bits, no infinities.  Exponent field 0 holds the subnormals m 2^-9; exponent
# e in 1..15 holds (1 + m/8) 2^(e-7), except exponent 15 with mantissa 7, which
# is NaN.  The largest finite magnitude is 1.75 2^8 = 448.

E4M3_MAX = 448.0


def e4m3_decode(codes) -> np.ndarray:
    """Exact float64 value of E4M3 codes (NaN for 0x7F / 0xFF)."""
    c = np.asarray(codes).astype(np.int64)
    sign = (c >> 7) & 1
    e = (c >> 3) & 15
    m = (c & 7).astype(np.float64)
    mag = np.where(e == 0, m * 2.0 ** -9, (1.0 + m / 8.0) * np.exp2(e.astype(np.float64) - 7.0))
    mag = np.where((e == 15) & (c & 7 == 7), np.nan, mag)
    return np.where(sign == 1, -mag, mag)


_E4M3_POS = e4m3_decode(np.arange(127))     # codes 0..126: the finite non-negative values, ascending


def e4m3_encode(x) -> np.ndarray:
    """Nearest E4M3 code of each value, ties to the even code, saturated to +-448; the sign
    of x is kept (a negative value that rounds to zero gives 0x80).  NaN gives 0x7F."""
    x = np.asarray(x, dtype=np.float64)
    a = np.minimum(np.abs(x), E4M3_MAX)
    hi = np.clip(np.searchsorted(_E4M3_POS, a, side="left"), 0, 126)   # first value >= a
    lo = np.maximum(hi - 1, 0)
    d_lo = a - _E4M3_POS[lo]
    d_hi = _E4M3_POS[hi] - a
    code = np.where(d_lo < d_hi, lo, hi)
    tie = d_lo == d_hi
    code = np.where(tie, np.where(lo % 2 == 0, lo, hi), code)
    code = np.where(np.signbit(x), code | 0x80, code)
    code = np.where(np.isnan(x), 0x7F, code)
    return code.astype(np.uint8)


# E5M2: 1 sign bit, 5 exponent bits with bias 15, 2 mantissa bits (the upper
# byte of an IEEE half).  Exponent field 0 holds the subnormals m 2^-16; 31 holds
# infinity (mantissa 0) and NaN.  The largest finite magnitude is 1.75 2^15.

E5M2_MAX = 57344.0


def e5m2_decode(codes) -> np.ndarray:
    """Exact float64 value of E5M2 codes (+-inf for 0x7C / 0xFC, NaN for the rest of exponent 31)."""
    c = np.asarray(codes).astype(np.int64)
    sign = (c >> 7) & 1
    e = (c >> 2) & 31
    m = (c & 3).astype(np.float64)
    mag = np.where(e == 0, m * 2.0 ** -16, (1.0 + m / 4.0) * np.exp2(e.astype(np.float64) - 15.0))
    mag = np.where(e == 31, np.where(c & 3 == 0, np.inf, np.nan), mag)
    return np.where(sign == 1, -mag, mag)


_E5M2_POS = e5m2_decode(np.arange(124))     # codes 0..123: the finite non-negative values, ascending


def _nearest_code(x, table, top: float, nan_code: int) -> np.ndarray:
    """Nearest code of |x| in an ascending table of finite values, ties to the even code,
    saturated to the table's top value; sign bit from x; NaN to nan_code."""
    x = np.asarray(x, dtype=np.float64)
    a = np.minimum(np.abs(x), top)
    last = len(table) - 1
    hi = np.clip(np.searchsorted(table, a, side="left"), 0, last)
    lo = np.maximum(hi - 1, 0)
    d_lo = a - table[lo]
    d_hi = table[hi] - a
    code = np.where(d_lo < d_hi, lo, hi)
    code = np.where(d_lo == d_hi, np.where(lo % 2 == 0, lo, hi), code)
    code = np.where(np.signbit(x), code | 0x80, code)
    code = np.where(np.isnan(x), nan_code, code)
    return code.astype(np.uint8)


def e5m2_encode(x) -> np.ndarray:
    """Nearest E5M2 code, ties to the even code, saturated to +-57344 (infinities included);
    the sign of x is kept.  NaN gives 0x7F."""
    return _nearest_code(x, _E5M2_POS, E5M2_MAX, 0x7F)


FP8_FORMATS = {"fp8_e4m3": (e4m3_encode, e4m3_decode), "fp8_e5m2": (e5m2_encode, e5m2_decode)}


def fp8_head_quantize(x_f32, scale_f32, fmt: str = "fp8_e4m3") -> np.ndarray:
    """Rows [..., d] of one kv head -> FP8 codes of x / s (the quotient rounded in fp32)."""
    q = np.asarray(x_f32, dtype=np.float32) / np.float32(scale_f32)
    return FP8_FORMATS[fmt][0](q.astype(np.float32))


def fp8_head_decode(codes, scale_f32, fmt: str = "fp8_e4m3") -> np.ndarray:
    """x_hat = value(code) * s in float64."""
    return FP8_FORMATS[fmt][1](codes) * np.float64(np.float32(scale_f32))


# ---- per-head asymmetric KV4 with a floating offset (M8.6 §0x09C) -----------
#
# One (scale, offset) pair per (token, kv head), separately for K and V, over
# the head's d channels.  Before storage rounding the page's parameters are
# s* = (max - min) / 15 and o* = -min / s*; both are stored as fp16 and the
# offset is a floating value that is NOT clamped to the code range (a range
# [1, 2] has o* = -15).  Codes are clip(rint(x / s + o), 0, 15) with the
# re-read stored s and o, the rounding done after the offset is added;
# x_hat = (code - o) * s.  Two codes per byte along d, the even channel in the
# low nibble (the same packing as the KIVI format).
#
# The page leaves the degenerate heads to the implementation and rejects them
# in its model; the readings taken here keep every stored value finite:
#  * a constant head (max == min) stores the sentinel s = 1 (M8.6 §0x02A) and
#    o = fp16(-min), so it decodes to fp16(min);
#  * a stored scale below 2^-14 (zero or subnormal fp16) is raised to 2^-14,
#    and the offset is then computed with that scale;
#  * fp16 conversions round to nearest even and saturate to +-65504.
# Arithmetic is fp32 (min / max exact, each divide and add correctly rounded).

def f16_saturated(x_f32) -> np.ndarray:
    """fp32 -> fp16, round to nearest even, saturated to the largest finite magnitude."""
    x = np.asarray(x_f32, dtype=np.float32)
    return np.clip(x, np.float32(-65504.0), np.float32(65504.0)).astype(np.float16)


def int4_head_qparams(x_f32):
    """Stored (s, o) fp16 of each (token, head) row along the last axis  (M8.6 §0x09C)."""
    x = np.asarray(x_f32, dtype=np.float32)
    mn = x.min(axis=-1)
    mx = x.max(axis=-1)
    width = (mx - mn).astype(np.float32)
    flat = width == 0
    with np.errstate(over="ignore"):
        base = np.where(flat, np.float32(1.0), width / np.float32(15.0)).astype(np.float32)
    s = f16_saturated(base)
    tiny = (s < F16_MIN_NORMAL) & ~flat
    s = np.where(tiny, F16_MIN_NORMAL, s).astype(np.float16)
    base = np.where(tiny, np.float32(F16_MIN_NORMAL), base).astype(np.float32)
    with np.errstate(over="ignore"):
        o = f16_saturated((-mn).astype(np.float32) / base)
    return s, o


def int4_head_encode(x_f32, s16, o16) -> np.ndarray:
    """codes = clip(rint_even(x / s + o), 0, 15), each fp32 operation rounded once."""
    x = np.asarray(x_f32, dtype=np.float32)
    s = np.asarray(s16, dtype=np.float16).astype(np.float32)[..., None]
    o = np.asarray(o16, dtype=np.float16).astype(np.float32)[..., None]
    with np.errstate(over="ignore"):
        u = (x / s).astype(np.float32) + o
    return np.clip(np.rint(u), 0, 15).astype(np.uint8)


def int4_head_quantize(x_f32):
    """(token, head) rows [..., d] -> codes uint8 [..., d] (unpacked), s, o fp16 [...]."""
    s, o = int4_head_qparams(x_f32)
    return int4_head_encode(x_f32, s, o), s, o


def int4_head_decode(codes, s16, o16) -> np.ndarray:
    """x_hat = (code - o) * s in float64 (s, o broadcast over the row)."""
    s = np.asarray(s16, dtype=np.float16).astype(np.float64)[..., None]
    o = np.asarray(o16, dtype=np.float16).astype(np.float64)[..., None]
    return (np.asarray(codes, dtype=np.float64) - o) * s


# ---- byte ledger, M8.6 §0x04A-B ---------------------------------------------

def served_bytes(T: int, L: int, H_kv: int, d_h: int, bits: int, G_t: int, G_d: int,
                 b_s: int, b_z: int, residual: int, b_res: int):
    """Code payload + K qparams + V qparams + residual for a synchronised tail (M8.6 §0x04B).

    Only the T - residual closed tokens carry codes and qparams.  K groups are
    per channel over G_t tokens; V groups per token over G_d channels.
    """
    n_q = T - residual
    codes = 2 * n_q * L * H_kv * d_h * bits // 8
    k_qp = (n_q // G_t) * L * H_kv * d_h * (b_s + b_z)
    v_qp = n_q * L * H_kv * (d_h // G_d) * (b_s + b_z)
    res = 2 * residual * L * H_kv * d_h * b_res
    return {"codes": codes, "k_qparams": k_qp, "v_qparams": v_qp, "residual": res,
            "total": codes + k_qp + v_qp + res}
