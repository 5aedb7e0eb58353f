"""Pins of the oracle's K/V quantizers and quantized cache (M8.6 §0x02A, §0x05B, §0x06A-B)."""

import math

import numpy as np
import pytest

from oracle import attention
from oracle import cache as cm
from oracle import quant
from tests.test_oracle_attention import _bf16


def _f32(bits):
    return quant.bf16_bits_to_f32(bits)


def test_int8_round_trip_bound_and_endpoints():
    rng = np.random.default_rng(20)
    x = _f32(_bf16(rng, (500, 128)))
    x[:, 5] *= 8
    codes, s, z = quant.int8_token_quantize(x)
    xh = quant.affine_decode(codes, s, z)
    s64 = s.astype(np.float64)[:, None]
    assert np.all(np.abs(xh - x) <= 0.5 * s64 * (1 + 1e-3) + 1e-6)
    assert np.all(codes[np.arange(500), x.argmin(axis=1)] == 0)
    assert np.all(codes[np.arange(500), x.argmax(axis=1)] >= 254)
    # scale is (max - min) / 255 up to fp16 rounding
    rng_ = (x.max(1) - x.min(1)).astype(np.float64)
    np.testing.assert_allclose(s.astype(np.float64), rng_ / 255, rtol=2 ** -10)


def test_int8_constant_row_sentinel_and_ties_to_even():
    codes, s, z = quant.int8_token_quantize(np.full((1, 8), 0.75, np.float32))
    assert s[0] == 1.0 and z[0] == 0.75 and not codes.any()
    row = np.zeros((1, 8), np.float32)
    row[0, :] = [0, 255, 2.5, 3.5, 4.5, 0.5, 1.5, 254.5]
    codes, s, z = quant.int8_token_quantize(row)
    assert s[0] == 1.0 and z[0] == 0.0
    assert codes[0].tolist() == [0, 255, 2, 4, 4, 0, 2, 254]


def test_tiny_range_scale_floor():
    row = np.array([[1.0, 1.0 + 2 ** -7]], np.float32)      # range / 255 is subnormal in fp16
    codes, s, z = quant.int8_token_quantize(row)
    assert s[0] == np.float16(2 ** -14)
    assert np.all(np.abs(quant.affine_decode(codes, s, z) - row) <= 2 ** -15)


def test_kivi_k_scales_per_channel_isolate_outlier():
    rng = np.random.default_rng(21)
    k = _f32(_bf16(rng, (32, 128)))
    k[:, 7] *= 8
    codes, s, z = quant.kivi_k_group_quantize(k)
    assert codes.shape == (32, 128) and s.shape == (128,)
    others = np.delete(s.astype(np.float64), 7)
    assert s[7] > 4 * np.median(others)
    xh = codes * s.astype(np.float64)[None, :] + z.astype(np.float64)[None, :]
    assert np.all(np.abs(xh - k) <= 0.5 * s.astype(np.float64)[None, :] * (1 + 1e-3) + 1e-6)
    for c in (0, 7, 100):                        # each channel: min -> 0, max -> 15 (or 14)
        assert codes[k[:, c].argmin(), c] == 0 and codes[k[:, c].argmax(), c] >= 14


def test_kivi_v_per_token_groups():
    rng = np.random.default_rng(22)
    v = _f32(_bf16(rng, (5, 128)))
    codes, s, z = quant.kivi_v_token_quantize(v, 32)
    assert s.shape == (5, 4) and codes.max() <= 15
    g = v.reshape(5, 4, 32)
    np.testing.assert_array_equal(z, g.min(axis=2).astype(np.float16))


def test_pack_unpack_int4():
    c = np.array([[1, 2, 15, 0]], np.uint8)
    p = quant.pack_int4(c)
    assert p.tolist() == [[0x21, 0x0F]]
    assert np.array_equal(quant.unpack_int4(p), c)


def test_kivi_frontier_replay():
    G, R = 32, 128
    for T in range(0, 700):
        n_q = quant.kivi_quantized_prefix(T, G, R)
        assert n_q % G == 0
        assert n_q == G * math.ceil(max(0, T - R) / G)
        if T > R:
            assert R - G < T - n_q <= R


def test_kivi_frontier_keeps_the_newest_128_rows_bf16_at_the_workload_residual():
    """The quantized workload keeps "the most recent 128 tokens" in bf16: with G = 32
    and R = 160 the closing loop never quantizes one of the newest 128 rows and never
    holds more than R residual rows (the ring); past R appends the residual stays in
    (128, 160], one group of G above the 128 rows it must keep."""
    import workloads as W
    G, R = 32, W.KIVI_RESIDUAL
    assert R == 160
    for T in range(0, 1200):
        n_q = quant.kivi_quantized_prefix(T, G, R)
        resid = T - n_q
        assert n_q % G == 0 and 0 <= n_q <= T
        assert resid >= min(T, 128)                      # rows T-128 .. T-1 stay bf16
        assert resid <= R                                # the ring of R rows holds them
        if T > R:
            assert 128 < resid <= 128 + G                # at most one group above the 128 kept rows
    w = W.quantized_history("kivi", B=2, S_q=1, H_q=4, H_kv=1, d=64, lens=[200, 33], P=16, seed=0,
                            device="cpu", fmt="int4_kivi")
    assert w.problem["kivi_residual"] == R


def test_quantized_cache_round_trip():
    rng = np.random.default_rng(23)
    lens = [300, 129, 40]
    H, d, P = 2, 64, 16
    n_pages = [-(-T // P) for T in lens]
    pool = sum(n_pages) + 2
    indices = rng.permutation(pool)[:sum(n_pages)]
    indptr = np.concatenate([[0], np.cumsum(n_pages)])
    ri = np.concatenate([[0], np.cumsum(lens)])
    k = _bf16(rng, (ri[-1], H, d))
    v = _bf16(rng, (ri[-1], H, d))
    ref = cm.empty_paged("bf16", pool, H, P, d, 3)
    cm.write_history(ref, indptr, indices, ri, k, v)
    for fmt, levels in (("int8", 255), ("int4_kivi", 15)):
        c = cm.empty_paged(fmt, pool, H, P, d, 3)
        cm.write_history(c, indptr, indices, ri, k, v)
        for b, T in enumerate(lens):
            for h in range(H):
                K0, V0 = cm.read_rows(ref, b, h, np.arange(T))
                K1, V1 = cm.read_rows(c, b, h, np.arange(T))
                span = 6.0 / levels * 4
                assert np.max(np.abs(K1 - K0)) < span and np.max(np.abs(V1 - V0)) < span
                if fmt == "int4_kivi":
                    n_q = quant.kivi_quantized_prefix(T)
                    assert np.array_equal(K1[n_q:], K0[n_q:]) and np.array_equal(V1[n_q:], V0[n_q:])
        problem = dict(B=3, S_q=1, H_q=4, H_kv=H, d=d)
        q = _bf16(rng, (3, 1, 4, d))
        O0, L0 = attention.decode_rows(problem, ref, q)
        O1, L1 = attention.decode_rows(problem, c, q)
        assert np.max(np.abs(O1 - O0)) < (0.05 if fmt == "int8" else 0.5)


# ---- FP8 E4M3 with a per-head scale (M8.6 §0x0A-0x0AA) -----------------------

def _torch_e4m3():
    torch = pytest.importorskip("torch")
    if not hasattr(torch, "float8_e4m3fn"):
        pytest.skip("torch without float8_e4m3fn")
    return torch


def test_e4m3_decode_matches_an_independent_implementation_on_all_codes():
    """PyTorch's float8_e4m3fn is an implementation of the same format written by others."""
    torch = _torch_e4m3()
    codes = np.arange(256)
    ours = quant.e4m3_decode(codes)
    theirs = torch.tensor(codes, dtype=torch.uint8).view(torch.float8_e4m3fn).double().numpy()
    assert np.array_equal(np.isnan(ours), np.isnan(theirs))
    assert np.array_equal(np.nan_to_num(ours), np.nan_to_num(theirs))
    assert np.array_equal(np.signbit(ours[~np.isnan(ours)]), np.signbit(theirs[~np.isnan(theirs)]))


def test_e4m3_decode_closed_forms():
    dec = quant.e4m3_decode
    assert dec(0x7E) == 448.0 and dec(0xFE) == -448.0          # 1.75 * 2^8, the largest finite value
    assert dec(0x01) == 2.0 ** -9 and dec(0x07) == 7 * 2.0 ** -9   # subnormals m 2^-9
    assert dec(0x08) == 2.0 ** -6                               # smallest normal
    assert dec(0x38) == 1.0 and dec(0x39) == 1.125               # exponent field 7 is 2^0
    assert np.isnan(dec(0x7F)) and np.isnan(dec(0xFF))           # no infinities, one NaN pattern
    assert dec(0x80) == 0.0 and np.signbit(dec(0x80))
    assert dec(0x77) == 240.0 and dec(0x78) == 256.0             # (1 + 7/8) 2^7, 2^8


def test_e4m3_encode_rounds_to_nearest_with_ties_to_even():
    enc = quant.e4m3_encode
    u = 2.0 ** -9
    assert enc(0.5 * u) == 0x00 and enc(1.5 * u) == 0x02 and enc(2.5 * u) == 0x02 and enc(3.5 * u) == 0x04
    assert enc(0.49 * u) == 0x00 and enc(0.51 * u) == 0x01
    assert enc(1.0625) == 0x38 and enc(1.1875) == 0x3A          # midpoints of [1, 1.125] and [1.125, 1.25]
    assert enc(-1.0625) == 0xB8
    assert enc(-1e-30) == 0x80                                  # the sign survives rounding to zero
    assert enc(float("nan")) == 0x7F


def test_e4m3_encode_saturates_and_agrees_with_torch_below_its_overflow():
    """Saturation to +-448 (the KV-cache convention); PyTorch instead gives NaN from 464
    up, so the two are compared on |x| < 464, with every midpoint included."""
    torch = _torch_e4m3()
    enc = quant.e4m3_encode
    assert enc(448.0) == 0x7E and enc(463.9) == 0x7E and enc(1000.0) == 0x7E and enc(-1e9) == 0xFE
    pos = quant.e4m3_decode(np.arange(127))
    mids = (pos[:-1] + pos[1:]) / 2
    rng = np.random.default_rng(30)
    x = np.concatenate([rng.uniform(-463.9, 463.9, 50000), rng.normal(0, 1, 50000),
                        rng.normal(0, 1e-3, 20000), mids, -mids, pos, -pos]).astype(np.float32)
    theirs = torch.tensor(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(enc(x), theirs)


def test_e4m3_round_trip_on_every_finite_code():
    codes = np.array([c for c in range(256) if c & 0x7F != 0x7F], np.uint8)
    assert np.array_equal(quant.e4m3_encode(quant.e4m3_decode(codes)), codes)


def test_fp8_head_quantize_divides_in_fp32_then_rounds():
    torch = _torch_e4m3()
    rng = np.random.default_rng(31)
    x = _f32(_bf16(rng, (64, 128)))
    for s in (1.0, 0.0137, 3.0, 1.7e-3):
        ours = quant.fp8_head_quantize(x, np.float32(s))
        q = torch.tensor(x) / torch.tensor(np.float32(s))        # fp32 quotient
        theirs = q.to(torch.float8_e4m3fn).view(torch.uint8).numpy()
        inside = np.abs(q.numpy()) < 464.0                       # PyTorch gives NaN beyond
        assert np.array_equal(ours[inside], theirs[inside])
        assert np.all(ours[~inside] & 0x7F == 0x7E)               # saturated to +-448
        err = np.abs(quant.fp8_head_decode(ours, np.float32(s)) - x)
        ok = np.abs(x) <= 448.0 * np.float32(s)
        assert np.all(err[ok] <= np.abs(x[ok]) * 2.0 ** -4 + np.float32(s) * 2.0 ** -10)   # half an ulp of 3 bits


def test_fp8_cache_round_trip_and_decode_close_to_bf16():
    rng = np.random.default_rng(32)
    lens = [300, 129, 40]
    H, d, P = 2, 64, 16
    n_pages = [-(-T // P) for T in lens]
    pool = sum(n_pages) + 2
    indices = rng.permutation(pool)[:sum(n_pages)]
    indptr = np.concatenate([[0], np.cumsum(n_pages)])
    ri = np.concatenate([[0], np.cumsum(lens)])
    k = _bf16(rng, (ri[-1], H, d))
    v = _bf16(rng, (ri[-1], H, d))
    ref = cm.empty_paged("bf16", pool, H, P, d, 3)
    cm.write_history(ref, indptr, indices, ri, k, v)
    ks = np.array([0.02, 1.0], np.float32)
    vs = np.array([1.0, 0.011], np.float32)
    c = cm.empty_paged("fp8_e4m3", pool, H, P, d, 3, k_scale=ks, v_scale=vs)
    cm.write_history(c, indptr, indices, ri, k, v)
    for b, T in enumerate(lens):
        for h in range(H):
            K0, V0 = cm.read_rows(ref, b, h, np.arange(T))
            K1, V1 = cm.read_rows(c, b, h, np.arange(T))
            assert np.all(np.abs(K1 - K0) <= np.abs(K0) / 16 + ks[h] * 2.0 ** -10)
            assert np.all(np.abs(V1 - V0) <= np.abs(V0) / 16 + vs[h] * 2.0 ** -10)
    problem = dict(B=3, S_q=1, H_q=4, H_kv=H, d=d)
    q = _bf16(rng, (3, 1, 4, d))
    O0, L0 = attention.decode_rows(problem, ref, q)
    O1, L1 = attention.decode_rows(problem, c, q)
    assert np.max(np.abs(O1 - O0)) < 0.05


def _torch_e5m2():
    torch = pytest.importorskip("torch")
    if not hasattr(torch, "float8_e5m2"):
        pytest.skip("torch without float8_e5m2")
    return torch


def test_e5m2_decode_matches_an_independent_implementation_on_all_codes():
    torch = _torch_e5m2()
    codes = np.arange(256)
    ours = quant.e5m2_decode(codes)
    theirs = torch.tensor(codes, dtype=torch.uint8).view(torch.float8_e5m2).double().numpy()
    assert np.array_equal(np.isnan(ours), np.isnan(theirs))
    fin = ~np.isnan(ours)
    assert np.array_equal(ours[fin], theirs[fin])
    assert np.array_equal(np.signbit(ours[fin]), np.signbit(theirs[fin]))


def test_e5m2_decode_closed_forms():
    dec = quant.e5m2_decode
    assert dec(0x7B) == 57344.0 and dec(0xFB) == -57344.0        # 1.75 * 2^15
    assert dec(0x7C) == np.inf and dec(0xFC) == -np.inf
    assert np.isnan(dec(0x7D)) and np.isnan(dec(0x7F))
    assert dec(0x01) == 2.0 ** -16 and dec(0x03) == 3 * 2.0 ** -16   # subnormals m 2^-16
    assert dec(0x04) == 2.0 ** -14 and dec(0x3C) == 1.0 and dec(0x3D) == 1.25
    # an E5M2 code is the upper byte of the IEEE half with the same value
    fin = [c for c in range(256) if (c >> 2) & 31 != 31]
    halves = (np.array(fin, np.uint16) << 8).view(np.float16).astype(np.float64)
    assert np.array_equal(dec(np.array(fin)), halves)


def test_e5m2_encode_ties_saturation_and_agreement_below_overflow():
    torch = _torch_e5m2()
    enc = quant.e5m2_encode
    u = 2.0 ** -16
    assert enc(0.5 * u) == 0x00 and enc(1.5 * u) == 0x02 and enc(2.5 * u) == 0x02
    assert enc(1.125) == 0x3C and enc(1.375) == 0x3E           # ties to the even code
    assert enc(57344.0) == 0x7B and enc(1e6) == 0x7B and enc(np.inf) == 0x7B and enc(-np.inf) == 0xFB
    pos = quant.e5m2_decode(np.arange(124))
    mids = (pos[:-1] + pos[1:]) / 2
    rng = np.random.default_rng(33)
    x = np.concatenate([rng.uniform(-61000, 61000, 50000), rng.normal(0, 1, 50000),
                        rng.normal(0, 1e-4, 20000), mids, -mids, pos, -pos]).astype(np.float32)
    theirs = torch.tensor(x).to(torch.float8_e5m2).view(torch.uint8).numpy()   # overflows to inf past 61440
    assert np.array_equal(enc(x), theirs)
    codes = np.array([c for c in range(256) if (c >> 2) & 31 != 31], np.uint8)
    assert np.array_equal(enc(quant.e5m2_decode(codes)), codes)


def test_fp8_e5m2_cache_decode_close_to_bf16():
    rng = np.random.default_rng(34)
    lens = [200, 33]
    H, d, P = 2, 64, 16
    n_pages = [-(-T // P) for T in lens]
    pool = sum(n_pages) + 1
    indices = rng.permutation(pool)[:sum(n_pages)]
    indptr = np.concatenate([[0], np.cumsum(n_pages)])
    ri = np.concatenate([[0], np.cumsum(lens)])
    k = _bf16(rng, (ri[-1], H, d))
    v = _bf16(rng, (ri[-1], H, d))
    ref = cm.empty_paged("bf16", pool, H, P, d, 2)
    cm.write_history(ref, indptr, indices, ri, k, v)
    c = cm.empty_paged("fp8_e5m2", pool, H, P, d, 2, k_scale=np.array([1e-4, 1.0], np.float32))
    cm.write_history(c, indptr, indices, ri, k, v)
    for b, T in enumerate(lens):
        for h in range(H):
            K0, V0 = cm.read_rows(ref, b, h, np.arange(T))
            K1, V1 = cm.read_rows(c, b, h, np.arange(T))
            s = c.k_qp[h]
            assert np.all(np.abs(K1 - K0) <= np.abs(K0) / 8 + s * 2.0 ** -17)
            assert np.all(np.abs(V1 - V0) <= np.abs(V0) / 8 + 2.0 ** -17)


# ---- per-head asymmetric KV4 with a floating offset (M8.6 §0x09C) ------------

def test_int4_head_positive_range_keeps_the_unclamped_offset():
    """§0x09C: a head whose values lie in [1, 2] has the ideal offset -15, outside the code
    range; clamping it to zero would bring both endpoints back near one."""
    row = np.array([[1.0, 2.0, 1.5, 1.25, 1.75, 1.0625, 1.9375, 1.5]], np.float32)
    codes, s, o = quant.int4_head_quantize(row)
    assert s[0] == np.float16(1.0 / 15.0)
    assert o[0] == -15.0
    assert codes[0, 0] == 0 and codes[0, 1] == 15
    xh = quant.int4_head_decode(codes, s, o)
    assert np.all(np.abs(xh - row) <= 0.5 * float(s[0]))
    clamped = quant.int4_head_decode(quant.int4_head_encode(row, s, np.float16([0.0])), s, np.float16([0.0]))
    assert abs(clamped[0, 0] - 1.0) < 0.01 and abs(clamped[0, 1] - 1.0) < 0.01   # 2 comes back near 1


def test_int4_head_round_trip_bound_and_endpoints():
    rng = np.random.default_rng(40)
    x = _f32(_bf16(rng, (600, 128)))
    x[:, 9] *= 8
    x[:300] = x[:300] * np.float32(0.125) + np.float32(6.0)   # positive rows: offsets below -15
    codes, s, o = quant.int4_head_quantize(x)
    xh = quant.int4_head_decode(codes, s, o)
    s64 = s.astype(np.float64)[:, None]
    assert np.all(np.abs(xh - x) <= 0.5 * s64 * (1 + 1e-5) + 1e-7)
    rows = np.arange(600)
    assert np.all(codes[rows, x.argmin(axis=1)] == 0)
    assert np.all(codes[rows, x.argmax(axis=1)] == 15)
    width = (x.max(1) - x.min(1)).astype(np.float64)
    np.testing.assert_allclose(s.astype(np.float64), width / 15, rtol=2 ** -11)
    np.testing.assert_allclose(o.astype(np.float64), -x.min(1) / (width / 15), rtol=2 ** -10)
    assert np.any(o[:300] < -15)                       # the offset is not clamped to [0, 15]


def test_int4_head_rounds_after_adding_the_offset_with_ties_to_even():
    row = np.array([[0, 15, 2.5, 3.5, 4.5, 0.5, 1.5, 14.5]], np.float32)   # s = 1, o = -0
    codes, s, o = quant.int4_head_quantize(row)
    assert s[0] == 1.0 and o[0] == 0.0
    assert codes[0].tolist() == [0, 15, 2, 4, 4, 0, 2, 14]
    shifted = row - np.float32(0.25)                   # o = 0.25: x / s + o lands on the same ties
    codes2, s2, o2 = quant.int4_head_quantize(shifted)
    assert s2[0] == 1.0 and o2[0] == 0.25
    assert codes2[0].tolist() == [0, 15, 2, 4, 4, 0, 2, 14]


def test_int4_head_degenerate_heads():
    # constant head: sentinel scale 1, decodes to fp16(min)
    for val in (0.75, 3.14159, -2.0):
        codes, s, o = quant.int4_head_quantize(np.full((1, 16), val, np.float32))
        assert s[0] == 1.0 and o[0] == np.float16(-val) and not codes.any()
        assert quant.int4_head_decode(codes, s, o)[0, 0] == float(np.float16(val))
    # range / 15 below the smallest normal fp16: scale 2^-14, offset computed with it
    codes, s, o = quant.int4_head_quantize(np.array([[1.0, 1.0 + 2 ** -12]], np.float32))
    assert s[0] == np.float16(2 ** -14) and o[0] == -16384.0
    assert codes[0].tolist() == [0, 4]
    assert np.array_equal(quant.int4_head_decode(codes, s, o)[0], [1.0, 1.0 + 2 ** -12])
    # stored values saturate to the largest finite fp16
    codes, s, o = quant.int4_head_quantize(np.array([[0.0, 1.0e6]], np.float32))
    assert s[0] == 65504.0 and codes[0].tolist() == [0, 15]
    codes, s, o = quant.int4_head_quantize(np.array([[1.0e5, 1.0e5 + 1.0]], np.float32))
    assert o[0] == -65504.0 and np.all(np.isfinite(quant.int4_head_decode(codes, s, o)))


def test_int4_head_fp32_encoding_agrees_with_fp64_away_from_ties():
    """The page's arithmetic model rounds x / s + o in float64; away from a tie fp32 gives the
    same code."""
    rng = np.random.default_rng(41)
    x = _f32(_bf16(rng, (400, 64)))
    codes, s, o = quant.int4_head_quantize(x)
    u64 = x.astype(np.float64) / s.astype(np.float64)[:, None] + o.astype(np.float64)[:, None]
    c64 = np.clip(np.rint(u64), 0, 15)
    near_tie = np.abs(u64 - np.floor(u64) - 0.5) < 2.0 ** -16
    assert np.array_equal(codes[~near_tie], c64[~near_tie])


def test_int4_head_cache_round_trip_and_decode_close_to_bf16():
    rng = np.random.default_rng(42)
    lens = [300, 129, 40]
    H, d, P = 2, 64, 16
    n_pages = [-(-T // P) for T in lens]
    pool = sum(n_pages) + 2
    indices = rng.permutation(pool)[:sum(n_pages)]
    indptr = np.concatenate([[0], np.cumsum(n_pages)])
    ri = np.concatenate([[0], np.cumsum(lens)])
    k = _bf16(rng, (ri[-1], H, d))
    v = _bf16(rng, (ri[-1], H, d))
    ref = cm.empty_paged("bf16", pool, H, P, d, 3)
    cm.write_history(ref, indptr, indices, ri, k, v)
    c = cm.empty_paged("int4_head", pool, H, P, d, 3)
    cm.write_history(c, indptr, indices, ri, k, v)
    assert c.k.shape == (pool, H, P, d // 2) and c.k_qp.shape == (pool, H, P, 2)
    for b, T in enumerate(lens):
        t = np.arange(T)
        pages = indices[indptr[b] + t // P]
        for h in range(H):
            K0, V0 = cm.read_rows(ref, b, h, t)
            K1, V1 = cm.read_rows(c, b, h, t)
            ks = c.k_qp[pages, h, t % P, 0].astype(np.float64)[:, None]
            vs = c.v_qp[pages, h, t % P, 0].astype(np.float64)[:, None]
            assert np.all(np.abs(K1 - K0) <= 0.5 * ks * (1 + 1e-5) + 1e-7)
            assert np.all(np.abs(V1 - V0) <= 0.5 * vs * (1 + 1e-5) + 1e-7)
            # the byte layout: even channel in the low nibble of byte c / 2
            kc = c.k[pages, h, t % P]
            assert np.array_equal(kc[:, 3] & 0xF, quant.int4_head_quantize(quant.bf16_bits_to_f32(
                k[ri[b]:ri[b + 1], h]))[0][:, 6])
    problem = dict(B=3, S_q=1, H_q=4, H_kv=H, d=d)
    q = _bf16(rng, (3, 1, 4, d))
    O0, L0 = attention.decode_rows(problem, ref, q)
    O1, L1 = attention.decode_rows(problem, c, q)
    assert np.max(np.abs(O1 - O0)) < 0.5
