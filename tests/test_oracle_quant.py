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
