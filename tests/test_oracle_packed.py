"""Pins of the oracle's ragged packed view (M5.4 §0x04C, the two-layer, two-K/V-head trace)."""

import numpy as np
import pytest

from oracle import attention
from oracle import cache as cm
from oracle import masks, quant
from tests.test_oracle_attention import _bf16

# the trace's frozen inputs: L = 2, H_kv = 2, T = 8, d = 4, positions per (layer, head)
_SETS = [[0, 2, 5, 7], [0, 1, 6, 7], [0, 3, 4, 7], [0, 2, 6, 7]]


def _symbolic(offset):
    """K[l, h, t, c] = 1000 l + 100 h + 10 t + c (+ 5000 for V), one slice per (l, h)."""
    t = np.arange(8)[:, None]
    c = np.arange(4)[None, :]
    return [offset + 1000 * l + 100 * h + 10 * t + c for l in range(2) for h in range(2)]


def test_packed_view_trace_values():
    K, V, pmap, offsets = cm.pack_view(_symbolic(0), _symbolic(5000), _SETS)
    assert pmap.tolist() == [0, 2, 5, 7, 0, 1, 6, 7, 0, 3, 4, 7, 0, 2, 6, 7]
    assert offsets.tolist() == [0, 4, 8, 12, 16]          # the trace's [[0,4,8],[8,12,16]], flattened
    r = offsets[2 * 1 + 0] + 1                            # layer 1, K/V head 0, packed row 1
    assert pmap[r] == 3
    assert K[r].tolist() == [1030, 1031, 1032, 1033]
    assert V[r].tolist() == [6030, 6031, 6032, 6033]
    # the byte terms of the trace: full cache, selected payload, position map, offsets
    b = 2 + 2
    assert 2 * 2 * 8 * 4 * b == 512 and len(pmap) * 4 * b == 256
    assert pmap.size * 4 == 64 and 2 * 3 * 4 == 24 and 256 + 64 + 24 == 344


def test_packed_row_is_not_the_position():
    K, V, pmap, offsets = cm.pack_view(_symbolic(0), _symbolic(5000), _SETS)
    c = cm.Cache("packed", "bf16", 2, 4, k=K, v=V, kv_len=np.array([8, 8]),
                 extra={"row_offsets": offsets, "position_map": pmap})
    assert cm.packed_rows(c, 1, 1, [2, 6]).tolist() == [13, 14]
    with pytest.raises(IndexError):
        cm.packed_rows(c, 1, 1, [3])                      # not retained by that slice
    with pytest.raises(ValueError):
        cm.pack_view(_symbolic(0)[:1], _symbolic(5000)[:1], [[2, 2]])


def test_attention_over_the_packed_view_equals_the_gather_over_the_source():
    """Decode over the packed rows (positions from the map) gives the same rows as the index-
    list program over the source cache: position identity survives packing."""
    rng = np.random.default_rng(50)
    B, H, d, T = 2, 2, 64, [40, 29]
    src = [_bf16(rng, (t, H, d)) for t in T]
    srcv = [_bf16(rng, (t, H, d)) for t in T]
    sets = [np.sort(rng.choice(T[b], size=min(T[b], 11), replace=False)) for b in range(B) for _ in range(H)]
    ks = [src[b][:, h] for b in range(B) for h in range(H)]
    vs = [srcv[b][:, h] for b in range(B) for h in range(H)]
    K, V, pmap, offsets = cm.pack_view(ks, vs, sets)
    packed = cm.Cache("packed", "bf16", H, d, k=K, v=V, kv_len=np.array(T),
                      extra={"row_offsets": offsets, "position_map": pmap})
    contig = cm.Cache("contig", "bf16", H, d, T_c=max(T), kv_len=np.array(T),
                      k=np.stack([np.pad(x, ((0, max(T) - len(x)), (0, 0), (0, 0))) for x in src]),
                      v=np.stack([np.pad(x, ((0, max(T) - len(x)), (0, 0), (0, 0))) for x in srcv]))
    p = dict(B=B, S_q=2, H_q=4, H_kv=H, d=d, mask="index_list", index_indptr=offsets, index_list=pmap)
    q = _bf16(rng, (B, 2, 4, d))
    O1, L1 = attention.decode_rows(p, packed, q)
    O2, L2 = attention.decode_rows(p, contig, q)
    assert np.array_equal(O1, O2) and np.array_equal(L1, L2, equal_nan=True)
    assert np.isfinite(L1).any()
