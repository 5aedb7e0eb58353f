"""Pins of the oracle's address translation (M4.5 §0x04A-§0x04I)."""

import numpy as np
import pytest

from oracle import address as ad
from oracle import cache as cm
from tests.conftest import golden


def test_gqa_head_map():
    g = golden("address_fixture.json")["gqa"]
    assert ad.kv_head(g["h_q"], g["H_q"], g["H_kv"]) == g["h_kv"]
    assert [ad.kv_head(h, 8, 2) for h in range(8)] == [0, 0, 0, 0, 1, 1, 1, 1]
    with pytest.raises(ValueError):
        ad.kv_head(0, 6, 4)


def test_contiguous_offsets():
    g = golden("address_fixture.json")["contiguous"]
    args = (g["c"], g["t"], g["h_kv"], g["x"], g["T_c"], g["H_kv"], g["d_h"])
    assert list(ad.contig_strides_nhd(g["T_c"], g["H_kv"], g["d_h"])) == g["nhd_strides"]
    assert list(ad.contig_strides_hnd(g["T_c"], g["H_kv"], g["d_h"])) == g["hnd_strides"]
    assert ad.offset_contig_nhd(*args) == g["nhd_offset"]
    assert ad.offset_contig_nhd(*args) * g["b_e"] == g["nhd_bytes"]
    assert ad.offset_contig_hnd(*args) == g["hnd_offset"]
    assert ad.offset_contig_hnd(*args) * g["b_e"] == g["hnd_bytes"]


def test_contiguous_offsets_match_numpy_ravel():
    """np.ravel_multi_index is an independent implementation of the stride dot product."""
    B_c, T_c, H, d = 3, 7, 2, 5
    for c in range(B_c):
        for t in range(T_c):
            for h in range(H):
                for x in range(d):
                    assert ad.offset_contig_nhd(c, t, h, x, T_c, H, d) == \
                        np.ravel_multi_index((c, t, h, x), (B_c, T_c, H, d))
                    assert ad.offset_contig_hnd(c, t, h, x, T_c, H, d) == \
                        np.ravel_multi_index((c, h, t, x), (B_c, H, T_c, d))


def test_ragged_rows():
    g = golden("address_fixture.json")["ragged"]
    assert list(np.concatenate([[0], np.cumsum(g["lengths"])])) == g["indptr"]
    assert ad.ragged_row(g["indptr"], g["request"], g["t"]) == g["row"]
    with pytest.raises(IndexError):
        ad.ragged_row(g["indptr"], 1, 7)


def test_page_segments_trace():
    g = golden("address_fixture.json")["paged"]
    a, e = g["split"]
    segs = ad.page_segments(lambda j: g["table"][j], a, e, g["P"])
    assert [list(s) for s in segs] == g["segments"]
    assert ad.n_segments(a, e, g["P"]) == len(g["segments"])
    # dense table and CSR list yield the same physical page for every visible block
    indptr, indices = [0, 3], g["table"]
    for j in range(3):
        assert ad.page_dense([g["table"]], 0, j) == ad.page_csr(indptr, indices, 0, j)


def test_n_segments_brute_force():
    for P in (1, 3, 4, 16):
        for a in range(0, 40):
            for e in range(a, 45):
                touched = {t // P for t in range(a, e)}
                assert ad.n_segments(a, e, P) == len(touched)


def test_page_tail_visibility_and_csr_length():
    g = golden("address_fixture.json")["page_tail"]
    assert ad.visible_rows_of_page(g["T"], 2, g["P"]) == g["visible_rows"]
    assert ad.csr_context_length(3, 2, 4) == g["T"]
    with pytest.raises(ValueError):
        ad.csr_context_length(3, 0, 4)


def test_metadata_bytes():
    g = golden("address_fixture.json")["metadata_bytes"]
    assert 4 * 3 * 4 == g["dense_bytes"] == g["dense_entries"] * 4
    # four row pointers, seven page ids, three last-page lengths
    assert (4 + 7 + 3) == g["csr_entries"] and g["csr_entries"] * 4 == g["csr_bytes"]


def test_payload_id_exhaustive_recovery_paged_hnd():
    """Write unique ids through the page walk, read every visible coordinate back."""
    rng = np.random.default_rng(3)
    H, d, P = 2, 4, 4
    lens = [10, 7, 5]
    n_pages = [(-(-T // P)) for T in lens]
    pool_pages = sum(n_pages) + 3
    perm = rng.permutation(pool_pages)
    indptr = np.concatenate([[0], np.cumsum(n_pages)])
    indices = perm[:indptr[-1]]
    pool = np.full((pool_pages, H, P, d), -1, np.int64)
    ids = {}
    for b, T in enumerate(lens):
        for t in range(T):
            for h in range(H):
                for x in range(d):
                    pid = 1000 * b + 100 * h + 10 * t + x
                    pi = ad.page_csr(indptr, indices, b, t // P)
                    o = ad.offset_paged_hnd(pi, t % P, h, x, P, H, d)
                    assert o not in ids, "address collision"
                    ids[o] = pid
                    pool.reshape(-1)[o] = pid
    c = cm.Cache("paged", "bf16", H, d, P=P, page_indptr=indptr, page_indices=indices,
                 kv_len=np.array(lens))
    for b, T in enumerate(lens):
        for h in range(H):
            pages, rows = cm._pages_and_rows(c, b, np.arange(T))
            got = pool[pages, h, rows, :]
            want = np.array([[1000 * b + 100 * h + 10 * t + x for x in range(d)] for t in range(T)])
            assert np.array_equal(got, want)
    with pytest.raises(IndexError):
        cm._pages_and_rows(c, 0, np.array([10]))      # allocated tail is not visible
