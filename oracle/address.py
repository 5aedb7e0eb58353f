"""Read-side K/V address translation, written out from the formulas.

Test infrastructure only (see ``oracle/__init__.py``).

Follows "M4.5 Decode Attention Kernels, Mask Programs, and Backend
Boundaries", §0x04A-§0x04F:

* §0x04A  request identity (cache_batch_idx) and GQA head h_kv = floor(h_q / g);
* §0x04B  contiguous NHD and HND element offsets;
* §0x04C  packed ragged rows p = indptr[r] + t;
* §0x04D  paged dense block table and CSR page list, NHD/HND page offsets,
          T = P (n_pages - 1) + last_page_len;
* §0x04E  page-segment iteration and n_seg;
* §0x04F  allocated tail rows are not visible.
"""

from __future__ import annotations


def kv_head(h_q: int, H_q: int, H_kv: int) -> int:
    """h_kv = floor(h_q / g) with g = H_q / H_kv  (§0x04A, §0x03A)."""
    if H_q % H_kv:
        raise ValueError("H_q must be a multiple of H_kv")
    return h_q // (H_q // H_kv)


def offset_contig_nhd(c, t, h_kv, x, T_c, H_kv, d_h):
    """o_NHD = ((c T_c + t) H_kv + h_kv) d_h + x  (§0x04B)."""
    return ((c * T_c + t) * H_kv + h_kv) * d_h + x


def offset_contig_hnd(c, t, h_kv, x, T_c, H_kv, d_h):
    """o_HND = ((c H_kv + h_kv) T_c + t) d_h + x  (§0x04B)."""
    return ((c * H_kv + h_kv) * T_c + t) * d_h + x


def contig_strides_nhd(T_c, H_kv, d_h):
    """Element strides of [B_c, T_c, H_kv, d_h]  (§0x04B)."""
    return (T_c * H_kv * d_h, H_kv * d_h, d_h, 1)


def contig_strides_hnd(T_c, H_kv, d_h):
    """Element strides of [B_c, H_kv, T_c, d_h]  (§0x04B)."""
    return (H_kv * T_c * d_h, T_c * d_h, d_h, 1)


def ragged_row(indptr, r, t):
    """Packed row p = indptr[r] + t, requiring 0 <= t < T_r  (§0x04C)."""
    if not 0 <= t < indptr[r + 1] - indptr[r]:
        raise IndexError("token outside the request's packed rows")
    return indptr[r] + t


def offset_ragged_nhd(p, h_kv, x, H_kv, d_h):
    """o_ragged = (p H_kv + h_kv) d_h + x  (§0x04C)."""
    return (p * H_kv + h_kv) * d_h + x


def page_dense(block_table, c, j):
    """pi = block_table[c, j]  (§0x04D)."""
    return block_table[c][j]


def page_csr(indptr, indices, i, j):
    """pi = indices[indptr[i] + j], requiring j < n_pages(i)  (§0x04D)."""
    if not 0 <= j < indptr[i + 1] - indptr[i]:
        raise IndexError("logical block outside the request's page list")
    return indices[indptr[i] + j]


def offset_paged_nhd(pi, r_p, h_kv, x, P, H_kv, d_h):
    """o_page,NHD = ((pi P + r_p) H_kv + h_kv) d_h + x  (§0x04D)."""
    return ((pi * P + r_p) * H_kv + h_kv) * d_h + x


def offset_paged_hnd(pi, r_p, h_kv, x, P, H_kv, d_h):
    """o_page,HND = ((pi H_kv + h_kv) P + r_p) d_h + x  (§0x04D)."""
    return ((pi * H_kv + h_kv) * P + r_p) * d_h + x


def csr_context_length(n_pages, last_page_len, P):
    """T = P (n_pages - 1) + last_page_len with 1 <= last <= P  (§0x04D)."""
    if n_pages == 0:
        return 0
    if not 1 <= last_page_len <= P:
        raise ValueError("last_page_len must lie in [1, P]")
    return P * (n_pages - 1) + last_page_len


def n_segments(a, e, P):
    """Pages touched by a non-empty [a, e): 1 + floor((e-1)/P) - floor(a/P)  (§0x04E)."""
    if e <= a:
        return 0
    return 1 + (e - 1) // P - a // P


def page_segments(lookup, a, e, P):
    """(physical page, first page row, rows) for each page touched by [a, e)  (§0x04E).

    ``lookup(j)`` maps a logical block j to its physical page.
    """
    out = []
    pos = a
    while pos < e:
        j, r = divmod(pos, P)
        seg_end = min(e, (j + 1) * P)
        out.append((lookup(j), r, seg_end - pos))
        pos = seg_end
    return out


def visible_rows_of_page(T, j, P):
    """Page rows of logical block j that hold visible tokens t < T  (§0x04F)."""
    return [r for r in range(P) if j * P + r < T]
