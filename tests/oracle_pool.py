"""The fp64 oracle over many query rows at once, in parallel worker processes.

Test infrastructure only.  The full-size parity tests compare every query row
of the benchmark workloads with the oracle; one process takes tens of seconds
on the larger ones, so the rows are split by request over a pool of
single-threaded workers.  The pool is started with "spawn" (never forked from
a process that has touched the GPU), the workers import only numpy and
``oracle``, and the inputs reach them as .npy files that each worker maps
read-only.

Two kinds of input:

* "cache": a bf16 cache as the GPU path stores it (paged, contiguous or
  packed rows); the worker builds the oracle's view of it and decodes.
* "history": packed bf16 history rows and page tables of a quantized cache;
  each worker writes its requests' histories with the oracle's own quantiser
  into a pool of its own (the requests' pages renumbered in order, so the
  pool holds only them) and decodes from it.
"""

from __future__ import annotations

import multiprocessing as mp
import os
import tempfile

import numpy as np


_THREAD_VARS = ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS")


def _load(path, name):
    f = os.path.join(path, name + ".npy")
    return np.load(f, mmap_mode="r") if os.path.exists(f) else None


def _cache_view(path, spec):
    from oracle import cache as ocache
    a = {n: _load(path, n) for n in ("k", "v", "page_indptr", "page_indices", "kv_len", "cache_batch_idx",
                                      "row_offsets", "position_map")}
    kv_len = np.asarray(a["kv_len"], np.int64)
    if spec["layout"] == "packed":
        return ocache.Cache("packed", "bf16", spec["H_kv"], spec["d"], k=a["k"], v=a["v"], kv_len=kv_len,
                            extra={"row_offsets": np.asarray(a["row_offsets"], np.int64),
                                   "position_map": np.asarray(a["position_map"], np.int64)})
    if spec["layout"] == "contig":
        c = ocache.Cache("contig", "bf16", spec["H_kv"], spec["d"], T_c=spec["T_cap"], k=a["k"], v=a["v"],
                         kv_len=kv_len)
        if a["cache_batch_idx"] is not None:
            c.cache_batch_idx = np.asarray(a["cache_batch_idx"])
        return c
    return ocache.Cache("paged", "bf16", spec["H_kv"], spec["d"], P=spec["P"], k=a["k"], v=a["v"],
                        page_indptr=np.asarray(a["page_indptr"], np.int64),
                        page_indices=np.asarray(a["page_indices"], np.int64), kv_len=kv_len)


def _history_view(path, spec, requests):
    """The oracle's own quantized cache holding only ``requests``' histories."""
    from oracle import cache as ocache
    k_rows, v_rows = _load(path, "k_rows"), _load(path, "v_rows")
    ri = np.asarray(_load(path, "rows_indptr"), np.int64)
    pi = np.asarray(_load(path, "page_indptr"), np.int64)
    px = np.asarray(_load(path, "page_indices"), np.int64)
    B = len(ri) - 1
    keep = np.zeros(B, bool)
    keep[list(requests)] = True
    n_rows = np.where(keep, np.diff(ri), 0)
    n_pages = np.where(keep, np.diff(pi), 0)
    sub_ri = np.concatenate([[0], np.cumsum(n_rows)])
    sub_pi = np.concatenate([[0], np.cumsum(n_pages)])
    mine = np.concatenate([px[pi[b]:pi[b + 1]] for b in range(B) if keep[b]])
    sub_px = np.argsort(np.argsort(mine))          # the requests' pages renumbered 0.. in pool order
    rows = np.concatenate([np.arange(ri[b], ri[b + 1]) for b in range(B) if keep[b]])
    c = ocache.empty_paged(spec["fmt"], len(mine), spec["H_kv"], spec["P"], spec["d"], B, G=spec["G"],
                           Gv=spec["Gv"], R=spec["R"], k_scale=spec.get("k_scale"), v_scale=spec.get("v_scale"))
    ocache.write_history(c, sub_pi, sub_px, sub_ri, np.asarray(k_rows[rows]), np.asarray(v_rows[rows]))
    c.kv_len = np.diff(ri)
    return c


def _job(args):
    path, spec, problem, requests, rows = args
    from oracle import attention
    cache = _history_view(path, spec, requests) if spec["kind"] == "history" else _cache_view(path, spec)
    q = np.load(os.path.join(path, "q.npy"), mmap_mode="r")
    return attention.decode_rows(problem, cache, np.asarray(q), rows)


def _balanced(units, cost, n):
    """Units of work dealt to n workers, heaviest first onto the least loaded."""
    load = [0.0] * n
    parts = [[] for _ in range(n)]
    for u in sorted(units, key=lambda u: -cost[u]):
        i = int(np.argmin(load))
        parts[i].append(u)
        load[i] += cost[u]
    return [p for p in parts if p]


def decode_rows_parallel(problem, spec, arrays, q_bits, rows, workers=None):
    """O [n, d], LSE [n] of ``rows`` = [(b, i, h_q), ...] by the oracle, in worker processes.

    ``spec`` names the input kind and its scalars; ``arrays`` maps the .npy
    names the kind reads to numpy arrays (bf16 data as uint16 bit patterns)."""
    # rows of one (request, kv head) share their K/V rows: the unit of work ("history"
    # inputs are written per request, so there the unit is the request)
    g = problem["H_q"] // problem["H_kv"]
    unit = (lambda r: r[0]) if spec["kind"] == "history" else (lambda r: (r[0], r[2] // g))
    by_req = {}
    for n, r in enumerate(rows):
        by_req.setdefault(unit(r), []).append(n)
    kv_len = np.asarray(arrays["kv_len"], np.int64)
    cost = {u: (1 + int(kv_len[rows[ix[0]][0]])) * len(ix) for u, ix in by_req.items()}
    workers = workers or min(16, os.cpu_count() or 1)
    parts = _balanced(by_req, cost, max(1, min(workers, len(by_req))))
    O = np.zeros((len(rows), int(spec["d"])))
    L = np.zeros(len(rows))
    with tempfile.TemporaryDirectory() as path:
        for name, a in arrays.items():
            if a is not None:
                np.save(os.path.join(path, name + ".npy"), np.ascontiguousarray(a))
        np.save(os.path.join(path, "q.npy"), np.ascontiguousarray(q_bits))
        jobs = []
        for part in parts:
            ix = [n for u in part for n in by_req[u]]
            requests = sorted({rows[n][0] for n in ix})
            jobs.append((ix, (path, spec, problem, requests, [rows[n] for n in ix])))
        if len(jobs) == 1:
            results = [_job(jobs[0][1])]
        else:
            # one BLAS thread per worker (the children read these when numpy loads)
            saved = {k: os.environ.get(k) for k in _THREAD_VARS}
            os.environ.update({k: "1" for k in _THREAD_VARS})
            try:
                with mp.get_context("spawn").Pool(len(jobs)) as pool:
                    results = pool.map(_job, [j[1] for j in jobs])
            finally:
                for k, v in saved.items():
                    if v is None:
                        os.environ.pop(k, None)
                    else:
                        os.environ[k] = v
        for (ix, _), (o, l) in zip(jobs, results):
            O[ix] = o
            L[ix] = l
    return O, L
