#!/usr/bin/env python3
"""Decode-attention benchmark: paged ragged GQA decode on GB300.

Headline workload (one "step" = one decode step over the whole batch): B=16
requests, S_q=1, H_q=32, H_kv=8, d=128, bf16 K/V in 16-token pages of a
10,000-page pool, lengths uniform in [1024, 8192] (seed 1).  The step runs
the whole hot path: partial kernel and LSE merge kernel over a work list
uploaded once per step (every layer of a model reuses it).

Metric: K/V bytes read per step / step time (GB/s), with the step time in
microseconds beside it.  Timing: CUDA events on the launching stream around
exactly --steps steps after --warmup steps, barrier + synchronize on both
sides, max over ranks.  Inside the region an event closes every batch of
--steps / 50 steps, so that at least 50 raw samples of the per-step time
give min / median / p95 / max.  The K/V read per step (~307 MB) is larger
than the 129 MB L2, so no flush runs between steps.

The same line carries every other configuration of the decode contract
(tiny contiguous, long context at S_q = 1 and 4, sink + window, index lists,
INT8 and KIVI INT4), each timed the same way in this process, with the fp64
CPU oracle's time on the same inputs beside it.

--impl reference times the fp64 CPU oracle (the parity reference) on the
host cores instead, one bounded sample of the headline workload per step.
"""

from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "decode-attn K/V HBM GB/s (% of GB300 peak); µs/step, B=16 paged GQA"
NOMINAL_HBM_GBS = 8000.0
FALLBACK_HBM_GBS = 6800.0
MIN_SAMPLES = 50

# The configurations of the decode contract carried by the default line, and the
# extra workloads --workload can time alone.
CONFIGS = ("tiny", "long-s1", "long-s4", "sink-window", "index-list", "int8", "int4-kivi")
OTHER_WORKLOADS = ("tiny", "long-s1", "long-s4", "sink-window", "index-list", "packed", "tree-verify", "mixed",
                   "int8", "fp8", "fp8-e5m2", "int4-head", "int4-kivi", "int4-kivi-s4", "int4-kivi-d64", "int4-kivi-p96",
                   "tree-verify@int8", "tree-verify@int4-head", "tree-verify@int4-kivi",
                   "mixed@int8", "mixed@int4-head", "mixed@int4-kivi")
CONFIG_LABEL = {"tiny": "1 tiny contiguous", "long-s1": "3 long context S_q=1", "long-s4": "3 long context S_q=4",
                "sink-window": "4a sink + window", "index-list": "4b index lists", "int8": "5a INT8",
                "int4-kivi": "5b KIVI INT4"}
QUANT = {"int8": "int8", "fp8": "fp8_e4m3", "fp8-e5m2": "fp8_e5m2", "int4-head": "int4_head",
         "int4-kivi": "int4_kivi", "int4-kivi-s4": "int4_kivi", "int4-kivi-d64": "int4_kivi",
         "int4-kivi-p96": "int4_kivi"}


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=50)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--e2e-steps", type=int, default=400)
    ap.add_argument("--config-steps", type=int, default=600,
                    help="timed steps of each other configuration in the default line (>= 50)")
    ap.add_argument("--no-configs", action="store_true", help="headline only")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--chunk", type=int, default=0, help="planner chunk width (0 = default)")
    ap.add_argument("--merge-tags", type=int, default=0, choices=(-1, 0, 1),
                    help="the plan's merge_tags (0 = library default)")
    ap.add_argument("--fused-merge", action="store_true", help="--workload: plan with fused_merge")
    ap.add_argument("--shared-shift", default=None, metavar="PHI,LO,HI",
                    help="bf16 partials in the common frame PHI with the guard LO < s - PHI < HI")
    ap.add_argument("--workload", choices=("paged",) + OTHER_WORKLOADS, default="paged",
                    help="paged: the benchmark line; the others print one timing line for a decode step "
                         "of that workload")
    ap.add_argument("--cpu-child", nargs="*", help=argparse.SUPPRESS)
    return ap.parse_args()


# ---- workload bookkeeping -------------------------------------------------------------

def kv_bytes_per_key(p):
    return 2 * p["d"] * 2          # K row + V row, bf16


def algorithmic_bytes(w, info, items):
    """Bytes each kernel of the step must move (no GQA re-reads, no tail waste)."""
    p = w.problem
    d, P, rows = p["d"], p["P"], info["rows"]
    kv = info["stream_keys"] * kv_bytes_per_key(p)
    pages = 0
    per_group = {}
    for it in items:
        per_group[(it["b"], it["h_kv"])] = per_group.get((it["b"], it["h_kv"]), 0) + 1
        if it["e"] > it["a"]:
            pages += (it["e"] - 1) // P - it["a"] // P + 1
    q = p["B"] * p["S_q"] * p["H_q"] * d * 2
    state = info["n_slots"] * rows * (d + 2) * 4
    direct_rows = max(0, len(per_group) - info["n_merge_groups"]) * rows    # groups that write O directly
    merged_rows = info["n_merge_groups"] * rows
    out_row = d * 2 + 4
    partial = kv + 4 * pages + q + state + direct_rows * out_row + info["blob_bytes"]
    merge = state + merged_rows * out_row
    return {"kv": kv, "partial": partial, "merge": merge, "page_list": 4 * pages, "q": q,
            "workspace_state": state, "out": (direct_rows + merged_rows) * out_row}


def stream_bytes(p, info, lens):
    """K/V bytes of the visible streams of one step (what the step must read)."""
    d = p["d"]
    fmt = p.get("fmt", "bf16")
    if fmt == "bf16":
        return info["stream_keys"] * 4 * d
    if fmt == "int8":
        return info["stream_keys"] * (2 * d + 8)
    if fmt in ("fp8_e4m3", "fp8_e5m2"):
        return info["stream_keys"] * 2 * d
    if fmt == "int4_head":
        return info["stream_keys"] * (d + 8)
    G, Gv, R = p["kivi_group"], p["kivi_v_group"], p["kivi_residual"]
    total = 0
    for T in lens:      # causal (the last query row sees every stored key) or FlashMask: the whole history
        nq = G * -(-max(0, T - R) // G)
        total += nq * (d + 4 * d // Gv) + (nq // G) * 4 * d + (T - nq) * 4 * d
    return total * p["H_kv"]


def kernel_hash():
    """Hash of the partial kernel's sources: DRAM counters taken on other sources are stale."""
    h = hashlib.sha256()
    for f in ("device.cuh", "internal.h", "stream.cuh", "tc_common.cuh", "partial_bf16.cu"):
        with open(os.path.join(ROOT, "split_kv_decode_flash_gb300", "csrc", f), "rb") as fh:
            h.update(f.encode() + fh.read())
    return h.hexdigest()[:16]


def measured_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["hbm_gbs"]), "of measured"
    except Exception:
        return FALLBACK_HBM_GBS, "of fallback"


def dram_traffic():
    """Per-launch DRAM bytes of the partial kernel from the committed ncu summary, when current."""
    path = os.path.join(ROOT, "profiles", "partial_kernel_traffic.json")
    try:
        with open(path) as f:
            t = json.load(f)
        if t.get("kernel_hash") == kernel_hash():
            return t.get("dram_bytes_per_launch")
    except Exception:
        pass
    return None


def summary(samples_us):
    s = sorted(samples_us)
    p95 = s[min(len(s) - 1, int(round(0.95 * (len(s) - 1))))]
    return {"n": len(s), "min": s[0], "median": statistics.median(s), "p95": p95, "max": s[-1]}


# ---- clocks -----------------------------------------------------------------------------

class Clocks:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, uuid=None):
        self.rows = []
        cmd = ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "50"]
        if uuid:
            cmd += ["-i", uuid]
        try:
            self.proc = subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
            return
        self.t = threading.Thread(target=self._read, daemon=True)
        self.t.start()

    def _read(self):
        for line in self.proc.stdout:
            self.rows.append([x.strip() for x in line.split(",")])

    def stop(self):
        if not self.proc:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.t.join(timeout=2)
        sm = [float(r[0]) for r in self.rows if len(r) >= 8 and r[0].replace(".", "").isdigit()]
        mx = [float(r[1]) for r in self.rows if len(r) >= 8 and r[1].replace(".", "").isdigit()]
        reasons = set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in self.rows:
            if len(r) < 8:
                continue
            for n, v in zip(names, r[4:8]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        loaded = [s for s in sm if mx and s > 0.5 * max(mx)] or sm
        return {"sm_mhz": statistics.median(loaded) if loaded else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": sorted(reasons),
                "samples": len(sm)}


# ---- CPU oracle baseline ----------------------------------------------------------------
#
# The oracle runs in fresh single-threaded processes (never forked from this
# process, which holds a CUDA context) over arrays saved as .npy files: the
# bf16 cache, or the codes, qparams and residual the GPU's kv_append wrote.

def _cpu_child(args):
    """Runs in a fresh single-threaded process: time the oracle on a list of (request, kv head) groups."""
    import numpy as np
    from oracle import attention
    from oracle import cache as ocache
    path, groups = args[0], [tuple(map(int, g.split(":"))) for g in args[1:]]
    with open(os.path.join(path, "meta.json")) as f:
        meta = json.load(f)

    def arr(n):
        fn = os.path.join(path, n + ".npy")
        return np.load(fn, mmap_mode="r") if os.path.exists(fn) else None

    i64 = lambda a: None if a is None else np.asarray(a, np.int64)
    if meta["layout"] == "contig":
        c = ocache.Cache("contig", "bf16", meta["H_kv"], meta["d"], T_c=meta["T_cap"], k=arr("k"), v=arr("v"),
                         kv_len=i64(arr("kv_len")))
    else:
        c = ocache.Cache("paged", meta["fmt"], meta["H_kv"], meta["d"], P=meta["P"], k=arr("k"), v=arr("v"),
                         k_qp=arr("k_qp"), v_qp=arr("v_qp"), k_res=arr("k_res"), v_res=arr("v_res"),
                         page_indptr=i64(arr("page_indptr")), page_indices=i64(arr("page_indices")),
                         kv_len=i64(arr("kv_len")), G=meta.get("G", 32), Gv=meta.get("Gv", 32),
                         R=meta.get("R", 128))
    problem = dict(meta["problem"])
    if arr("index_list") is not None:
        problem["index_indptr"] = np.asarray(arr("index_indptr"))
        problem["index_list"] = np.asarray(arr("index_list"))
    q = np.asarray(arr("q"))
    g = problem["H_q"] // problem["H_kv"]
    min_seconds = float(os.environ.get("DATTN_CPU_MIN_SECONDS", "0"))
    warm = int(os.environ.get("DATTN_CPU_WARMUP_GROUPS", "0"))
    for b, h in groups[:warm]:          # untimed
        attention.decode_rows(problem, c, q, [(b, i, h * g + j) for i in range(problem["S_q"]) for j in range(g)])
    groups = groups[warm:]
    t0 = time.perf_counter()
    passes = 0
    while True:              # whole passes over the groups until min_seconds of work
        for b, h in groups:
            rows = [(b, i, h * g + j) for i in range(problem["S_q"]) for j in range(g)]
            attention.decode_rows(problem, c, q, rows)
        passes += 1
        if time.perf_counter() - t0 >= min_seconds:
            break
    dt = time.perf_counter() - t0
    print(json.dumps({"seconds": dt, "passes": passes}))


def save_oracle_inputs(path, w, p, cache):
    """Everything the oracle reads for workload ``w`` (device data copied back), as .npy files."""
    import numpy as np
    import torch

    def host(t, bits=False):
        t = t.detach().cpu().contiguous()
        if bits:
            return t.view(torch.int16).numpy().view(np.uint16)
        return t.numpy()

    fmt = p.get("fmt", "bf16")
    arrays = {"q": host(w.q, True), "kv_len": w.kv_len.numpy().astype(np.int64)}
    meta = {"layout": p["layout"], "fmt": fmt, "H_kv": p["H_kv"], "d": p["d"], "P": p.get("P", 0),
            "T_cap": p.get("T_cap", 0), "G": p.get("kivi_group", 32), "Gv": p.get("kivi_v_group", 32),
            "R": p.get("kivi_residual", 128),
            "problem": {k: p[k] for k in ("B", "S_q", "H_q", "H_kv", "d", "mask", "n_sink", "window") if k in p}}
    if fmt == "bf16":
        arrays.update(k=host(cache["k"], True), v=host(cache["v"], True))
    else:
        arrays.update(k=host(cache["k"]), v=host(cache["v"]))
        if fmt in ("fp8_e4m3", "fp8_e5m2"):
            arrays.update(k_qp=host(cache["k_qparams"]), v_qp=host(cache["v_qparams"]))
        else:
            arrays.update(k_qp=host(cache["k_qparams"]), v_qp=host(cache["v_qparams"]))
        if fmt == "int4_kivi":
            arrays.update(k_res=host(cache["k_residual"], True), v_res=host(cache["v_residual"], True))
    if w.page_indptr is not None:
        arrays.update(page_indptr=w.page_indptr.numpy().astype(np.int64),
                      page_indices=w.page_indices.numpy().astype(np.int64))
    if w.index_list is not None:
        arrays.update(index_indptr=w.index_indptr.numpy().astype(np.int64),
                      index_list=w.index_list.numpy().astype(np.int64))
    for n, a in arrays.items():
        np.save(os.path.join(path, n + ".npy"), a)
    with open(os.path.join(path, "meta.json"), "w") as f:
        json.dump(meta, f)


def cpu_oracle_time(path, groups_per_worker, min_seconds=0.0, warmup_groups=0):
    """Times the oracle over groups split across single-threaded processes.

    Each process first decodes its first ``warmup_groups`` groups untimed, then
    repeats whole passes over the rest for at least ``min_seconds`` and times its
    own compute (process start-up and array loading excluded); returns the
    slowest process's seconds per pass."""
    env = dict(os.environ, OMP_NUM_THREADS="1", OPENBLAS_NUM_THREADS="1", MKL_NUM_THREADS="1",
               DATTN_CPU_MIN_SECONDS=str(min_seconds), DATTN_CPU_WARMUP_GROUPS=str(warmup_groups))
    procs = []
    for gl in groups_per_worker:
        cmd = [sys.executable, os.path.abspath(__file__), "--cpu-child", path] + [f"{b}:{h}" for b, h in gl]
        procs.append(subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.PIPE, text=True, env=env))
    per_pass = 0.0
    for pr in procs:
        out, err = pr.communicate()
        if pr.returncode != 0:
            raise RuntimeError("oracle timing child failed: " + err[-2000:])
        r = json.loads(out.strip().splitlines()[-1])
        per_pass = max(per_pass, r["seconds"] / r["passes"])
    return per_pass


def cpu_baseline(path, p, kv_bytes, one_core=False, min_seconds=1.0):
    """The oracle over one whole step (every (request, kv head) group) on all host cores,
    and optionally on one core."""
    groups = [(b, h) for b in range(p["B"]) for h in range(p["H_kv"])]
    workers = max(1, min(os.cpu_count() or 1, len(groups)))
    # deal the groups round robin by request length so that every process gets a share
    split = [groups[i::workers] for i in range(workers)]
    step_s = cpu_oracle_time(path, split, min_seconds)
    out = {"value": kv_bytes / step_s / 1e9, "unit": "GB/s", "cores": workers, "kind": "oracle",
           "step_s": step_s,
           "sample": f"one whole decode step: all {len(groups)} (request, kv head) groups, every query row, "
                     f"over {workers} single-threaded processes (float64 numpy), each repeating whole passes "
                     f"for >= {min_seconds:g} s; step time = the slowest process's time per pass"}
    if one_core:
        s1 = cpu_oracle_time(path, [groups], min_seconds)
        out["one_core"] = {"value": kv_bytes / s1 / 1e9, "unit": "GB/s", "step_s": s1, "cores": 1}
    return out


# ---- distributed helpers --------------------------------------------------------------

def dist_setup(gpus):
    import torch
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        dist.init_process_group(backend)
    elif torch.cuda.is_available():
        torch.cuda.set_device(0)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x, world):
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device="cuda" if torch.cuda.is_available() else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ---- building and timing one workload -------------------------------------------------

def quantized_cache(dattn, w, fmt, dev):
    """The workload's packed bf16 history written into a fresh cache by one kv_append call."""
    import torch

    p = dict(w.problem, fmt=fmt)
    H, P, d, B, n = p["H_kv"], p["P"], p["d"], p["B"], p["num_pages"]
    G, Gv, R = p["kivi_group"], p["kivi_v_group"], p["kivi_residual"]
    c = {}
    if fmt in ("int8", "int4_head"):
        c["k"] = torch.zeros((n, H, P, d if fmt == "int8" else d // 2), dtype=torch.uint8, device=dev)
        c["k_qparams"] = torch.zeros((n, H, P, 2), dtype=torch.float16, device=dev)
        c["v_qparams"] = torch.zeros_like(c["k_qparams"])
    elif fmt in ("fp8_e4m3", "fp8_e5m2"):
        c["k"] = torch.zeros((n, H, P, d), dtype=torch.uint8, device=dev)
        c["k_qparams"] = w.meta["k_scale"].to(dev, torch.float32)     # per-head scales
        c["v_qparams"] = w.meta["v_scale"].to(dev, torch.float32)
    else:
        c["k"] = torch.zeros((n, H, P, d // 2), dtype=torch.uint8, device=dev)
        c["k_qparams"] = torch.zeros((n, H, max(1, P // G), d, 2), dtype=torch.float16, device=dev)
        c["v_qparams"] = torch.zeros((n, H, P, d // Gv, 2), dtype=torch.float16, device=dev)
        c["k_residual"] = torch.zeros((B, R, H, d), dtype=torch.bfloat16, device=dev)
        c["v_residual"] = torch.zeros_like(c["k_residual"])
    c["v"] = torch.zeros_like(c["k"])
    c["page_indptr"] = w.page_indptr.to(dev)
    c["page_indices"] = w.page_indices.to(dev)
    ws = torch.empty(dattn.kv_append_workspace_bytes(p), dtype=torch.uint8, device=dev)
    dattn.kv_append(p, dattn.tensors_from(**c), w.k_rows.to(dev), w.v_rows.to(dev), [0] * B,
                    w.rows_indptr.tolist(), w.page_indptr, ws)
    torch.cuda.synchronize()
    assert int(ws[:4].view(torch.int32).item()) == 0, "kv_append device check fired"
    return p, c


def build_workload(dattn, name, dev):
    """(workload, problem, device cache tensors) of a named workload."""
    import workloads as W
    if "@" in name:
        # BASE@FMT: the tree-verify or mixed workload (its lengths, query, FlashMask intervals
        # and qo_indptr) over a cache of format FMT written by kv_append from bf16 history
        base, fq = name.split("@")
        src = {"tree-verify": W.tree_verify, "mixed": W.mixed_batch}[base]("cpu")
        fmt, p0 = QUANT[fq], src.problem
        w = W.quantized_history(f"{src.name}, {fmt} K/V", B=p0["B"], S_q=p0["S_q"], H_q=p0["H_q"],
                                H_kv=p0["H_kv"], d=p0["d"], lens=src.kv_len.tolist(), P=p0["P"], seed=7,
                                device=dev, fmt=fmt)
        w.problem = dict(w.problem, mask=p0["mask"])
        w.q, w.qo_indptr, w.fm_intervals = src.q.to(dev), src.qo_indptr, src.fm_intervals
        p, cache = quantized_cache(dattn, w, fmt, dev)
        if w.fm_intervals is not None:
            cache["fm_intervals"] = w.fm_intervals.to(dev).contiguous()
        w.k_rows = w.v_rows = None
        return w, p, cache
    if name in QUANT:
        # int4-kivi-s4: the quantized workload with 4 verify rows per request (16 rows per kv
        # head); int4-kivi-d64: 64-channel heads (V channel groups of 16); int4-kivi-p96:
        # 96-token pages, the KIVI shape that runs on the CUDA-core byte-format kernel
        w = W.quantized(dev, fmt=QUANT[name], S_q=4 if name.endswith("-s4") else 1,
                        d=64 if name.endswith("-d64") else 128, P=96 if name.endswith("-p96") else 16)
        p, cache = quantized_cache(dattn, w, QUANT[name], dev)
        w.k_rows = w.v_rows = None          # the bf16 history is no longer needed
        return w, p, cache
    w = {"paged": lambda: W.paged_ragged_gqa(dev), "tiny": lambda: W.tiny_contiguous(dev),
         "long-s1": lambda: W.long_context(dev, 1), "long-s4": lambda: W.long_context(dev, 4),
         "sink-window": lambda: W.retention(dev, "sink_window"),
         "index-list": lambda: W.retention(dev, "index_list"),
         "packed": lambda: W.packed_view(W.retention(dev, "index_list")),
         "tree-verify": lambda: W.tree_verify(dev), "mixed": lambda: W.mixed_batch(dev)}[name]()
    p = w.problem
    cache = dict(k=w.k, v=w.v)
    if w.page_indptr is not None:
        cache.update(page_indptr=w.page_indptr.to(dev), page_indices=w.page_indices.to(dev))
    if w.cache_batch_idx is not None:
        cache.update(cache_batch_idx=w.cache_batch_idx.to(dev))
    if w.index_list is not None:
        cache.update(index_indptr=w.index_indptr.to(dev), index_list=w.index_list.to(dev))
    if w.fm_intervals is not None:
        cache.update(fm_intervals=w.fm_intervals.to(dev).contiguous())
    return w, p, cache


class Step:
    """A planned decode step of one workload with its buffers, uploaded once."""

    def __init__(self, dattn, w, p, cache, dev, num_sms, chunk=0, shift=None, merge_tags=0, fused_merge=False):
        import torch
        self.dattn, self.p, self.shift = dattn, p, shift
        self.plan = dattn.dattn_plan(p, w.kv_len, page_indptr=w.page_indptr, index_indptr=w.index_indptr,
                                     index_list=w.index_list, num_sms=num_sms, chunk_tokens=chunk,
                                     qo_indptr=w.qo_indptr, merge_tags=merge_tags, fused_merge=fused_merge)
        self.info = self.plan.info
        n_rows = p["B"] * p["S_q"] if w.qo_indptr is None else int(w.qo_indptr[-1])   # packed query rows
        self.o = torch.empty((n_rows, p["H_q"], p["d"]), dtype=torch.bfloat16, device=dev)
        self.lse = torch.empty((n_rows, p["H_q"]), dtype=torch.float32, device=dev)
        self.t = dattn.tensors_from(q=w.q.to(dev), o=self.o, lse=self.lse, **cache)
        self.ws = torch.empty(self.plan.workspace_bytes, dtype=torch.uint8, device=dev)
        self.stream = torch.cuda.current_stream()
        dattn.dattn_plan_upload(self.plan, self.ws, self.stream)
        self.merges = 1 if self.info["n_merge_groups"] and not self.info["fused_merge"] else 0

    def run(self, events=None):
        self.dattn.dattn_run_ex(self.plan, self.p, self.t, self.ws, reuse_upload=True, events=events,
                                shared_shift=self.shift, stream=self.stream)

    def status(self):
        return self.dattn.dattn_device_status(self.ws, self.stream)


def timed_samples(step, K, warmup, world=1):
    """K steps back to back after ``warmup`` steps; an event closes every batch of
    max(1, K // MIN_SAMPLES) steps.  Returns (per-step µs samples, total ms)."""
    import torch
    m = max(1, K // MIN_SAMPLES)
    bounds = list(range(0, K, m)) + [K]
    if len(bounds) > 2 and bounds[-1] - bounds[-2] < m:
        bounds.pop(-2)            # the short last batch joins the one before
    evs = [torch.cuda.Event(enable_timing=True) for _ in bounds]
    for e in evs:
        e.record(step.stream)     # materialise the events before use
    for _ in range(warmup):
        step.run()
    barrier(world)
    torch.cuda.synchronize()
    j = 0
    for k in range(K + 1):
        if j < len(bounds) and bounds[j] == k:
            evs[j].record(step.stream)
            j += 1
        if k < K:
            step.run()
    torch.cuda.synchronize()
    barrier(world)
    samples = [evs[i].elapsed_time(evs[i + 1]) * 1e3 / (bounds[i + 1] - bounds[i]) for i in range(len(bounds) - 1)]
    return samples, evs[0].elapsed_time(evs[-1])


def timed_unbroken(step, K, warmup, world=1):
    """K steps back to back after ``warmup`` steps between two events only (no event
    inside the region can stop a kernel from launching under its predecessor's tail):
    total ms."""
    import torch
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    for _ in range(warmup):
        step.run()
    barrier(world)
    torch.cuda.synchronize()
    start.record(step.stream)
    for _ in range(K):
        step.run()
    end.record(step.stream)
    torch.cuda.synchronize()
    barrier(world)
    return start.elapsed_time(end)


def kernel_pass(step, K):
    """K steps with events around each kernel (this breaks the programmatic overlap of the
    two kernels, so it is a separate pass): mean partial and merge µs."""
    import torch
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(K)]
    for e3 in evs:
        for e in e3:
            e.record(step.stream)
    torch.cuda.synchronize()
    for k in range(K):
        step.run(events=evs[k])
    torch.cuda.synchronize()
    part = [evs[k][0].elapsed_time(evs[k][1]) * 1e3 for k in range(K)]
    merge = [evs[k][1].elapsed_time(evs[k][2]) * 1e3 for k in range(K)]
    return statistics.mean(part), statistics.mean(merge)


def timeline(step, n_steps=40, skip=10):
    """Per-step phases from the kernels' %globaltimer trace (bf16 K/V; dattn_run_options.trace):
    medians over steps of each phase in µs.  Steps run back to back as in the timed region."""
    import numpy as np
    import torch
    if step.p.get("fmt", "bf16") != "bf16":
        return None
    info = step.info
    n_ctas, words_m = info["n_ctas"], 2 * info["n_merge_groups"] * info["rows"]
    words = 16 * n_ctas + words_m
    buf = torch.zeros((n_steps, words), dtype=torch.int64, device=step.ws.device)
    torch.cuda.synchronize()
    for k in range(n_steps):
        step.dattn.dattn_run_ex(step.plan, step.p, step.t, step.ws, reuse_upload=True, trace=buf[k],
                                shared_shift=step.shift, stream=step.stream)
    torch.cuda.synchronize()
    tr = buf.cpu().numpy().astype(np.float64)
    rows = []
    prev_merge_end = None
    per_sm = {}
    for k in range(n_steps):
        P = tr[k, :16 * n_ctas].reshape(n_ctas, 16)
        if k >= skip:      # each CTA's streaming time by the SM it ran on
            for c in range(n_ctas):
                if P[c, 2] > 0:
                    per_sm.setdefault(int(P[c, 5]), []).append((P[c, 8:16].max() - P[c, 2]) / 1e3)
        M = tr[k, 16 * n_ctas:].reshape(-1, 2)
        M = M[M[:, 0] > 0]
        live = P[:, 2] > 0                                   # CTAs whose producer passed the wait
        wait = P[live, 2]
        end = P[:, 8:16].max(axis=1)
        merge_start = M[:, 0].min() if len(M) else end.max()
        merge_end = M[:, 1].max() if len(M) else end.max()
        if prev_merge_end is not None and k >= skip:
            rows.append({
                "wait_after_prev_step_us": (np.median(wait) - prev_merge_end) / 1e3,
                "first_page_after_wait_us": (np.median(P[live & (P[:, 6] > 0), 6] - P[live & (P[:, 6] > 0), 2]) / 1e3
                                             if (live & (P[:, 6] > 0)).any() else None),
                "first_copy_after_wait_us": np.median(P[live, 3] - wait) / 1e3,
                "first_stage_after_wait_us": np.median(P[live & (P[:, 4] > 0), 4] - P[live & (P[:, 4] > 0), 2]) / 1e3,
                "stream_median_cta_us": (np.median(end) - np.median(wait)) / 1e3,
                "tail_last_cta_us": (end.max() - np.median(end)) / 1e3,
                "cta_end_spread_p5_p95_us": (np.percentile(end, 95) - np.percentile(end, 5)) / 1e3,
                # the merge of a group starts once its states are tagged, so it may begin
                # before the last partial CTA ends (a negative wait)
                "merge_wait_after_last_cta_us": (merge_start - end.max()) / 1e3,
                "merge_us": (merge_end - merge_start) / 1e3,
                "merge_end_after_last_cta_us": (merge_end - end.max()) / 1e3,
                "period_us": (merge_end - prev_merge_end) / 1e3,
            })
        prev_merge_end = merge_end
    if not rows:
        return None
    out = {}
    for k in rows[0]:      # a phase the step's producer does not stamp is None
        vals = [r[k] for r in rows if r[k] is not None]
        out[k] = float(np.median(vals)) if vals else None
    # how much of the CTAs' spread belongs to the SM (same SM slow in every step) rather than
    # to the step: the variance of the per-SM means over the variance of all samples
    allv = [x for v in per_sm.values() for x in v]
    means = [np.mean(v) for v in per_sm.values() if len(v) > 1]
    if len(allv) > 2 and np.var(allv) > 0 and len(means) > 2:
        out["cta_time_share_of_variance_by_sm"] = float(np.var(means) / np.var(allv))
    return out


# ---- the two arms ---------------------------------------------------------------------

def run_reference(args):
    """Times the fp64 oracle on the host cores: each step is one (request, kv head) group."""
    import torch
    world, rank, _ = dist_setup(args.gpus)
    if rank != 0:
        return
    import workloads as W
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    w = W.paged_ragged_gqa(dev)
    p = w.problem
    groups = [(b, h) for b in range(p["B"]) for h in range(p["H_kv"])]
    seq = [groups[i % len(groups)] for i in range(args.warmup + args.steps)]
    with tempfile.TemporaryDirectory() as td:
        save_oracle_inputs(td, w, p, dict(k=w.k, v=w.v))
        wall = cpu_oracle_time(td, [seq], warmup_groups=args.warmup)
    nbytes = sum(int(w.kv_len[b]) for b, _ in seq[args.warmup:]) * kv_bytes_per_key(p)
    value = nbytes / wall / 1e9
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": wall * 1e3 / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic",
            "config": {"workload": w.name, "per_step": "one (request, kv head) group of the decode step",
                       "l2": "host run"},
            "cpu_baseline": {"value": value, "unit": "GB/s", "cores": 1, "kind": "oracle",
                             "sample": f"{args.steps} (request, kv head) groups cycled over the batch, "
                                       f"after {args.warmup} untimed ones, in one single-threaded process "
                                       f"(float64 numpy; its start-up and array loading not timed)"},
            "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def e2e_legs(dattn, w, p, info, dev, steps, world):
    """The headline metric through the public host-memory API, copies included.

    overlapped: dattn_step_host_submit_ex / _finish two steps deep, with the transfers
    on two streams of their own and one workspace per slot, so step k+1's inputs go up
    and step k-1's outputs come down while step k's kernels run; pipelined: the same
    with dattn_step_host_submit (transfers on the kernels' stream, one workspace), so
    only the host work overlaps; sync: one blocking dattn_step_host per step."""
    import torch
    props = torch.cuda.get_device_properties(dev)
    q_host = w.q.cpu().pin_memory()
    o_host = torch.empty((p["B"], p["S_q"], p["H_q"], p["d"]), dtype=torch.bfloat16).pin_memory()
    lse_host = torch.empty((p["B"], p["S_q"], p["H_q"]), dtype=torch.float32).pin_memory()
    io = dattn.host_step(q_host, w.kv_len, o_host, lse=lse_host, page_indptr=w.page_indptr,
                         page_indices=w.page_indices, num_sms=props.multi_processor_count)
    ws_bytes, staging_bytes = dattn.dattn_step_host_sizes(p, io)
    wss = [torch.empty(ws_bytes, dtype=torch.uint8, device=dev) for _ in range(2)]
    ws = wss[0]
    staging = [torch.empty(staging_bytes, dtype=torch.uint8).pin_memory() for _ in range(2)]
    done = [torch.cuda.Event(), torch.cuda.Event()]
    cache = dattn.tensors_from(k=w.k, v=w.v)
    stream = torch.cuda.current_stream()
    copy_streams = (torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev))
    side = [(torch.cuda.Event(), torch.cuda.Event()) for _ in range(2)]

    def overlapped(n):
        def submit(k):
            dattn.dattn_step_host_submit_ex(p, io, cache, staging[k % 2], wss[k % 2], done[k % 2], *copy_streams,
                                            *side[k % 2], stream=stream)
        submit(0)
        for k in range(1, n + 1):
            if k < n:
                submit(k)
            dattn.dattn_step_host_finish(p, io, staging[(k - 1) % 2], done[(k - 1) % 2])

    def pipelined(n):
        dattn.dattn_step_host_submit(p, io, cache, staging[0], ws, done[0], stream)
        for k in range(1, n + 1):
            if k < n:
                dattn.dattn_step_host_submit(p, io, cache, staging[k % 2], ws, done[k % 2], stream)
            dattn.dattn_step_host_finish(p, io, staging[(k - 1) % 2], done[(k - 1) % 2])

    def sync(n):
        for _ in range(n):
            dattn.dattn_step_host(p, io, cache, staging[0], ws, stream)

    out = {}
    for name, fn in (("overlapped", overlapped), ("pipelined", pipelined), ("sync", sync)):
        fn(5)
        barrier(world)
        t0 = time.perf_counter()
        fn(steps)
        out[name] = max_over_ranks((time.perf_counter() - t0) / steps, world)
    for x in wss:
        assert dattn.dattn_step_host_status(p, io, x, stream) == 0, "device bounds check fired (e2e)"
    h2d = (q_host.numel() * 2 + w.page_indptr.numel() * 4 + w.page_indices.numel() * 4 + info["blob_bytes"])
    d2h = o_host.numel() * 2 + lse_host.numel() * 4
    return out, h2d, d2h


def config_line(dattn, name, dev, num_sms, steps, cpu=True):
    """One configuration of the contract: samples, merge share and the CPU oracle beside."""
    import torch
    w, p, cache = build_workload(dattn, name, dev)
    step = Step(dattn, w, p, cache, dev, num_sms)
    for _ in range(3):
        step.run()
    torch.cuda.synchronize()
    assert step.status() == 0, f"device bounds check fired ({name})"
    total_ms = timed_unbroken(step, steps, 20)
    samples, _ = timed_samples(step, steps, 3)
    part_us, merge_us = kernel_pass(step, min(200, steps))
    tl = timeline(step)
    nb = stream_bytes(p, step.info, w.kv_len.tolist())
    peak, _ = measured_peak()
    s = summary(samples)
    out = {"config": CONFIG_LABEL.get(name, name), "workload": w.name, "us_per_step": s,
           "us_per_step_mean": total_ms * 1e3 / steps, "kv_bytes_per_step": nb,
           "GBps_median": nb / s["median"] / 1e3, "frac_of_nominal_8TBps": nb / s["median"] / 1e3 / NOMINAL_HBM_GBS,
           "frac_of_measured_hbm": nb / s["median"] / 1e3 / peak, "rows": step.info["rows"],
           "n_items": step.info["n_items"],
           "merge_share": merge_us / (part_us + merge_us) if step.merges else 0.0,
           "kernel_event_pass_us": {"partial": part_us, "merge": merge_us},
           "gpu_launches_per_step": 1 + step.merges}
    if tl:
        out["timeline"] = tl
    if cpu:
        try:
            with tempfile.TemporaryDirectory() as td:
                save_oracle_inputs(td, w, p, cache)
                out["cpu_oracle"] = cpu_baseline(td, p, nb, one_core=name in ("tiny", "index-list"))
        except Exception as e:  # reported, never required for the GPU numbers
            out["cpu_oracle"] = {"value": None, "sample": f"failed: {e}"[:300]}
    del step, cache, w
    torch.cuda.empty_cache()
    return out


def run_ours(args):
    import torch

    import split_kv_decode_flash_gb300 as dattn

    world, rank, local = dist_setup(args.gpus)
    assert torch.cuda.is_available(), "bench.py --impl ours needs a GPU"
    dattn.load()
    dev = torch.device("cuda", torch.cuda.current_device())
    props = torch.cuda.get_device_properties(dev)
    num_sms = props.multi_processor_count
    w, p, cache = build_workload(dattn, "paged", dev)
    step = Step(dattn, w, p, cache, dev, num_sms, chunk=args.chunk, shift=_shift(args), merge_tags=args.merge_tags)
    info = step.info
    ab = algorithmic_bytes(w, info, step.plan.items())
    for _ in range(max(3, args.warmup)):
        step.run()
    torch.cuda.synchronize()
    assert step.status() == 0, "device bounds check fired"

    uuid = None
    try:
        uuid = "GPU-" + str(props.uuid)
    except Exception:
        pass
    clocks = Clocks(uuid)
    time.sleep(0.2)
    # Timed region: K steps back to back, an event closing every batch of K / 50
    # steps (the raw samples).  Events between the partial and the merge kernel
    # would stop the merge from launching programmatically under the partial
    # kernel's tail, so the per-kernel events are taken in a separate pass.
    K = args.steps
    total_ms = timed_unbroken(step, K, max(3, args.warmup), world)
    samples, _ = timed_samples(step, K, 3, world)
    part_us, merge_us = kernel_pass(step, min(K, 500))
    tl = timeline(step)
    ck = clocks.stop()
    ms_step = max_over_ranks(total_ms / K, world)
    s = summary(samples)
    med_us = max_over_ranks(s["median"], world)
    value = world * ab["kv"] / (ms_step * 1e-3) / 1e9

    e2e, h2d, d2h = (None, 0, 0)
    if args.e2e_steps > 0:
        e2e, h2d, d2h = e2e_legs(dattn, w, p, info, dev, args.e2e_steps, world)

    peak, peak_src = measured_peak()
    # roofline of the partial kernel (the dominant one) from the headline region: its
    # algorithmic bytes over the median step, which bounds its duration from above
    achieved = ab["partial"] / (med_us * 1e-6) / 1e9
    line = {
        "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world, "steps": K, "warmup": args.warmup,
        "ms_per_step": ms_step, "us_per_step": ms_step * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": w.name, "B": p["B"], "S_q": p["S_q"], "H_q": p["H_q"], "H_kv": p["H_kv"],
                   "d": p["d"], "page_size": p["P"], "pool_pages": p["num_pages"],
                   "lengths": "uniform integers in [1024, 8192], seed 1",
                   "l2": "no flush: K/V read per step (%.0f MB) is larger than the 129 MB L2" % (ab["kv"] / 1e6),
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
                   "shared_shift": _shift(args),
                   "plan": {k: info[k] for k in ("n_items", "n_ctas", "n_slots", "n_merge_groups", "max_splits",
                                                 "stream_keys", "max_cta_keys", "workspace_bytes")}},
        "kv_bytes_per_step": ab["kv"],
        "us_per_step_samples": dict(s, what=f"{s['n']} samples, each the mean of {max(1, K // MIN_SAMPLES)} "
                                             f"consecutive steps between two events, in a second region of "
                                             f"K steps right after the timed one (the events between batches "
                                             f"cost a little: the timed region has none)"),
        "GBps_median": world * ab["kv"] / (med_us * 1e-6) / 1e9,
        "frac_of_nominal_8TBps": ab["kv"] / (med_us * 1e-6) / 1e9 / NOMINAL_HBM_GBS,
        "frac_of_measured_hbm": ab["kv"] / (med_us * 1e-6) / 1e9 / peak,
        "fractions_from": "the median per-step sample",
        "kernels": {"partial_us": part_us, "merge_us": merge_us, "merge_share": merge_us / (part_us + merge_us),
                    "timing": "CUDA events around each kernel on the launching stream, in a pass right after "
                              "the timed region; those events stop the merge from launching under the partial "
                              "kernel's tail, so partial_us + merge_us exceeds the step by the lost overlap",
                    "overlap_lost_us": part_us + merge_us - med_us},
        "roofline": {"bound": "hbm", "kernel": "dattn partial (bf16, d=128)", "achieved": achieved, "peak": peak,
                     "unit": "GB/s", "frac": achieved / peak, "peak_source": peak_src,
                     "algorithmic_bytes_per_launch": ab["partial"], "traffic": dram_traffic(),
                     "duration": "the median step of the headline region (an upper bound of the partial "
                                 "kernel's duration: the step also holds the merge's tail)",
                     "event_pass_frac": ab["partial"] / (part_us * 1e-6) / 1e9 / peak},
        "timeline": dict(tl or {}, what="medians over steps of the kernels' %globaltimer trace in a pass of "
                                         "back-to-back steps after the timed region (dattn_run_options.trace)"),
        "clocks": ck,
        "gpu_launches": K * (1 + step.merges),
    }
    if e2e:
        line["e2e"] = {"value": world * ab["kv"] / e2e["overlapped"] / 1e9, "unit": "GB/s",
                       "us_per_step": e2e["overlapped"] * 1e6, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                       "api": "dattn_step_host_submit_ex / dattn_step_host_finish, two steps in flight, "
                              "transfers on two copy streams, one workspace per slot",
                       "includes": "host planning, one pinned H2D of q, the page table and the work list, both "
                                   "kernels, one D2H of O and LSE, the wait for it, copy into the caller's host "
                                   "arrays",
                       "one_stream_us_per_step": e2e["pipelined"] * 1e6,
                       "one_stream_api": "dattn_step_host_submit / dattn_step_host_finish, transfers and "
                                         "kernels on one stream",
                       "sync_us_per_step": e2e["sync"] * 1e6,
                       "sync_api": "one blocking dattn_step_host call per step"}
    del step, cache
    torch.cuda.empty_cache()
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        try:
            with tempfile.TemporaryDirectory() as td:
                save_oracle_inputs(td, w, p, dict(k=w.k, v=w.v))
                line["cpu_baseline"] = cpu_baseline(td, p, ab["kv"])
        except Exception as e:  # the baseline is reported, never required for the GPU number
            line["cpu_baseline"] = {"value": None, "unit": "GB/s", "cores": 0, "kind": "oracle",
                                    "sample": f"failed: {e}"[:300]}
    del w
    if rank == 0 and world == 1 and not args.no_configs:
        clocks = Clocks(uuid)
        line["configs"] = {}
        for name in CONFIGS:
            line["configs"][name] = config_line(dattn, name, dev, num_sms, max(MIN_SAMPLES, args.config_steps),
                                                cpu=not args.no_cpu_baseline)
        line["configs_clocks"] = clocks.stop()
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def _shift(args):
    """(phi, lo, hi) of --shared-shift, or None."""
    return None if args.shared_shift is None else tuple(float(x) for x in args.shared_shift.split(","))


def run_other(args):
    import torch

    import split_kv_decode_flash_gb300 as dattn

    assert torch.cuda.is_available(), "bench.py --workload needs a GPU"
    dattn.load()
    dev = torch.device("cuda", torch.cuda.current_device())
    props = torch.cuda.get_device_properties(dev)
    w, p, cache = build_workload(dattn, args.workload, dev)
    step = Step(dattn, w, p, cache, dev, props.multi_processor_count, chunk=args.chunk, shift=_shift(args),
                merge_tags=args.merge_tags, fused_merge=args.fused_merge)
    for _ in range(3):
        step.run()
    torch.cuda.synchronize()
    assert step.status() == 0, "device bounds check fired"
    total_ms = timed_unbroken(step, max(MIN_SAMPLES, args.steps), max(3, args.warmup))
    samples, _ = timed_samples(step, max(MIN_SAMPLES, args.steps), 3)
    s = summary(samples)
    fallbacks = dattn.dattn_shift_fallbacks(step.ws, step.stream) if args.shared_shift else None
    tl = timeline(step)
    lens = w.kv_len.tolist()
    if w.qo_indptr is not None:      # an idle request (C_b = 0) reads nothing
        qo = [int(x) for x in w.qo_indptr]
        lens = [t if qo[b + 1] > qo[b] else 0 for b, t in enumerate(lens)]
    nb = stream_bytes(p, step.info, lens)
    peak, peak_src = measured_peak()
    print(json.dumps({"workload": w.name, "us_per_step": total_ms * 1e3 / max(MIN_SAMPLES, args.steps),
                      "us_per_step_samples": s, "kv_bytes_per_step": nb, "GBps": nb / s["median"] / 1e3,
                      "frac": nb / s["median"] / 1e3 / peak, "peak": peak, "peak_source": peak_src,
                      "rows": step.info["rows"], "n_items": step.info["n_items"], "merge_tags": step.info["merge_tags"],
                      "steps": args.steps,
                      "shared_shift": _shift(args), "shift_fallbacks": fallbacks, "timeline": tl,
                      "timing": "us_per_step: CUDA events around K back-to-back decode steps (partial + merge); "
                                "samples: a second region of K steps with an event after every K/50; GBps and "
                                "frac from the median sample"}), flush=True)


def main():
    args = parse()
    if args.cpu_child is not None:
        _cpu_child(args.cpu_child)
        return
    if args.impl == "reference":
        run_reference(args)
    elif args.workload != "paged":
        run_other(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
