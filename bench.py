#!/usr/bin/env python3
"""Decode-attention benchmark: paged ragged GQA decode on GB300.

Workload (one "step" = one decode step over the whole batch): B=16 requests,
S_q=1, H_q=32, H_kv=8, d=128, bf16 K/V in 16-token pages of a 10,000-page
pool, lengths uniform in [1024, 8192] (seed 1).  The step runs the whole hot
path: work-list upload, partial kernel, LSE merge kernel.

Metric: K/V bytes read per step / step time (GB/s), with the step time in
microseconds beside it.  Timing: CUDA events on the launching stream around
exactly --steps steps after --warmup steps, barrier + synchronize on both
sides, max over ranks.  The K/V read per step (~302 MB) is larger than the
129 MB L2, so no flush runs between steps.

--impl reference times the fp64 CPU oracle (the parity reference) on the
host cores instead, one bounded sample of the same workload per step.
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


OTHER_WORKLOADS = ("long-s1", "long-s4", "sink-window", "index-list", "packed", "tree-verify", "mixed", "int8", "fp8",
                   "fp8-e5m2", "int4-head", "int4-kivi")


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=50)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--e2e-steps", type=int, default=200)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--chunk", type=int, default=0, help="planner chunk width (0 = default)")
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
    direct_rows = sum(1 for n in per_group.values() if n == 1) * rows
    merged_rows = info["n_merge_groups"] * rows
    out_row = d * 2 + 4
    partial = kv + 4 * pages + q + state + direct_rows * out_row + info["blob_bytes"]
    merge = state + merged_rows * out_row
    return {"kv": kv, "partial": partial, "merge": merge, "page_list": 4 * pages, "q": q,
            "workspace_state": state, "out": (direct_rows + merged_rows) * out_row}


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

def _cpu_child(args):
    """Runs in a fresh single-threaded process: time the oracle on a list of groups."""
    import numpy as np
    from oracle import attention
    from oracle import cache as ocache
    path, groups = args[0], [tuple(map(int, g.split(":"))) for g in args[1:]]
    z = {n: np.load(os.path.join(path, n + ".npy"), mmap_mode="r")
         for n in ("k", "v", "q", "page_indptr", "page_indices", "kv_len")}
    with open(os.path.join(path, "meta.json")) as f:
        meta = json.load(f)
    c = ocache.Cache("paged", "bf16", meta["H_kv"], meta["d"], P=meta["P"], k=z["k"], v=z["v"],
                     page_indptr=z["page_indptr"], page_indices=z["page_indices"], kv_len=z["kv_len"])
    g = meta["H_q"] // meta["H_kv"]
    min_seconds = float(os.environ.get("DATTN_CPU_MIN_SECONDS", "0"))
    t0 = time.perf_counter()
    keys = passes = 0
    while True:              # whole passes over the groups until min_seconds of work
        for b, h in groups:
            rows = [(b, 0, h * g + j) for j in range(g)]
            attention.decode_rows(meta, c, z["q"], rows)
            keys += int(z["kv_len"][b])
        passes += 1
        if time.perf_counter() - t0 >= min_seconds:
            break
    dt = time.perf_counter() - t0
    print(json.dumps({"seconds": dt, "keys": keys, "passes": passes}))


def cpu_oracle_time(w, groups_per_worker, workers, tmpdir, min_seconds=0.0):
    """Times the oracle over groups split across ``workers`` single-threaded processes.

    Each process repeats whole passes over its groups for at least
    ``min_seconds`` and times its own compute (process start-up and array
    loading excluded); the sample's time is the slowest process's."""
    import numpy as np
    import torch

    def bits(t):
        return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)

    p = w.problem
    path = tmpdir
    if not os.path.exists(os.path.join(path, "meta.json")):
        arrays = dict(k=bits(w.k), v=bits(w.v), q=bits(w.q), page_indptr=w.page_indptr.numpy().astype(np.int64),
                      page_indices=w.page_indices.numpy().astype(np.int64), kv_len=w.kv_len.numpy().astype(np.int64))
        for n, a in arrays.items():
            np.save(os.path.join(path, n + ".npy"), a)
        with open(os.path.join(path, "meta.json"), "w") as f:
            json.dump(dict(B=p["B"], S_q=p["S_q"], H_q=p["H_q"], H_kv=p["H_kv"], d=p["d"], P=p["P"]), f)
    env = dict(os.environ, OMP_NUM_THREADS="1", OPENBLAS_NUM_THREADS="1", MKL_NUM_THREADS="1",
               DATTN_CPU_MIN_SECONDS=str(min_seconds))
    procs = []
    for gl in groups_per_worker[:workers]:
        cmd = [sys.executable, os.path.abspath(__file__), "--cpu-child", path] + [f"{b}:{h}" for b, h in gl]
        procs.append(subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.PIPE, text=True, env=env))
    keys, wall = 0, 0.0
    for pr in procs:
        out, err = pr.communicate()
        if pr.returncode != 0:
            raise RuntimeError("oracle timing child failed: " + err[-2000:])
        r = json.loads(out.strip().splitlines()[-1])
        keys += r["keys"]
        wall = max(wall, r["seconds"])
    return keys * kv_bytes_per_key(p), wall


def cpu_baseline(w, budget_groups=None):
    """Oracle over a bounded sample (whole (request, kv head) groups) on all host cores."""
    p = w.problem
    groups = [(b, h) for b in range(p["B"]) for h in range(p["H_kv"])]
    if budget_groups:
        groups = groups[:budget_groups]
    workers = max(1, min(os.cpu_count() or 1, len(groups)))
    split = [groups[i::workers] for i in range(workers)]
    with tempfile.TemporaryDirectory() as td:
        nbytes, wall = cpu_oracle_time(w, split, workers, td, min_seconds=1.0)
    return {"value": nbytes / wall / 1e9, "unit": "GB/s", "cores": workers, "kind": "oracle",
            "sample": f"all {len(groups)} (request, kv head) groups of one step "
                      f"({sum(int(w.kv_len[b]) for b, _ in groups)} keys), repeated in whole passes for "
                      f">= 1 s per process: {nbytes / kv_bytes_per_key(p):.0f} keys in {wall:.2f} s on "
                      f"{workers} single-threaded processes (float64 numpy, about {workers * wall:.0f} s of CPU work)"}


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
        cpu_oracle_time(w, [seq[:args.warmup]], 1, td) if args.warmup else None
        nbytes, wall = cpu_oracle_time(w, [seq[args.warmup:]], 1, td)
    value = nbytes / wall / 1e9
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": wall * 1e3 / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic",
            "config": {"workload": w.name, "per_step": "one (request, kv head) group of the decode step",
                       "l2": "host run"},
            "cpu_baseline": {"value": value, "unit": "GB/s", "cores": 1, "kind": "oracle",
                             "sample": f"{args.steps} (request, kv head) groups cycled over the batch"},
            "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def run_ours(args):
    import torch

    import split_kv_decode_flash_gb300 as dattn
    import workloads as W

    world, rank, local = dist_setup(args.gpus)
    assert torch.cuda.is_available(), "bench.py --impl ours needs a GPU"
    dattn.load()
    dev = torch.device("cuda", torch.cuda.current_device())
    w = W.paged_ragged_gqa(dev)
    p = w.problem
    props = torch.cuda.get_device_properties(dev)
    plan = dattn.dattn_plan(p, w.kv_len, page_indptr=w.page_indptr, num_sms=props.multi_processor_count,
                            chunk_tokens=args.chunk)
    info = plan.info
    items = plan.items()
    ab = algorithmic_bytes(w, info, items)
    o = torch.empty((p["B"], p["S_q"], p["H_q"], p["d"]), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((p["B"], p["S_q"], p["H_q"]), dtype=torch.float32, device=dev)
    ws = torch.empty(plan.workspace_bytes, dtype=torch.uint8, device=dev)
    pi_dev, pidx_dev = w.page_indptr.to(dev), w.page_indices.to(dev)
    t = dattn.tensors_from(q=w.q, k=w.k, v=w.v, o=o, lse=lse, page_indptr=pi_dev, page_indices=pidx_dev)
    stream = torch.cuda.current_stream()

    for _ in range(max(3, args.warmup)):
        dattn.dattn_run(plan, p, t, ws, stream)
    torch.cuda.synchronize()
    assert dattn.dattn_device_status(ws, stream) == 0, "device bounds check fired"

    K = args.steps
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(K)]
    for e3 in evs:
        for e in e3:
            e.record(stream)      # materialise the events before use
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    uuid = None
    try:
        uuid = "GPU-" + str(props.uuid)
    except Exception:
        pass
    clocks = Clocks(uuid)
    time.sleep(0.2)
    for _ in range(args.warmup):
        dattn.dattn_run(plan, p, t, ws, stream)
    barrier(world)
    torch.cuda.synchronize()
    dattn.dattn_plan_upload(plan, ws, stream)     # once per decode step; every layer reuses it
    # Timed region: K steps back to back, bracketed by two events.  An event
    # recorded between the partial and the merge kernel would stop the merge
    # from launching programmatically under the partial kernel's tail, so the
    # per-kernel events are taken in a second pass of K steps right after.
    start.record(stream)
    for k in range(K):
        dattn.dattn_run_ex(plan, p, t, ws, reuse_upload=True, shared_shift=_shift(args), stream=stream)
    end.record(stream)
    torch.cuda.synchronize()
    for k in range(K):
        dattn.dattn_run_ex(plan, p, t, ws, reuse_upload=True, events=evs[k], shared_shift=_shift(args),
                           stream=stream)
    torch.cuda.synchronize()
    barrier(world)
    ck = clocks.stop()
    total_ms = start.elapsed_time(end)
    partial_ms = [evs[k][0].elapsed_time(evs[k][1]) for k in range(K)]
    merge_ms = [evs[k][1].elapsed_time(evs[k][2]) for k in range(K)]
    ms_step = max_over_ranks(total_ms / K, world)
    value = world * ab["kv"] / (ms_step * 1e-3) / 1e9

    # end to end through the public API: one dattn_step_host call per step plans from the
    # host lengths, sends q, the page table and the work list in one transfer from pinned
    # memory, runs both kernels, brings O and LSE back in one transfer and synchronises
    q_host = w.q.cpu().pin_memory()
    o_host = torch.empty(o.shape, dtype=o.dtype).pin_memory()
    lse_host = torch.empty(lse.shape, dtype=lse.dtype).pin_memory()
    io = dattn.host_step(q_host, w.kv_len, o_host, lse=lse_host, page_indptr=w.page_indptr,
                         page_indices=w.page_indices, num_sms=props.multi_processor_count)
    ws_e2e_bytes, staging_bytes = dattn.dattn_step_host_sizes(p, io)
    ws_e2e = torch.empty(ws_e2e_bytes, dtype=torch.uint8, device=dev)
    staging = torch.empty(staging_bytes, dtype=torch.uint8).pin_memory()
    cache_e2e = dattn.tensors_from(k=w.k, v=w.v)

    def e2e_step():
        dattn.dattn_step_host(p, io, cache_e2e, staging, ws_e2e, stream)

    e2e_s = float("nan")
    if args.e2e_steps > 0:
        for _ in range(5):
            e2e_step()
        barrier(world)
        t0 = time.perf_counter()
        for _ in range(args.e2e_steps):
            e2e_step()
        e2e_s = max_over_ranks((time.perf_counter() - t0) / args.e2e_steps, world)
    h2d = (q_host.numel() * 2 + w.page_indptr.numel() * 4 + w.page_indices.numel() * 4 + info["blob_bytes"])
    d2h = o_host.numel() * 2 + lse_host.numel() * 4

    peak, peak_src = measured_peak()
    part_us = statistics.mean(partial_ms) * 1e3
    merge_us = statistics.mean(merge_ms) * 1e3
    achieved = ab["partial"] / (part_us * 1e-6) / 1e9
    traffic = dram_traffic()
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
        "frac_of_nominal_8TBps": value / world / NOMINAL_HBM_GBS,
        "frac_of_measured_hbm": value / world / peak,
        "kernels": {"partial_us": part_us, "merge_us": merge_us,
                    "partial_p50_us": statistics.median(partial_ms) * 1e3,
                    "timing": "CUDA events around each kernel on the launching stream, in a pass of K steps "
                              "right after the timed region (merge_us then includes its launch gap)"},
        "roofline": {"bound": "hbm", "kernel": "dattn partial (bf16, d=128)", "achieved": achieved, "peak": peak,
                     "unit": "GB/s", "frac": achieved / peak, "peak_source": peak_src,
                     "algorithmic_bytes_per_launch": ab["partial"], "traffic": traffic},
        "e2e": {"value": world * ab["kv"] / e2e_s / 1e9, "unit": "GB/s", "us_per_step": e2e_s * 1e6,
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "api": "dattn_step_host (one C call per step)",
                "includes": "host planning, one pinned H2D of q, the page table and the work list, both "
                            "kernels, one D2H of O and LSE, stream sync, copy into the caller's host arrays"},
        "clocks": ck,
        "gpu_launches": K * (1 + (1 if info["n_merge_groups"] and not info["fused_merge"] else 0)),
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        try:
            line["cpu_baseline"] = cpu_baseline(w)
        except Exception as e:  # the baseline is reported, never required for the GPU number
            line["cpu_baseline"] = {"value": None, "unit": "GB/s", "cores": 0, "kind": "oracle",
                                    "sample": f"failed: {e}"[:300]}
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


# ---- the other workloads: one timing line each ------------------------------------------

def _quantized_cache(dattn, w, fmt, dev):
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


def _shift(args):
    """(phi, lo, hi) of --shared-shift, or None."""
    return None if args.shared_shift is None else tuple(float(x) for x in args.shared_shift.split(","))


def _stream_bytes(p, info, lens):
    """K/V bytes of the visible streams (what the step must read)."""
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
    for T in lens:      # causal, S_q = 1: the stream is the whole history
        nq = G * -(-max(0, T - R) // G)
        total += nq * (d + 4 * d // Gv) + (nq // G) * 4 * d + (T - nq) * 4 * d
    return total * p["H_kv"]


def run_other(args):
    import torch

    import split_kv_decode_flash_gb300 as dattn
    import workloads as W

    assert torch.cuda.is_available(), "bench.py --workload needs a GPU"
    dattn.load()
    dev = torch.device("cuda", torch.cuda.current_device())
    name = args.workload
    if name in ("int8", "fp8", "fp8-e5m2", "int4-head", "int4-kivi"):
        fmt = {"int8": "int8", "fp8": "fp8_e4m3", "fp8-e5m2": "fp8_e5m2", "int4-head": "int4_head",
               "int4-kivi": "int4_kivi"}[name]
        w = W.quantized(dev, fmt=fmt)
        p, cache = _quantized_cache(dattn, w, fmt, dev)
    else:
        w = {"long-s1": lambda: W.long_context(dev, 1), "long-s4": lambda: W.long_context(dev, 4),
             "sink-window": lambda: W.retention(dev, "sink_window"),
             "index-list": lambda: W.retention(dev, "index_list"),
             "packed": lambda: W.packed_view(W.retention(dev, "index_list")),
             "tree-verify": lambda: W.tree_verify(dev), "mixed": lambda: W.mixed_batch(dev)}[name]()
        p = w.problem
        cache = dict(k=w.k, v=w.v)
        if w.page_indptr is not None:
            cache.update(page_indptr=w.page_indptr.to(dev), page_indices=w.page_indices.to(dev))
        if w.index_list is not None:
            cache.update(index_indptr=w.index_indptr.to(dev), index_list=w.index_list.to(dev))
        if w.fm_intervals is not None:
            cache.update(fm_intervals=w.fm_intervals.to(dev).contiguous())
    props = torch.cuda.get_device_properties(dev)
    plan = dattn.dattn_plan(p, w.kv_len, page_indptr=w.page_indptr, index_indptr=w.index_indptr,
                            index_list=w.index_list, num_sms=props.multi_processor_count, chunk_tokens=args.chunk,
                            qo_indptr=w.qo_indptr)
    n_rows = p["B"] * p["S_q"] if w.qo_indptr is None else int(w.qo_indptr[-1])   # packed query rows
    o = torch.empty((n_rows, p["H_q"], p["d"]), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((n_rows, p["H_q"]), dtype=torch.float32, device=dev)
    t = dattn.tensors_from(q=w.q.to(dev), o=o, lse=lse, **cache)
    ws = torch.empty(plan.workspace_bytes, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()
    dattn.dattn_plan_upload(plan, ws, stream)
    for _ in range(max(3, args.warmup)):
        dattn.dattn_run_ex(plan, p, t, ws, reuse_upload=True, shared_shift=_shift(args), stream=stream)
    torch.cuda.synchronize()
    assert dattn.dattn_device_status(ws, stream) == 0, "device bounds check fired"
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    start.record(stream)
    for _ in range(args.steps):
        dattn.dattn_run_ex(plan, p, t, ws, reuse_upload=True, shared_shift=_shift(args), stream=stream)
    end.record(stream)
    torch.cuda.synchronize()
    us = start.elapsed_time(end) / args.steps * 1e3
    fallbacks = dattn.dattn_shift_fallbacks(ws, stream) if args.shared_shift else None
    nb = _stream_bytes(p, plan.info, w.kv_len.tolist())
    peak, peak_src = measured_peak()
    print(json.dumps({"workload": w.name, "us_per_step": us, "kv_bytes_per_step": nb, "GBps": nb / us / 1e3,
                      "frac": nb / us / 1e3 / peak, "peak": peak, "peak_source": peak_src,
                      "rows": plan.info["rows"], "n_items": plan.info["n_items"], "steps": args.steps,
                      "shared_shift": _shift(args), "shift_fallbacks": fallbacks,
                      "timing": "CUDA events around K back-to-back decode steps (partial + merge)"}), flush=True)


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
