"""Python binding of libdattn: split-KV decode attention for GB300 (sm_103a).

A thin ctypes layer over the C ABI declared in ``include/dattn.h``.  Every
function keeps the C name and only marshals arguments (torch tensors become
device pointers, dicts become ``dattn_problem``); every step of the decode
path runs in the library's CUDA kernels.  There is no fallback: when the
library cannot be built or loaded, or a call fails, a ``DattnError`` is
raised.  PyTorch only provides device memory and streams.
"""

from __future__ import annotations

import ctypes
import math
import os

import numpy as np

from . import build as _build

__all__ = [
    "DattnError", "Problem", "load", "make_problem", "dattn_plan", "dattn_plan_get_info",
    "dattn_plan_get_items", "dattn_run", "dattn_run_ex", "dattn_run_noalloc", "dattn_noalloc_status", "dattn_plan_upload", "dattn_device_status", "dattn_shift_fallbacks", "kv_append",
    "kv_append_workspace_bytes", "dattn_debug_translate", "dattn_debug_classify",
    "dattn_debug_gather", "dattn_last_error", "dattn_version", "tensors_from", "decode",
    "LAYOUTS", "FORMATS", "MASKS", "TILE_CLASSES", "STATUS",
]

STATUS = {0: "DATTN_OK", 1: "DATTN_EINVAL", 2: "DATTN_EUNSUPPORTED", 3: "DATTN_EWORKSPACE",
          4: "DATTN_ESTALE_PLAN", 5: "DATTN_ECUDA", 6: "DATTN_EDEVICE_CHECK"}
LAYOUTS = {"contig": 0, "paged": 1, "packed": 2}
FORMATS = {"bf16": 0, "int8": 1, "int4_kivi": 2, "fp8_e4m3": 3, "fp8_e5m2": 4, "int4_head": 5}
MASKS = {"causal": 0, "sink_window": 1, "index_list": 2, "flashmask": 3}
TILE_CLASSES = {0: "SKIP", 1: "FULL", 2: "PARTIAL"}


class DattnError(RuntimeError):
    def __init__(self, status, where, text):
        self.status = status
        super().__init__(f"{where}: {STATUS.get(status, status)}: {text}")


class Problem(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in (
        "B", "S_q", "H_q", "H_kv", "d_h", "layout", "fmt", "page_size", "num_pages", "T_cap",
        "B_cache", "kivi_group", "kivi_v_group", "kivi_residual", "mask", "n_sink", "window")] + [
        ("sm_scale", ctypes.c_float), ("fixed_splits", ctypes.c_int32)]


class PlanInputs(ctypes.Structure):
    _fields_ = [("kv_len", ctypes.c_void_p), ("page_indptr", ctypes.c_void_p),
                ("index_indptr", ctypes.c_void_p), ("index_list", ctypes.c_void_p),
                ("num_sms", ctypes.c_int32), ("ctas_per_sm", ctypes.c_int32),
                ("chunk_tokens", ctypes.c_int32), ("fused_merge", ctypes.c_int32),
                ("qo_indptr", ctypes.c_void_p), ("item_cost_keys", ctypes.c_int32), ("merge_tags", ctypes.c_int32)]


class StepCopies(ctypes.Structure):
    _fields_ = [("h2d_stream", ctypes.c_void_p), ("d2h_stream", ctypes.c_void_p),
                ("inputs_event", ctypes.c_void_p), ("kernels_event", ctypes.c_void_p)]


class HostStep(ctypes.Structure):
    _fields_ = [("q", ctypes.c_void_p), ("kv_len", ctypes.c_void_p), ("page_indptr", ctypes.c_void_p),
                ("page_indices", ctypes.c_void_p), ("o", ctypes.c_void_p), ("lse", ctypes.c_void_p),
                ("num_sms", ctypes.c_int32)]


class Tensors(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in (
        "q", "k", "v", "k_qparams", "v_qparams", "k_residual", "v_residual", "page_indptr",
        "page_indices", "cache_batch_idx", "index_indptr", "index_list", "o", "lse", "fm_intervals")]


class PlanInfo(ctypes.Structure):
    _fields_ = [("workspace_bytes", ctypes.c_int64), ("blob_bytes", ctypes.c_int64),
                ("n_items", ctypes.c_int32), ("n_ctas", ctypes.c_int32), ("n_slots", ctypes.c_int32),
                ("n_merge_groups", ctypes.c_int32), ("max_splits", ctypes.c_int32),
                ("rows", ctypes.c_int32), ("stream_keys", ctypes.c_int64),
                ("max_cta_keys", ctypes.c_int64), ("fused_merge", ctypes.c_int32), ("merge_tags", ctypes.c_int32)]


class WorkItem(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in ("b", "h_kv", "a", "e", "slot", "cta")]


class RunOptions(ctypes.Structure):
    _fields_ = [("flags", ctypes.c_uint32), ("events", ctypes.c_void_p * 3),
                ("shift_phi", ctypes.c_float), ("shift_lo", ctypes.c_float), ("shift_hi", ctypes.c_float),
                ("wait_limit_us", ctypes.c_uint32), ("trace", ctypes.c_void_p)]


RUN_REUSE_UPLOAD = 1
RUN_SHARED_SHIFT = 2
RUN_TEST_SKIP_ARRIVAL = 4
NOALLOC_SCRATCH_BYTES = 16 << 20  # DATTN_NOALLOC_SCRATCH_BYTES


class AppendInputs(ctypes.Structure):
    _fields_ = [("kv_len_old", ctypes.c_void_p), ("new_indptr", ctypes.c_void_p),
                ("page_indptr", ctypes.c_void_p)]


_LIB = None
_VP = ctypes.c_void_p
_ST = ctypes.c_int


def load():
    """Build (if stale) and load libdattn.so; raises when that is impossible."""
    global _LIB
    if _LIB is not None:
        return _LIB
    path = _build.build()
    lib = ctypes.CDLL(path)
    sig = {
        "dattn_plan": (_ST, [ctypes.POINTER(Problem), ctypes.POINTER(PlanInputs), ctypes.POINTER(_VP),
                             ctypes.POINTER(ctypes.c_size_t)]),
        "dattn_plan_destroy": (None, [_VP]),
        "dattn_plan_get_info": (_ST, [_VP, ctypes.POINTER(PlanInfo)]),
        "dattn_plan_get_items": (_ST, [_VP, ctypes.POINTER(WorkItem), ctypes.c_int32,
                                       ctypes.POINTER(ctypes.c_int32)]),
        "dattn_run": (_ST, [_VP, ctypes.POINTER(Problem), ctypes.POINTER(Tensors), _VP, ctypes.c_size_t, _VP]),
        "dattn_run_ex": (_ST, [_VP, ctypes.POINTER(Problem), ctypes.POINTER(Tensors), _VP,
                               ctypes.c_size_t, _VP, ctypes.POINTER(RunOptions)]),
        "dattn_plan_upload": (_ST, [_VP, _VP, ctypes.c_size_t, _VP]),
        "dattn_run_noalloc": (_ST, [_VP, ctypes.POINTER(Problem), ctypes.POINTER(Tensors), _VP]),
        "dattn_noalloc_status": (_ST, [ctypes.POINTER(ctypes.c_int32), _VP]),
        "dattn_device_status": (_ST, [_VP, ctypes.POINTER(ctypes.c_int32), _VP]),
        "dattn_shift_fallbacks": (_ST, [_VP, ctypes.POINTER(ctypes.c_int32), _VP]),
        "kv_append_workspace_bytes": (ctypes.c_size_t, [ctypes.POINTER(Problem)]),
        "kv_append": (_ST, [ctypes.POINTER(Problem), ctypes.POINTER(AppendInputs), ctypes.POINTER(Tensors),
                            _VP, _VP, _VP, ctypes.c_size_t, _VP]),
        "dattn_debug_translate": (_ST, [ctypes.POINTER(Problem), ctypes.POINTER(Tensors), _VP, _VP,
                                        ctypes.c_int32, _VP, _VP]),
        "dattn_debug_classify": (_ST, [ctypes.POINTER(Problem), ctypes.POINTER(Tensors), _VP, _VP,
                                       ctypes.c_int32, _VP, _VP]),
        "dattn_debug_gather": (_ST, [_VP, ctypes.POINTER(Problem), ctypes.POINTER(Tensors), _VP,
                                     ctypes.c_size_t, ctypes.c_int32, ctypes.c_int32, _VP, ctypes.c_int32,
                                     ctypes.POINTER(ctypes.c_int32), _VP]),
        "dattn_step_host_sizes": (_ST, [ctypes.POINTER(Problem), ctypes.POINTER(HostStep),
                                        ctypes.POINTER(ctypes.c_size_t), ctypes.POINTER(ctypes.c_size_t)]),
        "dattn_step_host": (_ST, [ctypes.POINTER(Problem), ctypes.POINTER(HostStep), ctypes.POINTER(Tensors),
                                  _VP, ctypes.c_size_t, _VP, ctypes.c_size_t, _VP]),
        "dattn_step_host_status": (_ST, [ctypes.POINTER(Problem), ctypes.POINTER(HostStep), _VP,
                                         ctypes.POINTER(ctypes.c_int32), _VP]),
        "dattn_step_host_submit": (_ST, [ctypes.POINTER(Problem), ctypes.POINTER(HostStep), ctypes.POINTER(Tensors),
                                         _VP, ctypes.c_size_t, _VP, ctypes.c_size_t, _VP, _VP]),
        "dattn_step_host_finish": (_ST, [ctypes.POINTER(Problem), ctypes.POINTER(HostStep), _VP, ctypes.c_size_t,
                                         _VP]),
        "dattn_step_host_submit_ex": (_ST, [ctypes.POINTER(Problem), ctypes.POINTER(HostStep),
                                            ctypes.POINTER(Tensors), _VP, ctypes.c_size_t, _VP, ctypes.c_size_t,
                                            _VP, _VP, ctypes.POINTER(StepCopies)]),
        "dattn_last_error": (ctypes.c_char_p, []),
        "dattn_version": (ctypes.c_int32, []),
    }
    for name, (res, args) in sig.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _LIB = lib
    return lib


def dattn_last_error() -> str:
    return load().dattn_last_error().decode()


def dattn_version() -> int:
    return load().dattn_version()


def _check(status, where):
    if status != 0:
        raise DattnError(status, where, dattn_last_error())


def make_problem(d: dict) -> Problem:
    """dattn_problem from a dict with the keys of ``workloads.Workload.problem``."""
    p = Problem()
    p.B, p.S_q, p.H_q, p.H_kv = d["B"], d["S_q"], d["H_q"], d["H_kv"]
    p.d_h = d["d"]
    p.layout = LAYOUTS[d.get("layout", "paged")]
    p.fmt = FORMATS[d.get("fmt", "bf16")]
    p.page_size = d.get("P", 0)
    p.num_pages = d.get("num_pages", 0)
    p.T_cap = d.get("T_cap", 0)
    p.B_cache = d.get("B_cache", 0)
    p.kivi_group = d.get("kivi_group", 32)
    p.kivi_v_group = d.get("kivi_v_group", 32)
    p.kivi_residual = d.get("kivi_residual", 128)
    p.mask = MASKS[d.get("mask", "causal")]
    p.n_sink = d.get("n_sink", 0)
    p.window = d.get("window", 0)
    p.sm_scale = d.get("sm_scale", 0.0) or 0.0
    p.fixed_splits = d.get("fixed_splits", 0)
    return p


def _i32_host(x):
    if x is None:
        return None
    if hasattr(x, "detach"):
        x = x.detach().cpu().numpy()
    return np.ascontiguousarray(np.asarray(x, dtype=np.int32))


def _ptr(a):
    if a is None:
        return None
    if isinstance(a, np.ndarray):
        return a.ctypes.data
    return a.data_ptr()


def _stream_ptr(stream):
    if stream is None:
        import torch
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


class Plan:
    """Owns a dattn_plan_t; destroyed with the object."""

    def __init__(self, handle, problem, ws_bytes):
        self.handle = handle
        self.problem = problem
        self.workspace_bytes = ws_bytes

    @property
    def info(self) -> dict:
        return dattn_plan_get_info(self)

    def items(self):
        return dattn_plan_get_items(self)

    def __del__(self):
        if getattr(self, "handle", None) and _LIB is not None:
            _LIB.dattn_plan_destroy(self.handle)
            self.handle = None


def dattn_plan(problem, kv_len, *, page_indptr=None, index_indptr=None, index_list=None, num_sms=None,
               ctas_per_sm=0, chunk_tokens=0, fused_merge=False, qo_indptr=None, item_cost_keys=0,
               merge_tags=0) -> Plan:
    """Host-only planning (see dattn_plan in dattn.h).  Arrays are host int32."""
    lib = load()
    prob = problem if isinstance(problem, Problem) else make_problem(problem)
    if num_sms is None:
        import torch
        num_sms = torch.cuda.get_device_properties(torch.cuda.current_device()).multi_processor_count
    keep = [_i32_host(kv_len), _i32_host(page_indptr), _i32_host(index_indptr), _i32_host(index_list),
            _i32_host(qo_indptr)]
    inp = PlanInputs(_ptr(keep[0]), _ptr(keep[1]), _ptr(keep[2]), _ptr(keep[3]), int(num_sms),
                     int(ctas_per_sm), int(chunk_tokens), int(bool(fused_merge)), _ptr(keep[4]),
                     int(item_cost_keys), int(merge_tags))
    handle = ctypes.c_void_p()
    ws = ctypes.c_size_t()
    _check(lib.dattn_plan(ctypes.byref(prob), ctypes.byref(inp), ctypes.byref(handle), ctypes.byref(ws)),
           "dattn_plan")
    return Plan(handle, prob, ws.value)


def dattn_plan_get_info(plan: Plan) -> dict:
    info = PlanInfo()
    _check(load().dattn_plan_get_info(plan.handle, ctypes.byref(info)), "dattn_plan_get_info")
    return {n: getattr(info, n) for n, _ in PlanInfo._fields_}


def dattn_plan_get_items(plan: Plan):
    lib = load()
    n = ctypes.c_int32()
    _check(lib.dattn_plan_get_items(plan.handle, None, 0, ctypes.byref(n)), "dattn_plan_get_items")
    arr = (WorkItem * max(1, n.value))()
    _check(lib.dattn_plan_get_items(plan.handle, arr, n.value, ctypes.byref(n)), "dattn_plan_get_items")
    return [{f: getattr(arr[i], f) for f, _ in WorkItem._fields_} for i in range(n.value)]


def tensors_from(**kw) -> Tensors:
    """dattn_tensors from torch tensors (or None) keyed by the C field names.

    The returned struct holds references to the tensors, so their device
    memory stays allocated while the struct (and any work queued with it)
    is alive."""
    t = Tensors()
    keep = []
    for name, _ in Tensors._fields_:
        v = kw.pop(name, None)
        setattr(t, name, None if v is None else v.data_ptr())
        if v is not None:
            keep.append(v)
    if kw:
        raise TypeError(f"unknown tensor fields {sorted(kw)}")
    t._keep = keep
    return t


def dattn_run(plan: Plan, problem, tensors: Tensors, workspace, stream=None) -> None:
    """Enqueue one decode step on ``stream`` (see dattn_run in dattn.h)."""
    prob = problem if isinstance(problem, Problem) else make_problem(problem)
    _check(load().dattn_run(plan.handle, ctypes.byref(prob), ctypes.byref(tensors), workspace.data_ptr(),
                            workspace.numel() * workspace.element_size(), _stream_ptr(stream)), "dattn_run")


def dattn_run_noalloc(plan: Plan, problem, tensors: Tensors, stream=None) -> None:
    """dattn_run on the library's own static scratch array instead of a caller workspace
    (see dattn_run_noalloc in dattn.h); raises DattnError when the plan's workspace
    exceeds NOALLOC_SCRATCH_BYTES."""
    prob = problem if isinstance(problem, Problem) else make_problem(problem)
    _check(load().dattn_run_noalloc(plan.handle, ctypes.byref(prob), ctypes.byref(tensors), _stream_ptr(stream)),
           "dattn_run_noalloc")


def dattn_noalloc_status(stream=None) -> int:
    """Device status word of the last dattn_run_noalloc on the current device (0: no check fired)."""
    flags = ctypes.c_int32()
    st = load().dattn_noalloc_status(ctypes.byref(flags), _stream_ptr(stream))
    if st not in (0, 6):
        _check(st, "dattn_noalloc_status")
    return flags.value


def dattn_plan_upload(plan: Plan, workspace, stream=None) -> None:
    """Copy the plan's work list into ``workspace`` (see dattn_plan_upload in dattn.h)."""
    _check(load().dattn_plan_upload(plan.handle, workspace.data_ptr(), workspace.numel() * workspace.element_size(),
                                    _stream_ptr(stream)), "dattn_plan_upload")


def dattn_run_ex(plan: Plan, problem, tensors: Tensors, workspace, *, reuse_upload=False, events=None,
                 shared_shift=None, wait_limit_us=0, test_skip_arrival=False, trace=None, stream=None) -> None:
    """dattn_run with options: reuse an uploaded work list, record three torch.cuda.Events
    (before the partial kernel, after it, after the merge kernel), ``shared_shift =
    (phi, lo, hi)``: partials in the fixed frame phi, guarded by lo < s - phi < hi,
    ``wait_limit_us``: the bounded waits' limit, and ``test_skip_arrival``: the hook that
    makes one wait run out (DATTN_RUN_TEST_SKIP_ARRIVAL)."""
    prob = problem if isinstance(problem, Problem) else make_problem(problem)
    opt = RunOptions()
    opt.flags = (RUN_REUSE_UPLOAD if reuse_upload else 0) | (RUN_TEST_SKIP_ARRIVAL if test_skip_arrival else 0)
    opt.wait_limit_us = int(wait_limit_us)
    opt.trace = None if trace is None else trace.data_ptr()
    if shared_shift is not None:
        opt.flags |= RUN_SHARED_SHIFT
        opt.shift_phi, opt.shift_lo, opt.shift_hi = (float(x) for x in shared_shift)
    for i, e in enumerate(events or ()):
        opt.events[i] = None if e is None else e.cuda_event
    _check(load().dattn_run_ex(plan.handle, ctypes.byref(prob), ctypes.byref(tensors), workspace.data_ptr(),
                               workspace.numel() * workspace.element_size(), _stream_ptr(stream), ctypes.byref(opt)),
           "dattn_run_ex")


def dattn_device_status(workspace, stream=None) -> int:
    flags = ctypes.c_int32()
    st = load().dattn_device_status(workspace.data_ptr(), ctypes.byref(flags), _stream_ptr(stream))
    if st not in (0, 6):
        _check(st, "dattn_device_status")
    return flags.value


def dattn_shift_fallbacks(workspace, stream=None) -> int:
    """Groups of the last shared-shift run whose scores left the guard and took the online-max path."""
    count = ctypes.c_int32()
    _check(load().dattn_shift_fallbacks(workspace.data_ptr(), ctypes.byref(count), _stream_ptr(stream)),
           "dattn_shift_fallbacks")
    return count.value


def kv_append_workspace_bytes(problem) -> int:
    prob = problem if isinstance(problem, Problem) else make_problem(problem)
    return load().kv_append_workspace_bytes(ctypes.byref(prob))


def kv_append(problem, cache: Tensors, k_new, v_new, kv_len_old, new_indptr, page_indptr, workspace,
              stream=None) -> None:
    """Append packed bf16 rows (device) at kv_len_old (host int32 arrays)."""
    prob = problem if isinstance(problem, Problem) else make_problem(problem)
    keep = [_i32_host(kv_len_old), _i32_host(new_indptr), _i32_host(page_indptr)]
    inp = AppendInputs(_ptr(keep[0]), _ptr(keep[1]), _ptr(keep[2]))
    _check(load().kv_append(ctypes.byref(prob), ctypes.byref(inp), ctypes.byref(cache),
                            None if k_new is None else k_new.data_ptr(),
                            None if v_new is None else v_new.data_ptr(),
                            workspace.data_ptr(), workspace.numel() * workspace.element_size(),
                            _stream_ptr(stream)), "kv_append")


def dattn_debug_translate(problem, tensors: Tensors, kv_len_dev, coords_dev, out_dev, stream=None) -> None:
    prob = problem if isinstance(problem, Problem) else make_problem(problem)
    _check(load().dattn_debug_translate(ctypes.byref(prob), ctypes.byref(tensors), kv_len_dev.data_ptr(),
                                        coords_dev.data_ptr(), coords_dev.shape[0], out_dev.data_ptr(),
                                        _stream_ptr(stream)), "dattn_debug_translate")


def dattn_debug_classify(problem, tensors: Tensors, kv_len_dev, tiles_dev, out_dev, stream=None) -> None:
    prob = problem if isinstance(problem, Problem) else make_problem(problem)
    _check(load().dattn_debug_classify(ctypes.byref(prob), ctypes.byref(tensors), kv_len_dev.data_ptr(),
                                       tiles_dev.data_ptr(), tiles_dev.shape[0], out_dev.data_ptr(),
                                       _stream_ptr(stream)), "dattn_debug_classify")


def dattn_debug_gather(plan: Plan, problem, tensors: Tensors, workspace, b, h_kv, out_dev, stream=None) -> int:
    prob = problem if isinstance(problem, Problem) else make_problem(problem)
    n = ctypes.c_int32()
    _check(load().dattn_debug_gather(plan.handle, ctypes.byref(prob), ctypes.byref(tensors), workspace.data_ptr(),
                                     workspace.numel() * workspace.element_size(), int(b), int(h_kv),
                                     out_dev.data_ptr(), out_dev.numel(), ctypes.byref(n), _stream_ptr(stream)),
           "dattn_debug_gather")
    return n.value


def decode(problem, plan: Plan, workspace, *, q, o, lse=None, stream=None, **cache) -> None:
    """Convenience: dattn_run with tensors given as keyword arguments."""
    dattn_run(plan, problem, tensors_from(q=q, o=o, lse=lse, **cache), workspace, stream)


def default_scale(d: int) -> float:
    return 1.0 / math.sqrt(d)


# ---- one step from host memory -------------------------------------------------------------

def host_step(q, kv_len, o, *, page_indptr=None, page_indices=None, lse=None, num_sms=None) -> HostStep:
    """dattn_host_step from host arrays (torch CPU tensors, pinned for asynchronous copies,
    or numpy arrays).  The struct keeps references to the arrays it points to."""
    if num_sms is None:
        import torch
        num_sms = torch.cuda.get_device_properties(torch.cuda.current_device()).multi_processor_count
    keep = [q, _i32_host(kv_len), _i32_host(page_indptr), _i32_host(page_indices), o, lse]
    io = HostStep(_ptr(keep[0]), _ptr(keep[1]), _ptr(keep[2]), _ptr(keep[3]), _ptr(keep[4]), _ptr(keep[5]),
                  int(num_sms))
    io._keep = keep
    return io


def dattn_step_host_sizes(problem, io: HostStep):
    """(workspace bytes, staging bytes) that dattn_step_host needs for this call."""
    prob = problem if isinstance(problem, Problem) else make_problem(problem)
    ws, sg = ctypes.c_size_t(), ctypes.c_size_t()
    _check(load().dattn_step_host_sizes(ctypes.byref(prob), ctypes.byref(io), ctypes.byref(ws), ctypes.byref(sg)),
           "dattn_step_host_sizes")
    return ws.value, sg.value


def dattn_step_host(problem, io: HostStep, cache: Tensors, staging, workspace, stream=None) -> None:
    """One decode step from host memory: returns with O (and LSE) in the host arrays of io.
    ``staging`` is a pinned host uint8 tensor, ``workspace`` a device uint8 tensor."""
    prob = problem if isinstance(problem, Problem) else make_problem(problem)
    _check(load().dattn_step_host(ctypes.byref(prob), ctypes.byref(io), ctypes.byref(cache), staging.data_ptr(),
                                  staging.numel(), workspace.data_ptr(), workspace.numel(), _stream_ptr(stream)),
           "dattn_step_host")


def dattn_step_host_submit(problem, io: HostStep, cache: Tensors, staging, workspace, done_event,
                           stream=None) -> None:
    """Enqueue one decode step from host memory and return at once; ``done_event`` (a
    torch.cuda.Event) is recorded after its output transfer (see dattn.h)."""
    prob = problem if isinstance(problem, Problem) else make_problem(problem)
    if not done_event.cuda_event:      # torch creates the CUDA event at its first record
        done_event.record(stream if stream is not None else None)
    _check(load().dattn_step_host_submit(ctypes.byref(prob), ctypes.byref(io), ctypes.byref(cache),
                                         staging.data_ptr(), staging.numel(), workspace.data_ptr(),
                                         workspace.numel(), _stream_ptr(stream), done_event.cuda_event),
           "dattn_step_host_submit")


def dattn_step_host_submit_ex(problem, io: HostStep, cache: Tensors, staging, workspace, done_event,
                              h2d_stream, d2h_stream, inputs_event, kernels_event, stream=None) -> None:
    """dattn_step_host_submit with the transfers on ``h2d_stream`` and ``d2h_stream``
    (torch.cuda.Stream), ordered against the kernels by ``inputs_event`` and
    ``kernels_event`` (torch.cuda.Event); ``done_event`` is recorded on the device->host
    stream after the output transfer (see dattn.h)."""
    prob = problem if isinstance(problem, Problem) else make_problem(problem)
    for ev in (done_event, inputs_event, kernels_event):
        if not ev.cuda_event:          # torch creates the CUDA event at its first record
            ev.record(h2d_stream)
    cp = StepCopies(h2d_stream.cuda_stream, d2h_stream.cuda_stream, inputs_event.cuda_event,
                    kernels_event.cuda_event)
    _check(load().dattn_step_host_submit_ex(ctypes.byref(prob), ctypes.byref(io), ctypes.byref(cache),
                                            staging.data_ptr(), staging.numel(), workspace.data_ptr(),
                                            workspace.numel(), _stream_ptr(stream), done_event.cuda_event,
                                            ctypes.byref(cp)), "dattn_step_host_submit_ex")


def dattn_step_host_finish(problem, io: HostStep, staging, done_event) -> None:
    """Wait for a submitted step and copy its O (and LSE) into the host arrays of io."""
    prob = problem if isinstance(problem, Problem) else make_problem(problem)
    _check(load().dattn_step_host_finish(ctypes.byref(prob), ctypes.byref(io), staging.data_ptr(), staging.numel(),
                                         done_event.cuda_event), "dattn_step_host_finish")


def dattn_step_host_status(problem, io: HostStep, workspace, stream=None) -> int:
    prob = problem if isinstance(problem, Problem) else make_problem(problem)
    flags = ctypes.c_int32()
    st = load().dattn_step_host_status(ctypes.byref(prob), ctypes.byref(io), workspace.data_ptr(),
                                       ctypes.byref(flags), _stream_ptr(stream))
    if st not in (0, 6):
        _check(st, "dattn_step_host_status")
    return flags.value
