"""ctypes binding of libca.so (include/ca.h), argument marshalling only.

Every computation runs in the library's CUDA kernels.  If libca.so is missing
or cannot be loaded, every entry point raises: there is no fallback.  Torch
tensors are accepted for device buffers (their data pointers are passed);
torch is used here only for memory and streams.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional, Sequence

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "lib", "libca.so")

CA_OK = 0
CA_ERR_INVALID_ARG = 1
CA_ERR_UNSUPPORTED = 2
CA_ERR_CUDA = 3
CA_ERR_DEVICE_TIMEOUT = 4
CA_ERR_DEVICE_BOUNDS = 5
CA_ERR_NO_DEVICE = 6
CA_DTYPE_BF16 = 0
CA_DTYPE_FP32 = 1
CA_BWD_KERNEL_AUTO = 0
CA_BWD_KERNEL_SINGLE = 1
CA_BWD_KERNEL_PAIR = 2

# names declared in include/ca.h and include/ca_sched.h, in order
EXPORTS = [
    "ca_plan_create", "ca_plan_dry_run", "ca_plan_create_masked", "ca_plan_dry_run_masked", "ca_plan_set_kv_split",
    "ca_plan_set_backward_kernel", "ca_plan_info",
    "ca_plan_task_pairs", "ca_plan_destroy",
    "ca_forward", "ca_backward", "ca_backward_noalloc", "ca_merge", "ca_device_status", "ca_plan_set_wait_limit",
    "ca_watchdog_selftest", "ca_plan_set_timing_events", "ca_status_string", "ca_last_error", "ca_version",
    "ca_profile_create", "ca_profile_predict", "ca_profile_peak", "ca_profile_destroy", "ca_optimal_shard",
    "ca_schedule", "ca_shard_2n",
]


class CAError(RuntimeError):
    def __init__(self, status: int, msg: str):
        super().__init__(f"[{status}] {msg}")
        self.status = status


class Task(ctypes.Structure):
    _fields_ = [("doc_id", ctypes.c_int32), ("reserved", ctypes.c_int32), ("q_start", ctypes.c_int64),
                ("q_len", ctypes.c_int64), ("kv_start", ctypes.c_int64), ("kv_len", ctypes.c_int64)]


class Mask(ctypes.Structure):
    _fields_ = [("sink", ctypes.c_int64), ("lo", ctypes.c_int64), ("window", ctypes.c_int64)]


class Shape(ctypes.Structure):
    _fields_ = [("num_q_heads", ctypes.c_int32), ("num_kv_heads", ctypes.c_int32), ("head_dim", ctypes.c_int32),
                ("softmax_scale", ctypes.c_float), ("o_dtype", ctypes.c_int32)]


class PlanInfo(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int64) for n in (
        "total_q", "total_kv", "n_tasks", "n_docs", "causal_pairs", "flops_fwd", "flops_bwd",
        "workspace_bytes", "n_fwd_items", "n_bwd_items", "fwd_tile_pairs", "bwd_tile_pairs")]

    def as_dict(self):
        return {n: int(getattr(self, n)) for n, _ in self._fields_}


class SchedParams(ctypes.Structure):
    _fields_ = [("n_servers", ctypes.c_int32), ("tolerance", ctypes.c_double), ("min_score", ctypes.c_double),
                ("bytes_q", ctypes.c_double), ("bytes_kv", ctypes.c_double), ("min_shard_tokens", ctypes.c_int64)]


class SchedTask(ctypes.Structure):
    _fields_ = [("server", ctypes.c_int32), ("home", ctypes.c_int32), ("doc_id", ctypes.c_int32),
                ("reserved", ctypes.c_int32), ("q_start", ctypes.c_int64), ("q_len", ctypes.c_int64),
                ("kv_len", ctypes.c_int64), ("pairs", ctypes.c_int64)]


class SchedResult(ctypes.Structure):
    _fields_ = [("target_pairs_x1000", ctypes.c_int64), ("max_load", ctypes.c_int64), ("min_load", ctypes.c_int64),
                ("n_tasks", ctypes.c_int64), ("n_migrations", ctypes.c_int64), ("n_splits", ctypes.c_int64),
                ("comm_bytes", ctypes.c_double)]

    def as_dict(self):
        return {n: (float(getattr(self, n)) if n == "comm_bytes" else int(getattr(self, n))) for n, _ in self._fields_}


_lib = None


def load(path: Optional[str] = None) -> ctypes.CDLL:
    """Load libca.so (raises if it is missing: build it with
    ``document_masked_core_gb300.build.build()``)."""
    global _lib
    if _lib is not None and path is None:
        return _lib
    p = path or LIB_PATH
    if not os.path.exists(p):
        raise RuntimeError(f"libca.so not found at {p}; run document_masked_core_gb300.build.build() first")
    L = ctypes.CDLL(p)
    vp, i32, i64, st = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_int
    L.ca_plan_create.restype = st
    L.ca_plan_create.argtypes = [ctypes.POINTER(Task), i32, vp, vp, i32, ctypes.POINTER(Shape), vp,
                                 ctypes.POINTER(vp)]
    L.ca_plan_dry_run.restype = st
    L.ca_plan_dry_run.argtypes = [ctypes.POINTER(Task), i32, vp, vp, i32, ctypes.POINTER(Shape),
                                  ctypes.POINTER(PlanInfo), vp]
    L.ca_plan_create_masked.restype = st
    L.ca_plan_create_masked.argtypes = [ctypes.POINTER(Task), vp, i32, vp, vp, i32, ctypes.POINTER(Shape), vp,
                                        ctypes.POINTER(vp)]
    L.ca_plan_dry_run_masked.restype = st
    L.ca_plan_dry_run_masked.argtypes = [ctypes.POINTER(Task), vp, i32, vp, vp, i32, ctypes.POINTER(Shape),
                                         ctypes.POINTER(PlanInfo), vp]
    L.ca_plan_set_kv_split.restype = st
    L.ca_plan_set_kv_split.argtypes = [vp, i32]
    L.ca_plan_set_backward_kernel.restype = st
    L.ca_plan_set_backward_kernel.argtypes = [vp, i32]
    L.ca_plan_info.restype = st
    L.ca_plan_info.argtypes = [vp, ctypes.POINTER(PlanInfo)]
    L.ca_plan_task_pairs.restype = st
    L.ca_plan_task_pairs.argtypes = [vp, vp]
    L.ca_plan_destroy.restype = None
    L.ca_plan_destroy.argtypes = [vp]
    L.ca_forward.restype = st
    L.ca_forward.argtypes = [vp] * 8
    L.ca_backward.restype = st
    L.ca_backward.argtypes = [vp] * 12
    L.ca_backward_noalloc.restype = st
    L.ca_backward_noalloc.argtypes = [vp] * 11
    L.ca_merge.restype = st
    L.ca_merge.argtypes = [i32, vp, vp, i32, i64, i32, i32, vp, i32, vp, vp]
    L.ca_device_status.restype = st
    L.ca_device_status.argtypes = [vp, vp]
    L.ca_plan_set_wait_limit.restype = st
    L.ca_plan_set_wait_limit.argtypes = [vp, i64]
    L.ca_watchdog_selftest.restype = st
    L.ca_watchdog_selftest.argtypes = [vp, i64, vp]
    L.ca_plan_set_timing_events.restype = st
    L.ca_plan_set_timing_events.argtypes = [vp, vp, i32]
    L.ca_status_string.restype = ctypes.c_char_p
    L.ca_status_string.argtypes = [st]
    L.ca_last_error.restype = ctypes.c_char_p
    L.ca_last_error.argtypes = []
    L.ca_version.restype = i32
    L.ca_version.argtypes = []
    dbl = ctypes.c_double
    L.ca_profile_create.restype = st
    L.ca_profile_create.argtypes = [vp, i32, vp, i32, vp, dbl, ctypes.POINTER(vp)]
    L.ca_profile_predict.restype = st
    L.ca_profile_predict.argtypes = [vp, i64, i64, ctypes.POINTER(dbl)]
    L.ca_profile_peak.restype = st
    L.ca_profile_peak.argtypes = [vp, ctypes.POINTER(dbl)]
    L.ca_profile_destroy.restype = None
    L.ca_profile_destroy.argtypes = [vp]
    L.ca_optimal_shard.restype = st
    L.ca_optimal_shard.argtypes = [i64, i64, dbl, i64, dbl, dbl, ctypes.POINTER(i64), ctypes.POINTER(i64),
                                   ctypes.POINTER(dbl)]
    L.ca_shard_2n.restype = st
    L.ca_shard_2n.argtypes = [vp, i32, i32, ctypes.POINTER(SchedTask), i64, ctypes.POINTER(i64)]
    L.ca_schedule.restype = st
    L.ca_schedule.argtypes = [vp, i32, ctypes.POINTER(SchedParams), ctypes.POINTER(SchedTask), i64,
                              ctypes.POINTER(SchedResult)]
    if path is None:
        _lib = L
    return L


def _check(status: int):
    if status != CA_OK:
        L = load()
        raise CAError(status, f"{L.ca_status_string(status).decode()}: {L.ca_last_error().decode()}")


def _ptr(x) -> Optional[int]:
    if x is None:
        return None
    if isinstance(x, int):
        return x
    return int(x.data_ptr())


def _stream(stream) -> Optional[int]:
    if stream is None:
        import torch
        return int(torch.cuda.current_stream().cuda_stream)
    if isinstance(stream, int):
        return stream
    return int(stream.cuda_stream)


def _task_array(task_doc, task_q_start, task_q_len, task_kv_start, task_kv_len):
    n = len(task_q_len)
    arr = (Task * max(n, 1))()
    for i in range(n):
        arr[i].doc_id = int(task_doc[i])
        arr[i].reserved = 0
        arr[i].q_start = int(task_q_start[i])
        arr[i].q_len = int(task_q_len[i])
        arr[i].kv_start = int(task_kv_start[i])
        arr[i].kv_len = int(task_kv_len[i])
    return arr, n


def _mask_array(masks, n):
    """(sink, lo, window) triples (or None) -> ca_mask_t array (or None)."""
    if masks is None:
        return None
    m = np.asarray(masks, dtype=np.int64).reshape(-1, 3)
    if len(m) != n:
        raise ValueError("one mask per task")
    if not m.any():
        return None
    arr = (Mask * n)()
    for i in range(n):
        arr[i].sink, arr[i].lo, arr[i].window = (int(x) for x in m[i])
    return arr


def _workload_masks(w):
    return np.stack(w.masks(), axis=1) if getattr(w, "masked", False) else None


def dry_run(task_doc, task_q_start, task_q_len, task_kv_start, task_kv_len, doc_len, doc_kv_offset,
            num_q_heads: int, num_kv_heads: int, head_dim: int, softmax_scale: Optional[float] = None,
            o_dtype: int = CA_DTYPE_BF16, masks=None):
    """ca_plan_dry_run(_masked): validation and integer accounting without a
    device.  Returns (info dict, per-task pairs)."""
    L = load()
    arr, n = _task_array(task_doc, task_q_start, task_q_len, task_kv_start, task_kv_len)
    marr = _mask_array(masks, n)
    dl = np.ascontiguousarray(doc_len, dtype=np.int64)
    do = np.ascontiguousarray(doc_kv_offset, dtype=np.int64)
    if softmax_scale is None:
        softmax_scale = head_dim ** -0.5
    shape = Shape(num_q_heads, num_kv_heads, head_dim, float(softmax_scale), int(o_dtype))
    info = PlanInfo()
    pairs = np.zeros(max(n, 1), dtype=np.int64)
    _check(L.ca_plan_dry_run_masked(arr, marr, n, dl.ctypes.data, do.ctypes.data, len(dl), ctypes.byref(shape),
                                    ctypes.byref(info), pairs.ctypes.data))
    return info.as_dict(), pairs[:n]


def dry_run_workload(w):
    return dry_run(w.task_doc, w.task_q_start, w.task_q_len, w.task_kv_start, w.task_kv_len, w.doc_len,
                   w.doc_kv_offset, w.num_q_heads, w.num_kv_heads, w.head_dim, w.softmax_scale,
                   masks=_workload_masks(w))


class Plan:
    """A validated CA-task pool uploaded to the current device (ca_plan_create)."""

    def __init__(self, task_doc, task_q_start, task_q_len, task_kv_start, task_kv_len, doc_len, doc_kv_offset,
                 num_q_heads: int, num_kv_heads: int, head_dim: int, softmax_scale: Optional[float] = None,
                 o_dtype: int = CA_DTYPE_BF16, stream=None, masks=None):
        L = load()
        arr, n = _task_array(task_doc, task_q_start, task_q_len, task_kv_start, task_kv_len)
        marr = _mask_array(masks, n)
        self._doc_len = np.ascontiguousarray(doc_len, dtype=np.int64)
        self._doc_off = np.ascontiguousarray(doc_kv_offset, dtype=np.int64)
        if softmax_scale is None:
            softmax_scale = head_dim ** -0.5
        shape = Shape(num_q_heads, num_kv_heads, head_dim, float(softmax_scale), int(o_dtype))
        h = ctypes.c_void_p()
        _check(L.ca_plan_create_masked(arr, marr, n, self._doc_len.ctypes.data, self._doc_off.ctypes.data,
                                       len(self._doc_len), ctypes.byref(shape), _stream(stream), ctypes.byref(h)))
        self._h = h
        self.num_q_heads, self.num_kv_heads, self.head_dim = num_q_heads, num_kv_heads, head_dim
        self.o_dtype = o_dtype
        self.n_tasks = n

    @classmethod
    def from_workload(cls, w, o_dtype: int = CA_DTYPE_BF16, stream=None) -> "Plan":
        return cls(w.task_doc, w.task_q_start, w.task_q_len, w.task_kv_start, w.task_kv_len, w.doc_len,
                   w.doc_kv_offset, w.num_q_heads, w.num_kv_heads, w.head_dim, w.softmax_scale, o_dtype, stream,
                   masks=_workload_masks(w))

    @property
    def handle(self) -> int:
        if self._h is None or not self._h.value:
            raise RuntimeError("plan is closed")
        return self._h.value

    def info(self) -> dict:
        out = PlanInfo()
        _check(load().ca_plan_info(self.handle, ctypes.byref(out)))
        return out.as_dict()

    def set_kv_split(self, visits_per_part: int):
        """ca_plan_set_kv_split: cut forward items longer than this many key
        tiles into parts merged in the launch (0 = automatic, < 0 = never).
        The workspace size may change: allocate it after this call."""
        _check(load().ca_plan_set_kv_split(self.handle, int(visits_per_part)))

    def set_backward_kernel(self, kind: int):
        """Which backward main kernel runs: CA_BWD_KERNEL_AUTO or
        CA_BWD_KERNEL_SINGLE (the one-CTA kernel), CA_BWD_KERNEL_PAIR (the
        CTA-pair kernel where it applies)."""
        _check(load().ca_plan_set_backward_kernel(self.handle, int(kind)))

    def task_pairs(self) -> np.ndarray:
        out = np.zeros(self.n_tasks, dtype=np.int64)
        _check(load().ca_plan_task_pairs(self.handle, out.ctypes.data))
        return out

    def forward(self, q, k, v, o, lse, workspace=None, stream=None):
        """ca_forward: O and LSE of every task row.  q [total_q, H_q, d] and
        k, v [total_kv, H_kv, d] are bf16 CUDA tensors; o [total_q, H_q, d] is
        bf16 or float32 as the plan's o_dtype; lse [total_q, H_q] float32;
        workspace holds at least info()["workspace_bytes"] bytes.  Runs on
        ``stream`` (default: torch's current stream); nothing is allocated."""
        _check(load().ca_forward(self.handle, _ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(workspace),
                                 _stream(stream)))

    def backward(self, q, k, v, o, lse, d_o, dq, dk, dv, workspace, stream=None):
        """ca_backward: dQ, dK, dV from the forward's O and LSE and the
        upstream gradient d_o (bf16, shaped like q).  dq is shaped like q, dk
        and dv like k (bf16); dk and dv are overwritten with the sum over every
        task of the document (rows no task sees get 0)."""
        _check(load().ca_backward(self.handle, _ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(d_o),
                                  _ptr(dq), _ptr(dk), _ptr(dv), _ptr(workspace), _stream(stream)))

    def backward_noalloc(self, q, k, v, o, lse, d_o, dq, dk, dv, stream=None):
        """ca_backward_noalloc: the backward with the library's own 16 MiB
        scratch array instead of a caller workspace (for callers that cannot
        allocate device memory; calls on one device must not overlap)."""
        _check(load().ca_backward_noalloc(self.handle, _ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(d_o),
                                          _ptr(dq), _ptr(dk), _ptr(dv), _stream(stream)))

    def device_status(self, stream=None) -> int:
        """Sync the stream and return (and clear) the device error status."""
        return int(load().ca_device_status(self.handle, _stream(stream)))

    def set_wait_limit(self, ns: int):
        _check(load().ca_plan_set_wait_limit(self.handle, int(ns)))

    def watchdog_selftest(self, limit_ns: int, stream=None):
        _check(load().ca_watchdog_selftest(self.handle, int(limit_ns), _stream(stream)))

    def set_timing_events(self, events):
        """Bracket each kernel launch with the given 6 torch.cuda.Events (or None)."""
        if events is None:
            self._events_arr = None
            _check(load().ca_plan_set_timing_events(self.handle, None, 0))
            return
        arr = (ctypes.c_void_p * len(events))(*[int(e.cuda_event) for e in events])
        self._events_arr = (arr, list(events))  # keep the array and the events alive
        _check(load().ca_plan_set_timing_events(self.handle, arr, len(events)))

    def close(self):
        if getattr(self, "_h", None) is not None and self._h.value:
            load().ca_plan_destroy(self._h.value)
        self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def merge(o_parts: Sequence, lse_parts: Sequence, rows: int, heads: int, head_dim: int, o_out, lse_out=None,
          parts_dtype: int = CA_DTYPE_FP32, out_dtype: int = CA_DTYPE_BF16, stream=None):
    """ca_merge over n partial (O, LSE) results."""
    n = len(o_parts)
    op = (ctypes.c_void_p * n)(*[_ptr(x) for x in o_parts])
    lp = (ctypes.c_void_p * n)(*[_ptr(x) for x in lse_parts])
    _check(load().ca_merge(n, op, lp, int(parts_dtype), int(rows), int(heads), int(head_dim), _ptr(o_out),
                           int(out_dtype), _ptr(lse_out), _stream(stream)))


def version() -> int:
    return int(load().ca_version())


# ---------------------------------------------------------------- host planning (include/ca_sched.h)

class Profile:
    """Profiler cost model (ca_profile_*): measured fwd+bwd seconds on a grid
    of (query length, context length) CA-task shapes."""

    def __init__(self, nq_grid, nkv_grid, seconds, flops_per_pair: float):
        L = load()
        self.nq_grid = np.ascontiguousarray(nq_grid, dtype=np.int64)
        self.nkv_grid = np.ascontiguousarray(nkv_grid, dtype=np.int64)
        sec = np.ascontiguousarray(seconds, dtype=np.float64).reshape(len(self.nq_grid), len(self.nkv_grid))
        h = ctypes.c_void_p()
        _check(L.ca_profile_create(self.nq_grid.ctypes.data, len(self.nq_grid), self.nkv_grid.ctypes.data,
                                   len(self.nkv_grid), sec.ctypes.data, float(flops_per_pair), ctypes.byref(h)))
        self._h = h

    def predict(self, n_q: int, n_kv: int) -> float:
        out = ctypes.c_double()
        _check(load().ca_profile_predict(self._h.value, int(n_q), int(n_kv), ctypes.byref(out)))
        return float(out.value)

    def peak(self) -> float:
        out = ctypes.c_double()
        _check(load().ca_profile_peak(self._h.value, ctypes.byref(out)))
        return float(out.value)

    def close(self):
        if getattr(self, "_h", None) is not None and self._h.value:
            load().ca_profile_destroy(self._h.value)
        self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def optimal_shard(L_q: int, L_kv: int, alpha: float, target_pairs: int, bytes_q: float, bytes_kv: float):
    """ca_optimal_shard: (n_q, n_kv, continuous optimum) of a split."""
    nq, nkv, real = ctypes.c_int64(), ctypes.c_int64(), ctypes.c_double()
    _check(load().ca_optimal_shard(int(L_q), int(L_kv), float(alpha), int(target_pairs), float(bytes_q),
                                   float(bytes_kv), ctypes.byref(nq), ctypes.byref(nkv), ctypes.byref(real)))
    return int(nq.value), int(nkv.value), float(real.value)


def schedule(doc_len, n_servers: int, bytes_q: float, bytes_kv: float, tolerance: float = 0.0,
             min_score: float = 0.0, min_shard_tokens: int = 0):
    """ca_schedule: returns (tasks as a structured numpy array, result dict)."""
    L = load()
    dl = np.ascontiguousarray(doc_len, dtype=np.int64)
    prm = SchedParams(int(n_servers), float(tolerance), float(min_score), float(bytes_q), float(bytes_kv),
                      int(min_shard_tokens))
    res = SchedResult()
    cap = max(16, 4 * len(dl) + 4 * n_servers)
    while True:
        buf = (SchedTask * cap)()
        st = L.ca_schedule(dl.ctypes.data, len(dl), ctypes.byref(prm), buf, cap, ctypes.byref(res))
        if st == CA_OK:
            break
        if st == CA_ERR_INVALID_ARG and res.n_tasks > cap:
            cap = int(res.n_tasks)
            continue
        _check(st)
    return _sched_tasks(buf, int(res.n_tasks)), res.as_dict()


_SCHED_DTYPE = np.dtype([("server", np.int32), ("home", np.int32), ("doc_id", np.int32), ("reserved", np.int32),
                         ("q_start", np.int64), ("q_len", np.int64), ("kv_len", np.int64), ("pairs", np.int64)])


def _sched_tasks(buf, n):
    return np.frombuffer(bytes(buf)[: n * ctypes.sizeof(SchedTask)], dtype=_SCHED_DTYPE).copy()


def shard_2n(doc_len, n_ranks: int):
    """ca_shard_2n: 2N-chunk load-balanced shards of every document."""
    L = load()
    dl = np.ascontiguousarray(doc_len, dtype=np.int64)
    n = ctypes.c_int64()
    cap = 2 * len(dl) * int(n_ranks)
    buf = (SchedTask * max(cap, 1))()
    _check(L.ca_shard_2n(dl.ctypes.data, len(dl), int(n_ranks), buf, cap, ctypes.byref(n)))
    return _sched_tasks(buf, int(n.value))
