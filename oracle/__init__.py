"""fp64 CPU oracle for document-masked core attention (test infrastructure).

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline
leg may import this package.  The product path (``document_masked_core_gb300``)
never imports, links or runs it, and this package never imports the product.

The arithmetic lives in ``ca_oracle.c`` (plain C, double precision, one row or
one key column at a time, following the definitions written at its top).  This
file compiles it with gcc, marshals numpy arrays through ctypes, and decides
which rows a sampled check needs.  See ``ca_oracle.c`` for the formulas and
the passages they follow.

Parity pins for every function here live in ``tests/test_oracle_pins.py``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "ca_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "libca_oracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile ca_oracle.c into oracle/_build/libca_oracle.so (gcc, OpenMP)."""
    os.makedirs(_BUILD, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O3", "-fopenmp", "-shared", "-fPIC", "-std=c11", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


class _Problem(ctypes.Structure):
    _fields_ = [
        ("n_tasks", ctypes.c_int32),
        ("t_doc", ctypes.c_void_p),
        ("t_q_start", ctypes.c_void_p),
        ("t_q_len", ctypes.c_void_p),
        ("t_kv_start", ctypes.c_void_p),
        ("t_kv_len", ctypes.c_void_p),
        ("t_row0", ctypes.c_void_p),
        ("t_sink", ctypes.c_void_p),
        ("t_lo", ctypes.c_void_p),
        ("t_win", ctypes.c_void_p),
        ("n_docs", ctypes.c_int32),
        ("doc_len", ctypes.c_void_p),
        ("doc_kv_offset", ctypes.c_void_p),
        ("hq", ctypes.c_int32),
        ("hkv", ctypes.c_int32),
        ("d", ctypes.c_int32),
        ("scale", ctypes.c_double),
        ("q", ctypes.c_void_p),
        ("k", ctypes.c_void_p),
        ("v", ctypes.c_void_p),
        ("dout", ctypes.c_void_p),
    ]


def lib():
    global _lib
    with _lock:
        if _lib is None:
            build()
            L = ctypes.CDLL(_LIB_PATH)
            vp, i64, i32, dp = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32, ctypes.c_void_p
            L.orc_version.restype = ctypes.c_int
            L.orc_num_threads.restype = ctypes.c_int
            L.orc_visible_count.restype = i64
            L.orc_visible_count.argtypes = [i64, i64, i64]
            L.orc_visible_count_masked.restype = i64
            L.orc_visible_count_masked.argtypes = [i64, i64, i64, i64, i64, i64]
            L.orc_task_pairs.restype = None
            L.orc_task_pairs.argtypes = [i32, vp, vp, vp, vp, vp]
            pb = ctypes.POINTER(_Problem)
            L.orc_forward_rows.argtypes = [pb, i64, vp, vp, dp, dp]
            L.orc_forward_all.argtypes = [pb, i64, dp, dp]
            L.orc_dq_rows.argtypes = [pb, i64, vp, vp, dp]
            L.orc_row_stats.argtypes = [pb, i64, vp, dp, dp]
            L.orc_dkdv_cols.argtypes = [pb, i64, vp, vp, vp, dp, dp, dp, dp]
            L.orc_merge.restype = None
            L.orc_merge.argtypes = [i32, i64, i32, dp, dp, dp, dp]
            _lib = L
    return _lib


def num_threads() -> int:
    return int(lib().orc_num_threads())


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def _bits(x) -> np.ndarray:
    """bf16 values (torch CPU tensor, or numpy uint16 bit patterns) -> contiguous uint16."""
    if x is None:
        return None
    if isinstance(x, np.ndarray):
        if x.dtype != np.uint16:
            raise TypeError("numpy inputs must be uint16 bf16 bit patterns")
        return np.ascontiguousarray(x)
    import torch
    if x.dtype != torch.bfloat16:
        raise TypeError("torch inputs must be bfloat16")
    return x.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


class Problem:
    """A workload plus its bf16 inputs, ready for the C oracle."""

    def __init__(self, w, q, k, v, do=None):
        self.w = w
        self.q, self.k, self.v, self.do = _bits(q), _bits(k), _bits(v), _bits(do)
        self.t_doc = np.ascontiguousarray(w.task_doc, dtype=np.int32)
        self.t_q_start = np.ascontiguousarray(w.task_q_start, dtype=np.int64)
        self.t_q_len = np.ascontiguousarray(w.task_q_len, dtype=np.int64)
        self.t_kv_start = np.ascontiguousarray(w.task_kv_start, dtype=np.int64)
        self.t_kv_len = np.ascontiguousarray(w.task_kv_len, dtype=np.int64)
        self.t_row0 = np.ascontiguousarray(w.task_row_offset(), dtype=np.int64)
        sink, lo, win = w.masks()
        self.t_sink = np.ascontiguousarray(sink, dtype=np.int64)
        self.t_lo = np.ascontiguousarray(lo, dtype=np.int64)
        self.t_win = np.ascontiguousarray(win, dtype=np.int64)
        masked = bool(self.t_sink.any() or self.t_lo.any() or self.t_win.any())
        self.doc_len = np.ascontiguousarray(w.doc_len, dtype=np.int64)
        self.doc_kv_offset = np.ascontiguousarray(w.doc_kv_offset, dtype=np.int64)
        self.total_q = w.total_q
        hq, hkv, d = w.num_q_heads, w.num_kv_heads, w.head_dim
        if self.q.size != self.total_q * hq * d:
            raise ValueError("q has the wrong size")
        if self.k.size != w.total_kv * hkv * d or self.v.size != self.k.size:
            raise ValueError("k/v have the wrong size")
        self.s = _Problem(
            w.n_tasks, _ptr(self.t_doc).value, _ptr(self.t_q_start).value, _ptr(self.t_q_len).value,
            _ptr(self.t_kv_start).value, _ptr(self.t_kv_len).value, _ptr(self.t_row0).value,
            (_ptr(self.t_sink).value if masked else None), (_ptr(self.t_lo).value if masked else None),
            (_ptr(self.t_win).value if masked else None),
            w.n_docs, _ptr(self.doc_len).value, _ptr(self.doc_kv_offset).value,
            hq, hkv, d, float(w.softmax_scale),
            _ptr(self.q).value, _ptr(self.k).value, _ptr(self.v).value,
            (_ptr(self.do).value if self.do is not None else None))

    @property
    def ref(self):
        return ctypes.byref(self.s)


def task_pairs(w) -> np.ndarray:
    """Visible (token, key) pairs of every task, per head, int64."""
    n = w.n_tasks
    out = np.zeros(n, dtype=np.int64)
    a = [np.ascontiguousarray(x, dtype=np.int64) for x in
         (w.task_q_start, w.task_q_len, w.task_kv_start, w.task_kv_len)]
    lib().orc_task_pairs(n, *[_ptr(x) for x in a], _ptr(out))
    sink, lo, win = w.masks()
    for t in range(n):  # masked tasks: the per-key count of the visibility rule
        if sink[t] or lo[t] or win[t]:
            qs, ql, ks, kl = (int(x[t]) for x in a)
            out[t] = sum(lib().orc_visible_count_masked(p, ks, kl, int(sink[t]), int(lo[t]), int(win[t]))
                         for p in range(qs, qs + ql))
    return out


def visible_count_masked(p, kv_start, kv_len, sink, lo, window) -> int:
    return int(lib().orc_visible_count_masked(p, kv_start, kv_len, sink, lo, window))


def flops(w):
    """(forward, backward) FLOPs: 4 d and 8 d per causal pair per query head."""
    pairs = int(task_pairs(w).sum())
    base = pairs * w.num_q_heads * w.head_dim
    return 4 * base, 8 * base


def forward(pb: Problem):
    """O [total_q, hq, d] and LSE [total_q, hq], float64."""
    w = pb.w
    o = np.zeros((pb.total_q, w.num_q_heads, w.head_dim), dtype=np.float64)
    lse = np.zeros((pb.total_q, w.num_q_heads), dtype=np.float64)
    if lib().orc_forward_all(pb.ref, pb.total_q, _ptr(o), _ptr(lse)):
        raise MemoryError("oracle forward failed")
    return o, lse


def forward_rows(pb: Problem, rows, heads):
    rows = np.ascontiguousarray(rows, dtype=np.int64)
    heads = np.ascontiguousarray(heads, dtype=np.int32)
    o = np.zeros((len(rows), pb.w.head_dim), dtype=np.float64)
    lse = np.zeros(len(rows), dtype=np.float64)
    if lib().orc_forward_rows(pb.ref, len(rows), _ptr(rows), _ptr(heads), _ptr(o), _ptr(lse)):
        raise MemoryError("oracle forward_rows failed")
    return o, lse


def dq_rows(pb: Problem, rows, heads):
    if pb.do is None:
        raise ValueError("problem has no dO")
    rows = np.ascontiguousarray(rows, dtype=np.int64)
    heads = np.ascontiguousarray(heads, dtype=np.int32)
    dq = np.zeros((len(rows), pb.w.head_dim), dtype=np.float64)
    if lib().orc_dq_rows(pb.ref, len(rows), _ptr(rows), _ptr(heads), _ptr(dq)):
        raise MemoryError("oracle dq_rows failed")
    return dq


def dependent_rows_mask(w, col_doc, col_pos, col_g) -> np.ndarray:
    """uint8 [total_q, hq]: the (row, head) pairs whose statistics the given
    key columns need (rows p >= j of tasks of the column's document whose KV
    block holds j, heads of the column's group)."""
    G = w.num_q_heads // w.num_kv_heads
    mark = np.zeros((w.total_q, w.num_q_heads), dtype=np.uint8)
    row0 = w.task_row_offset()
    col_doc = np.asarray(col_doc)
    col_pos = np.asarray(col_pos)
    col_g = np.asarray(col_g)
    for t in range(w.n_tasks):
        sel = col_doc == w.task_doc[t]
        if not sel.any():
            continue
        ks, kl = int(w.task_kv_start[t]), int(w.task_kv_len[t])
        inblk = sel & (col_pos >= ks) & (col_pos < ks + kl)
        if not inblk.any():
            continue
        for g in np.unique(col_g[inblk]):
            jmin = int(col_pos[inblk & (col_g == g)].min())
            i0 = max(0, jmin - int(w.task_q_start[t]))
            if i0 >= int(w.task_q_len[t]):
                continue
            r0 = int(row0[t])
            mark[r0 + i0:r0 + int(w.task_q_len[t]), g * G:(g + 1) * G] = 1
    return mark


def row_stats(pb: Problem, mark: np.ndarray):
    """LSE and D = dO . O for the marked (row, head) pairs (others left 0)."""
    mark = np.ascontiguousarray(mark, dtype=np.uint8)
    lse = np.zeros(mark.shape, dtype=np.float64)
    D = np.zeros(mark.shape, dtype=np.float64)
    if lib().orc_row_stats(pb.ref, pb.total_q, _ptr(mark), _ptr(lse), _ptr(D)):
        raise MemoryError("oracle row_stats failed")
    return lse, D


def dkdv_cols(pb: Problem, col_doc, col_pos, col_g, stats=None):
    """dK, dV [n, d] of key columns (document, position in document, kv head)."""
    if pb.do is None:
        raise ValueError("problem has no dO")
    col_doc = np.ascontiguousarray(col_doc, dtype=np.int32)
    col_pos = np.ascontiguousarray(col_pos, dtype=np.int64)
    col_g = np.ascontiguousarray(col_g, dtype=np.int32)
    if stats is None:
        stats = row_stats(pb, dependent_rows_mask(pb.w, col_doc, col_pos, col_g))
    lse, D = stats
    n, d = len(col_doc), pb.w.head_dim
    dk = np.zeros((n, d), dtype=np.float64)
    dv = np.zeros((n, d), dtype=np.float64)
    if lib().orc_dkdv_cols(pb.ref, n, _ptr(col_doc), _ptr(col_pos), _ptr(col_g),
                           _ptr(np.ascontiguousarray(lse)), _ptr(np.ascontiguousarray(D)),
                           _ptr(dk), _ptr(dv)):
        raise MemoryError("oracle dkdv_cols failed")
    return dk, dv


def backward(pb: Problem):
    """Full dQ [total_q, hq, d], dK, dV [total_kv, hkv, d] (float64).  Key rows
    outside every document stay 0, as do keys no task sees."""
    w = pb.w
    hq, hkv, d = w.num_q_heads, w.num_kv_heads, w.head_dim
    rows = np.repeat(np.arange(pb.total_q, dtype=np.int64), hq)
    heads = np.tile(np.arange(hq, dtype=np.int32), pb.total_q)
    dq = dq_rows(pb, rows, heads).reshape(pb.total_q, hq, d)
    col_doc, col_pos, col_g, col_row = [], [], [], []
    for i in range(w.n_docs):
        L = int(w.doc_len[i])
        pos = np.arange(L, dtype=np.int64)
        for g in range(hkv):
            col_doc.append(np.full(L, i, dtype=np.int32))
            col_pos.append(pos)
            col_g.append(np.full(L, g, dtype=np.int32))
            col_row.append(int(w.doc_kv_offset[i]) + pos)
    dk = np.zeros((w.total_kv, hkv, d))
    dv = np.zeros((w.total_kv, hkv, d))
    if col_doc:
        cd, cp, cg, cr = (np.concatenate(x) for x in (col_doc, col_pos, col_g, col_row))
        mark = np.ones((pb.total_q, hq), dtype=np.uint8)
        a, b = dkdv_cols(pb, cd, cp, cg, stats=row_stats(pb, mark))
        dk[cr, cg] = a
        dv[cr, cg] = b
    return dq, dk, dv


def merge(o_parts: np.ndarray, lse_parts: np.ndarray):
    """Eq. 4 merge.  o_parts [n, rows, d], lse_parts [n, rows] -> O [rows, d], LSE [rows]."""
    o_parts = np.ascontiguousarray(o_parts, dtype=np.float64)
    lse_parts = np.ascontiguousarray(lse_parts, dtype=np.float64)
    n, rows, d = o_parts.shape
    o = np.zeros((rows, d))
    lse = np.zeros(rows)
    lib().orc_merge(n, rows, d, _ptr(o_parts), _ptr(lse_parts), _ptr(o), _ptr(lse))
    return o, lse
