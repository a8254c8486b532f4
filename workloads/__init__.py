"""Seeded synthetic workloads for document-masked core attention.

This module is the one piece shared by the fp64 oracle side (``oracle/``,
``tests/``) and the CUDA side (``document_masked_core_gb300``).  It draws
document lengths, cuts documents into CA-tasks and draws the Q/K/V/dO values.
It holds none of the attention arithmetic: no pair counts, no FLOPs, no mask
logic beyond the descriptor fields themselves.

A CA-task (Efficient Long-context Language Model Training by Core Attention
Disaggregation, §3.4 "The CA-Task Abstraction") is a contiguous query shard
``[q_start, q_start + q_len)`` of one document plus the keys/values it attends
to.  Here a task also carries ``kv_start``/``kv_len`` so that a KV block of a
split context (Context Parallelism for Scalable Million-Token Inference,
§3.5.2 pass-KV, Appendix B merge) is one task.  The prefix form of the CA-task
is ``kv_start = 0, kv_len = q_start + q_len``.

Layouts (token-major, the same on host and device):
  Q, O, dQ, dO : [total_q, H_q, d]  -- rows of all tasks packed in task order
  K, V, dK, dV : [total_kv, H_kv, d] -- document ``i`` owns rows
                 [doc_kv_offset[i], doc_kv_offset[i] + doc_len[i])
  LSE          : [total_q, H_q] float32
"""
from __future__ import annotations

import dataclasses
import math
from typing import List, Optional

import numpy as np

__all__ = [
    "Workload",
    "tiny_chunk",
    "llama8b_chunk",
    "rebatched_pool",
    "long_context_chunk",
    "split_kv_prefill",
    "custom",
    "lambda_chunk",
    "blockwise_chunk",
    "shared_question_pool",
    "decode_batch",
    "WORKLOADS",
    "MASKED_WORKLOADS",
    "make_tensors",
]


@dataclasses.dataclass
class Workload:
    """Documents, CA-tasks and head shape of one synthetic batch."""

    name: str
    doc_len: np.ndarray          # int64 [n_docs]
    doc_kv_offset: np.ndarray    # int64 [n_docs]
    task_doc: np.ndarray         # int32 [n_tasks]
    task_q_start: np.ndarray     # int64 [n_tasks]
    task_q_len: np.ndarray       # int64 [n_tasks]
    task_kv_start: np.ndarray    # int64 [n_tasks]
    task_kv_len: np.ndarray      # int64 [n_tasks]
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    seed: int = 0
    note: str = ""
    # sparse mask per task ("DCP: Addressing Input Dynamism In Long-Context
    # Training via Dynamic Context Parallelism", §2.4, Figure 6), None = plain
    task_sink: Optional[np.ndarray] = None
    task_lo: Optional[np.ndarray] = None
    task_win: Optional[np.ndarray] = None

    def masks(self):
        """(sink, lo, window) int64 arrays, zeros for plain tasks."""
        z = np.zeros(self.n_tasks, dtype=np.int64)
        pick = lambda a: z.copy() if a is None else np.asarray(a, dtype=np.int64)  # noqa: E731
        return pick(self.task_sink), pick(self.task_lo), pick(self.task_win)

    @property
    def masked(self) -> bool:
        return any(a is not None and np.any(a) for a in (self.task_sink, self.task_lo, self.task_win))

    @property
    def n_docs(self) -> int:
        return int(self.doc_len.shape[0])

    @property
    def n_tasks(self) -> int:
        return int(self.task_q_len.shape[0])

    @property
    def total_q(self) -> int:
        return int(self.task_q_len.sum())

    @property
    def total_kv(self) -> int:
        if self.n_docs == 0:
            return 0
        return int((self.doc_kv_offset + self.doc_len).max())

    @property
    def softmax_scale(self) -> float:
        return 1.0 / math.sqrt(self.head_dim)

    def task_row_offset(self) -> np.ndarray:
        """First packed query row of every task (tasks are packed in order)."""
        off = np.zeros(self.n_tasks, dtype=np.int64)
        if self.n_tasks > 1:
            off[1:] = np.cumsum(self.task_q_len)[:-1]
        return off

    def describe(self) -> dict:
        return {
            "workload": self.name,
            "n_docs": self.n_docs,
            "n_tasks": self.n_tasks,
            "total_q": self.total_q,
            "total_kv": self.total_kv,
            "num_q_heads": self.num_q_heads,
            "num_kv_heads": self.num_kv_heads,
            "head_dim": self.head_dim,
            "seed": self.seed,
        }


def _packed_offsets(lengths: np.ndarray) -> np.ndarray:
    off = np.zeros(len(lengths), dtype=np.int64)
    if len(lengths) > 1:
        off[1:] = np.cumsum(lengths)[:-1]
    return off


def _whole_document_tasks(name, doc_len, hq, hkv, d, seed, note="") -> Workload:
    doc_len = np.asarray(doc_len, dtype=np.int64)
    n = len(doc_len)
    return Workload(
        name=name,
        doc_len=doc_len,
        doc_kv_offset=_packed_offsets(doc_len),
        task_doc=np.arange(n, dtype=np.int32),
        task_q_start=np.zeros(n, dtype=np.int64),
        task_q_len=doc_len.copy(),
        task_kv_start=np.zeros(n, dtype=np.int64),
        task_kv_len=doc_len.copy(),
        num_q_heads=hq,
        num_kv_heads=hkv,
        head_dim=d,
        seed=seed,
        note=note,
    )


def _lognormal_fill(rng, total: int, median: float, sigma: float,
                    lo: int, hi: int, prefix: Optional[List[int]] = None) -> np.ndarray:
    """Append round(exp(ln median + sigma z)) clipped to [lo, hi] until the
    lengths reach ``total``; the last document is truncated to fill exactly."""
    lens = list(prefix or [])
    acc = sum(lens)
    while acc < total:
        z = rng.standard_normal()
        l = int(round(math.exp(math.log(median) + sigma * z)))
        l = min(max(l, lo), hi)
        l = min(l, total - acc)
        lens.append(l)
        acc += l
    return np.asarray(lens, dtype=np.int64)


def tiny_chunk(seed: int = 0) -> Workload:
    """2048-token chunk of documents [1024, 512, 256, 256], 4 q heads / 1 kv
    head, head_dim 64; each document is one CA-task."""
    return _whole_document_tasks("tiny_chunk_2k_g4_d64", [1024, 512, 256, 256], 4, 1, 64, seed)


def llama8b_chunk(seed: int = 0, total: int = 65536) -> Workload:
    """One packed chunk of ``total`` tokens (65536 by default) of documents with
    lognormal lengths (median 2048, sigma 1.5) clipped to [128, total]; 32 q /
    8 kv heads, head_dim 128; one CA-task per document."""
    rng = np.random.default_rng(seed)
    lens = _lognormal_fill(rng, total, 2048.0, 1.5, 128, total)
    return _whole_document_tasks(f"llama8b_chunk_{total // 1024}k_h32x8_d128", lens, 32, 8, 128, seed)


def rebatched_pool(seed: int = 0, n_docs: int = 16, doc_lo: int = 8192, doc_hi: int = 131072,
                   shard_lo: int = 512, shard_hi: int = 8192, total_q: int = 131072,
                   hq: int = 32, hkv: int = 8, d: int = 128) -> Workload:
    """Rebatched CA-task pool: ``n_docs`` documents with lengths uniform in
    [doc_lo, doc_hi], each cut front to back into shards of length uniform in
    [shard_lo, shard_hi] (last shard = remainder); the shard list is shuffled
    and taken in order until exactly ``total_q`` query tokens (the last taken
    shard is truncated).  Each task is a shard with its document's KV prefix."""
    rng = np.random.default_rng(seed)
    doc_len = rng.integers(doc_lo, doc_hi, size=n_docs, endpoint=True).astype(np.int64)
    shards = []
    for i, L in enumerate(doc_len):
        pos = 0
        while pos < L:
            s = int(rng.integers(shard_lo, shard_hi, endpoint=True))
            s = min(s, int(L) - pos)
            shards.append((i, pos, s))
            pos += s
    order = rng.permutation(len(shards))
    taken = []
    acc = 0
    for k in order:
        if acc >= total_q:
            break
        doc, q0, ql = shards[k]
        ql = min(ql, total_q - acc)
        taken.append((doc, q0, ql))
        acc += ql
    if acc < total_q:
        raise ValueError("documents too short for the requested query total")
    t = np.asarray(taken, dtype=np.int64)
    return Workload(
        name=f"rebatched_pool_{total_q // 1024}k_h{hq}x{hkv}_d{d}",
        doc_len=doc_len,
        doc_kv_offset=_packed_offsets(doc_len),
        task_doc=t[:, 0].astype(np.int32),
        task_q_start=t[:, 1].copy(),
        task_q_len=t[:, 2].copy(),
        task_kv_start=np.zeros(len(t), dtype=np.int64),
        task_kv_len=(t[:, 1] + t[:, 2]).copy(),
        num_q_heads=hq, num_kv_heads=hkv, head_dim=d, seed=seed,
    )


def long_context_chunk(seed: int = 0, total: int = 524288, first: int = 262144,
                       hq: int = 64, hkv: int = 8, d: int = 128) -> Workload:
    """Long-context chunk: one ``first``-token document, then lognormal
    documents (median 8192, sigma 1.2) clipped to [128, total] until ``total``."""
    rng = np.random.default_rng(seed)
    lens = _lognormal_fill(rng, total, 8192.0, 1.2, 128, total, prefix=[first])
    return _whole_document_tasks(f"long_context_chunk_{total // 1024}k_h{hq}x{hkv}_d{d}", lens, hq, hkv, d, seed)


def split_kv_prefill(seed: int = 0, n_new: int = 4096, cached: int = 131072, n_blocks: int = 8,
                     hq: int = 128, hkv: int = 8, d: int = 128, split: bool = True) -> Workload:
    """Partial prefill: ``n_new`` query tokens at positions cached..cached+n_new-1
    of one document of cached+n_new tokens.  With ``split`` the KV is cut into
    ``n_blocks`` contiguous equal blocks, one task per block (each yields a
    partial (O, LSE)); otherwise one task sees the whole prefix."""
    L = cached + n_new
    if split:
        if L % n_blocks:
            raise ValueError("context length must split evenly")
        b = L // n_blocks
        kv_start = np.arange(n_blocks, dtype=np.int64) * b
        kv_len = np.full(n_blocks, b, dtype=np.int64)
    else:
        kv_start = np.zeros(1, dtype=np.int64)
        kv_len = np.full(1, L, dtype=np.int64)
    n = len(kv_start)
    return Workload(
        name=f"split_kv_prefill_{n_new}x{L}_{'b%d' % n_blocks if split else 'whole'}_h{hq}x{hkv}_d{d}",
        doc_len=np.asarray([L], dtype=np.int64),
        doc_kv_offset=np.zeros(1, dtype=np.int64),
        task_doc=np.zeros(n, dtype=np.int32),
        task_q_start=np.full(n, cached, dtype=np.int64),
        task_q_len=np.full(n, n_new, dtype=np.int64),
        task_kv_start=kv_start,
        task_kv_len=kv_len,
        num_q_heads=hq, num_kv_heads=hkv, head_dim=d, seed=seed,
    )


def custom(name: str, doc_len, tasks, hq: int, hkv: int, d: int, seed: int = 0,
           doc_kv_offset=None, masks=None) -> Workload:
    """Explicit documents and tasks.  ``tasks`` is a list of
    (doc, q_start, q_len, kv_start, kv_len); ``masks`` an optional list of
    (sink, lo, window) per task."""
    doc_len = np.asarray(doc_len, dtype=np.int64)
    t = np.asarray(tasks, dtype=np.int64).reshape(-1, 5)
    m = None if masks is None else np.asarray(masks, dtype=np.int64).reshape(-1, 3)
    return Workload(
        name=name,
        doc_len=doc_len,
        doc_kv_offset=(_packed_offsets(doc_len) if doc_kv_offset is None
                       else np.asarray(doc_kv_offset, dtype=np.int64)),
        task_doc=t[:, 0].astype(np.int32),
        task_q_start=t[:, 1].copy(),
        task_q_len=t[:, 2].copy(),
        task_kv_start=t[:, 3].copy(),
        task_kv_len=t[:, 4].copy(),
        num_q_heads=hq, num_kv_heads=hkv, head_dim=d, seed=seed,
        task_sink=None if m is None else m[:, 0].copy(),
        task_lo=None if m is None else m[:, 1].copy(),
        task_win=None if m is None else m[:, 2].copy(),
    )


# ---------------------------------------------------------------- sparse mask families

def lambda_chunk(seed: int = 0, total: int = 65536, sink: int = 64, window: int = 4096,
                 hq: int = 32, hkv: int = 8, d: int = 128) -> Workload:
    """The 64K lognormal chunk with a lambda-shaped mask on every document:
    an attention sink of ``sink`` tokens plus a sliding window of ``window``
    tokens ("DCP ...", §2.4, Figure 6b; window 4096 as in its Figure 14)."""
    w = llama8b_chunk(seed=seed, total=total)
    tasks = [(i, 0, int(L), 0, int(L)) for i, L in enumerate(w.doc_len)]
    masks = [(min(sink, int(L)), 0, min(window, int(L))) for L in w.doc_len]
    out = custom(f"lambda_chunk_{total // 1024}k_s{sink}_w{window}", w.doc_len, tasks, hq, hkv, d, seed, masks=masks)
    return out


def blockwise_chunk(seed: int = 0, total: int = 65536, block: int = 256, sink_blocks: int = 1,
                    window_blocks: int = 2, hq: int = 32, hkv: int = 8, d: int = 128) -> Workload:
    """The 64K lognormal chunk with a causal blockwise mask on every document
    ("DCP ...", §2.4, Figure 6c): blocks of ``block`` tokens (in-context
    examples); a token of a non-final block sees, causally, the first
    ``sink_blocks`` blocks and the last ``window_blocks`` blocks up to its
    own; the final block (the test example) sees everything before it.  One
    task per block."""
    w = llama8b_chunk(seed=seed, total=total)
    tasks, masks = [], []
    for i, L in enumerate(int(x) for x in w.doc_len):
        nb = -(-L // block)
        for b in range(nb):
            q0, q1 = b * block, min((b + 1) * block, L)
            tasks.append((i, q0, q1 - q0, 0, q1))
            if b == nb - 1:
                masks.append((0, 0, 0))
            else:
                masks.append((min(sink_blocks * block, L), max(0, b - window_blocks + 1) * block, 0))
    return custom(f"blockwise_chunk_{total // 1024}k_b{block}", w.doc_len, tasks, hq, hkv, d, seed, masks=masks)


def shared_question_pool(seed: int = 0, total: int = 65536, q_lo: int = 512, q_hi: int = 4096,
                         n_ans_lo: int = 2, n_ans_hi: int = 8, a_lo: int = 256, a_hi: int = 2048,
                         hq: int = 32, hkv: int = 8, d: int = 128) -> Workload:
    """Documents made of one question and several answers that share it
    ("DCP ...", §2.4, Figure 6d): the question is causal; answer i sees the
    whole question and itself causally, not the other answers.  Lengths
    uniform in the given ranges (numpy PCG64 from ``seed``), documents
    appended until ``total`` tokens (the last one truncated)."""
    rng = np.random.default_rng(seed)
    doc_len, tasks, masks = [], [], []
    used = 0
    while used < total:
        qn = int(rng.integers(q_lo, q_hi, endpoint=True))
        na = int(rng.integers(n_ans_lo, n_ans_hi, endpoint=True))
        ans = [int(x) for x in rng.integers(a_lo, a_hi, na, endpoint=True)]
        L = qn + sum(ans)
        if used + L > total:  # the last document: keep what fits, cut the answer that crosses
            room = total - used
            qn = min(qn, room)
            keep, acc = [], qn
            for a in ans:
                if acc >= room:
                    break
                keep.append(min(a, room - acc))
                acc += keep[-1]
            ans = keep
            L = qn + sum(ans)
        d_ = len(doc_len)
        doc_len.append(L)
        tasks.append((d_, 0, qn, 0, qn))
        masks.append((0, 0, 0))
        s = qn
        for a in ans:
            tasks.append((d_, s, a, 0, s + a))
            masks.append((qn, s, 0))
            s += a
        used += L
    return custom(f"shared_question_{total // 1024}k", doc_len, tasks, hq, hkv, d, seed, masks=masks)


def decode_batch(seed: int = 0, n_seq: int = 16, context: int = 131072, q_len: int = 1, jitter: int = 0,
                 hq: int = 32, hkv: int = 8, d: int = 128) -> Workload:
    """Decode / pass-Q shape (Context Parallelism for Scalable Million-Token
    Inference, §3.5.3-3.5.4: T new tokens per sequence, T = 1 for decode,
    against a long cached context P): ``n_seq`` documents of ``context``
    cached tokens (minus a uniform jitter in [0, jitter]) followed by
    ``q_len`` new tokens, one task per sequence with the prefix context."""
    rng = np.random.default_rng(seed)
    ctx = [context - int(rng.integers(0, jitter, endpoint=True)) if jitter else context for _ in range(n_seq)]
    doc_len = [c + q_len for c in ctx]
    tasks = [(i, c, q_len, 0, c + q_len) for i, c in enumerate(ctx)]
    return custom(f"decode_{n_seq}x{context}_t{q_len}_h{hq}x{hkv}_d{d}", doc_len, tasks, hq, hkv, d, seed)


WORKLOADS = {
    "tiny": tiny_chunk,
    "llama8b": llama8b_chunk,
    "pool": rebatched_pool,
    "long": long_context_chunk,
    "splitkv": split_kv_prefill,
}

MASKED_WORKLOADS = {
    "lambda": lambda_chunk,
    "blockwise": blockwise_chunk,
    "shared_question": shared_question_pool,
}


def make_tensors(w: Workload, device="cpu", need_grad_inputs: bool = True, chunk_rows: int = 1 << 16):
    """Draw Q, K, V (and dO) ~ N(0, 1) in float32 from seeded torch generators
    on ``device`` and round them to bf16 (round-to-nearest-even).  Stream k of
    the seed: Q = seed+1, K = seed+2, V = seed+3, dO = seed+4.  Large tensors
    are drawn in row chunks so the float32 temporary stays small."""
    import torch

    def draw(rows, heads, k):
        g = torch.Generator(device=device)
        g.manual_seed(w.seed * 16 + k)
        out = torch.empty((rows, heads, w.head_dim), dtype=torch.bfloat16, device=device)
        for r0 in range(0, rows, chunk_rows):
            r1 = min(rows, r0 + chunk_rows)
            out[r0:r1] = torch.randn((r1 - r0, heads, w.head_dim), generator=g,
                                     dtype=torch.float32, device=device).to(torch.bfloat16)
        return out

    q = draw(w.total_q, w.num_q_heads, 1)
    k = draw(w.total_kv, w.num_kv_heads, 2)
    v = draw(w.total_kv, w.num_kv_heads, 3)
    do = draw(w.total_q, w.num_q_heads, 4) if need_grad_inputs else None
    return q, k, v, do
