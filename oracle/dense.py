"""Whole-document fp64 oracle written with matrix products (test infrastructure).

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline
leg may import this module; it never imports the product.

It computes the same definitions as ``ca_oracle.c`` (core attention over
CA-tasks, forward and backward with recompute; Efficient Long-context Language
Model Training by Core Attention Disaggregation, §3.4 "The CA-Task
Abstraction", "Property 1: Statelessness" and §3.2 "Information flow (backward
pass)"), but for all rows of one document and one kv head at once, so that
full-size documents can be checked column by column:

  for each task t of the document, each block of its query rows, each query
  head h of kv head g (G = H_q / H_kv, contiguous groups):
      S    = scale * Q K^T                  over keys [kv_start, last visible + 1)
      S_pj = -inf where row p does not see key j (block, causal and sparse rules)
      LSE  = logsumexp_j S                   (natural log of the scaled scores)
      P    = exp(S - LSE),  O = P V,  D = rowsum(dO * O)
      dP   = dO V^T,  dS = P * (dP - D)
      dQ   = scale dS K,  dK += scale dS^T Q,  dV += P^T dO

Every product is a library matrix product in float64 (torch CPU); each row's
statistics use its full visible key set, and rows are taken in blocks only to
bound memory, so no row's arithmetic changes.  dK and dV sum over every task
of the document, every row block and every head of the group.  Rows with an
empty visible set get LSE = -inf, O = 0 and no gradient.  Inputs are the exact
bf16 values widened to float64.

Pins: ``tests/test_oracle_dense_pins.py`` (equal to ``ca_oracle.c`` on the
small edge and mask cases to 1e-10, and to torch float64 autograd).
"""
from __future__ import annotations

import os

import numpy as np
import torch


def _threads():
    n = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()
    torch.set_num_threads(max(1, int(n or 1)))


def _visible(p, j, kv_start, kv_len, sink, lo, win):
    """bool [len(p), len(j)]: row p sees key j (document positions)."""
    P = p[:, None]
    J = j[None, :]
    vis = (J >= kv_start) & (J < kv_start + kv_len) & (J <= P)
    if sink or lo or win:
        allow = (J < sink) | ((J >= lo) & ((win == 0) | (J >= P - win + 1)))
        vis &= allow
    return vis


class DocResult:
    """Results for one (document, kv head): per-task row ranges of O, LSE, dQ
    ([rows, G, d] / [rows, G]) and dK, dV of the document's keys [L, d] (or of
    the requested columns only)."""

    def __init__(self):
        self.rows = []      # (packed row 0, n rows) per task, in task order
        self.o = []         # [n, G, d] per task
        self.lse = []       # [n, G]
        self.dq = []        # [n, G, d]
        self.dk = None
        self.dv = None


def document_group(w, q, k, v, do, doc: int, g: int, columns=None, want_dq=True, block=None) -> DocResult:
    """O, LSE, dQ of every row of every task of document ``doc`` for the query
    heads of kv head ``g``, and dK, dV of the document's keys of head ``g``.

    q, k, v, do: torch bf16 CPU tensors in the library's layouts.  With
    ``columns`` (document positions), dK/dV are computed only at those columns
    and dQ is skipped; since key j is seen only by rows p >= j, rows before
    the first column are skipped too (their O and LSE are left NaN).  The LSE
    and O of every row that is computed still come from all its visible keys.
    """
    _threads()
    hq, hkv, d = w.num_q_heads, w.num_kv_heads, w.head_dim
    G = hq // hkv
    scale = float(w.softmax_scale)
    L = int(w.doc_len[doc])
    off = int(w.doc_kv_offset[doc])
    K = k[off:off + L, g].to(torch.float64)
    V = v[off:off + L, g].to(torch.float64)
    row0 = w.task_row_offset()
    sink_a, lo_a, win_a = w.masks()
    res = DocResult()
    cols = None
    if columns is not None:
        cols = torch.as_tensor(np.asarray(columns, dtype=np.int64))
        if len(torch.unique(cols)) != len(cols) or (len(cols) and (int(cols.min()) < 0 or int(cols.max()) >= L)):
            raise ValueError("columns must be distinct positions inside the document")
        res.dk = torch.zeros((len(cols), d), dtype=torch.float64)
        res.dv = torch.zeros((len(cols), d), dtype=torch.float64)
        want_dq = False
    else:
        res.dk = torch.zeros((L, d), dtype=torch.float64)
        res.dv = torch.zeros((L, d), dtype=torch.float64)
    for t in range(w.n_tasks):
        if int(w.task_doc[t]) != doc:
            continue
        qs, ql = int(w.task_q_start[t]), int(w.task_q_len[t])
        ks, kl = int(w.task_kv_start[t]), int(w.task_kv_len[t])
        sink, lo, win = int(sink_a[t]), int(lo_a[t]), int(win_a[t])
        r0 = int(row0[t])
        o_t = torch.zeros((ql, G, d), dtype=torch.float64)
        lse_t = torch.full((ql, G), -np.inf, dtype=torch.float64)
        dq_t = torch.zeros((ql, G, d), dtype=torch.float64) if want_dq else None
        nb_max = block or max(64, min(1024, int(2 ** 25 // max(1, min(L, qs + ql)))))
        b0 = 0
        if cols is not None:
            if len(cols) == 0:
                continue
            b0 = max(0, int(cols.min()) - qs) // nb_max * nb_max
            o_t[:b0] = np.nan
            lse_t[:b0] = np.nan
        for b in range(b0, ql, nb_max):
            nb = min(nb_max, ql - b)
            p = torch.arange(qs + b, qs + b + nb, dtype=torch.int64)
            kend = min(ks + kl, qs + b + nb)  # one past the last key any row of the block may see
            if kend <= ks:
                continue
            j = torch.arange(ks, kend, dtype=torch.int64)
            hidden = ~_visible(p, j, ks, kl, sink, lo, win)
            Kb, Vb = K[ks:kend], V[ks:kend]
            if cols is not None:
                csel = (cols >= ks) & (cols < kend)
                cidx = torch.nonzero(csel).flatten()
                cj = cols[cidx] - ks
            for hh in range(G):
                h = g * G + hh
                Q = q[r0 + b:r0 + b + nb, h].to(torch.float64)
                S = scale * (Q @ Kb.T)
                S.masked_fill_(hidden, -np.inf)
                lse = torch.logsumexp(S, dim=1)
                # P = exp(S - LSE); hidden keys give exp(-inf) = 0, and a row
                # with no visible key (LSE = -inf) is taken against 0 so that
                # its P stays 0
                P = S.sub_(torch.where(torch.isinf(lse), torch.zeros_like(lse), lse)[:, None]).exp_()
                O = P @ Vb
                o_t[b:b + nb, hh] = O
                lse_t[b:b + nb, hh] = lse
                if do is None:
                    continue
                dO = do[r0 + b:r0 + b + nb, h].to(torch.float64)
                D = (dO * O).sum(dim=1)
                if cols is None:
                    dS = (dO @ Vb.T).sub_(D[:, None]).mul_(P)  # P * (dP - D)
                    if want_dq:
                        dq_t[b:b + nb, hh] = scale * (dS @ Kb)
                    res.dk[ks:kend] += scale * (dS.T @ Q)
                    res.dv[ks:kend] += P.T @ dO
                elif len(cidx):
                    Pc = P[:, cj]
                    dSc = (dO @ Vb[cj].T).sub_(D[:, None]).mul_(Pc)
                    res.dk[cidx] += scale * (dSc.T @ Q)
                    res.dv[cidx] += Pc.T @ dO
        res.rows.append((r0, ql))
        res.o.append(o_t)
        res.lse.append(lse_t)
        res.dq.append(dq_t)
    return res


def full(w, q, k, v, do=None):
    """O [total_q, hq, d], LSE [total_q, hq], dQ, dK [total_kv, hkv, d], dV of a
    whole workload (float64 numpy), assembled from document_group over every
    document and kv head.  Key rows outside every document stay 0."""
    hq, hkv, d = w.num_q_heads, w.num_kv_heads, w.head_dim
    G = hq // hkv
    O = np.zeros((w.total_q, hq, d))
    LSE = np.full((w.total_q, hq), -np.inf)
    dQ = np.zeros((w.total_q, hq, d))
    dK = np.zeros((w.total_kv, hkv, d))
    dV = np.zeros((w.total_kv, hkv, d))
    for doc in range(w.n_docs):
        off, L = int(w.doc_kv_offset[doc]), int(w.doc_len[doc])
        for g in range(hkv):
            r = document_group(w, q, k, v, do, doc, g, want_dq=do is not None)
            for (r0, n), o, lse, dq in zip(r.rows, r.o, r.lse, r.dq):
                O[r0:r0 + n, g * G:(g + 1) * G] = o.numpy()
                LSE[r0:r0 + n, g * G:(g + 1) * G] = lse.numpy()
                if dq is not None:
                    dQ[r0:r0 + n, g * G:(g + 1) * G] = dq.numpy()
            if do is not None:
                dK[off:off + L, g] = r.dk.numpy()
                dV[off:off + L, g] = r.dv.numpy()
    return O, LSE, dQ, dK, dV
