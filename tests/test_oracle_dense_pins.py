"""Pins of the whole-document oracle form (oracle/dense.py), CPU only.

It is checked against two things outside itself: the row-by-row C oracle
(ca_oracle.c, itself pinned by brute force, autograd, finite differences and
closed forms in test_oracle_pins.py), on the small edge cases that span several
tiles, sharded documents, KV blocks with empty rows, gaps in the KV buffer and
every sparse mask family; and torch float64 autograd of the masked softmax.
Its column mode must equal its full mode at the chosen columns.
"""
import numpy as np
import pytest
import torch

import oracle
from oracle import dense
import workloads as W
from cases import EDGE

MASKED = [
    W.lambda_chunk(seed=1, total=700, sink=70, window=150, hq=4, hkv=2, d=64),
    W.blockwise_chunk(seed=3, total=800, block=96, sink_blocks=2, window_blocks=3, hq=4, hkv=1, d=64),
    W.shared_question_pool(seed=4, total=900, q_lo=100, q_hi=200, a_lo=40, a_hi=150, hq=4, hkv=1, d=64),
    W.custom("mixed_masks", [300, 200], [(0, 0, 300, 0, 300), (1, 40, 120, 20, 160), (0, 120, 80, 0, 250)],
             4, 2, 64, seed=6, masks=[(10, 0, 90), (0, 100, 0), (30, 150, 41)]),
]

CASES = EDGE + MASKED


def c_oracle(w, q, k, v, do):
    pb = oracle.Problem(w, q, k, v, do)
    O, LSE = oracle.forward(pb)
    dQ, dK, dV = oracle.backward(pb)
    return O, LSE, dQ, dK, dV


def close(a, b, tol=1e-10):
    scale = max(1.0, float(np.abs(b).max()) if b.size else 1.0)
    return float(np.abs(a - b).max()) <= tol * scale if b.size else True


@pytest.mark.parametrize("w", CASES, ids=lambda w: w.name)
def test_dense_equals_row_oracle(w):
    q, k, v, do = W.make_tensors(w, device="cpu")
    O, LSE, dQ, dK, dV = dense.full(w, q, k, v, do)
    Oc, LSEc, dQc, dKc, dVc = c_oracle(w, q, k, v, do)
    fin = np.isfinite(LSEc)
    assert np.array_equal(np.isfinite(LSE), fin)
    assert np.all(LSE[~fin] == -np.inf)
    assert close(LSE[fin], LSEc[fin])
    assert close(O, Oc)
    assert close(dQ, dQc)
    assert close(dK, dKc)
    assert close(dV, dVc)


@pytest.mark.parametrize("w", [EDGE[1], EDGE[3], MASKED[0]], ids=lambda w: w.name)
def test_dense_columns_equal_full(w):
    q, k, v, do = W.make_tensors(w, device="cpu")
    rng = np.random.default_rng(11)
    for doc in range(w.n_docs):
        L = int(w.doc_len[doc])
        for g in range(w.num_kv_heads):
            whole = dense.document_group(w, q, k, v, do, doc, g)
            for cols in (np.unique(np.concatenate([[0, L - 1], rng.integers(0, L, 7)])),
                         np.unique(rng.integers(L // 2, L, 5))):  # late columns: early rows skipped
                part = dense.document_group(w, q, k, v, do, doc, g, columns=cols, block=64)
                assert torch.allclose(part.dk, whole.dk[cols], rtol=0, atol=1e-12)
                assert torch.allclose(part.dv, whole.dv[cols], rtol=0, atol=1e-12)
            for a, b in zip(part.lse, whole.lse):  # rows the column mode computed
                done = ~torch.isnan(a)
                assert torch.allclose(a[done], b[done], rtol=0, atol=1e-12)


def test_dense_equals_torch_autograd():
    """torch float64 autograd of sum(O * dO) over the masked softmax, written
    with plain torch ops (no blocking), on sharded tasks, KV blocks with an
    empty row and a sparse mask."""
    w = W.custom("autograd", [90, 40], [(0, 0, 30, 0, 30), (0, 30, 60, 0, 90), (1, 5, 35, 12, 20),
                                       (0, 60, 30, 0, 90)], 4, 2, 16, seed=9,
                 masks=[(0, 0, 0), (0, 0, 0), (0, 0, 0), (5, 0, 17)])
    q, k, v, do = W.make_tensors(w, device="cpu")
    O, LSE, dQ, dK, dV = dense.full(w, q, k, v, do)
    hq, hkv = w.num_q_heads, w.num_kv_heads
    G = hq // hkv
    Q = q.to(torch.float64).requires_grad_(True)
    K = k.to(torch.float64).requires_grad_(True)
    V = v.to(torch.float64).requires_grad_(True)
    row0 = w.task_row_offset()
    sink, lo, win = w.masks()
    loss = torch.zeros((), dtype=torch.float64)
    for t in range(w.n_tasks):
        doc = int(w.task_doc[t])
        off, L = int(w.doc_kv_offset[doc]), int(w.doc_len[doc])
        r0, ql = int(row0[t]), int(w.task_q_len[t])
        p = int(w.task_q_start[t]) + torch.arange(ql)[:, None]
        j = torch.arange(L)[None, :]
        ks, kl = int(w.task_kv_start[t]), int(w.task_kv_len[t])
        vis = (j >= ks) & (j < ks + kl) & (j <= p)
        if sink[t] or lo[t] or win[t]:
            vis &= (j < int(sink[t])) | ((j >= int(lo[t])) & ((int(win[t]) == 0) | (j >= p - int(win[t]) + 1)))
        live = vis.any(1)
        rows = torch.arange(r0, r0 + ql)[live]
        for h in range(hq):
            S = w.softmax_scale * Q[rows, h] @ K[off:off + L, h // G].T
            P = torch.softmax(S.masked_fill(~vis[live], float("-inf")), dim=1)
            loss = loss + ((P @ V[off:off + L, h // G]) * do[rows, h].to(torch.float64)).sum()
    loss.backward()
    assert close(dQ, Q.grad.numpy())
    assert close(dK, K.grad.numpy())
    assert close(dV, V.grad.numpy())
