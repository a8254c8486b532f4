"""Pins of the oracle's sparse masks (CPU only), each against a route that
does not use the (sink, lo, window) encoding or the oracle's own loops:

  * numpy brute force and torch fp64 autograd with the visible sets built
    from each family's own description ("DCP: Addressing Input Dynamism In
    Long-Context Training via Dynamic Context Parallelism", §2.4, Figure 6):
    lambda = sink tokens plus a sliding window, causal blockwise = block ids,
    shared question = question / answer segment ids;
  * closed forms: a window covering the document is the plain causal rule; a
    window of 1 gives O_p = v_p and LSE_p = s_pp;
  * Eq. 4 of the million-token paper's Appendix B: a window-free mask is the
    union of two plain KV blocks, so the masked rows equal the LSE merge of
    the two blocks' partial results;
  * shared-question answer rows equal plain causal attention over a document
    made of the question followed by that one answer.
"""
import numpy as np
import pytest
import scipy.special
import torch

import oracle
import workloads as W


def f64(x):
    return x.to(torch.float64).numpy()


def family_visibility(kind, w, t, L):
    """[q_len, L] boolean visible set of task t from the family's own
    description (block ids, segment ids, sink + window)."""
    q0, ql = int(w.task_q_start[t]), int(w.task_q_len[t])
    p = q0 + np.arange(ql)[:, None]
    j = np.arange(L)[None, :]
    causal = (j <= p) & (j >= int(w.task_kv_start[t])) & (j < int(w.task_kv_start[t] + w.task_kv_len[t]))
    if kind == "plain":
        return causal
    if kind == "lambda":
        sink, window = w.params
        return causal & ((j < sink) | (p - j < window))
    if kind == "blockwise":
        B, sb, wb = w.params
        nb = -(-L // B)
        bp, bj = p // B, j // B
        return causal & ((bp == nb - 1) | (bj < sb) | (bp - bj < wb))
    if kind == "shared":
        seg = w.segments[int(w.task_doc[t])]  # segment id per position: 0 = question, i = answer i
        sp, sj = seg[p], seg[j]
        return causal & ((sj == 0) | (sj == sp))
    raise ValueError(kind)


def small_cases():
    lam = W.lambda_chunk(seed=3, total=400, sink=5, window=37, hq=4, hkv=2, d=16)
    lam.kind, lam.params = "lambda", (5, 37)
    blk = W.blockwise_chunk(seed=4, total=420, block=32, sink_blocks=1, window_blocks=2, hq=4, hkv=1, d=16)
    blk.kind, blk.params = "blockwise", (32, 1, 2)
    sq = W.shared_question_pool(seed=5, total=360, q_lo=20, q_hi=60, n_ans_lo=2, n_ans_hi=4, a_lo=10, a_hi=50,
                                hq=4, hkv=2, d=16)
    sq.kind = "shared"
    sq.segments = {}
    for d_ in range(sq.n_docs):
        L = int(sq.doc_len[d_])
        seg = np.zeros(L, dtype=np.int64)
        ts = [t for t in range(sq.n_tasks) if int(sq.task_doc[t]) == d_]
        for i, t in enumerate(ts):
            seg[int(sq.task_q_start[t]):int(sq.task_q_start[t] + sq.task_q_len[t])] = i
        sq.segments[d_] = seg
    return [lam, blk, sq]


CASES = small_cases()


def brute(w, q, k, v, do):
    """O, LSE by numpy; dQ, dK, dV by torch autograd; both with the family
    visibility."""
    hq, d = w.num_q_heads, w.head_dim
    G = hq // w.num_kv_heads
    row0 = w.task_row_offset()
    O = np.zeros((w.total_q, hq, d))
    LSE = np.zeros((w.total_q, hq))
    Q = q.to(torch.float64).requires_grad_(True)
    K = k.to(torch.float64).requires_grad_(True)
    V = v.to(torch.float64).requires_grad_(True)
    loss = torch.zeros((), dtype=torch.float64)
    for t in range(w.n_tasks):
        doc = int(w.task_doc[t])
        off, L = int(w.doc_kv_offset[doc]), int(w.doc_len[doc])
        r0, ql = int(row0[t]), int(w.task_q_len[t])
        vis = family_visibility(w.kind, w, t, L)
        live = vis.any(1)
        for h in range(hq):
            S = w.softmax_scale * f64(q[r0:r0 + ql, h]) @ f64(k[off:off + L, h // G]).T
            S = np.where(vis, S, -np.inf)
            with np.errstate(divide="ignore", invalid="ignore"):
                lse = scipy.special.logsumexp(S, axis=1)
                P = np.where(vis, np.exp(S - lse[:, None]), 0.0)
            O[r0:r0 + ql, h] = P @ f64(v[off:off + L, h // G])
            LSE[r0:r0 + ql, h] = np.where(live, lse, -np.inf)
            rows = torch.arange(r0, r0 + ql)[torch.as_tensor(live)]
            St = w.softmax_scale * Q[rows, h] @ K[off:off + L, h // G].T
            St = St.masked_fill(~torch.as_tensor(vis[live]), float("-inf"))
            Ot = torch.softmax(St, dim=1) @ V[off:off + L, h // G]
            loss = loss + (Ot * do[rows, h].to(torch.float64)).sum()
    loss.backward()
    return O, LSE, Q.grad.numpy(), K.grad.numpy(), V.grad.numpy()


@pytest.mark.parametrize("w", CASES, ids=lambda w: w.kind)
def test_masked_oracle_matches_family_brute_force(w):
    q, k, v, do = W.make_tensors(w, device="cpu")
    O, LSE, dQ, dK, dV = brute(w, q, k, v, do)
    pb = oracle.Problem(w, q, k, v, do)
    Oo, Lo = oracle.forward(pb)
    assert np.allclose(Oo, O, rtol=0, atol=1e-12)
    assert np.array_equal(np.isinf(Lo), np.isinf(LSE))
    fin = np.isfinite(LSE)
    assert np.allclose(Lo[fin], LSE[fin], rtol=0, atol=1e-12)
    dq, dk, dv = oracle.backward(pb)
    assert np.allclose(dq, dQ, rtol=0, atol=1e-10)
    assert np.allclose(dk, dK, rtol=0, atol=1e-10)
    assert np.allclose(dv, dV, rtol=0, atol=1e-10)


@pytest.mark.parametrize("w", CASES, ids=lambda w: w.kind)
def test_masked_pair_counts_match_family_enumeration(w):
    ref = []
    for t in range(w.n_tasks):
        L = int(w.doc_len[int(w.task_doc[t])])
        ref.append(int(family_visibility(w.kind, w, t, L).sum()))
    assert np.array_equal(oracle.task_pairs(w), np.asarray(ref))


def test_window_covering_the_document_is_causal():
    docs = [40, 23]
    tasks = [(0, 0, 40, 0, 40), (1, 5, 18, 0, 23)]
    plain = W.custom("plain", docs, tasks, hq=2, hkv=1, d=8, seed=11)
    wide = W.custom("wide", docs, tasks, hq=2, hkv=1, d=8, seed=11, masks=[(0, 0, 40), (3, 0, 23)])
    q, k, v, do = W.make_tensors(plain, device="cpu")
    Op, Lp = oracle.forward(oracle.Problem(plain, q, k, v))
    Ow, Lw = oracle.forward(oracle.Problem(wide, q, k, v))
    assert np.array_equal(Op, Ow) and np.array_equal(Lp, Lw)
    assert np.array_equal(oracle.task_pairs(plain), oracle.task_pairs(wide))


def test_window_of_one_returns_own_value():
    L = 30
    w = W.custom("self", [L], [(0, 0, L, 0, L)], hq=2, hkv=1, d=8, seed=12, masks=[(0, 0, 1)])
    q, k, v, _ = W.make_tensors(w, device="cpu")
    O, LSE = oracle.forward(oracle.Problem(w, q, k, v))
    for h in range(2):
        assert np.array_equal(O[:, h], f64(v[:, 0]))
        s = w.softmax_scale * (f64(q[:, h]) * f64(k[:, 0])).sum(1)
        assert np.allclose(LSE[:, h], s, rtol=0, atol=1e-12)
    assert oracle.task_pairs(w)[0] == L


@pytest.mark.parametrize("sink,lo", [(8, 20), (12, 12), (0, 25), (16, 5)])
def test_window_free_mask_is_the_merge_of_two_kv_blocks(sink, lo):
    """[0, sink) U [lo, p]: the plain blocks [0, sink) and [max(sink, lo), L)
    merged by Eq. 4 give the masked rows."""
    L, q0 = 48, 28
    nq = L - q0
    masked = W.custom("masked", [L], [(0, q0, nq, 0, L)], hq=2, hkv=1, d=8, seed=13, masks=[(sink, lo, 0)])
    a = max(sink, lo)
    parts = [(0, q0, nq, a, L - a)] + ([(0, q0, nq, 0, sink)] if sink > 0 else [])
    split = W.custom("split", [L], parts, hq=2, hkv=1, d=8, seed=13)
    q, k, v, _ = W.make_tensors(masked, device="cpu")
    Om, Lm = oracle.forward(oracle.Problem(masked, q, k, v))
    n = len(parts)
    Os, Ls = oracle.forward(oracle.Problem(split, q.repeat(n, 1, 1), k, v))
    Og, Lg = oracle.merge(Os.reshape(n, nq * 2, 8), Ls.reshape(n, nq * 2))
    assert np.allclose(Og, Om.reshape(nq * 2, 8), rtol=0, atol=1e-12)
    assert np.allclose(Lg, Lm.reshape(-1), rtol=0, atol=1e-12)


def test_shared_question_answer_equals_question_plus_answer_document():
    qn, answers = 17, [9, 14, 6]
    L = qn + sum(answers)
    tasks, masks, s = [(0, 0, qn, 0, qn)], [(0, 0, 0)], qn
    for a in answers:
        tasks.append((0, s, a, 0, s + a))
        masks.append((qn, s, 0))
        s += a
    shared = W.custom("shared", [L], tasks, hq=4, hkv=2, d=8, seed=14, masks=masks)
    q, k, v, do = W.make_tensors(shared, device="cpu")
    pb = oracle.Problem(shared, q, k, v, do)
    O, LSE = oracle.forward(pb)
    dQ, _, _ = oracle.backward(pb)
    s = qn
    for a in answers:
        # a plain document: the question's tokens followed by this answer's tokens
        idx = np.concatenate([np.arange(qn), np.arange(s, s + a)])
        one = W.custom("one", [qn + a], [(0, qn, a, 0, qn + a)], hq=4, hkv=2, d=8, seed=14)
        po = oracle.Problem(one, q[s:s + a], k[idx], v[idx], do[s:s + a])
        O1, L1 = oracle.forward(po)
        dq1, _, _ = oracle.backward(po)
        assert np.allclose(O1, O[s:s + a], rtol=0, atol=1e-12)
        assert np.allclose(L1, LSE[s:s + a], rtol=0, atol=1e-12)
        assert np.allclose(dq1, dQ[s:s + a], rtol=0, atol=1e-11)
        s += a
