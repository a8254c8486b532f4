"""Pins of the fp64 oracle against facts fixed outside it (CPU only).

Each test checks the oracle against something other than itself: numpy brute
force of the full masked score matrix with scipy's logsumexp, torch fp64
autograd, central finite differences, closed forms (Q = 0, constant V, first
token of a document, pair counts l(l+1)/2), the imbalance ratios the pages
print, composability of shards, and the LSE-merge identity.
"""
import math
import os

import numpy as np
import pytest
import scipy.special
import torch

import oracle
import workloads as W

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def f64(x):
    return x.to(torch.float64).numpy()


def inputs(w, zero_q=False, const_v=None):
    q, k, v, do = W.make_tensors(w, device="cpu")
    if zero_q:
        q.zero_()
    if const_v is not None:
        v.copy_(const_v.to(torch.bfloat16).expand_as(v))
    return q, k, v, do


def brute_scores(w, q, k, t, h):
    """Masked scaled scores of task t, head h: rows = task rows, cols = all
    keys of the task's document; -inf where the key is not visible."""
    G = w.num_q_heads // w.num_kv_heads
    g = h // G
    doc = int(w.task_doc[t])
    L = int(w.doc_len[doc])
    off = int(w.doc_kv_offset[doc])
    r0 = int(w.task_row_offset()[t])
    ql = int(w.task_q_len[t])
    Q = f64(q[r0:r0 + ql, h])
    K = f64(k[off:off + L, g])
    S = w.softmax_scale * Q @ K.T
    p = int(w.task_q_start[t]) + np.arange(ql)[:, None]
    j = np.arange(L)[None, :]
    ks, kl = int(w.task_kv_start[t]), int(w.task_kv_len[t])
    vis = (j >= ks) & (j < ks + kl) & (j <= p)
    return np.where(vis, S, -np.inf), vis


def brute_forward(w, q, k, v):
    hq, d = w.num_q_heads, w.head_dim
    G = hq // w.num_kv_heads
    O = np.zeros((w.total_q, hq, d))
    LSE = np.zeros((w.total_q, hq))
    row0 = w.task_row_offset()
    for t in range(w.n_tasks):
        doc = int(w.task_doc[t])
        off, L = int(w.doc_kv_offset[doc]), int(w.doc_len[doc])
        r0, ql = int(row0[t]), int(w.task_q_len[t])
        for h in range(hq):
            S, vis = brute_scores(w, q, k, t, h)
            with np.errstate(divide="ignore", invalid="ignore"):
                lse = scipy.special.logsumexp(S, axis=1)
                P = np.where(vis, np.exp(S - lse[:, None]), 0.0)
            O[r0:r0 + ql, h] = P @ f64(v[off:off + L, h // G])
            LSE[r0:r0 + ql, h] = lse
    return O, LSE


def torch_autograd(w, q, k, v, do):
    """dQ, dK, dV of sum(O * dO) by torch fp64 autograd over the masked
    softmax written with torch ops."""
    hq, hkv = w.num_q_heads, w.num_kv_heads
    G = hq // hkv
    Q = q.to(torch.float64).requires_grad_(True)
    K = k.to(torch.float64).requires_grad_(True)
    V = v.to(torch.float64).requires_grad_(True)
    row0 = w.task_row_offset()
    loss = torch.zeros((), dtype=torch.float64)
    for t in range(w.n_tasks):
        doc = int(w.task_doc[t])
        off, L = int(w.doc_kv_offset[doc]), int(w.doc_len[doc])
        r0, ql = int(row0[t]), int(w.task_q_len[t])
        p = int(w.task_q_start[t]) + torch.arange(ql)[:, None]
        j = torch.arange(L)[None, :]
        ks, kl = int(w.task_kv_start[t]), int(w.task_kv_len[t])
        vis = (j >= ks) & (j < ks + kl) & (j <= p)
        live = vis.any(1)  # rows with an empty visible set have O = 0 and no gradient
        rows = torch.arange(r0, r0 + ql)[live]
        for h in range(hq):
            S = w.softmax_scale * Q[rows, h] @ K[off:off + L, h // G].T
            S = S.masked_fill(~vis[live], float("-inf"))
            P = torch.softmax(S, dim=1)
            O = P @ V[off:off + L, h // G]
            loss = loss + (O * do[rows, h].to(torch.float64)).sum()
    loss.backward()
    return Q.grad.numpy(), K.grad.numpy(), V.grad.numpy()


SMALL = [
    # two documents, one split into three shards, GQA 2
    W.custom("two_docs_sharded", [37, 20], [(0, 0, 10, 0, 10), (0, 10, 15, 0, 25), (0, 25, 12, 0, 37),
                                           (1, 0, 20, 0, 20)], hq=4, hkv=2, d=16, seed=3),
    # KV blocks that start inside the document, including a row with an empty visible set
    W.custom("kv_blocks", [24], [(0, 16, 8, 0, 8), (0, 16, 8, 8, 8), (0, 16, 8, 16, 8), (0, 2, 3, 8, 8)],
             hq=2, hkv=1, d=8, seed=5),
    # G = 4, tasks out of document order, a gap in the KV buffer between documents
    W.custom("unordered_gap", [9, 13], [(1, 4, 9, 0, 13), (0, 0, 9, 0, 9)], hq=4, hkv=1, d=32, seed=7,
             doc_kv_offset=[20, 2]),
]


@pytest.mark.parametrize("w", SMALL, ids=lambda w: w.name)
def test_forward_matches_brute_force(w):
    q, k, v, _ = inputs(w)
    pb = oracle.Problem(w, q, k, v)
    O, LSE = oracle.forward(pb)
    Ob, LSEb = brute_forward(w, q, k, v)
    assert np.allclose(O, Ob, rtol=0, atol=1e-12)
    fin = np.isfinite(LSEb)
    assert np.array_equal(fin, np.isfinite(LSE))
    assert np.all(LSE[~fin] == -np.inf)
    assert np.allclose(LSE[fin], LSEb[fin], rtol=0, atol=1e-12)


@pytest.mark.parametrize("w", SMALL, ids=lambda w: w.name)
def test_forward_rows_equal_full(w):
    q, k, v, _ = inputs(w)
    pb = oracle.Problem(w, q, k, v)
    O, LSE = oracle.forward(pb)
    rng = np.random.default_rng(0)
    rows = rng.integers(0, w.total_q, 30)
    heads = rng.integers(0, w.num_q_heads, 30)
    o, l = oracle.forward_rows(pb, rows, heads)
    assert np.array_equal(o, O[rows, heads])
    assert np.array_equal(l, LSE[rows, heads])


@pytest.mark.parametrize("w", SMALL, ids=lambda w: w.name)
def test_backward_matches_torch_autograd(w):
    q, k, v, do = inputs(w)
    pb = oracle.Problem(w, q, k, v, do)
    dq, dk, dv = oracle.backward(pb)
    tq, tk, tv = torch_autograd(w, q, k, v, do)
    for a, b in ((dq, tq), (dk, tk), (dv, tv)):
        assert np.allclose(a, b, rtol=0, atol=1e-11), np.abs(a - b).max()


def test_backward_central_differences():
    """dL/dx for L = sum(O . dO) by central differences.  The probed inputs
    are set to 0 so x +- 2^-20 are exact bf16 values."""
    w = W.custom("fd", [12, 7], [(0, 0, 12, 0, 12), (1, 2, 5, 1, 6)], hq=2, hkv=1, d=8, seed=11)
    q, k, v, do = inputs(w)
    probes = [("q", 3, 1, 2), ("q", 14, 0, 5), ("k", 4, 0, 1), ("k", 13, 0, 7), ("v", 0, 0, 3), ("v", 15, 0, 0)]
    T = {"q": q, "k": k, "v": v}
    for name, r, h, c in probes:
        T[name][r, h, c] = 0.0
    pb = oracle.Problem(w, q, k, v, do)
    dq, dk, dv = oracle.backward(pb)
    G = {"q": dq, "k": dk, "v": dv}
    eps = 2.0 ** -20
    dof = f64(do)

    def loss():
        O, _ = oracle.forward(oracle.Problem(w, q, k, v))
        return float((O * dof).sum())

    for name, r, h, c in probes:
        T[name][r, h, c] = eps
        lp = loss()
        T[name][r, h, c] = -eps
        lm = loss()
        T[name][r, h, c] = 0.0
        fd = (lp - lm) / (2 * eps)
        an = G[name][r, h, c]
        assert abs(fd - an) <= 1e-6 * max(1.0, abs(an)), (name, r, h, c, fd, an)


def test_q_zero_closed_forms():
    """Q = 0: every visible key has score 0, so O_p is the mean of the visible
    v_j, LSE_p = ln |V(p)|, and dV_j = sum over (p, h) seeing j of dO_p / |V(p)|."""
    w = SMALL[0]
    q, k, v, do = inputs(w, zero_q=True)
    pb = oracle.Problem(w, q, k, v, do)
    O, LSE = oracle.forward(pb)
    dq, dk, dv = oracle.backward(pb)
    G = w.num_q_heads // w.num_kv_heads
    row0 = w.task_row_offset()
    vv, dof = f64(v), f64(do)
    dv_ref = np.zeros_like(dv)
    for t in range(w.n_tasks):
        off = int(w.doc_kv_offset[w.task_doc[t]])
        for i in range(int(w.task_q_len[t])):
            p = int(w.task_q_start[t]) + i
            ks = int(w.task_kv_start[t])
            hi = min(ks + int(w.task_kv_len[t]), p + 1)
            n = hi - ks
            for h in range(w.num_q_heads):
                r = int(row0[t]) + i
                assert LSE[r, h] == pytest.approx(math.log(n), abs=1e-13)
                assert np.allclose(O[r, h], vv[off + ks:off + hi, h // G].mean(0), atol=1e-13)
                dv_ref[off + ks:off + hi, h // G] += dof[r, h] / n
    assert np.allclose(dv, dv_ref, atol=1e-12)


def test_constant_v_and_first_token():
    w = SMALL[0]
    c = torch.linspace(-2, 2, w.head_dim)
    q, k, v, _ = inputs(w, const_v=c)
    O, _ = oracle.forward(oracle.Problem(w, q, k, v))
    assert np.allclose(O, f64(c.to(torch.bfloat16))[None, None, :], atol=1e-13)
    # first token of a document with kv_start = 0 sees only itself: O = v_0, LSE = s_00
    q, k, v, _ = inputs(w)
    O, LSE = oracle.forward(oracle.Problem(w, q, k, v))
    G = w.num_q_heads // w.num_kv_heads
    row0 = w.task_row_offset()
    for t in range(w.n_tasks):
        if int(w.task_q_start[t]) != 0:
            continue
        r = int(row0[t])
        off = int(w.doc_kv_offset[w.task_doc[t]])
        for h in range(w.num_q_heads):
            assert np.array_equal(O[r, h], f64(v[off, h // G]))
            s = w.softmax_scale * float(f64(q[r, h]) @ f64(k[off, h // G]))
            assert LSE[r, h] == pytest.approx(s, abs=1e-13)


def test_rows_sum_to_one_via_constant_value_column():
    """Softmax rows sum to 1: with v = e_c in one channel, O[:, :, c] = 1."""
    w = SMALL[1]
    q, k, v, _ = inputs(w)
    v.zero_()
    v[..., 3] = 1.0
    O, LSE = oracle.forward(oracle.Problem(w, q, k, v))
    fin = np.isfinite(LSE)
    assert np.allclose(O[..., 3][fin], 1.0, atol=1e-14)
    assert np.all(O[..., 3][~fin] == 0.0)


def test_composability_sharded_equals_unsharded():
    """A document's CA is the union of the outputs of tasks whose query shards
    partition it; dK/dV are the sums over the shards."""
    whole = W.custom("whole", [50, 31], [(0, 0, 50, 0, 50), (1, 0, 31, 0, 31)], hq=4, hkv=2, d=16, seed=2)
    shards = [(1, 20, 11, 0, 31), (0, 0, 7, 0, 7), (0, 33, 17, 0, 50), (1, 0, 20, 0, 20), (0, 7, 26, 0, 33)]
    sharded = W.custom("sharded", [50, 31], shards, hq=4, hkv=2, d=16, seed=2)
    q, k, v, do = inputs(whole)
    # the same token's row in the sharded packing
    rows = []
    for (doc, q0, ql, _, _) in shards:
        base = 0 if doc == 0 else 50
        rows.extend(range(base + q0, base + q0 + ql))
    rows = np.asarray(rows)
    pw = oracle.Problem(whole, q, k, v, do)
    ps = oracle.Problem(sharded, q[rows], k, v, do[rows])
    Ow, Lw = oracle.forward(pw)
    Os, Ls = oracle.forward(ps)
    assert np.array_equal(Os, Ow[rows]) and np.array_equal(Ls, Lw[rows])
    dqw, dkw, dvw = oracle.backward(pw)
    dqs, dks, dvs = oracle.backward(ps)
    assert np.allclose(dqs, dqw[rows], atol=1e-13)
    assert np.allclose(dks, dkw, atol=1e-12) and np.allclose(dvs, dvw, atol=1e-12)


def test_merge_of_kv_blocks_equals_unsplit():
    """Eq. 4: merging the partial (O, LSE) of KV blocks reproduces attention
    over the whole context."""
    L, nq, nb = 96, 16, 4
    whole = W.custom("whole", [L], [(0, L - nq, nq, 0, L)], hq=4, hkv=1, d=16, seed=9)
    blk = L // nb
    split = W.custom("split", [L], [(0, L - nq, nq, b * blk, blk) for b in range(nb)], hq=4, hkv=1, d=16, seed=9)
    q, k, v, _ = inputs(whole)
    Ow, Lw = oracle.forward(oracle.Problem(whole, q, k, v))
    qs = q.repeat(nb, 1, 1)
    Os, Ls = oracle.forward(oracle.Problem(split, qs, k, v))
    Om, Lm = oracle.merge(Os.reshape(nb, nq * 4, 16), Ls.reshape(nb, nq * 4))
    assert np.allclose(Om, Ow.reshape(nq * 4, 16), rtol=0, atol=1e-12)
    assert np.allclose(Lm, Lw.reshape(-1), rtol=0, atol=1e-12)


def test_merge_empty_parts():
    o = np.random.default_rng(0).standard_normal((3, 4, 5))
    lse = np.array([[0.5, -np.inf, -np.inf, 2.0], [-np.inf, -np.inf, 1.0, 2.0], [1.5, -np.inf, -np.inf, 2.0]])
    O, L = oracle.merge(o, lse)
    # a part with LSE = -inf has weight 0; all parts empty -> O = 0, LSE = -inf
    w0 = np.exp(lse[[0, 2], 0] - 1.5)
    assert np.allclose(O[0], (w0[0] * o[0, 0] + w0[1] * o[2, 0]) / w0.sum(), atol=1e-15)
    assert L[1] == -np.inf and np.all(O[1] == 0)
    assert np.array_equal(O[2], o[1, 2]) and L[2] == 1.0
    assert np.allclose(O[3], o[:, 3].mean(0)) and L[3] == pytest.approx(2.0 + math.log(3))


def test_backward_sum_invariants():
    """Each row's dS sums to 0 over its visible keys, so sum_j dK_j = 0 over
    every document and kv head; sum_j dV_j = sum of dO over rows that see a key."""
    w = SMALL[0]
    q, k, v, do = inputs(w)
    pb = oracle.Problem(w, q, k, v, do)
    dq, dk, dv = oracle.backward(pb)
    G = w.num_q_heads // w.num_kv_heads
    for doc in range(w.n_docs):
        off, L = int(w.doc_kv_offset[doc]), int(w.doc_len[doc])
        assert np.allclose(dk[off:off + L].sum(0), 0.0, atol=1e-11)
        rows = [r for t in range(w.n_tasks) if w.task_doc[t] == doc
                for r in range(int(w.task_row_offset()[t]), int(w.task_row_offset()[t] + w.task_q_len[t]))]
        dsum = f64(do)[rows].reshape(len(rows), w.num_kv_heads, G, -1).sum((0, 2))
        assert np.allclose(dv[off:off + L].sum(0), dsum, atol=1e-11)


# ---------------------------------------------------------------- integer accounting

def brute_pairs(w):
    out = []
    for t in range(w.n_tasks):
        p = int(w.task_q_start[t]) + np.arange(int(w.task_q_len[t]))[:, None]
        j = np.arange(int(w.doc_len[w.task_doc[t]]))[None, :]
        ks, kl = int(w.task_kv_start[t]), int(w.task_kv_len[t])
        out.append(int(((j >= ks) & (j < ks + kl) & (j <= p)).sum()))
    return np.asarray(out)


@pytest.mark.parametrize("w", SMALL + [W.tiny_chunk()], ids=lambda w: w.name)
def test_pairs_brute_force(w):
    assert np.array_equal(oracle.task_pairs(w), brute_pairs(w))


def test_pairs_closed_forms():
    # whole document: l(l+1)/2
    for L in (1, 2, 127, 128, 129, 4000, 65536, 262144):
        w = W.custom("doc", [L], [(0, 0, L, 0, L)], 1, 1, 64)
        assert oracle.task_pairs(w)[0] == L * (L + 1) // 2
    # prefix task of a shard: q_len * q_start + q_len (q_len + 1) / 2
    for (q0, ql) in ((0, 5), (100, 1), (131072, 4096), (777, 333)):
        w = W.custom("shard", [q0 + ql], [(0, q0, ql, 0, q0 + ql)], 1, 1, 64)
        assert oracle.task_pairs(w)[0] == ql * q0 + ql * (ql + 1) // 2
    # tiny chunk: docs [1024, 512, 256, 256]
    assert oracle.task_pairs(W.tiny_chunk()).sum() == 721920
    # split-KV prefill: the eight blocks add up to the unsplit prefix task
    s = oracle.task_pairs(W.split_kv_prefill()).sum()
    u = oracle.task_pairs(W.split_kv_prefill(split=False)).sum()
    assert s == u == 4096 * 131072 + 4096 * 4097 // 2


def _golden(name):
    rows = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if line:
                key, *vals = line.split()
                rows[key] = vals
    return rows


def test_imbalance_examples_from_the_pages():
    """Two equal-token chunks differ in attention work by the printed factors."""
    g = _golden("imbalance_examples.txt")
    for key, (a, b, factor) in g.items():
        da = [int(x) for x in a.split(",")]
        db = [int(x) for x in b.split(",")]
        assert sum(da) == sum(db)
        wa = W.custom("a", da, [(i, 0, l, 0, l) for i, l in enumerate(da)], 1, 1, 64)
        wb = W.custom("b", db, [(i, 0, l, 0, l) for i, l in enumerate(db)], 1, 1, 64)
        ratio = oracle.task_pairs(wa).sum() / oracle.task_pairs(wb).sum()
        # the pages count l^2; causal pairs l(l+1)/2 give the factor to within 0.1 %
        assert ratio == pytest.approx(float(factor), rel=1e-3), key


def test_flops_convention():
    w = W.tiny_chunk()
    f, b = oracle.flops(w)
    assert f == 4 * 64 * 4 * 721920 and b == 2 * f


@pytest.mark.parametrize("w", SMALL, ids=lambda w: w.name)
def test_sampled_columns_and_rows_equal_full_backward(w):
    """The sampled paths (dq_rows, dkdv_cols with only the dependent rows'
    statistics computed) give the same values as the full backward."""
    q, k, v, do = inputs(w)
    pb = oracle.Problem(w, q, k, v, do)
    dq, dk, dv = oracle.backward(pb)
    rng = np.random.default_rng(1)
    docs = rng.integers(0, w.n_docs, 12).astype(np.int32)
    pos = np.array([rng.integers(0, int(w.doc_len[i])) for i in docs])
    g = rng.integers(0, w.num_kv_heads, 12).astype(np.int32)
    a, b = oracle.dkdv_cols(pb, docs, pos, g)
    rows = w.doc_kv_offset[docs] + pos
    assert np.allclose(a, dk[rows, g], atol=1e-13) and np.allclose(b, dv[rows, g], atol=1e-13)
    r = rng.integers(0, w.total_q, 12)
    h = rng.integers(0, w.num_q_heads, 12)
    assert np.array_equal(oracle.dq_rows(pb, r, h), dq[r, h])
