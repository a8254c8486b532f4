"""Parity at the full workload sizes, in the launch configuration bench.py
times (plans built from the same generators, bf16 O), on sampled outputs the
oracle computes one by one:

  * 4096 (token, query head) rows of O and LSE (float32-output run; the bf16
    output the bench uses must be the round-to-nearest-even of it),
  * 4096 (token, query head) rows of dQ,
  * (key, kv head) columns of dK / dV drawn uniformly over the keys some row
    sees and kept while the rows they depend on stay within a fixed oracle
    budget (so columns late in their document and short documents dominate;
    every column of the long documents is compared in
    test_fullsize_dense_gpu.py),
  * the sum invariants at every size: per document and kv head,
    sum_j dK_j ~ 0 and sum_j dV_j = sum of dO over the rows that see a key.
Split-KV prefill: the eight KV-block partials merged by ca_merge are checked
against the oracle's unsplit rows and against the GPU's unsplit launch.
"""
import numpy as np
import pytest
import torch

import document_masked_core_gb300 as ca
import oracle
import workloads as W
from parity import check_grad, check_lse, check_o, to64

pytestmark = pytest.mark.gpu

N_ROWS = 4096
COL_BUDGET = 3e8  # (row, head, key) evaluations the oracle spends on dK/dV columns


@pytest.fixture(scope="module", autouse=True)
def built():
    from document_masked_core_gb300 import build
    build.build()


def sample_rows(w, seed, n=N_ROWS):
    rng = np.random.default_rng(seed + 1000)
    return rng.integers(0, w.total_q, n), rng.integers(0, w.num_q_heads, n)


def sample_cols(w, seed, budget=COL_BUDGET, max_cols=N_ROWS):
    """Key columns in uniform random order, kept while the union of their
    dependent rows (rows p >= j of the document, all heads of the group)
    costs at most `budget` (row, head, key) evaluations."""
    rng = np.random.default_rng(seed + 2000)
    G = w.num_q_heads // w.num_kv_heads
    starts = np.concatenate([[0], np.cumsum(w.doc_len)[:-1]])
    total = int(w.doc_len.sum())
    # last position any task of each document reaches: keys past it are seen by
    # no row (both sides 0), which would make the check vacuous
    last_row = np.full(w.n_docs, -1)
    for t in range(w.n_tasks):
        d = int(w.task_doc[t])
        last_row[d] = max(last_row[d], int(w.task_q_start[t] + w.task_q_len[t]) - 1)
    jmin = {}
    cost = 0.0
    out = []

    tasks_of = {}
    for t in range(w.n_tasks):
        tasks_of.setdefault(int(w.task_doc[t]), []).append((int(w.task_q_start[t]), int(w.task_q_len[t])))

    def union_cost(d, j):  # the document's task rows p >= j, each seeing ~p+1 keys, G heads
        c = 0.0
        for q0, ql in tasks_of.get(d, []):
            a, e = max(j, q0), q0 + ql  # rows [a, e)
            if e > a:
                c += (e * (e + 1) - a * (a + 1)) / 2.0
        return G * c

    for flat in rng.permutation(total)[: 200 * max_cols]:
        d = int(np.searchsorted(starts, flat, side="right") - 1)
        j = int(flat - starts[d])
        g = int(rng.integers(0, w.num_kv_heads))
        if j > last_row[d]:
            continue
        L = int(w.doc_len[d])
        old = jmin.get((d, g), L)
        new = min(old, j)
        extra = union_cost(d, new) - union_cost(d, old)
        if cost + extra > budget:
            continue
        cost += extra
        jmin[(d, g)] = new
        out.append((d, j, g))
        if len(out) >= max_cols:
            break
    a = np.asarray(out, dtype=np.int64)
    return a[:, 0], a[:, 1], a[:, 2]


def run(w, o_dtype, inputs):
    q, k, v, do = inputs
    plan = ca.Plan.from_workload(w, o_dtype=o_dtype)
    ws = ca.workspace(plan)
    o, lse = ca.alloc_forward(plan)
    plan.forward(q, k, v, o, lse, ws)
    torch.cuda.synchronize()
    assert plan.device_status() == 0
    return plan, ws, o, lse


def host(x, rows=None):
    return (x if rows is None else x[rows]).cpu()


@pytest.mark.parametrize("name", ["llama8b", "pool", "long"])
def test_fullsize_forward_backward_sampled(name):
    w = W.WORKLOADS[name]()
    inputs = W.make_tensors(w, device="cuda")
    q, k, v, do = inputs
    plan, ws, o16, lse = run(w, ca.CA_DTYPE_BF16, inputs)
    _, _, o32, lse32 = run(w, ca.CA_DTYPE_FP32, inputs)
    assert torch.equal(lse, lse32)
    rows, heads = sample_rows(w, w.seed)
    rt, ht = torch.as_tensor(rows, device="cuda"), torch.as_tensor(heads, device="cuda")
    assert torch.equal(o16[rt, ht].view(torch.int16), o32[rt, ht].to(torch.bfloat16).view(torch.int16))
    pb = oracle.Problem(w, host(q), host(k), host(v), host(do))
    O, LSE = oracle.forward_rows(pb, rows, heads)
    check_o(to64(o32[rt, ht]), O)
    check_lse(to64(lse[rt, ht]), LSE)
    del o32, lse32
    # backward in the bench's configuration (bf16 O)
    dq, dk, dv = ca.alloc_backward(plan)
    plan.backward(q, k, v, o16, lse, do, dq, dk, dv, ws)
    torch.cuda.synchronize()
    assert plan.device_status() == 0
    dQ = oracle.dq_rows(pb, rows, heads)
    check_grad(to64(dq[rt, ht]), dQ, "dQ (sampled rows)")
    cd, cj, cg = sample_cols(w, w.seed)
    assert len(cd) >= 256
    dK, dV = oracle.dkdv_cols(pb, cd, cj, cg)
    kr = torch.as_tensor(w.doc_kv_offset[cd] + cj, device="cuda")
    gt = torch.as_tensor(cg, device="cuda")
    check_grad(to64(dk[kr, gt]), dK, "dK (sampled columns)")
    check_grad(to64(dv[kr, gt]), dV, "dV (sampled columns)")
    # sum invariants over every document and kv head (all sizes)
    G = w.num_q_heads // w.num_kv_heads
    row0 = w.task_row_offset()
    dof = do.float()
    for d in range(w.n_docs):
        off, L = int(w.doc_kv_offset[d]), int(w.doc_len[d])
        dkd = dk[off:off + L].float()
        assert torch.all(dkd.sum(0).abs() <= 2e-2 * (dkd.abs().sum(0) + 1e-3))
        sel = [(int(row0[t]), int(w.task_q_len[t])) for t in range(w.n_tasks) if w.task_doc[t] == d]
        if not sel:
            continue
        ref = sum(dof[r0:r0 + n].sum(0) for r0, n in sel).reshape(w.num_kv_heads, G, -1).sum(1)
        dvd = dv[off:off + L].float()
        assert torch.all((dvd.sum(0) - ref).abs() <= 1e-2 * (dvd.abs().sum(0) + 1e-3))


def test_fullsize_split_kv_prefill_merge():
    ws_ = W.split_kv_prefill()
    whole = W.split_kv_prefill(split=False)
    nb = ws_.n_tasks
    qd, k, v, _ = W.make_tensors(whole, device="cuda", need_grad_inputs=False)
    nq, hq, d = qd.shape
    # the eight tasks share the query rows; they are packed one block after another
    q8 = qd.repeat(nb, 1, 1)
    plan_s = ca.Plan.from_workload(ws_, o_dtype=ca.CA_DTYPE_FP32)
    o_p, lse_p = ca.alloc_forward(plan_s)
    plan_s.forward(q8, k, v, o_p, lse_p, ca.workspace(plan_s))
    o_m = torch.empty((nq, hq, d), dtype=torch.float32, device="cuda")
    lse_m = torch.empty((nq, hq), dtype=torch.float32, device="cuda")
    o_parts = [o_p[b * nq:(b + 1) * nq] for b in range(nb)]
    l_parts = [lse_p[b * nq:(b + 1) * nq] for b in range(nb)]
    ca.merge(o_parts, l_parts, nq, hq, d, o_m, lse_m, parts_dtype=ca.CA_DTYPE_FP32, out_dtype=ca.CA_DTYPE_FP32)
    torch.cuda.synchronize()
    assert plan_s.device_status() == 0
    plan_w, _, o_w, lse_w = run(whole, ca.CA_DTYPE_FP32, (qd, k, v, None))
    rows, heads = sample_rows(whole, whole.seed)
    rt, ht = torch.as_tensor(rows, device="cuda"), torch.as_tensor(heads, device="cuda")
    pb = oracle.Problem(whole, host(qd), host(k), host(v))
    O, LSE = oracle.forward_rows(pb, rows, heads)
    check_o(to64(o_m[rt, ht]), O, "merged O")
    check_lse(to64(lse_m[rt, ht]), LSE, "merged LSE")
    check_o(to64(o_w[rt, ht]), O, "unsplit O")
    # merged partials against the GPU's unsplit launch, every row
    assert (o_m - o_w).abs().max().item() <= 1e-2
    rel = ((lse_m - lse_w).abs() / lse_w.abs().clamp(min=1.0)).max().item()
    assert rel <= 1e-3
    # the partials themselves: each KV block's rows against the oracle
    pbs = oracle.Problem(ws_, host(q8), host(k), host(v))
    r8 = rows[:512] + nq * (np.arange(512) % nb)
    Ob, Lb = oracle.forward_rows(pbs, r8, heads[:512])
    r8t = torch.as_tensor(r8, device="cuda")
    check_o(to64(o_p[r8t, ht[:512]]), Ob, "partial O")
    check_lse(to64(lse_p[r8t, ht[:512]]), Lb, "partial LSE")
