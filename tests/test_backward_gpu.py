"""GPU parity of ca_backward against the fp64 oracle."""
import numpy as np
import pytest
import torch

import document_masked_core_gb300 as ca
import oracle
import workloads as W
from cases import EDGE
from parity import check_grad, to64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    from document_masked_core_gb300 import build
    build.build()


def run_fwd_bwd(w, o_dtype=ca.CA_DTYPE_BF16, inputs=None, sentinel=7.0):
    if inputs is None:
        inputs = W.make_tensors(w, device="cuda")
    q, k, v, do = inputs
    plan = ca.Plan.from_workload(w, o_dtype=o_dtype)
    ws = ca.workspace(plan)
    o, lse = ca.alloc_forward(plan)
    plan.forward(q, k, v, o, lse, ws)
    dq, dk, dv = ca.alloc_backward(plan)
    dq.fill_(float("nan"))
    dk.fill_(sentinel)
    dv.fill_(sentinel)
    plan.backward(q, k, v, o, lse, do, dq, dk, dv, ws)
    torch.cuda.synchronize()
    assert plan.device_status() == 0
    return plan, (q, k, v, do), (o, lse), (dq, dk, dv)


def doc_rows(w):
    rows = np.zeros(w.total_kv, dtype=bool)
    for off, L in zip(w.doc_kv_offset, w.doc_len):
        rows[int(off):int(off + L)] = True
    return rows


@pytest.mark.parametrize("w", [W.tiny_chunk()] + EDGE, ids=lambda w: w.name)
@pytest.mark.parametrize("o_dtype", [ca.CA_DTYPE_BF16, ca.CA_DTYPE_FP32], ids=["obf16", "ofp32"])
def test_backward_matches_oracle(w, o_dtype):
    _, (q, k, v, do), _, (dq, dk, dv) = run_fwd_bwd(w, o_dtype)
    dQ, dK, dV = oracle.backward(oracle.Problem(w, q.cpu(), k.cpu(), v.cpu(), do.cpu()))
    inside = doc_rows(w)
    check_grad(to64(dq), dQ, "dQ")
    check_grad(to64(dk)[inside], dK[inside], "dK")
    check_grad(to64(dv)[inside], dV[inside], "dV")
    # keys that no task sees are exactly 0; rows outside every document are untouched
    unseen = inside[:, None] & (np.abs(dK).sum(-1) == 0) & (np.abs(dV).sum(-1) == 0)
    assert np.all(to64(dk)[unseen] == 0) and np.all(to64(dv)[unseen] == 0)
    assert np.all(to64(dk)[~inside] == 7.0) and np.all(to64(dv)[~inside] == 7.0)


def test_backward_sum_invariants_on_gpu():
    """Each row's dS sums to zero, so per document and kv head sum_j dK_j ~ 0
    and sum_j dV_j = sum of dO over the group's heads."""
    w = EDGE[1]
    _, (q, k, v, do), _, (dq, dk, dv) = run_fwd_bwd(w)
    G = w.num_q_heads // w.num_kv_heads
    dof = to64(do)
    row0 = w.task_row_offset()
    for d in range(w.n_docs):
        off, L = int(w.doc_kv_offset[d]), int(w.doc_len[d])
        dkd, dvd = to64(dk)[off:off + L], to64(dv)[off:off + L]
        assert np.all(np.abs(dkd.sum(0)) <= 2e-2 * (np.abs(dkd).sum(0) + 1e-6))
        # rows whose visible set is empty (p < kv_start) contribute nothing to dV
        rows = [int(row0[t]) + i for t in range(w.n_tasks) if w.task_doc[t] == d
                for i in range(int(w.task_q_len[t])) if int(w.task_q_start[t]) + i >= int(w.task_kv_start[t])]
        ref = dof[rows].reshape(len(rows), w.num_kv_heads, G, -1).sum((0, 2))
        assert np.all(np.abs(dvd.sum(0) - ref) <= 1e-2 * (np.abs(dvd).sum(0) + 1e-6))


def test_backward_is_deterministic_for_dk_dv():
    w = EDGE[3]
    _, inp, _, (dq1, dk1, dv1) = run_fwd_bwd(w)
    _, _, _, (dq2, dk2, dv2) = run_fwd_bwd(w, inputs=inp)
    assert torch.equal(dk1, dk2) and torch.equal(dv1, dv2)
    # dQ sums fp32 atomics in arbitrary order: equal to rounding
    assert (dq1.float() - dq2.float()).abs().max().item() <= 1e-2


def test_overlapping_buffers_are_refused_before_any_launch():
    """Outputs that share a byte with another output or with an input are
    rejected with CA_ERR_INVALID_ARG (sizes from the plan), on the host."""
    w = EDGE[0]
    q, k, v, do = W.make_tensors(w, device="cuda")
    plan = ca.Plan.from_workload(w)
    ws = ca.workspace(plan)
    o, lse = ca.alloc_forward(plan)
    dq, dk, dv = ca.alloc_backward(plan)
    big = torch.empty(q.numel() * 4 + 4096, dtype=torch.uint8, device="cuda")

    def refused(fn):
        with pytest.raises(ca.CAError) as ei:
            fn()
        assert ei.value.status == ca.capi.CA_ERR_INVALID_ARG
    # forward: O overlapping Q (offset by one 16-byte row chunk), LSE inside O, workspace over V
    q_in_big = big[:q.numel() * 2].view(torch.bfloat16).view_as(q).copy_(q)
    o_shift = big[16:16 + o.numel() * 2].view(torch.bfloat16).view_as(o)
    refused(lambda: plan.forward(q_in_big, k, v, o_shift, lse, ws))
    refused(lambda: plan.forward(q, k, v, o, o.view(torch.float32).view(-1)[:lse.numel()].view_as(lse), ws))
    refused(lambda: plan.forward(q, k, v, o, lse, v.view(torch.uint8)))
    plan.forward(q, k, v, o, lse, ws)
    # backward: dK over V, dQ over the workspace, dV over dK
    refused(lambda: plan.backward(q, k, v, o, lse, do, dq, v, dv, ws))
    refused(lambda: plan.backward(q, k, v, o, lse, do, ws.view(torch.bfloat16)[:dq.numel()].view_as(dq), dk, dv, ws))
    refused(lambda: plan.backward(q, k, v, o, lse, do, dq, dk, dk, ws))
    # the refused calls launched nothing: a real backward still matches the first one
    plan.backward(q, k, v, o, lse, do, dq, dk, dv, ws)
    torch.cuda.synchronize()
    assert plan.device_status() == 0
    ref = oracle.backward(oracle.Problem(w, q.cpu(), k.cpu(), v.cpu(), do.cpu()))
    inside = doc_rows(w)
    check_grad(to64(dq), ref[0], "dQ")
    check_grad(to64(dk)[inside], ref[1][inside], "dK")


def test_forward_backward_replay_from_a_cuda_graph():
    """ca_forward + ca_backward captured into a CUDA graph (stream capture; the
    calls allocate nothing and every counter they use is reset on the device
    each call) replay with the eager results: O, LSE, dK, dV bit for bit, dQ
    (fp32 reduce-adds in any order) within the gradient tolerance of the
    oracle, twice in a row."""
    w = W.tiny_chunk()
    q, k, v, do = W.make_tensors(w, device="cuda")
    plan = ca.Plan.from_workload(w)
    ws = ca.workspace(plan)
    o, lse = ca.alloc_forward(plan)
    dq, dk, dv = ca.alloc_backward(plan)
    plan.forward(q, k, v, o, lse, ws)
    plan.backward(q, k, v, o, lse, do, dq, dk, dv, ws)
    torch.cuda.synchronize()
    o2, lse2 = ca.alloc_forward(plan)
    dq2, dk2, dv2 = ca.alloc_backward(plan)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        plan.forward(q, k, v, o2, lse2, ws)
        plan.backward(q, k, v, o2, lse2, do, dq2, dk2, dv2, ws)
    ref = oracle.backward(oracle.Problem(w, q.cpu(), k.cpu(), v.cpu(), do.cpu()))
    for _ in range(2):
        for t in (o2, dq2, dk2, dv2):
            t.fill_(float("nan"))
        lse2.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        assert plan.device_status() == 0
        assert torch.equal(o2.view(torch.int16), o.view(torch.int16)) and torch.equal(lse2, lse)
        assert torch.equal(dk2.view(torch.int16), dk.view(torch.int16))
        assert torch.equal(dv2.view(torch.int16), dv.view(torch.int16))
        check_grad(to64(dq2), ref[0], "dQ (graph replay)")
