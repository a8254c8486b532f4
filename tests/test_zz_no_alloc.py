"""ca_backward_noalloc: the backward for callers that cannot allocate device
memory (for example code inside a framework that owns every device
allocation, or plug-in code handed only its inputs and outputs).  It uses the
library's own 16 MiB device scratch array instead of a caller workspace.

This file is collected last so that a run stopping at the first failure has
already run every other test.  It checks, through the C ABI, that two calls in
a row give the results of ca_backward (with a caller workspace) and of the fp64
oracle within the gradient tolerance of the parity tests, that a decode-shaped
plan whose workspace is large only because of the forward's split-KV scratch
is accepted, and that a plan whose backward needs more scratch than the array
holds is refused before any launch."""
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


def test_noalloc_backward_matches_workspace_backward_twice():
    w = EDGE[1]  # G = 8, shards out of order, KV blocks with empty rows, ragged tails
    q, k, v, do = W.make_tensors(w, device="cuda")
    plan = ca.Plan.from_workload(w)
    assert plan.info()["workspace_bytes"] <= 16 << 20
    ws = ca.workspace(plan)
    o, lse = ca.alloc_forward(plan)
    plan.forward(q, k, v, o, lse, ws)
    ref = ca.alloc_backward(plan)
    plan.backward(q, k, v, o, lse, do, *ref, ws)
    torch.cuda.synchronize()
    assert plan.device_status() == 0
    for _ in range(2):
        out = ca.alloc_backward(plan)
        for t in out:
            t.fill_(3.0)  # stale contents must not survive
        plan.backward_noalloc(q, k, v, o, lse, do, *out)
        torch.cuda.synchronize()
        assert plan.device_status() == 0
        for name, x, r in zip(("dQ", "dK", "dV"), out, ref):
            check_grad(to64(x), to64(r), name)
    # the last call's results against the fp64 oracle (independent of ca_backward)
    dQ, dK, dV = oracle.backward(oracle.Problem(w, q.cpu(), k.cpu(), v.cpu(), do.cpu()))
    inside = torch.zeros(w.total_kv, dtype=torch.bool)
    for off, L in zip(w.doc_kv_offset, w.doc_len):
        inside[int(off):int(off + L)] = True
    check_grad(to64(out[0]), dQ, "dQ vs oracle")
    check_grad(to64(out[1])[inside.numpy()], dK[inside.numpy()], "dK vs oracle")
    check_grad(to64(out[2])[inside.numpy()], dV[inside.numpy()], "dV vs oracle")


def test_noalloc_accepts_decode_plan_with_large_forward_scratch():
    """Four decode rows against 32K cached tokens: the forward's split-KV
    partials make the workspace larger than 16 MiB, while the backward needs
    only 66 KB of it."""
    w = W.decode_batch(n_seq=4, context=32768)
    q, k, v, do = W.make_tensors(w, device="cuda")
    plan = ca.Plan.from_workload(w)
    assert plan.info()["workspace_bytes"] > 16 << 20
    ws = ca.workspace(plan)
    o, lse = ca.alloc_forward(plan)
    plan.forward(q, k, v, o, lse, ws)
    ref = ca.alloc_backward(plan)
    plan.backward(q, k, v, o, lse, do, *ref, ws)
    out = ca.alloc_backward(plan)
    plan.backward_noalloc(q, k, v, o, lse, do, *out)
    torch.cuda.synchronize()
    assert plan.device_status() == 0
    for name, x, r in zip(("dQ", "dK", "dV"), out, ref):
        check_grad(to64(x), to64(r), name)


def test_noalloc_rejects_plans_beyond_the_scratch():
    w = W.custom("big", [40000], [(0, 0, 40000, 0, 40000)], hq=32, hkv=8, d=128)
    plan = ca.Plan.from_workload(w)
    assert plan.info()["workspace_bytes"] > 16 << 20
    t = torch.empty(16, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(ca.CAError) as ei:
        plan.backward_noalloc(t, t, t, t, t, t, t, torch.empty_like(t), torch.empty_like(t))
    assert ei.value.status == ca.capi.CA_ERR_UNSUPPORTED
