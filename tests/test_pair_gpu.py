"""GPU parity of the CTA-pair backward main kernel (ca_plan_set_backward_kernel
with CA_BWD_KERNEL_PAIR): against the fp64 oracle on small cases, and against
the one-CTA kernel on the same inputs -- dK and dV bit for bit (both
accumulate the same products in the same order; query tiles that see only one
of the pair's key tiles add exact zeros to the other), dQ to fp32 summation
order (the reduce-adds land in a different order)."""
import numpy as np
import pytest
import torch

import document_masked_core_gb300 as ca
import oracle
import workloads as W
from cases import EDGE
from parity import check_grad, rel_fro, to64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    from document_masked_core_gb300 import build
    build.build()


def pair_applies(w):
    G = w.num_q_heads // w.num_kv_heads
    return w.head_dim == 128 and 64 % G == 0


SMALL = [w for w in EDGE if pair_applies(w)] + [
    # odd numbers of key tiles: the last pair's second tile lies past the document
    W.custom("pair_odd_tiles", [384, 129, 1000], [(i, 0, l, 0, l) for i, l in enumerate([384, 129, 1000])],
             hq=32, hkv=8, d=128, seed=11),
    # G = 1, 2, 64: 128, 64 and 2 query tokens per tile, 64, 32 and 1 per CTA of the pair
    W.custom("pair_g1", [700, 300], [(0, 0, 700, 0, 700), (1, 0, 300, 0, 300)], hq=2, hkv=2, d=128, seed=12),
    W.custom("pair_g2", [500], [(0, 0, 500, 0, 500)], hq=4, hkv=2, d=128, seed=13),
    W.custom("pair_g64", [90, 200], [(0, 0, 90, 0, 90), (1, 0, 200, 0, 200)], hq=64, hkv=1, d=128, seed=14),
    # sparse masks: sink + window narrower than a tile, a sliding window, causal blockwise
    W.custom("pair_window40", [1500], [(0, 0, 1500, 0, 1500)], hq=32, hkv=8, d=128, seed=15, masks=[(0, 0, 40)]),
    W.custom("pair_lambda", [2500, 700], [(0, 0, 2500, 0, 2500), (1, 0, 700, 0, 700)], hq=32, hkv=8, d=128, seed=16,
             masks=[(64, 0, 512), (64, 0, 512)]),
    W.blockwise_chunk(seed=17, total=2048, block=256),
]


def fwd_bwd_both(w, inputs=None):
    if inputs is None:
        inputs = W.make_tensors(w, device="cuda")
    torch.cuda.synchronize()
    q, k, v, do = inputs
    plan = ca.Plan.from_workload(w)
    ws = ca.workspace(plan)
    o, lse = ca.alloc_forward(plan)
    plan.forward(q, k, v, o, lse, ws)
    out = {}
    for kind in (ca.capi.CA_BWD_KERNEL_SINGLE, ca.capi.CA_BWD_KERNEL_PAIR):
        plan.set_backward_kernel(kind)
        dq, dk, dv = ca.alloc_backward(plan)
        dq.fill_(float("nan"))
        dk.fill_(7.0)
        dv.fill_(7.0)
        plan.backward(q, k, v, o, lse, do, dq, dk, dv, ws)
        torch.cuda.synchronize()
        assert plan.device_status() == 0
        out[kind] = (dq, dk, dv)
    return (q, k, v, do), out[ca.capi.CA_BWD_KERNEL_SINGLE], out[ca.capi.CA_BWD_KERNEL_PAIR]


def doc_rows(w):
    rows = np.zeros(w.total_kv, dtype=bool)
    for off, L in zip(w.doc_kv_offset, w.doc_len):
        rows[int(off):int(off + L)] = True
    return rows


@pytest.mark.parametrize("w", SMALL, ids=lambda w: w.name)
def test_pair_backward_matches_oracle_and_single(w):
    (q, k, v, do), single, pair = fwd_bwd_both(w)
    dq, dk, dv = pair
    dQ, dK, dV = oracle.backward(oracle.Problem(w, q.cpu(), k.cpu(), v.cpu(), do.cpu()))
    inside = doc_rows(w)
    check_grad(to64(dq), dQ, "dQ")
    check_grad(to64(dk)[inside], dK[inside], "dK")
    check_grad(to64(dv)[inside], dV[inside], "dV")
    # rows outside every document are not written
    assert np.all(to64(dk)[~inside] == 7.0) and np.all(to64(dv)[~inside] == 7.0)
    assert torch.equal(dk, single[1]) and torch.equal(dv, single[2])
    assert rel_fro(to64(dq), to64(single[0])) <= 1e-4


@pytest.mark.parametrize("make", [lambda: W.llama8b_chunk(seed=0), lambda: W.rebatched_pool(seed=0)],
                         ids=["llama8b_chunk_64k", "rebatched_pool_128k"])
def test_pair_backward_equals_single_at_full_size(make):
    """The bench workload and the rebatched pool of shards at full size: every
    dK and dV bit for bit, dQ to summation order (the one-CTA kernel is
    compared with the oracle on every row and column of these elsewhere)."""
    w = make()
    _, single, pair = fwd_bwd_both(w)
    assert torch.equal(pair[1], single[1]) and torch.equal(pair[2], single[2])
    assert bool(torch.isfinite(pair[0]).all())
    a, b = pair[0].double(), single[0].double()
    assert float((a - b).norm() / b.norm()) <= 1e-4


def test_pair_selection_falls_back_where_it_does_not_apply():
    """head_dim 64 or G = 128: CA_BWD_KERNEL_PAIR runs the one-CTA kernel."""
    for w in (W.tiny_chunk(), [x for x in EDGE if x.name == "g128_d128"][0]):
        assert not pair_applies(w)
        _, single, pair = fwd_bwd_both(w)
        assert torch.equal(pair[1], single[1]) and torch.equal(pair[2], single[2])
        assert rel_fro(to64(pair[0]), to64(single[0])) <= 1e-4


def test_set_backward_kernel_rejects_unknown_kinds():
    plan = ca.Plan.from_workload(W.tiny_chunk())
    with pytest.raises(ca.CAError):
        plan.set_backward_kernel(3)
    with pytest.raises(ca.CAError):
        plan.set_backward_kernel(-1)


def test_pair_backward_with_float32_o():
    """The preprocess reads a float32 O; the pair kernel is the same."""
    w = [x for x in EDGE if x.name == "g8_shards_blocks"][0]
    q, k, v, do = W.make_tensors(w, device="cuda")
    torch.cuda.synchronize()
    plan = ca.Plan.from_workload(w, o_dtype=ca.CA_DTYPE_FP32)
    plan.set_backward_kernel(ca.capi.CA_BWD_KERNEL_PAIR)
    ws = ca.workspace(plan)
    o, lse = ca.alloc_forward(plan)
    plan.forward(q, k, v, o, lse, ws)
    dq, dk, dv = ca.alloc_backward(plan)
    plan.backward(q, k, v, o, lse, do, dq, dk, dv, ws)
    torch.cuda.synchronize()
    assert plan.device_status() == 0
    dQ, dK, dV = oracle.backward(oracle.Problem(w, q.cpu(), k.cpu(), v.cpu(), do.cpu()))
    inside = doc_rows(w)
    check_grad(to64(dq), dQ, "dQ")
    check_grad(to64(dk)[inside], dK[inside], "dK")
    check_grad(to64(dv)[inside], dV[inside], "dV")


def test_pair_backward_replays_from_a_cuda_graph():
    """Forward + pair backward captured into a CUDA graph replay with the
    eager results (dK, dV bit for bit, dQ within the gradient tolerance of the
    oracle), twice in a row."""
    w = [x for x in SMALL if x.name == "pair_odd_tiles"][0]  # odd numbers of key tiles per document
    q, k, v, do = W.make_tensors(w, device="cuda")
    torch.cuda.synchronize()
    plan = ca.Plan.from_workload(w)
    plan.set_backward_kernel(ca.capi.CA_BWD_KERNEL_PAIR)
    ws = ca.workspace(plan)
    o, lse = ca.alloc_forward(plan)
    dq, dk, dv = ca.alloc_backward(plan)
    plan.forward(q, k, v, o, lse, ws)
    plan.backward(q, k, v, o, lse, do, dq, dk, dv, ws)
    torch.cuda.synchronize()
    assert plan.device_status() == 0
    o2, lse2 = ca.alloc_forward(plan)
    dq2, dk2, dv2 = ca.alloc_backward(plan)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        plan.forward(q, k, v, o2, lse2, ws)
        plan.backward(q, k, v, o2, lse2, do, dq2, dk2, dv2, ws)
    ref = oracle.backward(oracle.Problem(w, q.cpu(), k.cpu(), v.cpu(), do.cpu()))
    for _ in range(2):
        for t in (dq2, dk2, dv2):
            t.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        assert plan.device_status() == 0
        assert torch.equal(dk2, dk) and torch.equal(dv2, dv)
        check_grad(to64(dq2), ref[0], "dQ (graph replay)")


def test_pair_backward_without_a_workspace():
    """ca_backward_noalloc with the pair kernel selected gives the workspace
    call's dK, dV bit for bit and its dQ to summation order."""
    w = [x for x in EDGE if x.name == "g8_shards_blocks"][0]
    q, k, v, do = W.make_tensors(w, device="cuda")
    torch.cuda.synchronize()
    plan = ca.Plan.from_workload(w)
    plan.set_backward_kernel(ca.capi.CA_BWD_KERNEL_PAIR)
    ws = ca.workspace(plan)
    o, lse = ca.alloc_forward(plan)
    plan.forward(q, k, v, o, lse, ws)
    ref = ca.alloc_backward(plan)
    plan.backward(q, k, v, o, lse, do, *ref, ws)
    out = ca.alloc_backward(plan)
    plan.backward_noalloc(q, k, v, o, lse, do, *out)
    torch.cuda.synchronize()
    assert plan.device_status() == 0
    assert torch.equal(out[1], ref[1]) and torch.equal(out[2], ref[2])
    assert rel_fro(to64(out[0]), to64(ref[0])) <= 1e-4
