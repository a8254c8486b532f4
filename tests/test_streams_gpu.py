"""One plan used on several streams at once, each call with its own workspace
and outputs (the concurrency rule of include/ca.h): the results equal those of
the same calls run one after another -- O, LSE, dK and dV bit for bit, dQ to
the summation order of its reduce-adds."""
import pytest
import torch

import document_masked_core_gb300 as ca
import workloads as W
from cases import EDGE
from parity import rel_fro, to64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    from document_masked_core_gb300 import build
    build.build()


def step(plan, inputs, ws, stream):
    q, k, v, do = inputs
    o, lse = ca.alloc_forward(plan)
    dq, dk, dv = ca.alloc_backward(plan)
    dk.fill_(7.0)  # rows outside every document are written by no call
    dv.fill_(7.0)
    plan.forward(q, k, v, o, lse, ws, stream=stream)
    plan.backward(q, k, v, o, lse, do, dq, dk, dv, ws, stream=stream)
    return o, lse, dq, dk, dv


@pytest.mark.parametrize("make", [lambda: [x for x in EDGE if x.name == "g8_shards_blocks"][0],
                                  lambda: W.rebatched_pool(seed=3, total_q=16384, doc_lo=2000, doc_hi=12000,
                                                           shard_lo=200, shard_hi=3000)],
                         ids=["g8_shards_blocks", "pool_16k"])
def test_one_plan_on_four_streams(make):
    w = make()
    inputs = W.make_tensors(w, device="cuda")
    torch.cuda.synchronize()
    plan = ca.Plan.from_workload(w)
    ref = step(plan, inputs, ca.workspace(plan), torch.cuda.current_stream())
    torch.cuda.synchronize()
    assert plan.device_status() == 0
    streams = [torch.cuda.Stream() for _ in range(4)]
    spaces = [ca.workspace(plan) for _ in streams]
    outs = []
    for _ in range(2):  # two rounds, so the streams' launches overlap one another
        for s, ws in zip(streams, spaces):
            with torch.cuda.stream(s):
                outs.append(step(plan, inputs, ws, s))
    torch.cuda.synchronize()
    assert plan.device_status() == 0
    for o, lse, dq, dk, dv in outs:
        assert torch.equal(o.view(torch.int16), ref[0].view(torch.int16)) and torch.equal(lse, ref[1])
        assert torch.equal(dk, ref[3]) and torch.equal(dv, ref[4])
        # the reduce-adds of dQ land in any order, and a few bf16 roundings of
        # dQ flip with it (about 1e-5 relative on this pool; the same bound as
        # the other kernel-against-kernel dQ checks)
        assert rel_fro(to64(dq), to64(ref[2])) <= 1e-4
