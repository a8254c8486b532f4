"""GPU parity of the sparse mask families ("DCP: Addressing Input Dynamism
In Long-Context Training via Dynamic Context Parallelism", §2.4, Figure 6)
against the fp64 oracle: small cases element by element (every row, every
key), the 64K-token chunks of each family on sampled rows and key columns,
plus the sum invariants of dK / dV at full size."""
import numpy as np
import pytest
import torch

import document_masked_core_gb300 as ca
import oracle
import workloads as W
from parity import check_grad, check_lse, check_o, to64

pytestmark = pytest.mark.gpu

SMALL = [
    W.lambda_chunk(seed=1, total=3000, sink=70, window=300, hq=8, hkv=2, d=64),
    W.lambda_chunk(seed=2, total=3000, sink=0, window=129, hq=4, hkv=1, d=128),
    W.blockwise_chunk(seed=3, total=3000, block=96, sink_blocks=2, window_blocks=3, hq=8, hkv=1, d=64),
    W.blockwise_chunk(seed=5, total=2600, block=256, sink_blocks=1, window_blocks=2, hq=32, hkv=8, d=128),
    W.shared_question_pool(seed=4, total=3000, q_lo=100, q_hi=400, a_lo=40, a_hi=300, hq=4, hkv=1, d=64),
    W.custom("mixed_masks", [700, 500], [(0, 0, 700, 0, 700), (1, 100, 300, 50, 400), (0, 300, 200, 0, 600)],
             8, 2, 128, seed=6, masks=[(10, 0, 200), (0, 256, 0), (130, 400, 77)]),
]


@pytest.fixture(scope="module", autouse=True)
def built():
    from document_masked_core_gb300 import build
    build.build()


def run(w, o_dtype, inputs):
    q, k, v, do = inputs
    plan = ca.Plan.from_workload(w, o_dtype=o_dtype)
    ws = ca.workspace(plan)
    o, lse = ca.alloc_forward(plan)
    plan.forward(q, k, v, o, lse, ws)
    dq, dk, dv = ca.alloc_backward(plan)
    dk.fill_(7.0)
    dv.fill_(7.0)
    plan.backward(q, k, v, o, lse, do, dq, dk, dv, ws)
    torch.cuda.synchronize()
    assert plan.device_status() == 0
    return o, lse, dq, dk, dv


@pytest.mark.parametrize("w", SMALL, ids=lambda w: w.name)
def test_masked_small_match_oracle(w):
    inputs = W.make_tensors(w, device="cuda")
    q, k, v, do = inputs
    o32, lse32, _, _, _ = run(w, ca.CA_DTYPE_FP32, inputs)
    o16, lse16, dq, dk, dv = run(w, ca.CA_DTYPE_BF16, inputs)
    assert torch.equal(lse16, lse32)
    assert torch.equal(o16.view(torch.int16), o32.to(torch.bfloat16).view(torch.int16))
    pb = oracle.Problem(w, q.cpu(), k.cpu(), v.cpu(), do.cpu())
    O, LSE = oracle.forward(pb)
    check_o(to64(o32), O)
    check_lse(to64(lse32), LSE)
    dQ, dK, dV = oracle.backward(pb)
    check_grad(to64(dq), dQ, "dQ")
    inside = np.zeros(w.total_kv, dtype=bool)
    for off, L in zip(w.doc_kv_offset, w.doc_len):
        inside[int(off):int(off + L)] = True
    check_grad(to64(dk)[inside], dK[inside], "dK")
    check_grad(to64(dv)[inside], dV[inside], "dV")


@pytest.mark.parametrize("name", list(W.MASKED_WORKLOADS))
def test_masked_fullsize_sampled(name):
    w = W.MASKED_WORKLOADS[name]()
    inputs = W.make_tensors(w, device="cuda")
    q, k, v, do = inputs
    o32, lse32, _, _, _ = run(w, ca.CA_DTYPE_FP32, inputs)
    o16, lse, dq, dk, dv = run(w, ca.CA_DTYPE_BF16, inputs)
    rng = np.random.default_rng(w.seed + 1000)
    rows, heads = rng.integers(0, w.total_q, 2048), rng.integers(0, w.num_q_heads, 2048)
    rt, ht = torch.as_tensor(rows, device="cuda"), torch.as_tensor(heads, device="cuda")
    pb = oracle.Problem(w, q.cpu(), k.cpu(), v.cpu(), do.cpu())
    O, LSE = oracle.forward_rows(pb, rows, heads)
    check_o(to64(o32[rt, ht]), O)
    check_lse(to64(lse[rt, ht]), LSE)
    check_grad(to64(dq[rt, ht]), oracle.dq_rows(pb, rows, heads), "dQ (sampled rows)")
    # key columns late in their documents (few dependent rows under any mask)
    G = w.num_q_heads // w.num_kv_heads
    cd, cj, cg = [], [], []
    for d_ in range(w.n_docs):
        L = int(w.doc_len[d_])
        for j in rng.integers(max(0, L - 256), L, 8):
            cd.append(d_)
            cj.append(int(j))
            cg.append(int(rng.integers(0, w.num_kv_heads)))
    dK, dV = oracle.dkdv_cols(pb, np.asarray(cd), np.asarray(cj), np.asarray(cg))
    kr = torch.as_tensor(w.doc_kv_offset[np.asarray(cd)] + np.asarray(cj), device="cuda")
    gt = torch.as_tensor(np.asarray(cg), device="cuda")
    check_grad(to64(dk[kr, gt]), dK, "dK (sampled columns)")
    check_grad(to64(dv[kr, gt]), dV, "dV (sampled columns)")
    # sum over every document and kv head: sum_j dK_j = 0 (each row's dS sums to 0)
    for d_ in range(w.n_docs):
        off, L = int(w.doc_kv_offset[d_]), int(w.doc_len[d_])
        dkd = dk[off:off + L].float()
        assert torch.all(dkd.sum(0).abs() <= 2e-2 * (dkd.abs().sum(0) + 1e-3))
    assert G >= 1
