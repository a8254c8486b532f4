"""In-launch split-KV (ca_plan_set_kv_split): forward items cut into parts
whose partial (O, LSE) rows are merged inside the launch by the last part to
finish (the pass-KV merge, "Context Parallelism for Scalable Million-Token
Inference", Appendix B, Eq. 4).  Forced splits on small cases and the
automatic split of decode-shaped batches are checked against the fp64 oracle
and against the unsplit launch."""
import numpy as np
import pytest
import torch

import document_masked_core_gb300 as ca
import oracle
import workloads as W
from cases import EDGE
from parity import LSE_RTOL, O_ATOL, check_grad, check_lse, check_o, to64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    from document_masked_core_gb300 import build
    build.build()


def forward(w, inputs, split, o_dtype=ca.CA_DTYPE_FP32, backward=False):
    q, k, v, do = inputs
    plan = ca.Plan.from_workload(w, o_dtype=o_dtype)
    plan.set_kv_split(split)
    info = plan.info()
    ws = ca.workspace(plan)
    o, lse = ca.alloc_forward(plan)
    plan.forward(q, k, v, o, lse, ws)
    grads = None
    if backward:
        dq, dk, dv = ca.alloc_backward(plan)
        plan.backward(q, k, v, o, lse, do, dq, dk, dv, ws)
        grads = (dq, dk, dv)
    torch.cuda.synchronize()
    assert plan.device_status() == 0
    return info, o, lse, grads


SMALL = [W.tiny_chunk()] + EDGE + [
    W.lambda_chunk(seed=1, total=3000, sink=70, window=300, hq=8, hkv=2, d=64),
    # long enough contexts (> 2 x 64 key tiles) for the automatic rule to split
    W.decode_batch(seed=2, n_seq=6, context=20000, q_len=1, jitter=3000, hq=8, hkv=2, d=128),
    W.decode_batch(seed=3, n_seq=5, context=17000, q_len=5, jitter=300, hq=16, hkv=1, d=64),
]


@pytest.mark.parametrize("w", SMALL, ids=lambda w: w.name)
@pytest.mark.parametrize("split", [1, 3])
def test_forced_split_matches_oracle_and_unsplit(w, split):
    inputs = W.make_tensors(w, device="cuda")
    q, k, v, do = inputs
    info_s, o_s, l_s, _ = forward(w, inputs, split)
    info_n, o_n, l_n, _ = forward(w, inputs, -1)
    assert info_s["fwd_tile_pairs"] == info_n["fwd_tile_pairs"]
    assert info_s["n_fwd_items"] >= info_n["n_fwd_items"]
    O, LSE = oracle.forward(oracle.Problem(w, q.cpu(), k.cpu(), v.cpu()))
    check_o(to64(o_s), O, "O (split)")
    check_lse(to64(l_s), LSE, "LSE (split)")
    assert np.array_equal(np.isinf(to64(l_s)), np.isinf(to64(l_n)))
    # each part rounds its bf16 P against its own row max, so split and unsplit
    # agree to the O tolerance, not bit for bit
    assert (o_s - o_n).abs().max().item() <= O_ATOL


@pytest.mark.parametrize("w", SMALL[-2:], ids=lambda w: w.name)
def test_decode_automatic_split_forward_backward(w):
    inputs = W.make_tensors(w, device="cuda")
    q, k, v, do = inputs
    info, o, lse, (dq, dk, dv) = forward(w, inputs, 0, o_dtype=ca.CA_DTYPE_BF16, backward=True)
    assert info["n_fwd_items"] > w.n_tasks * w.num_kv_heads  # the automatic rule split these
    _, o32, l32, _ = forward(w, inputs, 0)
    assert torch.equal(o.view(torch.int16), o32.to(torch.bfloat16).view(torch.int16))
    pb = oracle.Problem(w, q.cpu(), k.cpu(), v.cpu(), do.cpu())
    O, LSE = oracle.forward(pb)
    check_o(to64(o32), O)
    check_lse(to64(lse), LSE)
    dQ, dK, dV = oracle.backward(pb)
    check_grad(to64(dq), dQ, "dQ")
    check_grad(to64(dk), dK, "dK")
    check_grad(to64(dv), dV, "dV")


def test_decode_fullsize_split_vs_unsplit_and_sampled_rows():
    w = W.decode_batch(seed=0, n_seq=16, context=131072, q_len=1)
    inputs = W.make_tensors(w, device="cuda", need_grad_inputs=False)
    q, k, v, _ = inputs
    info_a, o_a, l_a, _ = forward(w, inputs, 0)
    info_n, o_n, l_n, _ = forward(w, inputs, -1)
    assert info_a["n_fwd_items"] > info_n["n_fwd_items"]
    assert (o_a - o_n).abs().max().item() <= O_ATOL
    assert ((l_a - l_n).abs() / l_n.abs().clamp(min=1)).max().item() <= LSE_RTOL
    rng = np.random.default_rng(7)
    rows, heads = rng.integers(0, w.total_q, 64), rng.integers(0, w.num_q_heads, 64)
    pb = oracle.Problem(w, q.cpu(), k.cpu(), v.cpu())
    O, LSE = oracle.forward_rows(pb, rows, heads)
    rt, ht = torch.as_tensor(rows, device="cuda"), torch.as_tensor(heads, device="cuda")
    check_o(to64(o_a[rt, ht]), O)
    check_lse(to64(l_a[rt, ht]), LSE)
