"""GPU parity of ca_forward against the fp64 oracle (element by element)."""
import numpy as np
import pytest
import torch

import document_masked_core_gb300 as ca
import oracle
import workloads as W
from cases import EDGE
from parity import check_lse, check_o, to64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    from document_masked_core_gb300 import build
    build.build()


def run_forward(w, o_dtype, inputs=None):
    if inputs is None:
        inputs = W.make_tensors(w, device="cuda", need_grad_inputs=False)
    q, k, v, _ = inputs
    plan = ca.Plan.from_workload(w, o_dtype=o_dtype)
    o, lse = ca.alloc_forward(plan)
    o.fill_(float("nan"))
    lse.fill_(float("nan"))
    ws = ca.workspace(plan)
    plan.forward(q, k, v, o, lse, ws)
    torch.cuda.synchronize()
    assert plan.device_status() == 0
    return plan, (q, k, v), o, lse


@pytest.mark.parametrize("w", [W.tiny_chunk()] + EDGE, ids=lambda w: w.name)
def test_forward_matches_oracle(w):
    plan, (q, k, v), o32, lse = run_forward(w, ca.CA_DTYPE_FP32)
    O, LSE = oracle.forward(oracle.Problem(w, q.cpu(), k.cpu(), v.cpu()))
    check_o(to64(o32), O)
    check_lse(to64(lse), LSE)
    # empty rows: O = 0
    empty = ~np.isfinite(LSE)
    assert np.all(to64(o32)[empty] == 0.0)
    # bf16 output = round-to-nearest-even of the float32 output
    _, _, o16, lse16 = run_forward(w, ca.CA_DTYPE_BF16, inputs=(q, k, v, None))
    assert torch.equal(o16.view(torch.int16), o32.to(torch.bfloat16).view(torch.int16))
    assert torch.equal(lse16, lse)


def test_forward_is_deterministic():
    w = EDGE[1]
    _, inp, o1, l1 = run_forward(w, ca.CA_DTYPE_FP32)
    _, _, o2, l2 = run_forward(w, ca.CA_DTYPE_FP32, inputs=inp + (None,))
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_sharded_equals_unsharded_on_gpu():
    """Composability: rebatched shards of a document give exactly the rows of
    the one-task-per-document launch (key tiles sit at document coordinates)."""
    w = W.rebatched_pool(seed=6, n_docs=4, doc_lo=600, doc_hi=1100, shard_lo=40, shard_hi=300, total_q=2000,
                         hq=8, hkv=2, d=128)
    whole = W.custom("whole", w.doc_len, [(i, 0, int(l), 0, int(l)) for i, l in enumerate(w.doc_len)],
                     hq=8, hkv=2, d=128, seed=6)
    qw, k, v, _ = W.make_tensors(whole, device="cuda", need_grad_inputs=False)
    rows = np.concatenate([int(whole.doc_kv_offset[d]) + np.arange(q0, q0 + ql)
                           for d, q0, ql in zip(w.task_doc, w.task_q_start, w.task_q_len)])
    rows_t = torch.as_tensor(rows, device="cuda")
    _, _, ow, lw = run_forward(whole, ca.CA_DTYPE_FP32, inputs=(qw, k, v, None))
    _, _, os_, ls = run_forward(w, ca.CA_DTYPE_FP32, inputs=(qw[rows_t].contiguous(), k, v, None))
    assert torch.equal(os_, ow[rows_t]) and torch.equal(ls, lw[rows_t])
