"""GPU parity of ca_merge (Eq. 4 of the merge appendix) against the oracle's
merge, and the device watchdog self-test."""
import numpy as np
import pytest
import torch

import document_masked_core_gb300 as ca
import oracle
import workloads as W
from parity import check_lse, check_o, to64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    from document_masked_core_gb300 import build
    build.build()


@pytest.mark.parametrize("n,rows,heads,d", [(1, 7, 3, 64), (8, 333, 4, 128), (3, 50, 2, 8), (16, 64, 1, 256)])
@pytest.mark.parametrize("parts_dtype,out_dtype", [(ca.CA_DTYPE_FP32, ca.CA_DTYPE_FP32),
                                                   (ca.CA_DTYPE_BF16, ca.CA_DTYPE_FP32),
                                                   (ca.CA_DTYPE_FP32, ca.CA_DTYPE_BF16)])
def test_merge_matches_oracle(n, rows, heads, d, parts_dtype, out_dtype):
    g = torch.Generator(device="cuda").manual_seed(n * 1000 + rows)
    pdt = torch.float32 if parts_dtype == ca.CA_DTYPE_FP32 else torch.bfloat16
    o = [torch.randn((rows, heads, d), generator=g, device="cuda").to(pdt) for _ in range(n)]
    lse = [torch.randn((rows, heads), generator=g, device="cuda") * 3 for _ in range(n)]
    # empty parts (LSE = -inf): a few per part, and rows where every part is empty
    for s in range(n):
        lse[s][(torch.arange(rows, device="cuda") % (s + 2)) == 0] = float("-inf")
    for s in range(n):
        lse[s][rows // 2] = float("-inf")
    odt = torch.float32 if out_dtype == ca.CA_DTYPE_FP32 else torch.bfloat16
    out = torch.full((rows, heads, d), float("nan"), dtype=odt, device="cuda")
    lse_out = torch.empty((rows, heads), device="cuda")
    ca.merge(o, lse, rows, heads, d, out, lse_out, parts_dtype=parts_dtype, out_dtype=out_dtype)
    torch.cuda.synchronize()
    O, L = oracle.merge(np.stack([to64(x).reshape(rows * heads, d) for x in o]),
                        np.stack([to64(x).reshape(-1) for x in lse]))
    got = to64(out).reshape(rows * heads, d)
    if out_dtype == ca.CA_DTYPE_FP32:
        check_o(got, O, "merged O")
    else:  # bf16 output: half an ulp of |O| on top of the tolerance
        assert np.all(np.abs(got - O) <= 1e-2 + np.abs(O) * 2.0 ** -8)
    check_lse(to64(lse_out).reshape(-1), L, "merged LSE")
    assert np.all(got[~np.isfinite(L)] == 0)


def test_merge_rejects_bad_arguments():
    t = torch.zeros((4, 1, 64), device="cuda")
    l = torch.zeros((4, 1), device="cuda")
    with pytest.raises(ca.CAError):
        ca.merge([t] * 65, [l] * 65, 4, 1, 64, t)          # too many parts
    with pytest.raises(ca.CAError):
        ca.merge([t], [l], 4, 1, 60, t)                      # head_dim not a multiple of 8


def test_watchdog_reports_timeout_and_context_survives():
    w = W.tiny_chunk()
    plan = ca.Plan.from_workload(w, o_dtype=ca.CA_DTYPE_FP32)
    plan.watchdog_selftest(5_000_000)  # 5 ms wait on a barrier nothing arrives on
    assert plan.device_status() == ca.capi.CA_ERR_DEVICE_TIMEOUT
    assert plan.device_status() == 0  # the word is cleared on read
    # the context is still usable: a normal forward runs and is correct
    q, k, v, _ = W.make_tensors(w, device="cuda", need_grad_inputs=False)
    o, lse = ca.alloc_forward(plan)
    plan.forward(q, k, v, o, lse, ca.workspace(plan))
    torch.cuda.synchronize()
    assert plan.device_status() == 0
    O, LSE = oracle.forward(oracle.Problem(w, q.cpu(), k.cpu(), v.cpu()))
    check_o(to64(o), O)
