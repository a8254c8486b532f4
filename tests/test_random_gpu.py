"""GPU parity on seeded random CA-task pools against the fp64 oracle: forward
(float32 O element by element, LSE, bf16 O = RNE of float32 O), backward
(dQ, dK, dV), the forward with its items cut into parts of 1 and 2 key tiles
(in-launch split-KV and merge) and, where it applies, the CTA-pair backward
(dK, dV bit for bit with the one-CTA kernel).  The pools mix what the fixed cases test one at a
time: G from 1 to 128, head_dim 64 and 128, shards in random order, rows no
task asks for, KV blocks starting past 0 or ending before a shard's rows,
gaps between documents in K/V, and random (sink, lo, window) masks."""
import numpy as np
import pytest
import torch

import document_masked_core_gb300 as ca
import oracle
import workloads as W
from cases import random_pool
from parity import O_ATOL, check_grad, check_lse, check_o, rel_fro, to64

pytestmark = pytest.mark.gpu

# A sliding window over a KV block that ends before the shard's last rows:
# rows past kv_end + window - 2 see only the sink, so a query tile's last row
# sees fewer key tiles than the rows before it (the forward must visit the
# furthest key tile of any row, not of the last row).
WINDOW_PAST_KV_END = W.custom("window_past_kv_end", [9, 594, 253],
                              [(0, 0, 9, 0, 9), (1, 0, 594, 283, 311), (2, 30, 223, 0, 172)],
                              hq=8, hkv=1, d=64, seed=31, doc_kv_offset=[35, 48, 657],
                              masks=[(0, 6, 1), (132, 0, 0), (36, 0, 34)])
WINDOW_PAST_KV_END_D128 = W.custom("window_past_kv_end_g4_d128", [700],
                                   [(0, 0, 700, 0, 300), (0, 100, 600, 64, 400)],
                                   hq=16, hkv=4, d=128, seed=32, masks=[(10, 0, 90), (0, 200, 150)])

CASES = [WINDOW_PAST_KV_END, WINDOW_PAST_KV_END_D128] + [random_pool(s) for s in range(24)]


@pytest.fixture(scope="module", autouse=True)
def built():
    from document_masked_core_gb300 import build
    build.build()


def doc_rows(w):
    rows = np.zeros(w.total_kv, dtype=bool)
    for off, L in zip(w.doc_kv_offset, w.doc_len):
        rows[int(off):int(off + L)] = True
    return rows


def pair_applies(w):
    return w.head_dim == 128 and 64 % (w.num_q_heads // w.num_kv_heads) == 0


@pytest.mark.parametrize("w", CASES, ids=lambda w: w.name)
def test_random_pool_matches_oracle(w):
    q, k, v, do = W.make_tensors(w, device="cuda")
    torch.cuda.synchronize()
    pb = oracle.Problem(w, q.cpu(), k.cpu(), v.cpu(), do.cpu())
    O, LSE = oracle.forward(pb)
    dQ, dK, dV = oracle.backward(pb)
    inside = doc_rows(w)

    plan32 = ca.Plan.from_workload(w, o_dtype=ca.CA_DTYPE_FP32)
    ws = ca.workspace(plan32)
    o32, lse = ca.alloc_forward(plan32)
    o32.fill_(float("nan"))
    plan32.forward(q, k, v, o32, lse, ws)
    torch.cuda.synchronize()
    assert plan32.device_status() == 0
    check_o(to64(o32), O)
    check_lse(to64(lse), LSE)

    plan = ca.Plan.from_workload(w)
    o16, lse16 = ca.alloc_forward(plan)
    plan.forward(q, k, v, o16, lse16, ws)
    torch.cuda.synchronize()
    assert torch.equal(o16.view(torch.int16), o32.to(torch.bfloat16).view(torch.int16))
    assert torch.equal(lse16, lse)

    kinds = [ca.capi.CA_BWD_KERNEL_SINGLE] + ([ca.capi.CA_BWD_KERNEL_PAIR] if pair_applies(w) else [])
    out = {}
    for kind in kinds:
        plan.set_backward_kernel(kind)
        dq, dk, dv = ca.alloc_backward(plan)
        dq.fill_(float("nan"))
        dk.fill_(7.0)
        dv.fill_(7.0)
        plan.backward(q, k, v, o16, lse16, do, dq, dk, dv, ws)
        torch.cuda.synchronize()
        assert plan.device_status() == 0
        check_grad(to64(dq), dQ, "dQ")
        check_grad(to64(dk)[inside], dK[inside], "dK")
        check_grad(to64(dv)[inside], dV[inside], "dV")
        assert np.all(to64(dk)[~inside] == 7.0) and np.all(to64(dv)[~inside] == 7.0)
        out[kind] = (dq, dk, dv)
    if len(out) == 2:
        s, p = out[kinds[0]], out[kinds[1]]
        assert torch.equal(s[1], p[1]) and torch.equal(s[2], p[2])
        assert rel_fro(to64(p[0]), to64(s[0])) <= 1e-4


@pytest.mark.parametrize("w", CASES, ids=lambda w: w.name)
@pytest.mark.parametrize("split", [1, 2])
def test_random_pool_split_forward_matches_oracle(w, split):
    """Every item cut into parts of `split` key tiles, merged in the launch."""
    q, k, v, _ = W.make_tensors(w, device="cuda", need_grad_inputs=False)
    torch.cuda.synchronize()
    O, LSE = oracle.forward(oracle.Problem(w, q.cpu(), k.cpu(), v.cpu()))
    res = {}
    for kv_split in (split, -1):
        plan = ca.Plan.from_workload(w, o_dtype=ca.CA_DTYPE_FP32)
        plan.set_kv_split(kv_split)
        ws = ca.workspace(plan)
        o, lse = ca.alloc_forward(plan)
        o.fill_(float("nan"))
        plan.forward(q, k, v, o, lse, ws)
        torch.cuda.synchronize()
        assert plan.device_status() == 0
        res[kv_split] = (plan.info(), o, lse)
    info_s, o_s, l_s = res[split]
    info_n, o_n, l_n = res[-1]
    assert info_s["fwd_tile_pairs"] == info_n["fwd_tile_pairs"]
    check_o(to64(o_s), O, "O (split)")
    check_lse(to64(l_s), LSE, "LSE (split)")
    assert (o_s - o_n).abs().max().item() <= O_ATOL
