"""The scheduler's shards and the 2N-chunk shards run on simulated attention
servers / ranks (one after another on this GPU): per server one rebatched
launch of its CA-tasks, query
rows gathered from the devices that hold them.  The forward rows equal the
one-task-per-document launch bit for bit (key tiles sit at document
coordinates); dQ rows and the dK / dV partials summed over servers match it
within the gradient tolerance.  The cost model built from a measured grid
reproduces its grid points and predicts each server's time to within a
factor of two."""
import numpy as np
import pytest
import torch

import document_masked_core_gb300 as ca
from document_masked_core_gb300 import capi, profiler
import workloads as W
from parity import GRAD_RFRO

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    from document_masked_core_gb300 import build
    build.build()


def rfro(x, ref):
    x, ref = x.double(), ref.double()
    return float((x - ref).norm() / ref.norm().clamp(min=1e-30))


def run_plan(w, q, k, v, do, o_dtype):
    plan = ca.Plan.from_workload(w, o_dtype=o_dtype)
    ws = ca.workspace(plan)
    o, lse = ca.alloc_forward(plan)
    plan.forward(q, k, v, o, lse, ws)
    dq, dk, dv = ca.alloc_backward(plan)
    plan.backward(q, k, v, o, lse, do, dq, dk, dv, ws)
    torch.cuda.synchronize()
    assert plan.device_status() == 0
    return o, lse, dq, dk, dv


def check_servers(docs, tasks, k, hq=32, hkv=8, d=128, seed=9):
    """Run every server's tasks as one launch and compare with the
    one-task-per-document launch."""
    whole = W.custom("whole", docs, [(i, 0, int(L), 0, int(L)) for i, L in enumerate(docs)], hq=hq, hkv=hkv, d=d,
                     seed=seed)
    q, kk, v, do = W.make_tensors(whole, device="cuda")
    ow, lw, _, _, _ = run_plan(whole, q, kk, v, do, ca.CA_DTYPE_FP32)
    _, _, dqw16, dkw16, dvw16 = run_plan(whole, q, kk, v, do, ca.CA_DTYPE_BF16)
    dk_sum = torch.zeros_like(dkw16, dtype=torch.float32)
    dv_sum = torch.zeros_like(dvw16, dtype=torch.float32)
    for s in range(k):
        mine = [t for t in tasks if t["server"] == s]
        assert mine, "every server gets work"
        ws_ = W.custom(f"server{s}", docs, [(int(t["doc_id"]), int(t["q_start"]), int(t["q_len"]), 0,
                                              int(t["kv_len"])) for t in mine], hq=hq, hkv=hkv, d=d, seed=seed)
        rows = torch.as_tensor(np.concatenate([int(whole.doc_kv_offset[int(t["doc_id"])]) +
                                               np.arange(int(t["q_start"]), int(t["q_start"] + t["q_len"]))
                                               for t in mine]), device="cuda")
        qs, dos = q[rows].contiguous(), do[rows].contiguous()
        os_, ls, _, _, _ = run_plan(ws_, qs, kk, v, dos, ca.CA_DTYPE_FP32)
        assert torch.equal(os_, ow[rows]) and torch.equal(ls, lw[rows])
        _, _, dqs, dks, dvs = run_plan(ws_, qs, kk, v, dos, ca.CA_DTYPE_BF16)
        assert rfro(dqs, dqw16[rows]) <= GRAD_RFRO / 4
        dk_sum += dks.float()
        dv_sum += dvs.float()
    assert rfro(dk_sum, dkw16) <= GRAD_RFRO / 4
    assert rfro(dv_sum, dvw16) <= GRAD_RFRO / 4


@pytest.mark.parametrize("k,min_shard", [(4, 0), (3, 128)])
def test_scheduled_servers_equal_unsharded(k, min_shard):
    docs = W.llama8b_chunk(seed=2, total=16384).doc_len
    tasks, _ = capi.schedule(docs, k, 32 * 128 * 2.0, 2 * 8 * 128 * 2.0, tolerance=0.01, min_shard_tokens=min_shard)
    check_servers(docs, tasks, k)


@pytest.mark.parametrize("n_ranks", [2, 4])
def test_2n_chunk_ranks_equal_unsharded(n_ranks):
    docs = W.llama8b_chunk(seed=4, total=16384).doc_len
    check_servers(docs, capi.shard_2n(docs, n_ranks), n_ranks)


def test_cost_model_from_a_measured_grid():
    grid = profiler.measure(nq_grid=[128, 512, 2048], nkv_grid=[512, 2048, 8192], q_budget=8192,
                            kv_budget=1 << 18, reps=3, warmup=1)
    prof = profiler.load_profile(grid)
    assert prof.peak() > 1e14
    for i, nq in enumerate(grid["nq_grid"]):
        for j, nkv in enumerate(grid["nkv_grid"]):
            if nq <= nkv:
                assert prof.predict(nq, nkv) == pytest.approx(grid["seconds"][i][j], rel=1e-12)
    docs = [int(x) for x in W.llama8b_chunk(seed=2, total=16384).doc_len]
    rows = profiler.report(grid, {"chunk16k": docs}, servers=(2,), reps=2, warmup=1)
    for p_, m_ in zip(rows[0]["pred_ms"], rows[0]["meas_ms"]):
        assert 0.5 * m_ <= p_ <= 2.0 * m_, (p_, m_)
