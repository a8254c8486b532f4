"""Element-wise parity at full workload sizes against the whole-document
oracle (oracle/dense.py), in the launch configuration bench.py times (bf16 O
for the backward; a float32-O forward for the O check):

  * the 64K Llama-8B-shaped chunk: every row (O, LSE, dQ) and every key column
    (dK, dV) of every kv head, checked per document;
  * the rebatched CA-task pool: every row and column of one kv head in its
    three longest documents (127K, 120K and 113K tokens, 15 shard tasks), so
    dK/dV accumulated over thousands of query tiles and over shard boundaries
    are compared column by column;
  * the 512K long-context chunk: the last 1024 key columns of its 262K
    document (each depends on ~1K rows that see up to 262K keys);
  * the three sparse-mask chunks: every row and column of one kv head,
    including every sink column and every window start.

Plus the composability check of the pool at full size: the 131,072-row shard
pool against one task per whole document over the same 16 documents (Efficient
Long-context Language Model Training by Core Attention Disaggregation, §3.4
"Property 2: Composability"): O and LSE of every pool row bit for bit, dQ and
the summed dK/dV (dO zero on rows outside the pool) within the gradient
tolerance.
"""
import os

import numpy as np
import pytest
import torch

import document_masked_core_gb300 as ca
import workloads as W
from oracle import dense
from parity import GRAD_RFRO, check_grad, check_lse, check_o, rel_fro

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    from document_masked_core_gb300 import build
    build.build()


def gpu_run(w, inputs, kv_split=None):
    """Forward (float32 O and bf16 O) and the backward on the bf16 O."""
    q, k, v, do = inputs
    out = {}
    for name, dt in (("f32", ca.CA_DTYPE_FP32), ("bf16", ca.CA_DTYPE_BF16)):
        plan = ca.Plan.from_workload(w, o_dtype=dt)
        if kv_split is not None:
            plan.set_kv_split(kv_split)
        ws = ca.workspace(plan)
        o, lse = ca.alloc_forward(plan)
        plan.forward(q, k, v, o, lse, ws)
        torch.cuda.synchronize()
        assert plan.device_status() == 0
        if name == "f32":
            out["o32"], out["lse32"] = o, lse
            del ws
            continue
        out["o16"], out["lse"] = o, lse
        if do is not None:
            dq, dk, dv = ca.alloc_backward(plan)
            plan.backward(q, k, v, o, lse, do, dq, dk, dv, ws)
            torch.cuda.synchronize()
            assert plan.device_status() == 0
            out["dq"], out["dk"], out["dv"] = dq, dk, dv
    assert torch.equal(out["lse"], out["lse32"])
    return out


def check_doc(w, res, gpu, doc, g, what):
    """Compare one (document, kv head) of the GPU results with the oracle's."""
    G = w.num_q_heads // w.num_kv_heads
    hs = slice(g * G, (g + 1) * G)
    for (r0, n), o, lse, dq in zip(res.rows, res.o, res.lse, res.dq):
        o_ref, l_ref = o.numpy(), lse.numpy()
        done = ~np.isnan(l_ref[:, 0])  # column mode leaves rows before its first column out
        if not done.any():
            continue
        r = slice(r0, r0 + n)
        o_gpu = gpu["o32"][r, hs].double().cpu().numpy()
        l_gpu = gpu["lse"][r, hs].double().cpu().numpy()
        check_o(o_gpu[done], o_ref[done], f"{what}: O")
        check_lse(l_gpu[done], l_ref[done], f"{what}: LSE")
        o16 = gpu["o16"][r, hs]
        assert torch.equal(o16.view(torch.int16), gpu["o32"][r, hs].to(torch.bfloat16).view(torch.int16))
        if dq is not None:
            check_grad(gpu["dq"][r, hs].double().cpu().numpy(), dq.numpy(), f"{what}: dQ")


def check_cols(w, res, gpu, doc, g, cols, what):
    off = int(w.doc_kv_offset[doc])
    kr = torch.as_tensor(off + np.asarray(cols), device="cuda")
    dk = gpu["dk"][kr, g].double().cpu().numpy()
    dv = gpu["dv"][kr, g].double().cpu().numpy()
    e_k = check_grad(dk, res.dk.numpy(), f"{what}: dK")
    e_v = check_grad(dv, res.dv.numpy(), f"{what}: dV")
    return e_k, e_v


def host_inputs(inputs):
    return tuple(None if x is None else x.cpu() for x in inputs)


# --------------------------------------------------------------- 64K chunk
@pytest.fixture(scope="module")
def llama8b():
    w = W.llama8b_chunk()
    inputs = W.make_tensors(w, device="cuda")
    gpu = gpu_run(w, inputs)
    return w, host_inputs(inputs), gpu


@pytest.mark.parametrize("g", range(8))
def test_llama8b_every_row_and_column(llama8b, g):
    w, (q, k, v, do), gpu = llama8b
    worst = 0.0
    for doc in range(w.n_docs):
        res = dense.document_group(w, q, k, v, do, doc, g)
        what = f"doc {doc} (len {int(w.doc_len[doc])}) kv head {g}"
        check_doc(w, res, gpu, doc, g, what)
        worst = max(worst, *check_cols(w, res, gpu, doc, g, np.arange(int(w.doc_len[doc])), what))
    print(f"kv head {g}: worst per-document dK/dV relative Frobenius error {worst:.2e}")


# --------------------------------------------------------------- rebatched pool
def test_pool_longest_documents_every_row_and_column():
    w = W.rebatched_pool()
    inputs = W.make_tensors(w, device="cuda")
    gpu = gpu_run(w, inputs)
    q, k, v, do = host_inputs(inputs)
    g = 5
    longest = [int(d) for d in np.argsort(-w.doc_len, kind="stable")[:3]]
    n_tasks = 0
    for doc in longest:
        res = dense.document_group(w, q, k, v, do, doc, g)
        n_tasks += len(res.rows)
        what = f"pool doc {doc} (len {int(w.doc_len[doc])}, {len(res.rows)} shards) kv head {g}"
        check_doc(w, res, gpu, doc, g, what)
        check_cols(w, res, gpu, doc, g, np.arange(int(w.doc_len[doc])), what)
    assert min(int(w.doc_len[d]) for d in longest) > 100_000 and n_tasks >= 10


def test_pool_sharded_equals_whole_documents():
    """The shard pool against one task per whole document, same documents,
    same K/V, the pool's Q/dO rows copied from the whole documents' rows."""
    w = W.rebatched_pool()
    whole = W.custom("pool_whole_documents", w.doc_len,
                     [(d, 0, int(L), 0, int(L)) for d, L in enumerate(w.doc_len)],
                     w.num_q_heads, w.num_kv_heads, w.head_dim, seed=w.seed, doc_kv_offset=w.doc_kv_offset)
    qw, k, v, dow = W.make_tensors(whole, device="cuda")
    # pool row r of task t = whole row (row0 of its document) + q_start + i
    wrow0 = whole.task_row_offset()
    src = np.concatenate([wrow0[int(d)] + int(s) + np.arange(int(n))
                          for d, s, n in zip(w.task_doc, w.task_q_start, w.task_q_len)])
    src_t = torch.as_tensor(src, device="cuda")
    q = qw[src_t].contiguous()
    do = dow[src_t].contiguous()
    keep = torch.zeros(whole.total_q, dtype=torch.bool, device="cuda")
    keep[src_t] = True
    dow[~keep] = 0  # rows outside the pool add nothing to dK/dV
    pool = gpu_run(w, (q, k, v, do), kv_split=-1)
    full = gpu_run(whole, (qw, k, v, dow), kv_split=-1)
    assert torch.equal(pool["lse"], full["lse"][src_t])
    assert torch.equal(pool["o16"].view(torch.int16), full["o16"][src_t].view(torch.int16))
    assert torch.equal(pool["o32"], full["o32"][src_t])
    e_q = rel_fro(pool["dq"].double().cpu().numpy(), full["dq"][src_t].double().cpu().numpy())
    assert e_q <= GRAD_RFRO
    inside = torch.zeros(w.total_kv, dtype=torch.bool, device="cuda")
    for off, L in zip(w.doc_kv_offset, w.doc_len):
        inside[int(off):int(off + L)] = True
    for name in ("dk", "dv"):
        e = rel_fro(pool[name][inside].double().cpu().numpy(), full[name][inside].double().cpu().numpy())
        assert e <= GRAD_RFRO, f"{name}: {e:.3e}"
    print(f"pool vs whole documents: dQ {e_q:.2e}")


# --------------------------------------------------------------- 512K chunk
def test_long_chunk_last_columns_of_262k_document():
    w = W.long_context_chunk()
    inputs = W.make_tensors(w, device="cuda")
    gpu = gpu_run(w, inputs)
    q, k, v, do = host_inputs(inputs)
    doc = int(np.argmax(w.doc_len))
    L = int(w.doc_len[doc])
    assert L == 262144
    g = 3
    cols = np.arange(L - 1024, L)
    res = dense.document_group(w, q, k, v, do, doc, g, columns=cols)
    what = f"long chunk doc {doc} (len {L}) kv head {g}, last 1024 columns"
    check_doc(w, res, gpu, doc, g, what)
    check_cols(w, res, gpu, doc, g, cols, what)


# --------------------------------------------------------------- sparse masks
@pytest.mark.parametrize("name", list(W.MASKED_WORKLOADS))
def test_masked_chunk_every_row_and_column(name):
    w = W.MASKED_WORKLOADS[name]()
    inputs = W.make_tensors(w, device="cuda")
    gpu = gpu_run(w, inputs)
    q, k, v, do = host_inputs(inputs)
    g = 6
    for doc in range(w.n_docs):
        res = dense.document_group(w, q, k, v, do, doc, g)
        what = f"{name} doc {doc} (len {int(w.doc_len[doc])}) kv head {g}"
        check_doc(w, res, gpu, doc, g, what)
        check_cols(w, res, gpu, doc, g, np.arange(int(w.doc_len[doc])), what)


@pytest.mark.skipif(os.environ.get("CA_LONG_PARITY") != "1",
                    reason="about 23 minutes of oracle time on 16 host cores: run with CA_LONG_PARITY=1")
def test_long_chunk_early_columns_of_262k_document():
    """The 262K document's earliest key columns (each depends on every later
    row, 262K rows seeing up to 262K keys, one kv head) and stratified
    columns across the document, element-wise against the oracle."""
    w = W.long_context_chunk()
    inputs = W.make_tensors(w, device="cuda")
    gpu = gpu_run(w, inputs)
    q, k, v, do = host_inputs(inputs)
    doc = int(np.argmax(w.doc_len))
    L = int(w.doc_len[doc])
    g = 5
    rng = np.random.default_rng(w.seed + 3000)
    cols = np.unique(np.concatenate([np.arange(0, 128), np.arange(128, L, 4096), rng.integers(0, L, 256)]))
    res = dense.document_group(w, q, k, v, do, doc, g, columns=cols)
    what = f"long chunk doc {doc} (len {L}) kv head {g}, {len(cols)} columns from 0"
    check_doc(w, res, gpu, doc, g, what)
    e_k, e_v = check_cols(w, res, gpu, doc, g, cols, what)
    print(f"{what}: dK {e_k:.2e}, dV {e_v:.2e}")
