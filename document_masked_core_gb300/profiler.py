"""Profiler of the cost model ("Efficient Long-context Language Model Training
by Core Attention Disaggregation", "The Profiler and Cost Model"): measures
fwd+bwd time of CA-tasks on a grid of (query length n_q, context length n_kv)
with this library's own kernels, and builds the interpolating cost model
(``capi.Profile``) the scheduler's loads are predicted with.

A grid point is measured as a rebatched launch of m identical CA-tasks (each a
query shard of n_q tokens ending at position n_kv of its own document; m as
large as a query-token and a context-token budget allow), the way the
scheduler's shards run; its time is the launch's fwd+bwd time divided by m.
Where n_q > n_kv the point is the whole-document task n_q = n_kv.

Run on a GPU:  python -m document_masked_core_gb300.profiler --out PATH.json
"""
from __future__ import annotations

import argparse
import json
import time

import numpy as np

from . import capi

NQ_GRID = [128, 256, 512, 1024, 2048, 4096, 8192, 16384]
NKV_GRID = [128, 256, 512, 1024, 2048, 4096, 8192, 16384, 32768, 65536]


def _launch_time(doc_len, tasks, hq, hkv, d, reps, warmup):
    """Median fwd+bwd seconds of one launch over ``tasks`` (CUDA events)."""
    import torch
    from . import alloc_backward, alloc_forward, workspace
    off = np.concatenate([[0], np.cumsum(doc_len)[:-1]]).astype(np.int64)
    t = np.asarray(tasks, dtype=np.int64)
    plan = capi.Plan(t[:, 0], t[:, 1], t[:, 2], t[:, 3], t[:, 4], doc_len, off, hq, hkv, d)
    info = plan.info()
    g = torch.Generator(device="cuda").manual_seed(1234)
    q = torch.randn((info["total_q"], hq, d), generator=g, device="cuda").to(torch.bfloat16)
    k = torch.randn((info["total_kv"], hkv, d), generator=g, device="cuda").to(torch.bfloat16)
    v = torch.randn((info["total_kv"], hkv, d), generator=g, device="cuda").to(torch.bfloat16)
    do = torch.randn((info["total_q"], hq, d), generator=g, device="cuda").to(torch.bfloat16)
    ws = workspace(plan)
    o, lse = alloc_forward(plan)
    dq, dk, dv = alloc_backward(plan)
    times = []
    for r in range(warmup + reps):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        plan.forward(q, k, v, o, lse, ws)
        plan.backward(q, k, v, o, lse, do, dq, dk, dv, ws)
        e1.record()
        e1.synchronize()
        if r >= warmup:
            times.append(e0.elapsed_time(e1) / 1e3)
    if plan.device_status() != 0:
        raise RuntimeError("device error during profiling")
    plan.close()
    return float(np.median(times))


def measure(hq=32, hkv=8, d=128, nq_grid=NQ_GRID, nkv_grid=NKV_GRID, q_budget=32768, kv_budget=1 << 20,
            reps=5, warmup=2):
    """Measured grid: dict with nq_grid, nkv_grid, seconds[i][j], flops_per_pair."""
    sec = [[0.0] * len(nkv_grid) for _ in nq_grid]
    for i, nq in enumerate(nq_grid):
        for j, nkv in enumerate(nkv_grid):
            q = min(nq, nkv)
            m = max(1, min(q_budget // q, kv_budget // nkv))
            tasks = [(t, nkv - q, q, 0, nkv) for t in range(m)]
            sec[i][j] = _launch_time(np.full(m, nkv, dtype=np.int64), tasks, hq, hkv, d, reps, warmup) / m
    return {"nq_grid": list(nq_grid), "nkv_grid": list(nkv_grid), "seconds": sec,
            "flops_per_pair": 12.0 * d * hq, "shape": {"num_q_heads": hq, "num_kv_heads": hkv, "head_dim": d},
            "how": f"rebatched launch of identical CA-tasks, q budget {q_budget} tokens, kv budget {kv_budget} "
                   f"tokens, median of {reps} fwd+bwd launches after {warmup} warm-up (CUDA events)"}


def load_profile(grid: dict) -> capi.Profile:
    return capi.Profile(grid["nq_grid"], grid["nkv_grid"], grid["seconds"], grid["flops_per_pair"])


def report(grid: dict, doc_sets: dict, servers=(2, 4, 8), hq=32, hkv=8, d=128, reps=3, warmup=1):
    """For each document set and server count: the schedule (host time,
    balance before and after, bytes moved) and every server's fwd+bwd time,
    predicted by the cost model and measured by running the server's shards
    as one launch on this GPU (the servers run one after another)."""
    prof = load_profile(grid)
    bq, bkv = float(hq * d * 2), float(2 * hkv * d * 2)
    rows = []
    for name, docs in doc_sets.items():
        docs = [int(x) for x in docs]
        for k in servers:
            t0 = time.perf_counter()
            tasks, res = capi.schedule(docs, k, bq, bkv, tolerance=0.01)
            host_ms = (time.perf_counter() - t0) * 1e3
            # balance before: the devices that hold the tokens compute their own
            T = -(-sum(docs) // k)
            before = [0] * k
            off = 0
            for L in docs:
                pos = off
                while pos < off + L:
                    s = min(pos // T, k - 1)
                    stop = min(off + L, (s + 1) * T)
                    a, b = pos - off, stop - off
                    before[s] += b * (b + 1) // 2 - a * (a + 1) // 2
                    pos = stop
                off += L
            pred, meas = [], []
            for s in range(k):
                mine = [t for t in tasks if t["server"] == s]
                pred.append(sum(prof.predict(int(t["q_len"]), int(t["kv_len"])) for t in mine))
                tl = [(int(t["doc_id"]), int(t["q_start"]), int(t["q_len"]), 0, int(t["kv_len"])) for t in mine]
                meas.append(_launch_time(np.asarray(docs, dtype=np.int64), tl, hq, hkv, d, reps, warmup))
            mean = sum(before) / k
            rows.append({"docs": name, "servers": k, "host_ms": host_ms, "n_tasks": res["n_tasks"],
                         "splits": res["n_splits"], "migrations": res["n_migrations"],
                         "comm_MB": res["comm_bytes"] / 1e6, "imbalance_before": max(before) / mean,
                         "imbalance_after": res["max_load"] / mean,
                         "pred_ms": [x * 1e3 for x in pred], "meas_ms": [x * 1e3 for x in meas],
                         "pred_err_max": max(abs(p_ - m_) / m_ for p_, m_ in zip(pred, meas))})
    return rows


SHARD_LENGTHS = [8, 16, 32, 64, 128, 256, 512, 1024, 2048, 4096]


def sweep_shard_lengths(lengths=SHARD_LENGTHS, total_q=32768, n_docs=16, doc_len=32768, hq=32, hkv=8, d=128,
                        reps=5, warmup=2, seed=0):
    """Throughput of one rebatched launch of total_q query tokens made of shards
    of one length s, each placed at a uniformly random position of one of
    n_docs documents of doc_len tokens (so contexts vary from s to doc_len),
    for every s (the composability measurement of "Efficient Long-context
    Language Model Training by Core Attention Disaggregation", "Property 2:
    Composability", Figure 5).  TFLOP/s over 12*d*H_q*causal pairs."""
    rng = np.random.default_rng(seed)
    docs = np.full(n_docs, doc_len, dtype=np.int64)
    rows = []
    for s in lengths:
        m = total_q // s
        tasks = []
        for t in range(m):
            q0 = int(rng.integers(0, doc_len - s + 1))
            tasks.append((t % n_docs, q0, s, 0, q0 + s))
        pairs = sum(s * (q0 + s) - s * (s - 1) // 2 for _, q0, _, _, _ in tasks)
        sec = _launch_time(docs, tasks, hq, hkv, d, reps, warmup)
        rows.append({"shard_tokens": s, "shards": m, "causal_pairs": pairs, "fwd_bwd_ms": sec * 1e3,
                     "tflops": 12.0 * d * hq * pairs / sec / 1e12})
    return rows


def rank_balance(doc_sets: dict, ranks=(2, 4, 8)):
    """Max / mean causal pairs per rank: contiguous token ranges of the whole
    chunk vs the 2N-chunk shards of every document."""
    out = []
    for name, docs in doc_sets.items():
        docs = [int(x) for x in docs]
        total = sum(docs)
        for n in ranks:
            T = -(-total // n)
            cont = [0] * n
            off = 0
            for L in docs:
                pos = off
                while pos < off + L:
                    r = min(pos // T, n - 1)
                    stop = min(off + L, (r + 1) * T)
                    a, b = pos - off, stop - off
                    cont[r] += b * (b + 1) // 2 - a * (a + 1) // 2
                    pos = stop
                off += L
            two = [0] * n
            for t in capi.shard_2n(docs, n):
                two[int(t["server"])] += int(t["pairs"])
            out.append({"docs": name, "ranks": n, "contiguous": max(cont) / (sum(cont) / n),
                        "two_n_chunk": max(two) / (sum(two) / n)})
    return out


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__)
    ap.add_argument("--out", help="grid JSON to write (or read with --report-only)")
    ap.add_argument("--hq", type=int, default=32)
    ap.add_argument("--hkv", type=int, default=8)
    ap.add_argument("--head-dim", type=int, default=128)
    ap.add_argument("--report", help="also schedule the bench's document sets and write this JSON")
    ap.add_argument("--report-only", action="store_true", help="read the grid from --out instead of measuring")
    ap.add_argument("--sweep", help="measure throughput vs shard length and write this JSON (no grid)")
    a = ap.parse_args(argv)
    if a.sweep:
        import workloads as W
        rows = sweep_shard_lengths(hq=a.hq, hkv=a.hkv, d=a.head_dim)
        bal = rank_balance({"llama8b_chunk_64k": W.llama8b_chunk(seed=0).doc_len,
                            "pool_16_docs": W.rebatched_pool().doc_len,
                            "long_chunk_512k": W.long_context_chunk().doc_len})
        with open(a.sweep, "w") as f:
            json.dump({"sweep": rows, "rank_balance": bal}, f, indent=1)
        for r in rows + bal:
            print(json.dumps({k: (round(v, 4) if isinstance(v, float) else v) for k, v in r.items()}))
        return
    if a.report_only:
        with open(a.out) as f:
            grid = json.load(f)
    else:
        t0 = time.time()
        grid = measure(a.hq, a.hkv, a.head_dim)
        grid["measure_seconds"] = time.time() - t0
        with open(a.out, "w") as f:
            json.dump(grid, f, indent=1)
    prof = load_profile(grid)
    print(json.dumps({"grid": a.out, "peak_tflops": prof.peak() / 1e12, "seconds": grid.get("measure_seconds")}))
    if a.report:
        import workloads as W
        sets = {"llama8b_chunk_64k": W.llama8b_chunk(seed=0).doc_len,
                "pool_16_docs": W.rebatched_pool().doc_len,
                "long_chunk_512k": W.long_context_chunk().doc_len}
        rows = report(grid, sets, hq=a.hq, hkv=a.hkv, d=a.head_dim)
        with open(a.report, "w") as f:
            json.dump(rows, f, indent=1)
        for r in rows:
            print(json.dumps({k: (round(v, 4) if isinstance(v, float) else v) for k, v in r.items()
                              if k not in ("pred_ms", "meas_ms")}))


if __name__ == "__main__":
    main()
