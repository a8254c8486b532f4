"""Oracle for the host planning steps (test infrastructure).

Only ``tests/`` may import this module; the product never does, and this
module imports nothing from the product.  Plain Python, written from
"Efficient Long-context Language Model Training by Core Attention
Disaggregation":

  * ``profile_predict``  -- "The Profiler and Cost Model": bilinear
    interpolation over the four grid points around (n_q, n_kv); beyond the
    grid, FLOPs / peak measured throughput.
  * ``optimal_shard``    -- "Appendix B: Optimal Shard Dimension Computation":
    minimise n_q*bytes_q + n_kv*bytes_kv subject to the work fraction
    n_q(2 n_kv - n_q) / (L_q(2 L_kv - L_q)) = alpha, by the appendix's closed
    form and its boundary rule; then the integer shard.
  * ``schedule``         -- "The Communication-Aware Greedy Scheduler", steps
    1 to 4, in the order the section gives them.
  * ``shard_2n``         -- "Context Parallelism for Scalable Million-Token
    Inference", §3.5.1: 2N chunks per sequence, rank i takes C_i and
    C_{2N-i-1} (padding not materialised: the last chunks are shorter).

Readings where the pages leave a step open (the same ones the library states
in include/ca_sched.h): work is counted in exact causal pairs; devices hold
consecutive equal token ranges of the document stream; a split takes the
sub-shard [n_kv - n_q, n_kv) and leaves up to two pieces; ties go to the
earliest Item; the integer shard rounds n_q to the nearest integer and then
takes the context length whose exact pair count is nearest the target.

Pins: ``tests/test_sched_cpu.py`` (brute-force minimisation of the split,
closed forms of the interpolation, a schedule worked by hand, invariants).
"""
from __future__ import annotations

import math


def pairs_of_range(a: int, b: int) -> int:
    """Causal pairs of query positions [a, b) that see the prefix [0, p]."""
    return sum(p + 1 for p in range(a, b)) if b - a < 64 else (b * (b + 1) - a * (a + 1)) // 2


def shard_pairs(n_q: int, n_kv: int) -> int:
    """Pairs of the n_q queries that end the context [0, n_kv)."""
    return pairs_of_range(n_kv - n_q, n_kv)


# ---------------------------------------------------------------- profiler

def profile_peak(nq_grid, nkv_grid, seconds, flops_per_pair):
    best = 0.0
    for i, nq in enumerate(nq_grid):
        for j, nkv in enumerate(nkv_grid):
            q = min(nq, nkv)
            best = max(best, shard_pairs(q, nkv) * flops_per_pair / seconds[i][j])
    return best


def _axis(grid, x):
    """Cell index i and fraction t in [0, 1] of x between grid[i], grid[i+1]."""
    if len(grid) == 1 or x <= grid[0]:
        return 0, 0.0
    i = 0
    while i + 1 < len(grid) and grid[i + 1] <= x:
        i += 1
    if i >= len(grid) - 1:
        i = len(grid) - 2
    return i, (x - grid[i]) / (grid[i + 1] - grid[i])


def profile_predict(nq_grid, nkv_grid, seconds, flops_per_pair, n_q, n_kv):
    assert 1 <= n_q <= n_kv
    if n_q > nq_grid[-1] or n_kv > nkv_grid[-1]:
        return shard_pairs(n_q, n_kv) * flops_per_pair / profile_peak(nq_grid, nkv_grid, seconds, flops_per_pair)
    i, tq = _axis(nq_grid, n_q)
    j, tk = _axis(nkv_grid, n_kv)
    i1 = min(i + 1, len(nq_grid) - 1)
    j1 = min(j + 1, len(nkv_grid) - 1)
    lo = (1 - tk) * seconds[i][j] + tk * seconds[i][j1]
    hi = (1 - tk) * seconds[i1][j] + tk * seconds[i1][j1]
    return (1 - tq) * lo + tq * hi


# ---------------------------------------------------------------- Appendix B

def optimal_shard_real(L_q, L_kv, alpha, bytes_q, bytes_kv):
    """Continuous optimum n_q of the split and the feasible interval."""
    beta = bytes_kv / bytes_q
    A = alpha * L_q * (2 * L_kv - L_q)
    n_opt = math.sqrt(alpha * beta * L_q * (2 * L_kv - L_q) / (beta + 2))
    # feasibility: n_kv = (A/n_q + n_q)/2 within [n_q + L_kv - L_q, L_kv], n_q <= L_q
    c = L_kv - L_q
    lo = A / (L_kv + math.sqrt(max(L_kv * L_kv - A, 0.0)))
    hi = min(L_q, A / (math.sqrt(c * c + A) + c))
    return min(max(n_opt, lo), max(hi, lo)), lo, hi


def optimal_shard(L_q, L_kv, alpha, target_pairs, bytes_q, bytes_kv):
    n_real, _, _ = optimal_shard_real(L_q, L_kv, alpha, bytes_q, bytes_kv)
    n_q = int(math.floor(n_real + 0.5))
    n_q = min(max(n_q, 1), L_q)
    lo_kv, hi_kv = n_q + L_kv - L_q, L_kv
    best = None
    for n_kv in range(lo_kv, hi_kv + 1):  # brute force over the feasible context lengths
        gap = abs(shard_pairs(n_q, n_kv) - target_pairs)
        if best is None or gap < best[0]:
            best = (gap, n_kv)
    return n_q, best[1], n_real


# ---------------------------------------------------------------- greedy scheduler

def initial_items(doc_len, k):
    """Items of the devices that hold the tokens: device s holds [sT, (s+1)T)."""
    total = sum(doc_len)
    T = -(-total // k)
    items = []
    off = 0
    for d, L in enumerate(doc_len):
        pos = off
        while pos < off + L:
            s = min(pos // T, k - 1)
            stop = min(off + L, (s + 1) * T)
            items.append({"doc": d, "q0": pos - off, "q1": stop - off, "server": s, "home": s, "alive": True})
            pos = stop
        off += L
    return items


def schedule(doc_len, k, bytes_q, bytes_kv, tolerance=0.0, min_score=0.0, min_shard_tokens=0):
    items = initial_items(doc_len, k)
    load = [0] * k
    for it in items:
        load[it["server"]] += pairs_of_range(it["q0"], it["q1"])
    total = sum(load)
    target = total / k                                              # step 1
    deficit = [s for s in range(k) if load[s] < target]
    deficit.sort(key=lambda s: (target - load[s]) * -1)              # step 2: largest deficit first (stable)
    stats = {"n_migrations": 0, "n_splits": 0, "comm_bytes": 0.0}
    for dst in deficit:
        while target - load[dst] > tolerance * target:
            D = target - load[dst]
            best = None
            for idx, it in enumerate(items):
                if not it["alive"] or it["server"] == dst:
                    continue
                S = load[it["server"]] - target
                if not S > 0:
                    continue
                f = pairs_of_range(it["q0"], it["q1"])
                dF = min(f, S, D)
                L_q, L_kv = it["q1"] - it["q0"], it["q1"]
                split = dF < f
                nq, nkv = L_q, L_kv
                if split:
                    nq, nkv, _ = optimal_shard(L_q, L_kv, dF / f, max(1, int(math.floor(dF + 0.5))), bytes_q, bytes_kv)
                    if nq == L_q and nkv == L_kv:
                        split = False
                    elif min_shard_tokens > 0:
                        left, right = (nkv - nq) - it["q0"], it["q1"] - nkv
                        if nq < min_shard_tokens or 0 < left < min_shard_tokens or 0 < right < min_shard_tokens:
                            continue
                nbytes = nq * bytes_q + nkv * bytes_kv
                e = dF / nbytes                                      # E = transferred work per byte
                if best is None or e > best[0]:
                    best = (e, idx, split, nq, nkv, nbytes)
            if best is None or not best[0] > min_score:                # step 4
                break
            e, idx, split, nq, nkv, nbytes = best                    # step 3
            it = items[idx]
            src = it["server"]
            stats["comm_bytes"] += nbytes
            if not split:
                f = pairs_of_range(it["q0"], it["q1"])
                load[src] -= f
                load[dst] += f
                it["server"] = dst
                stats["n_migrations"] += 1
            else:
                a, b = nkv - nq, nkv
                moved = pairs_of_range(a, b)
                load[src] -= moved
                load[dst] += moved
                it["alive"] = False
                if a > it["q0"]:
                    items.append({"doc": it["doc"], "q0": it["q0"], "q1": a, "server": src, "home": it["home"],
                                  "alive": True})
                items.append({"doc": it["doc"], "q0": a, "q1": b, "server": dst, "home": it["home"], "alive": True})
                if it["q1"] > b:
                    items.append({"doc": it["doc"], "q0": b, "q1": it["q1"], "server": src, "home": it["home"],
                                  "alive": True})
                stats["n_splits"] += 1
    live = sorted((it for it in items if it["alive"]), key=lambda it: (it["server"], it["doc"], it["q0"]))
    tasks = [(it["server"], it["home"], it["doc"], it["q0"], it["q1"] - it["q0"], it["q1"],
              pairs_of_range(it["q0"], it["q1"])) for it in live]
    stats.update({"max_load": max(load), "min_load": min(load), "target": target, "loads": load})
    return tasks, stats


# ---------------------------------------------------------------- 2N-chunk sharding

def shard_2n(doc_len, N):
    """(rank, rank, doc, q_start, q_len, kv_len, pairs) for every non-empty chunk."""
    out = []
    for r in range(N):
        for d, L in enumerate(doc_len):
            c = -(-L // (2 * N))
            chunks = [[p for p in range(L) if p // c == j] for j in range(2 * N)]  # positions of chunk j
            for j in sorted({r, 2 * N - 1 - r}):
                pos = chunks[j]
                if pos:
                    out.append((r, r, d, pos[0], len(pos), pos[-1] + 1, pairs_of_range(pos[0], pos[-1] + 1)))
    return out
