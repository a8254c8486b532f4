"""Host-side checks of libca.so that need no GPU: every symbol include/*.h
declares is exported, the integer accounting of the plan equals the oracle's
enumeration bit-exactly, and invalid descriptors are rejected."""
import ctypes
import os
import re

import numpy as np
import pytest

import document_masked_core_gb300 as ca
from document_masked_core_gb300 import build, capi
import oracle
import workloads as W
from cases import random_pool

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module", autouse=True)
def built():
    build.build()


def declared_symbols():
    names = set()
    for h in sorted(os.listdir(os.path.join(ROOT, "include"))):
        if h.endswith(".h"):
            text = open(os.path.join(ROOT, "include", h)).read()
            text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
            names |= set(re.findall(r"\b(ca_[a-z_0-9]+)\s*\(", text))
    return sorted(names)


def test_library_exports_every_declared_symbol():
    L = ctypes.CDLL(capi.LIB_PATH)
    names = declared_symbols()
    assert names, "no declarations parsed"
    for n in names:
        assert hasattr(L, n), n
    assert sorted(capi.EXPORTS) == names


def test_set_backward_kernel_needs_a_plan():
    L = capi.load()
    assert L.ca_plan_set_backward_kernel(None, capi.CA_BWD_KERNEL_PAIR) == capi.CA_ERR_INVALID_ARG


def test_status_strings_and_version():
    L = capi.load()
    for s in range(7):
        assert L.ca_status_string(s)
    assert ca.version() >> 16 == 1


WORKLOADS = [W.tiny_chunk(), W.llama8b_chunk(), W.rebatched_pool(), W.long_context_chunk(),
             W.split_kv_prefill(), W.split_kv_prefill(split=False),
             W.custom("kv_blocks", [300], [(0, 200, 100, 0, 64), (0, 200, 100, 64, 200), (0, 5, 20, 100, 7)],
                      4, 1, 128),
             W.lambda_chunk(total=16384), W.blockwise_chunk(total=16384), W.shared_question_pool(total=16384)]

MASKED_SMALL = [
    W.lambda_chunk(seed=1, total=3000, sink=70, window=300, hq=8, hkv=2, d=64),
    W.lambda_chunk(seed=2, total=3000, sink=0, window=129, hq=4, hkv=1, d=128),
    W.blockwise_chunk(seed=3, total=3000, block=96, sink_blocks=2, window_blocks=3, hq=8, hkv=1, d=64),
    W.shared_question_pool(seed=4, total=3000, q_lo=100, q_hi=400, a_lo=40, a_hi=300, hq=4, hkv=1, d=64),
    W.custom("mixed_masks", [700, 500], [(0, 0, 700, 0, 700), (1, 100, 300, 50, 400), (0, 300, 200, 0, 600)],
             8, 2, 64, masks=[(10, 0, 200), (0, 256, 0), (130, 400, 77)]),
]


@pytest.mark.parametrize("w", WORKLOADS, ids=lambda w: w.name)
def test_pair_accounting_bit_exact(w):
    info, pairs = ca.dry_run_workload(w)
    ref = oracle.task_pairs(w)
    assert np.array_equal(pairs, ref)
    assert info["causal_pairs"] == int(ref.sum())
    fwd, bwd = oracle.flops(w)
    assert info["flops_fwd"] == fwd and info["flops_bwd"] == bwd
    assert info["total_q"] == w.total_q and info["total_kv"] == w.total_kv


def visible_block(w, t, p_lo, p_hi, k0, k1):
    """Whether any row p in [p_lo, p_hi] of task t sees any key in [k0, k1]."""
    sink, lo, win = (int(x[t]) for x in w.masks())
    a, e = int(w.task_kv_start[t]), int(w.task_kv_start[t] + w.task_kv_len[t])
    p = np.arange(p_lo, p_hi + 1)[:, None]
    j = np.arange(k0, k1 + 1)[None, :]
    vis = (j >= a) & (j < e) & (j <= p)
    if sink or lo or win:
        vis &= (j < sink) | ((j >= lo) & ((win == 0) | (j >= p - win + 1)))
    return bool(vis.any())


def masked_tile_pairs_reference(w):
    G = w.num_q_heads // w.num_kv_heads
    T = 128 // G
    n = 0
    for t in range(w.n_tasks):
        q0, ql = int(w.task_q_start[t]), int(w.task_q_len[t])
        L = int(w.doc_len[w.task_doc[t]])
        for tile in range((ql + T - 1) // T):
            p_lo = q0 + tile * T
            p_hi = min(q0 + ql, p_lo + T) - 1
            for jt in range((L + 127) // 128):
                n += visible_block(w, t, p_lo, p_hi, jt * 128, min(L, jt * 128 + 128) - 1)
    return n * w.num_kv_heads


@pytest.mark.parametrize("w", MASKED_SMALL, ids=lambda w: w.name)
def test_masked_tile_lists(w):
    """Backward: exactly the (key tile, query tile) pairs with a visible pair.
    Forward: those, plus at most one extra key tile per query tile where the
    two tiles of an item start their windows in different key tiles."""
    info, pairs = ca.dry_run_workload(w)
    assert np.array_equal(pairs, oracle.task_pairs(w))
    ref = masked_tile_pairs_reference(w)
    assert info["bwd_tile_pairs"] == ref
    G = w.num_q_heads // w.num_kv_heads
    n_qtiles = sum(-(-int(x) // (128 // G)) for x in w.task_q_len) * w.num_kv_heads
    assert ref <= info["fwd_tile_pairs"] <= ref + n_qtiles


def tile_pairs_reference(w):
    """Visible (query tile, key tile) pairs by enumerating tiles: a query tile
    (128/G tokens of one task) and a 128-key tile of the document meet when
    some row of the tile sees some key of the tile."""
    G = w.num_q_heads // w.num_kv_heads
    T = 128 // G
    n = 0
    for t in range(w.n_tasks):
        q0, ql = int(w.task_q_start[t]), int(w.task_q_len[t])
        a, e = int(w.task_kv_start[t]), int(w.task_kv_start[t] + w.task_kv_len[t])
        for tile in range((ql + T - 1) // T):
            p_lo = q0 + tile * T
            p_hi = min(q0 + ql, p_lo + T) - 1
            L = int(w.doc_len[w.task_doc[t]])
            for jt in range((L + 127) // 128):
                k0, k1 = jt * 128, jt * 128 + 127
                lo, hi = max(k0, a), min(k1, e - 1, p_hi)
                n += hi >= lo
    return n * w.num_kv_heads


@pytest.mark.parametrize("w", [WORKLOADS[0], WORKLOADS[6], W.rebatched_pool(total_q=4096, doc_lo=1000,
                                                                              doc_hi=3000, shard_lo=50,
                                                                              shard_hi=700)],
                         ids=lambda w: w.name)
def test_tile_lists_cover_visible_tiles(w):
    info, _ = ca.dry_run_workload(w)
    ref = tile_pairs_reference(w)
    assert info["fwd_tile_pairs"] == ref
    assert info["bwd_tile_pairs"] == ref


@pytest.mark.parametrize("seed", range(64))
def test_random_pools_accounting_and_tile_lists(seed):
    """Seeded random pools (shards, KV blocks, gaps between documents, masks,
    G from 1 to 128): per-task pairs, FLOPs and the backward's tile list equal
    the oracle's and the enumeration's exactly; the forward's list covers every
    visible tile, and equals the enumeration on unmasked pools."""
    w = random_pool(seed)
    info, pairs = ca.dry_run_workload(w)
    ref = oracle.task_pairs(w)
    assert np.array_equal(pairs, ref)
    assert info["causal_pairs"] == int(ref.sum())
    assert (info["flops_fwd"], info["flops_bwd"]) == oracle.flops(w)
    tiles = masked_tile_pairs_reference(w)
    assert info["bwd_tile_pairs"] == tiles
    if not w.masked:
        assert info["fwd_tile_pairs"] == tiles
    else:
        G = w.num_q_heads // w.num_kv_heads
        n_qtiles = sum(-(-int(x) // (128 // G)) for x in w.task_q_len) * w.num_kv_heads
        assert tiles <= info["fwd_tile_pairs"] <= tiles + n_qtiles


def test_invalid_descriptors_rejected():
    base = dict(task_doc=[0], task_q_start=[0], task_q_len=[10], task_kv_start=[0], task_kv_len=[10],
                doc_len=[10], doc_kv_offset=[0], num_q_heads=4, num_kv_heads=1, head_dim=64)
    ca.dry_run(**base)
    bad = [
        dict(task_q_len=[0]),
        dict(task_q_start=[5]),                 # runs past the document
        dict(task_kv_len=[11]),
        dict(task_kv_start=[-1]),
        dict(task_doc=[1]),                     # unknown document
        dict(num_q_heads=6, num_kv_heads=4),    # not a multiple
        dict(doc_len=[10, 5], doc_kv_offset=[0, 8]),  # overlapping documents
        dict(softmax_scale=-1.0),
        # sums that would overflow int64 if the host formed them
        dict(task_q_start=[2 ** 63 - 5]),
        dict(task_kv_start=[2 ** 63 - 5]),
        dict(doc_kv_offset=[2 ** 63 - 5]),
        dict(task_q_len=[2 ** 63 - 1]),
    ]
    for b in bad:
        kw = dict(base, **b)
        with pytest.raises(ca.CAError) as ei:
            ca.dry_run(**kw)
        assert ei.value.status == capi.CA_ERR_INVALID_ARG, b
    for b in (dict(head_dim=96), dict(num_q_heads=3, num_kv_heads=1), dict(num_q_heads=8192, num_kv_heads=64)):
        with pytest.raises(ca.CAError) as ei:
            ca.dry_run(**dict(base, **b))
        assert ei.value.status == capi.CA_ERR_UNSUPPORTED, b


def _descriptor(w):
    return dict(task_doc=w.task_doc.astype(np.int64).copy(), task_q_start=w.task_q_start.copy(),
                task_q_len=w.task_q_len.copy(), task_kv_start=w.task_kv_start.copy(),
                task_kv_len=w.task_kv_len.copy(), doc_len=w.doc_len.copy(), doc_kv_offset=w.doc_kv_offset.copy(),
                num_q_heads=w.num_q_heads, num_kv_heads=w.num_kv_heads, head_dim=w.head_dim,
                masks=np.stack(w.masks(), axis=1))


def _break_one_rule(kw, rng):
    """Violate exactly one of ca_plan_create's INVALID_ARG rules (include/ca.h)
    in one randomly chosen task or document; returns the rule's name."""
    n, nd = len(kw["task_doc"]), len(kw["doc_len"])
    t = int(rng.integers(n))
    L = int(kw["doc_len"][kw["task_doc"][t]])
    rules = ["q_len_zero", "q_len_negative", "q_past_doc", "q_start_negative", "q_start_huge", "kv_len_zero",
             "kv_past_doc", "kv_start_negative", "doc_id_unknown", "doc_id_negative", "doc_shrunk",
             "mask_negative", "mask_past_doc", "q_len_huge", "scale_bad"]
    if nd > 1:
        rules.append("docs_overlap")
    rule = str(rng.choice(rules))
    q0, ql, k0, kl = (int(kw[f][t]) for f in ("task_q_start", "task_q_len", "task_kv_start", "task_kv_len"))
    if rule == "q_len_zero":
        kw["task_q_len"][t] = 0
    elif rule == "q_len_negative":
        kw["task_q_len"][t] = -int(rng.integers(1, 1 << 40))
    elif rule == "q_past_doc":
        kw["task_q_len"][t] = L - q0 + int(rng.integers(1, 100))
    elif rule == "q_start_negative":
        kw["task_q_start"][t] = -int(rng.integers(1, 1 << 40))
    elif rule == "q_start_huge":
        kw["task_q_start"][t] = (1 << 63) - int(rng.integers(1, 1000))
    elif rule == "q_len_huge":
        kw["task_q_len"][t] = (1 << 63) - int(rng.integers(1, 1000))
    elif rule == "kv_len_zero":
        kw["task_kv_len"][t] = 0
    elif rule == "kv_past_doc":
        kw["task_kv_len"][t] = L - k0 + int(rng.integers(1, 100))
    elif rule == "kv_start_negative":
        kw["task_kv_start"][t] = -int(rng.integers(1, 1 << 40))
    elif rule == "doc_id_unknown":
        kw["task_doc"][t] = nd + int(rng.integers(0, 5))
    elif rule == "doc_id_negative":
        kw["task_doc"][t] = -int(rng.integers(1, 5))
    elif rule == "doc_shrunk":  # the document ends before one of its tasks
        d = int(kw["task_doc"][t])
        kw["doc_len"][d] = max(q0 + ql, k0 + kl) - 1
        if kw["doc_len"][d] < 1:
            kw["task_q_start"][t] = kw["doc_len"][d] = 1
    elif rule == "mask_negative":
        kw["masks"][t, int(rng.integers(3))] = -int(rng.integers(1, 100))
    elif rule == "mask_past_doc":
        kw["masks"][t, int(rng.integers(3))] = L + int(rng.integers(1, 100))
    elif rule == "scale_bad":
        kw["softmax_scale"] = float(rng.choice([0.0, -0.5, np.inf, np.nan]))
    elif rule == "docs_overlap":  # document b starts inside document a
        a, b = (int(x) for x in rng.choice(nd, 2, replace=False))
        kw["doc_kv_offset"][b] = kw["doc_kv_offset"][a] + int(rng.integers(0, kw["doc_len"][a]))
    return rule


@pytest.mark.parametrize("seed", range(32))
def test_random_invalid_descriptors_rejected(seed):
    """Random pools with one rule of ca_plan_create broken at a time are
    refused with CA_ERR_INVALID_ARG on the host (and planned when intact)."""
    rng = np.random.default_rng(30_000 + seed)
    w = random_pool(seed)
    ca.dry_run(**_descriptor(w))
    for _ in range(12):
        kw = _descriptor(w)
        rule = _break_one_rule(kw, rng)
        with pytest.raises(ca.CAError) as ei:
            ca.dry_run(**kw)
        assert ei.value.status == capi.CA_ERR_INVALID_ARG, (rule, str(ei.value))


def test_merge_rejects_sizes_that_overflow_the_launch():
    """ca_merge validates its sizes on the host before any CUDA call."""
    with pytest.raises(ca.CAError) as ei:
        capi.merge([16], [16], 2 ** 62, 1, 64, 16, stream=0)
    assert ei.value.status == capi.CA_ERR_INVALID_ARG
    with pytest.raises(ca.CAError) as ei:
        capi.merge([16], [16], 4, 1, 60, 16, stream=0)  # head_dim not a multiple of 8
    assert ei.value.status == capi.CA_ERR_INVALID_ARG
