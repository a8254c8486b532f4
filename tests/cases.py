"""Small workloads shared by the GPU parity tests: sizes the oracle finishes
in seconds that still span several tiles, ragged tails and the edge cases of
the CA-task descriptor."""
import numpy as np

import workloads as W

EDGE = [
    # G = 1, head_dim 128: documents shorter than, equal to and just past one tile
    W.custom("g1_d128_edges", [1, 127, 128, 129, 300], [(i, 0, l, 0, l) for i, l in enumerate([1, 127, 128, 129, 300])],
             hq=2, hkv=2, d=128, seed=1),
    # G = 8, sharded tasks out of order, KV blocks with empty rows, ragged tails
    W.custom("g8_shards_blocks", [700, 260],
             [(0, 300, 400, 0, 700), (1, 0, 260, 0, 260), (0, 0, 300, 0, 300), (0, 650, 50, 128, 300),
              (0, 10, 40, 37, 90)], hq=16, hkv=2, d=128, seed=2),
    # G = 16, head_dim 64, one long row crossing many key tiles, a gap between documents
    W.custom("g16_d64_long", [1500, 33], [(0, 1400, 100, 0, 1500), (1, 0, 33, 0, 33)], hq=16, hkv=1, d=64, seed=3,
             doc_kv_offset=[40, 1]),
    # G = 2, head_dim 64, many short shards (the composability case of Fig. 5: shards below the tile size)
    W.rebatched_pool(seed=4, n_docs=3, doc_lo=500, doc_hi=900, shard_lo=20, shard_hi=200, total_q=1200,
                     hq=4, hkv=2, d=64),
    # split KV: four blocks of one document (pass-KV partials)
    W.split_kv_prefill(seed=5, n_new=96, cached=416, n_blocks=4, hq=8, hkv=1, d=128),
    # G = 32, 64, 128: 4, 2 and 1 tokens per 128-row query tile; shards and ragged ends
    W.custom("g32_d128_shards", [77, 300], [(1, 0, 150, 0, 150), (0, 0, 77, 0, 77), (1, 150, 150, 0, 300)],
             hq=32, hkv=1, d=128, seed=6),
    W.custom("g64_d64_blocks", [150], [(0, 0, 150, 0, 150), (0, 100, 50, 30, 100)], hq=64, hkv=1, d=64, seed=7),
    W.custom("g128_d128", [40, 129], [(0, 0, 40, 0, 40), (1, 0, 129, 0, 129)], hq=128, hkv=1, d=128, seed=8),
]




def random_pool(seed: int, max_len: int = 1600, max_rows_x_heads: int = 100_000):
    """A seeded random CA-task pool: 1-4 documents of log-uniform length (with
    gaps between them in K/V half the time), each cut into 1-3 query shards
    that keep a random subset of its rows, some shards with a KV block that
    starts past 0, and on two pools in five a random (sink, lo, window) mask
    per task.  G is drawn from 1..128 and head_dim from {64, 128}; documents
    shrink with the head count so that the oracle stays within seconds."""
    rng = np.random.default_rng(20_000 + seed)
    d = int(rng.choice([64, 128]))
    G = int(rng.choice([1, 2, 4, 8, 16, 32, 64, 128]))
    hkv = 1 if G >= 64 else int(rng.choice([1, 2]))
    hq = G * hkv
    n_docs = int(rng.integers(1, 5))
    cap = int(min(max_len, max(16, max_rows_x_heads // hq // n_docs)))
    doc_len = np.exp(rng.uniform(0.0, np.log(cap), n_docs)).astype(np.int64) + 1
    gaps = rng.integers(0, 48, n_docs) if rng.random() < 0.5 else np.zeros(n_docs, dtype=np.int64)
    off = np.cumsum(gaps + np.concatenate([[0], doc_len[:-1]])).astype(np.int64)
    tasks = []
    for doc, L in enumerate(int(x) for x in doc_len):
        cuts = sorted(set(int(c) for c in rng.integers(1, L, int(rng.integers(0, 3)))) if L > 1 else set())
        edges = [0] + cuts + [L]
        for a, b in zip(edges[:-1], edges[1:]):
            if rng.random() < 0.2 and len(edges) > 2:
                continue                                   # rows no task asks for
            kv0 = 0
            if rng.random() < 0.3:
                kv0 = int(rng.integers(0, b))                  # a KV block, possibly past some rows
            kv1 = int(rng.integers(max(kv0 + 1, 1), L + 1)) if rng.random() < 0.3 else b
            tasks.append((doc, a, b - a, kv0, max(1, kv1 - kv0)))
    if not tasks:
        tasks.append((0, 0, int(doc_len[0]), 0, int(doc_len[0])))
    order = rng.permutation(len(tasks))
    tasks = [tasks[i] for i in order]
    masks = None
    if rng.random() < 0.4:
        masks = []
        for doc, *_ in tasks:
            L = int(doc_len[doc])
            pick = lambda: int(rng.integers(0, L + 1)) if rng.random() < 0.7 else 0  # noqa: E731
            masks.append((pick(), pick(), pick()))
    return W.custom(f"random_pool_{seed}", doc_len, tasks, hq=hq, hkv=hkv, d=d, seed=100 + seed,
                    doc_kv_offset=off, masks=masks)
