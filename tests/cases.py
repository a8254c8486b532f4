"""Small workloads shared by the GPU parity tests: sizes the oracle finishes
in seconds that still span several tiles, ragged tails and the edge cases of
the CA-task descriptor."""
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


