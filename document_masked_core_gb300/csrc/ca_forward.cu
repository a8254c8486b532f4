// Forward core attention over a rebatched pool of CA-tasks (sm_103a).
//
// One persistent CTA per SM takes the plan's forward items (longest first)
// from a global work queue.
// An item is two consecutive 128-row query tiles A and B of one task and one
// kv head g; a tile row is one (token, head) pair, 128 / G tokens x G heads,
// so one 128-key K/V tile of head g serves both tiles (GQA sharing by packing
// heads into the MMA M dimension).  For each visible key tile j:
//   S_X = Q_X K_j^T        tcgen05.mma, bf16 x bf16 -> fp32 in TMEM
//   online softmax         one thread per row reads its S row from TMEM,
//                          masks the causal / block edges, keeps the running
//                          max m and sum l (log2 domain), writes P (bf16)
//                          over S in TMEM
//   O_X += P_X V_j         tcgen05.mma with A = P from TMEM, B = V (MN-major)
// and finally O /= l, LSE = ln 2 (m + log2 l).  The online-softmax recurrence
// with saved row statistics is what the disaggregation paper relies on
// (Efficient Long-context Language Model Training by Core Attention
// Disaggregation, §3.4 "Property 1: Statelessness"); fully masked key tiles
// are never visited (the plan lists only visible tiles).
//
// The two tiles ping-pong on the tensor core: while warpgroup A computes the
// softmax of S_A(j), the MMA warp runs PV_B(j-1) and S_B(j), and vice versa.
// The running max is rescaled lazily: a row's O and l are rescaled only when
// its max grows by more than 2^8, otherwise exponentials are taken against
// the stale max (values up to 2^8, exact in the final normalisation).
//
// Warp roles (320 threads): warps 0-3 softmax + epilogue of tile A, warps 4-7
// of tile B (thread i of a warpgroup <-> TMEM lane i <-> tile row i), warp 8
// TMA producer, warp 9 TMEM owner + MMA issuer.  The producer and MMA warps
// run their loops with all 32 lanes (every wait, count and descriptor is the
// same in each lane) and one elected lane issues each copy or tcgen05 op: the
// MMA warp's instruction stream is what paces the tensor core here, and with
// a single lane issuing inside a lane-0 branch the forward ran 10-15 % slower.
//
// Across items the MMA warp keeps the tensor core fed: Q tiles go through a
// three-slot ring, each slot released after its tile's last S product, and in
// an item's last visit the next item's first S products take the places of
// the missing S(j+1) products when their Q and K tiles have landed.
#include <algorithm>
#include <cmath>

#include <cuda_bf16.h>

#include "ca_sm100.cuh"

namespace ca {
namespace {

using namespace dev;

struct FwdParams {
    const DevTask *tasks;
    const FwdItem *items;
    int32_t n_items;
    int32_t hq, G, tpt;
    float scale_log2;  // softmax_scale * log2(e)
    void *o;
    int32_t o_v8;  // O is 32-byte aligned: the epilogue stores whole 32-byte sectors
    float *lse;
    int32_t *sched;  // work-queue counter (zeroed before the launch)
    SplitScratch split;  // partial rows of split items and their row counters (zeroed before the launch)
    DevCtl ctl;
};

template <int D>
struct FwdCfg {
    static constexpr int kStages = 2;
    // Q tiles go through a ring of three slots in the order they are loaded
    // (an item's tile A, then its tile B): the next item's first tile loads
    // into the free slot while the current item runs.
    static constexpr int kQSlots = 3;
    static constexpr int kHalfBytes = 128 * 128;              // 128 rows x 64 bf16
    static constexpr int kTileBytes = (D / 64) * kHalfBytes;  // 128 rows x D bf16
    static constexpr int kOffQ = 0;
    static constexpr int kOffK = kOffQ + kQSlots * kTileBytes;
    static constexpr int kOffV = kOffK + kStages * kTileBytes;
    static constexpr int kOffBar = kOffV + kStages * kTileBytes;
    static constexpr int kBarBytes = 512;  // FwdBars (checked below)
    static constexpr int kOffRec = kOffBar + kBarBytes;
    static constexpr int kRecBytes = 4 * 128;  // ItemRec ring (checked below)
    static constexpr int kSmemRaw = kOffRec + kRecBytes;
    static constexpr int kSmemBytes = kSmemRaw > 122880 ? kSmemRaw : 122880;  // one CTA per SM
    static_assert(kSmemBytes <= 232448, "forward tiles exceed 227 KB of shared memory");
    static constexpr uint32_t kTmemCols = 512;
    // TMEM columns: S/P of tile X at 128 X, O of tile X at 256 + D X
    static constexpr uint32_t kColS = 0;
    static constexpr uint32_t kColO = 256;
    static constexpr uint32_t kIdescQK = idesc_bf16(128, 128, false, false);
    static constexpr uint32_t kIdescPV = idesc_bf16(128, D, false, true);
};

constexpr float kRescaleThreshold = 8.0f;  // log2 units: rescale when the max grows by > 2^8

// warps that read each work-queue ring entry: MMA and the 8 softmax warps
constexpr uint32_t kRingConsumers = 9;

struct FwdBars {
    uint64_t ring_full[4], ring_empty[4];
    uint64_t q_full[3], q_empty[3];  // Q slot s (q_empty: committed after the tile's last S product)
    uint64_t k_full[2], v_full[2];
    uint64_t k_empty[2];  // committed after the last S product that reads the K tile
    uint64_t v_empty[2];  // committed after the last PV product that reads the V tile
    uint64_t s_full[2], p_full[2];
    uint64_t o_full[2], o_empty[2];
    uint64_t mma_done;
    uint32_t tmem_base;
    uint32_t abort_flag;
};

static_assert(sizeof(FwdBars) <= 512, "barrier block exceeds its shared-memory reservation");

struct TileGeo {
    int32_t row0, p_first, ntok, n_kv;  // n_kv = 0: tile absent or sees nothing
};

// Key tiles of an item: the sequence of key_tile_ranges over the rows of its
// two query tiles; tile x visits the prefix of n_kv(x) entries that reaches
// the furthest key any of its rows sees (the same rule as the host plan).
struct ItemGeo {
    int32_t g, kv_off, n_kv, i0;
    int32_t part, nparts, split, slot0;
    KeyTileRanges kr;
    DevTask task;
    TileGeo t[2];
};

__device__ __forceinline__ TileGeo tile_geo(const DevTask &t, int32_t tile, int32_t tpt) {
    TileGeo tg;
    const int32_t tok0 = tile * tpt;
    tg.row0 = t.row0 + tok0;
    tg.p_first = t.q_start + tok0;
    tg.ntok = max(0, min(tpt, t.q_len - tok0));
    tg.n_kv = 0;
    return tg;
}

__device__ __forceinline__ ItemGeo decode_item(const FwdParams &p, int32_t idx) {
    const FwdItem it = p.items[idx];
    ItemGeo gi;
    gi.task = p.tasks[it.task];
    const DevTask &t = gi.task;
    gi.g = it.g;
    gi.kv_off = t.kv_off;
    gi.t[0] = tile_geo(t, it.tile, p.tpt);
    gi.t[1] = tile_geo(t, it.tile + 1, p.tpt);
    const int32_t end0 = gi.t[0].p_first + gi.t[0].ntok - 1;
    const int32_t end1 = gi.t[1].ntok > 0 ? gi.t[1].p_first + gi.t[1].ntok - 1 : end0;
    gi.kr = key_tile_ranges(t, gi.t[0].p_first, end1);
    // this item covers visits [i0, i1) of the pair's sequence
    gi.i0 = it.i0;
    gi.part = it.part;
    gi.nparts = it.nparts;
    gi.split = it.split;
    gi.slot0 = it.slot0;
    const int32_t va = gi.t[0].ntok > 0 ? visits_upto(gi.kr, t, gi.t[0].p_first, end0) : 0;
    const int32_t vb = gi.t[1].ntok > 0 ? visits_upto(gi.kr, t, gi.t[1].p_first, end1) : 0;
    gi.t[0].n_kv = max(0, min(va, it.i1) - it.i0);
    gi.t[1].n_kv = max(0, min(vb, it.i1) - it.i0);
    gi.n_kv = max(gi.t[0].n_kv, gi.t[1].n_kv);
    return gi;
}

// A work-queue entry as the producer publishes it: the item's index (-1 once
// the queue is exhausted) and its decoded geometry, so the other roles read it
// from shared memory instead of chasing the item and task tables in global
// memory at each item start.
struct ItemRec {
    ItemGeo gi;
    int32_t idx;
};
static_assert(sizeof(ItemRec) <= 128, "work-queue record exceeds its shared-memory slot");

// Make the compiler treat the 32 registers as produced after the preceding
// tcgen05.wait::ld (their values are only valid after it).
__device__ __forceinline__ void reg_fence(uint32_t (&r)[32]) {
    asm volatile(""
                 : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]),
                   "+r"(r[7]), "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]), "+r"(r[12]), "+r"(r[13]),
                   "+r"(r[14]), "+r"(r[15]), "+r"(r[16]), "+r"(r[17]), "+r"(r[18]), "+r"(r[19]), "+r"(r[20]),
                   "+r"(r[21]), "+r"(r[22]), "+r"(r[23]), "+r"(r[24]), "+r"(r[25]), "+r"(r[26]), "+r"(r[27]),
                   "+r"(r[28]), "+r"(r[29]), "+r"(r[30]), "+r"(r[31])
                 :
                 : "memory");
}

template <int D, bool OUT_F32>
__device__ __forceinline__ void store_row_zero(const FwdParams &p, size_t out_idx) {
    if (OUT_F32) {
        float4 *dst = reinterpret_cast<float4 *>(static_cast<float *>(p.o) + out_idx * D);
#pragma unroll
        for (int c = 0; c < D / 4; ++c) dst[c] = make_float4(0.f, 0.f, 0.f, 0.f);
    } else {
        uint4 *dst = reinterpret_cast<uint4 *>(static_cast<__nv_bfloat16 *>(p.o) + out_idx * D);
#pragma unroll
        for (int c = 0; c < D / 8; ++c) dst[c] = make_uint4(0, 0, 0, 0);
    }
    p.lse[out_idx] = -INFINITY;
}

// Split items: merge of the parts' partial rows (Eq. 4 of the million-token
// paper's Appendix B) by the part that finished a row last.  Partials are
// read through L2 (other SMs wrote them).
template <int D, bool OUT_F32>
__device__ __noinline__ void merge_split_row(const FwdParams &p, int32_t nparts, int32_t slot0, int32_t rowslot,
                                             size_t out_idx) {
    float M = -INFINITY;
    for (int32_t s = 0; s < nparts; ++s) M = fmaxf(M, __ldcg(p.split.lse + (slot0 + s) * 256 + rowslot));
    if (M == -INFINITY) {
        store_row_zero<D, OUT_F32>(p, out_idx);
        return;
    }
    float wsum = 0.f;
    for (int32_t s = 0; s < nparts; ++s) wsum += expf(__ldcg(p.split.lse + (slot0 + s) * 256 + rowslot) - M);
    const float inv = 1.f / wsum;
#pragma unroll 1
    for (int c = 0; c < D / 32; ++c) {
        float acc[32];
#pragma unroll
        for (int e = 0; e < 32; ++e) acc[e] = 0.f;
        for (int32_t s = 0; s < nparts; ++s) {
            const float w = expf(__ldcg(p.split.lse + (slot0 + s) * 256 + rowslot) - M);
            const float4 *src =
                reinterpret_cast<const float4 *>(p.split.o + (static_cast<size_t>(slot0 + s) * 256 + rowslot) * D + c * 32);
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                const float4 v = __ldcg(src + e);
                acc[4 * e] += w * v.x;
                acc[4 * e + 1] += w * v.y;
                acc[4 * e + 2] += w * v.z;
                acc[4 * e + 3] += w * v.w;
            }
        }
        if (OUT_F32) {
            float4 *dst = reinterpret_cast<float4 *>(static_cast<float *>(p.o) + out_idx * D + c * 32);
#pragma unroll
            for (int e = 0; e < 8; ++e)
                dst[e] = make_float4(acc[4 * e] * inv, acc[4 * e + 1] * inv, acc[4 * e + 2] * inv, acc[4 * e + 3] * inv);
        } else {
            uint4 *dst = reinterpret_cast<uint4 *>(static_cast<__nv_bfloat16 *>(p.o) + out_idx * D + c * 32);
#pragma unroll
            for (int e = 0; e < 4; ++e)
                dst[e] = make_uint4(pack_bf16(acc[8 * e] * inv, acc[8 * e + 1] * inv),
                                    pack_bf16(acc[8 * e + 2] * inv, acc[8 * e + 3] * inv),
                                    pack_bf16(acc[8 * e + 4] * inv, acc[8 * e + 5] * inv),
                                    pack_bf16(acc[8 * e + 6] * inv, acc[8 * e + 7] * inv));
        }
    }
    p.lse[out_idx] = M + logf(wsum);
}

// A part's row is in the workspace: count it, and merge the row if this part
// was the last of the item's parts to get there.
template <int D, bool OUT_F32>
__device__ __forceinline__ void finish_split_row(const FwdParams &p, const ItemGeo &gi, int32_t rowslot,
                                                 size_t out_idx) {
    __threadfence();
    const int32_t done = atomicAdd(p.split.cnt + gi.split * 256 + rowslot, 1);
    if (done == gi.nparts - 1) {
        __threadfence();
        merge_split_row<D, OUT_F32>(p, gi.nparts, gi.slot0, rowslot, out_idx);
    }
}

template <int D, bool OUT_F32>
__global__ void __launch_bounds__(320, 1)
    ca_fwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                  const __grid_constant__ CUtensorMap tm_v, const FwdParams p) {
    using C = FwdCfg<D>;
    extern __shared__ __align__(1024) uint8_t smem[];
    if (smem_u32(smem) & 1023u) {  // the swizzled tiles need 1024-byte alignment
        if (threadIdx.x == 0) atomicOr(p.ctl.err, kErrBounds);
        return;
    }
    uint8_t *sQ = smem + C::kOffQ;
    uint8_t *sK = smem + C::kOffK;
    uint8_t *sV = smem + C::kOffV;
    FwdBars &bars = *reinterpret_cast<FwdBars *>(smem + C::kOffBar);
    ItemRec *recs = reinterpret_cast<ItemRec *>(smem + C::kOffRec);  // [4], one per ring entry

    const uint32_t warp = warp_id();
    const uint32_t lane = lane_id();

    if (threadIdx.x == 0) {
        for (int sl = 0; sl < C::kQSlots; ++sl) {
            mbar_init(&bars.q_full[sl], 1);
            mbar_init(&bars.q_empty[sl], 1);
        }
        for (int x = 0; x < 2; ++x) {
            mbar_init(&bars.s_full[x], 1);
            mbar_init(&bars.p_full[x], 4);  // one arrival per warp
            mbar_init(&bars.o_full[x], 1);
            mbar_init(&bars.o_empty[x], 4);
        }
        for (int s = 0; s < C::kStages; ++s) {
            mbar_init(&bars.k_full[s], 1);
            mbar_init(&bars.v_full[s], 1);
            mbar_init(&bars.k_empty[s], 1);
            mbar_init(&bars.v_empty[s], 1);
        }
        mbar_init(&bars.mma_done, 1);
        for (int r = 0; r < 4; ++r) {
            mbar_init(&bars.ring_full[r], 1);
            mbar_init(&bars.ring_empty[r], kRingConsumers);
        }
        bars.abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 9) {
        tmem_alloc(&bars.tmem_base, C::kTmemCols);
        tmem_relinquish();
    }
    if (warp == 8 && lane == 0) {
        tma_prefetch_desc(&tm_q);
        tma_prefetch_desc(&tm_k);
        tma_prefetch_desc(&tm_v);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = bars.tmem_base;
    const Watchdog wd{&p.ctl, &bars.abort_flag};

    if (warp == 8) {
        // ------------------------------------------------------------ producer
        // The producer publishes the work queue one item ahead of its own loads
        // (each ring entry carries the decoded item), then loads the item's Q
        // tiles into the Q slot ring and its K/V tiles into the two stages, in
        // the order the MMA warp consumes them: Q_A, K(0), Q_B, V(0), K(1), V(1), ...
        {
            // the whole warp runs the loop; one elected lane issues each copy
            auto wwait = [&](uint64_t *bar, uint32_t parity) -> bool {
                return __all_sync(0xffffffffu, mbar_wait_ool(bar, parity, wd));
            };
            uint32_t kv_it = 0, qi = 0;
            bool ok = true;
            auto publish = [&](uint32_t r, ItemGeo &gi) -> int32_t {
                if (!(ok = wwait(&bars.ring_empty[r & 3], ((r >> 2) & 1) ^ 1))) return -1;
                int32_t idx = 0;
                if (lane == 0) idx = atomicAdd(p.sched, 1);
                idx = __shfl_sync(0xffffffffu, idx, 0);
                if (idx >= p.n_items) idx = -1;
                if (idx >= 0) gi = decode_item(p, idx);
                if (lane == 0) {
                    if (idx >= 0) recs[r & 3].gi = gi;
                    recs[r & 3].idx = idx;
                    mbar_arrive(&bars.ring_full[r & 3]);  // release: the record is complete
                }
                __syncwarp();
                return idx;
            };
            auto load_q = [&](const ItemGeo &gi, int x) -> bool {
                const uint32_t sl = qi % C::kQSlots;
                if (!wwait(&bars.q_empty[sl], ((qi / C::kQSlots) & 1) ^ 1)) return false;
                mbar_arrive_expect_tx_w(&bars.q_full[sl], C::kTileBytes);
#pragma unroll
                for (int h = 0; h < D / 64; ++h)
                    tma_load_3d_w(sQ + sl * C::kTileBytes + h * C::kHalfBytes, &tm_q, &bars.q_full[sl], h * 64,
                                gi.g * p.G, gi.t[x].row0);
                ++qi;
                return true;
            };
            // K and V stages are released separately: K once both query tiles' S
            // products have read it (an iteration before V), so each K load has
            // about two iterations to land before its S product
            auto load_kv = [&](const ItemGeo &gi, int32_t i, bool v) -> bool {
                const uint32_t kvi = kv_it + i;
                const uint32_t st = kvi % C::kStages, ph = (kvi / C::kStages) & 1;
                if (!wwait(v ? &bars.v_empty[st] : &bars.k_empty[st], ph ^ 1)) return false;
                uint64_t *full = v ? &bars.v_full[st] : &bars.k_full[st];
                const int32_t key_row = gi.kv_off + gi.kr.tile(gi.i0 + i) * kTileKeys;
                mbar_arrive_expect_tx_w(full, C::kTileBytes);
                uint8_t *dst = (v ? sV : sK) + st * C::kTileBytes;
#pragma unroll
                for (int h = 0; h < D / 64; ++h)
                    tma_load_3d_w(dst + h * C::kHalfBytes, v ? &tm_v : &tm_k, full, h * 64, gi.g, key_row);
                return true;
            };
            // The next entry is published after the current item's first loads are
            // in flight, so its decode (dependent global loads) overlaps them.
            ItemGeo gi;
            int32_t idx = publish(0, gi);
            for (uint32_t r = 0; ok && idx >= 0; ++r) {
                if (gi.n_kv > 0)
                    ok = (gi.t[0].n_kv == 0 || load_q(gi, 0)) && load_kv(gi, 0, false) &&
                         (gi.t[1].n_kv == 0 || load_q(gi, 1)) && load_kv(gi, 0, true);
                if (!ok) break;
                ItemGeo nx;
                const int32_t nidx = publish(r + 1, nx);
                if (!ok) break;
                for (int32_t i = 1; i < gi.n_kv && ok; ++i) ok = load_kv(gi, i, false) && load_kv(gi, i, true);
                kv_it += gi.n_kv;
                gi = nx;
                idx = nidx;
            }
            if (!ok && lane == 0) __nanosleep(1000000);  // let copies already in flight land before the CTA drains
        }
    } else if (warp == 9) {
        // ------------------------------------------------------------ MMA issuer
        // Per visit i of an item: PV_A(i), S_A(i+1), PV_B(i), S_B(i+1).  In an
        // item's last visit, when both tiles end there, the next item's S_A(0)
        // and S_B(0) take the places of the missing S(i+1) products, so the
        // tensor core does not idle across the item boundary.
        {
            // the whole warp runs the loop; one elected lane issues each tcgen05 op
            auto wwait = [&](uint64_t *bar, uint32_t parity) -> bool {
                return __all_sync(0xffffffffu, mbar_wait_ool(bar, parity, wd));
            };
            uint32_t kv_it = 0, qi = 0, r = 0;
            uint32_t s_it[2] = {0, 0}, o_it[2] = {0, 0};
            bool ok = true;
            const uint32_t q_base = smem_u32(sQ), k_base = smem_u32(sK), v_base = smem_u32(sV);
            // S_x = Q K^T of the tile in Q ring slot q and the key tile of K ring index
            // kvi, into tile x's S columns.  The K stage is released after the last S
            // product that reads it (release_k: tile B's, or tile A's when B does not
            // visit that key tile), the Q slot after its tile's last S product.
            auto issue_s = [&](int x, uint32_t q, uint32_t kvi, bool release_k, bool release_q) -> bool {
                const uint32_t st = kvi % C::kStages;
                if (!wwait(&bars.k_full[st], (kvi / C::kStages) & 1)) return false;
                tc_fence_after();
                const uint32_t ad = sdesc_lo(q_base + (q % C::kQSlots) * C::kTileBytes, 16);
                const uint32_t bd = sdesc_lo(k_base + st * C::kTileBytes, 16);
                const uint32_t d_s = tmem + C::kColS + x * 128;
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint32_t off = (kk / 4) * C::kHalfBytes + (kk % 4) * 32;
                    umma_ss_w(d_s, sdesc_at(ad, off), sdesc_at(bd, off), C::kIdescQK, kk > 0 ? 1u : 0u);
                }
                umma_commit_w(&bars.s_full[x]);
                if (release_k) umma_commit_w(&bars.k_empty[st]);
                if (release_q) umma_commit_w(&bars.q_empty[q % C::kQSlots]);
                return true;
            };
            auto wait_q = [&](uint32_t q) -> bool {
                if (!wwait(&bars.q_full[q % C::kQSlots], (q / C::kQSlots) & 1)) return false;
                tc_fence_after();
                return true;
            };
            // the next ring entry with key tiles to visit: n = 0 once the queue is exhausted
            // Take the next ring entry with key tiles to visit (n = 0 once the queue is
            // exhausted).  Blocking, or (poll) only as far as entries are published:
            // then it returns false with fetched unset when the next one is not there.
            auto take = [&](int32_t (&nk)[2], int32_t &n, bool poll, bool &fetched) -> bool {
                fetched = false;
                while (true) {
                    if (poll) {
                        if (!__all_sync(0xffffffffu, mbar_try_wait(&bars.ring_full[r & 3], (r >> 2) & 1))) return true;
                    } else if (!wwait(&bars.ring_full[r & 3], (r >> 2) & 1)) {
                        return false;
                    }
                    const ItemRec &rc = recs[r & 3];
                    const int32_t idx = __shfl_sync(0xffffffffu, rc.idx, 0), a = __shfl_sync(0xffffffffu, rc.gi.t[0].n_kv, 0),
                                  b = __shfl_sync(0xffffffffu, rc.gi.t[1].n_kv, 0), m = __shfl_sync(0xffffffffu, rc.gi.n_kv, 0);
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&bars.ring_empty[r & 3]);
                    ++r;
                    if (idx < 0 || m > 0) {
                        nk[0] = idx < 0 ? 0 : a;
                        nk[1] = idx < 0 ? 0 : b;
                        n = idx < 0 ? 0 : m;
                        fetched = true;
                        return true;
                    }
                }
            };
            int32_t nk[2] = {0, 0}, n = 0;
            bool pre[2] = {false, false};  // S_x(0) already issued in the previous item's last visit
            bool fetched = false;
            ok = take(nk, n, false, fetched);
            while (ok && n > 0) {
                // Q ring indices of the item's tiles (A first), as the producer loads them
                const uint32_t qx[2] = {qi, qi + (nk[0] > 0 ? 1u : 0u)};
                const uint32_t qn = qx[1] + (nk[1] > 0 ? 1u : 0u);
#pragma unroll
                for (int x = 0; x < 2; ++x) {
                    if (nk[x] == 0 || pre[x]) continue;
                    if (!(ok = wait_q(qx[x]) && issue_s(x, qx[x], kv_it, x == 1 || nk[1] == 0, nk[x] == 1))) break;
                }
                int32_t mk[2] = {0, 0}, m = 0;  // the next item
                bool pre_next[2] = {false, false};
                fetched = false;
                for (int32_t i = 0; i < n && ok; ++i) {
                    const uint32_t kvi = kv_it + i;
                    const uint32_t st = kvi % C::kStages;
                    if (!(ok = wwait(&bars.v_full[st], (kvi / C::kStages) & 1))) break;
#pragma unroll
                    for (int x = 0; x < 2; ++x) {
                        if (i >= nk[x]) continue;
                        if (!(ok = wwait(&bars.p_full[x], s_it[x] & 1))) break;
                        if (i == 0 && !(ok = wwait(&bars.o_empty[x], (o_it[x] & 1) ^ 1))) break;
                        tc_fence_after();
                        const uint32_t bd = sdesc_lo(v_base + st * C::kTileBytes, C::kHalfBytes);
                        const uint32_t d_o = tmem + C::kColO + x * D, a_p = tmem + C::kColS + x * 128;
#pragma unroll
                        for (int kk = 0; kk < 8; ++kk)
                            umma_ts_w(d_o, a_p + kk * 8, sdesc_at(bd, kk * 2048), C::kIdescPV,
                                    (i > 0 || kk > 0) ? 1u : 0u);
                        ++s_it[x];
                        if (i + 1 < nk[x]) {
                            if (!(ok = issue_s(x, qx[x], kvi + 1, x == 1 || i + 1 >= nk[1], i + 2 == nk[x]))) break;
                            continue;
                        }
                        umma_commit_w(&bars.o_full[x]);  // O_x complete
                        ++o_it[x];
                        // Both tiles end here: the next item's S_x(0) takes the place of
                        // S_x(i+1) when its entry is published and its Q and K tiles have
                        // landed; otherwise the next item issues it (waiting here would
                        // hold back PV_B).  Tile B's goes only after tile A's, which the K
                        // release rule assumes.
                        if (nk[0] != nk[1]) continue;
                        if (x == 0 && !(ok = take(mk, m, true, fetched))) break;
                        const uint32_t q = qn + (x == 1 && mk[0] > 0 ? 1u : 0u);
                        const uint32_t kn = kv_it + n;
                        if (fetched && mk[x] > 0 && (x == 0 || mk[0] == 0 || pre_next[0]) &&
                            __all_sync(0xffffffffu, mbar_try_wait(&bars.q_full[q % C::kQSlots], (q / C::kQSlots) & 1) &&
                                                        mbar_try_wait(&bars.k_full[kn % C::kStages], (kn / C::kStages) & 1))) {
                            tc_fence_after();
                            if (!(ok = issue_s(x, q, kn, x == 1 || mk[1] == 0, mk[x] == 1))) break;
                            pre_next[x] = true;
                        }
                    }
                    if (!ok) break;
                    umma_commit_w(&bars.v_empty[st]);
                }
                if (!ok) break;
                if (!fetched && !(ok = take(mk, m, false, fetched))) break;
                pre[0] = pre_next[0];
                pre[1] = pre_next[1];
                kv_it += n;
                qi = qn;
                nk[0] = mk[0];
                nk[1] = mk[1];
                n = m;
            }
            umma_commit_w(&bars.mma_done);  // arrives once every MMA issued above has completed
            const DevCtl drain{p.ctl.err, p.ctl.wait_limit_ns};
            uint32_t zero = 0;
            const Watchdog wd2{&drain, &zero};
            mbar_wait_ool(&bars.mma_done, 0, wd2);
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------------ softmax + epilogue (tile x = warp / 4)
        const int x = static_cast<int>(warp >> 2);
        const uint32_t row = threadIdx.x & 127u;
        const uint32_t lane_addr = ((warp & 3u) * 32u) << 16;
        const uint32_t s_addr = tmem + lane_addr + C::kColS + x * 128;
        const uint32_t o_addr = tmem + lane_addr + C::kColO + x * D;
        uint32_t s_it = 0, o_it = 0;
        bool ok = true;
        for (uint32_t r = 0; ok; ++r) {
            ok = __all_sync(0xffffffffu, mbar_wait_ool(&bars.ring_full[r & 3], (r >> 2) & 1, wd));
            if (!ok) break;
            const int32_t idx = recs[r & 3].idx;
            const ItemGeo gi = recs[r & 3].gi;
            __syncwarp();
            if (lane == 0) mbar_arrive(&bars.ring_empty[r & 3]);
            if (idx < 0) break;
            const TileGeo tg = gi.t[x];
            const int32_t tok = row / p.G;
            const int32_t h = gi.g * p.G + (row % p.G);
            const bool valid = tok < tg.ntok;
            const int32_t pos = tg.p_first + min(tok, max(tg.ntok - 1, 0));
            const RowKeys rk = row_keys(gi.task, pos);  // visible keys: [a, r1) U [r2, hi)
            const size_t out_idx = static_cast<size_t>(tg.row0 + tok) * p.hq + h;
            const bool split = gi.nparts > 1;
            const int32_t rowslot = x * 128 + static_cast<int32_t>(row);
            float *part_o = p.split.o + (static_cast<size_t>(gi.slot0 + gi.part) * 256 + rowslot) * D;
            if (tg.n_kv == 0) {
                if (valid) {
                    if (split) {  // this part sees none of the tile's keys: an empty partial
                        float4 *dst = reinterpret_cast<float4 *>(part_o);
#pragma unroll
                        for (int c = 0; c < D / 4; ++c) dst[c] = make_float4(0.f, 0.f, 0.f, 0.f);
                        p.split.lse[(gi.slot0 + gi.part) * 256 + rowslot] = -INFINITY;
                        finish_split_row<D, OUT_F32>(p, gi, rowslot, out_idx);
                    } else {
                        store_row_zero<D, OUT_F32>(p, out_idx);
                    }
                }
                continue;
            }
            float m = -INFINITY, l = 0.f;
            for (int32_t i = 0; i < tg.n_kv; ++i, ++s_it) {
                ok = __all_sync(0xffffffffu, mbar_wait_ool(&bars.s_full[x], s_it & 1, wd));
                if (!ok) break;
                tc_fence_after();
                // s_full also implies that PV_x(i-1) has completed (issued before S_x(i))
                uint32_t sr[4][32];
#pragma unroll
                for (int c = 0; c < 4; ++c) tmem_ld32(s_addr + c * 32, sr[c]);
                tmem_ld_wait();
#pragma unroll
                for (int c = 0; c < 4; ++c) reg_fence(sr[c]);
                const int32_t key0 = gi.kr.tile(gi.i0 + i) * kTileKeys;
                const bool whole = (key0 >= rk.a && key0 + kTileKeys <= rk.r1) ||
                                   (key0 >= rk.a && key0 >= rk.r2 && key0 + kTileKeys <= rk.hi);
                if (!whole) {
#pragma unroll
                    for (int c = 0; c < 4; ++c)
#pragma unroll
                        for (int e = 0; e < 32; ++e) {
                            const int32_t key = key0 + c * 32 + e;
                            const bool vis = key >= rk.a && (key < rk.r1 || (key >= rk.r2 && key < rk.hi));
                            if (!vis) sr[c][e] = __float_as_uint(-INFINITY);
                        }
                }
                float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
                for (int c = 0; c < 4; ++c)
#pragma unroll
                    for (int e = 0; e < 32; e += 2) {
                        mx0 = fmaxf(mx0, __uint_as_float(sr[c][e]));
                        mx1 = fmaxf(mx1, __uint_as_float(sr[c][e + 1]));
                    }
                const float m_tile = fmaxf(mx0, mx1) * p.scale_log2;  // scale > 0 keeps the order
                float alpha = 1.f;
                bool rescale = false;
                if (m == -INFINITY) {
                    m = m_tile;  // nothing accumulated yet (l = 0, O = 0 or about to be overwritten)
                } else if (m_tile > m + kRescaleThreshold) {
                    alpha = ex2(m - m_tile);
                    m = m_tile;
                    rescale = true;
                }
                const float m_use = (m == -INFINITY) ? 0.f : m;
                // paired f32x2 arithmetic: the softmax is bound by instruction issue
                // (the two tiles' warps share each scheduler), not by the ex2 unit
                const float2 sc2 = make_float2(p.scale_log2, p.scale_log2);
                const float2 nm2 = make_float2(-m_use, -m_use);
                float2 sum2 = make_float2(0.f, 0.f);
                // P of keys 32c .. 32c+31 packed two per column into columns 16c ..: every S
                // column is in registers already, so each chunk is stored as soon as it is
                // ready (fewer live registers)
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    uint32_t pk[16];
#pragma unroll
                    for (int e = 0; e < 32; e += 2) {
                        const float2 x2 = __ffma2_rn(make_float2(__uint_as_float(sr[c][e]), __uint_as_float(sr[c][e + 1])),
                                                     sc2, nm2);
                        const float2 p2 = make_float2(ex2(x2.x), ex2(x2.y));
                        sum2 = __fadd2_rn(sum2, p2);
                        pk[e >> 1] = pack_bf16(p2.x, p2.y);
                    }
                    tmem_st16(s_addr + 16 * c, pk);
                }
                l = l * alpha + (sum2.x + sum2.y);
                if (i > 0 && __any_sync(0xffffffffu, rescale)) {
#pragma unroll
                    for (int c = 0; c < D / 32; ++c) {
                        uint32_t orr[32];
                        tmem_ld32(o_addr + c * 32, orr);
                        tmem_ld_wait();
                        reg_fence(orr);
#pragma unroll
                        for (int e = 0; e < 32; ++e) orr[e] = __float_as_uint(__uint_as_float(orr[e]) * alpha);
                        tmem_st32(o_addr + c * 32, orr);
                    }
                }
                tmem_st_wait();
                tc_fence_before();
                mbar_arrive_warp(&bars.p_full[x]);
            }
            if (!ok) break;
            // epilogue: O / l and LSE once the last PV of this tile has landed
            ok = __all_sync(0xffffffffu, mbar_wait_ool(&bars.o_full[x], o_it & 1, wd));
            if (!ok) break;
            ++o_it;
            tc_fence_after();
            const float inv_l = l > 0.f ? 1.f / l : 0.f;
#pragma unroll
            for (int c = 0; c < D / 32; ++c) {
                uint32_t orr[32];
                tmem_ld32(o_addr + c * 32, orr);
                tmem_ld_wait();
                reg_fence(orr);
                if (valid && split) {
                    float4 *dst = reinterpret_cast<float4 *>(part_o + c * 32);
#pragma unroll
                    for (int e = 0; e < 8; ++e)
                        dst[e] = make_float4(__uint_as_float(orr[4 * e]) * inv_l, __uint_as_float(orr[4 * e + 1]) * inv_l,
                                             __uint_as_float(orr[4 * e + 2]) * inv_l,
                                             __uint_as_float(orr[4 * e + 3]) * inv_l);
                } else if (valid) {
                    // a lane writes its own row: 16- or 32-byte pieces, each a separate
                    // sector of the warp's store, so the wider pieces halve the requests
                    if (OUT_F32) {
                        float *dst = static_cast<float *>(p.o) + out_idx * D + c * 32;
#pragma unroll
                        for (int e = 0; e < 32; ++e) orr[e] = __float_as_uint(__uint_as_float(orr[e]) * inv_l);
                        if (p.o_v8) {
#pragma unroll
                            for (int e = 0; e < 4; ++e)
                                st_global_v8(dst + 8 * e, orr[8 * e], orr[8 * e + 1], orr[8 * e + 2], orr[8 * e + 3],
                                             orr[8 * e + 4], orr[8 * e + 5], orr[8 * e + 6], orr[8 * e + 7]);
                        } else {
#pragma unroll
                            for (int e = 0; e < 8; ++e)
                                reinterpret_cast<uint4 *>(dst)[e] =
                                    make_uint4(orr[4 * e], orr[4 * e + 1], orr[4 * e + 2], orr[4 * e + 3]);
                        }
                    } else {
                        __nv_bfloat16 *dst = static_cast<__nv_bfloat16 *>(p.o) + out_idx * D + c * 32;
                        uint32_t w[16];
#pragma unroll
                        for (int e = 0; e < 16; ++e)
                            w[e] = pack_bf16(__uint_as_float(orr[2 * e]) * inv_l, __uint_as_float(orr[2 * e + 1]) * inv_l);
                        if (p.o_v8) {
                            st_global_v8(dst, w[0], w[1], w[2], w[3], w[4], w[5], w[6], w[7]);
                            st_global_v8(dst + 16, w[8], w[9], w[10], w[11], w[12], w[13], w[14], w[15]);
                        } else {
#pragma unroll
                            for (int e = 0; e < 4; ++e)
                                reinterpret_cast<uint4 *>(dst)[e] = make_uint4(w[4 * e], w[4 * e + 1], w[4 * e + 2], w[4 * e + 3]);
                        }
                    }
                }
            }
            tc_fence_before();
            mbar_arrive_warp(&bars.o_empty[x]);
            const float lse_row = l > 0.f ? (m + lg2(l)) * 0.69314718055994531f : -INFINITY;
            if (valid && split) {
                p.split.lse[(gi.slot0 + gi.part) * 256 + rowslot] = lse_row;
                finish_split_row<D, OUT_F32>(p, gi, rowslot, out_idx);
            } else if (valid) {
                p.lse[out_idx] = lse_row;
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 9) {
        tc_fence_after();
        tmem_dealloc(tmem, C::kTmemCols);
    }
}

template <int D, bool F32>
cudaError_t launch_fwd_t(const ca_plan *pl, const CUtensorMap &tq, const CUtensorMap &tk, const CUtensorMap &tv,
                         const FwdParams &prm, cudaStream_t stream) {
    using C = FwdCfg<D>;
    auto kern = ca_fwd_kernel<D, F32>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
    if (e != cudaSuccess) return e;
    const int grid = static_cast<int>(std::min<int64_t>(pl->n_fwd, pl->num_sms));
    if (grid <= 0) return cudaSuccess;
    if ((e = mark(pl, 0, stream)) != cudaSuccess) return e;
    kern<<<grid, 320, C::kSmemBytes, stream>>>(tq, tk, tv, prm);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    return mark(pl, 1, stream);
}

}  // namespace

cudaError_t launch_forward(const ca_plan *pl, const void *q, const void *k, const void *v, void *o, float *lse,
                           void *workspace, cudaStream_t stream) {
    if (pl->n_fwd == 0) return cudaSuccess;
    int32_t *sched = work_counters(pl, workspace) + 1;
    cudaError_t e0 = cudaMemsetAsync(sched, 0, sizeof(int32_t), stream);
    if (e0 != cudaSuccess) return e0;
    const SplitScratch split = split_scratch(pl, workspace);
    if (pl->n_split > 0) {  // row counters of the split items start at zero
        e0 = cudaMemsetAsync(split.cnt, 0, static_cast<size_t>(pl->n_split) * 256 * sizeof(int32_t), stream);
        if (e0 != cudaSuccess) return e0;
    }
    CUtensorMap tq, tk, tv;
    if (make_tmap_3d(&tq, q, pl->total_q, pl->hq, pl->d, pl->G, pl->tpt) != CA_OK ||
        make_tmap_3d(&tk, k, pl->total_kv, pl->hkv, pl->d, 1, kTileKeys) != CA_OK ||
        make_tmap_3d(&tv, v, pl->total_kv, pl->hkv, pl->d, 1, kTileKeys) != CA_OK)
        return cudaErrorInvalidValue;
    FwdParams prm;
    prm.tasks = pl->d_tasks;
    prm.items = pl->d_fwd;
    prm.n_items = static_cast<int32_t>(pl->n_fwd);
    prm.hq = pl->hq;
    prm.G = pl->G;
    prm.tpt = pl->tpt;
    prm.scale_log2 = pl->scale * 1.4426950408889634f;
    prm.o = o;
    prm.o_v8 = (reinterpret_cast<uintptr_t>(o) & 31u) == 0 ? 1 : 0;
    prm.lse = lse;
    prm.sched = sched;
    prm.split = split;
    prm.ctl.err = pl->d_err;
    prm.ctl.wait_limit_ns = static_cast<unsigned long long>(pl->wait_limit_ns);
    const bool f32 = pl->o_dtype == CA_DTYPE_FP32;
    if (pl->d == 128)
        return f32 ? launch_fwd_t<128, true>(pl, tq, tk, tv, prm, stream)
                   : launch_fwd_t<128, false>(pl, tq, tk, tv, prm, stream);
    return f32 ? launch_fwd_t<64, true>(pl, tq, tk, tv, prm, stream)
               : launch_fwd_t<64, false>(pl, tq, tk, tv, prm, stream);
}

}  // namespace ca
