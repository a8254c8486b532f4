// Backward main pass on CTA pairs (head_dim 128, a number of query heads per
// kv head that divides 64): the recompute backward of core attention (Efficient Long-context
// Language Model Training by Core Attention Disaggregation, §3.4 "Property 1:
// Statelessness"; §3.2 "Information flow (backward pass)") with the same
// products as the one-CTA kernel in ca_backward.cu, computed by two SMs at once.
//
// A cluster of two CTAs takes an item (document, kv head g, key-tile pair jp):
// CTA r holds key tile 2 jp + r (K, V resident) and, for every query tile of
// the document that sees either key tile, rank 0 issues tcgen05 pair products
// (cta_group::2) in which each SM computes the rows of its own key tile:
//   S^T  = K Q^T       M = 256 (128 keys per CTA), N = 128 query rows; each
//   dP^T = V dO^T      CTA supplies 64 of the query rows (B operand halves)
//   dV  += P^T dO      M = 256, N = 128 = head_dim; A = P^T from each CTA's
//   dK  += dS^T Q      TMEM, each CTA supplies half of head_dim of B
//   dQ   = dS K        M = 128: CTA r computes query rows 64 r .. 64 r + 63
//                      over both key tiles (K = 256), half of head_dim of B
// so each SM reads half of every B operand it used to read alone and reduces
// half of each query tile's dQ.  The element-wise passes (P^T, dS^T, one
// thread per key row of the CTA's own tile) are those of the one-CTA kernel;
// the only data that crosses the pair is dS: the warpgroup of CTA r that owns
// query rows 64 w .. 64 w + 63 writes its dS rows into CTA w's shared memory.
//
// Shared memory per CTA (226.5 KB): K, V of its key tile (K-major, 32 KB
// each); KD = both key tiles' K in its half of head_dim (B of dQ, 32 KB); two
// Q stages and two dO stages of 32 KB, each = its 64 query rows x head_dim
// (B of S^T / dP^T) + all 128 rows x its half of head_dim (B of dK / dV).  A
// dO stage then holds dS (256 key rows x its 64 query rows, A of dQ) and
// finally the dQ staging of its 64 rows for the TMA reduce-add.
//
// Barriers: the full barriers of the loads (both CTAs' TMA loads signal rank
// 0's) and every barrier the MMA thread waits on live in rank 0; the pair's
// commits arrive on both CTAs' barriers (multicast); each CTA's roles arrive
// on rank 0's barriers with cluster-scope release.  Every wait is bounded.
#include <algorithm>
#include <cmath>

#include <cuda_bf16.h>

#include "ca_sm100.cuh"

namespace ca {
namespace {

using namespace dev;

struct PairParams {
    const DevTask *tasks;
    const BwdItem *items;  // kv_tile = pair index jp
    const int32_t *doc_task_ptr;
    const int32_t *doc_tasks;
    const int32_t *doc_info;  // {kv_off, doc_len} per document
    int32_t n_items;
    int32_t hq, hkv, G, tpt;
    float scale, scale_log2;
    const float *lse;
    const float *Dvec;
    int32_t *sched;
    __nv_bfloat16 *dk, *dv;
    DevCtl ctl;
};

struct PairCfg {
    static constexpr int D = 128;
    static constexpr int kHalf = 128 * 128;     // 128 rows x 128 bytes (64 bf16)
    static constexpr int kQuarter = 64 * 128;   // 64 rows x 128 bytes
    static constexpr int kStage = 2 * kHalf;    // one Q or dO stage
    static constexpr int kOffK = 0;
    static constexpr int kOffV = kOffK + 2 * kHalf;
    static constexpr int kOffKD = kOffV + 2 * kHalf;
    static constexpr int kOffQ = kOffKD + 2 * kHalf;
    static constexpr int kOffDO = kOffQ + 2 * kStage;
    static constexpr int kOffRow = kOffDO + 2 * kStage;  // LSE2[2][128], -D[2][128]
    static constexpr int kOffBar = kOffRow + 4 * 128 * 4;
    static constexpr int kBarBytes = 512;
    static constexpr int kSmemBytes = kOffBar + kBarBytes;
    static_assert(kSmemBytes <= 232448, "pair backward tiles exceed 227 KB of shared memory");
    // Inside a stage: rows 64 r .. 64 r + 63 of the tile, both halves of
    // head_dim (two 8 KB boxes), then all 128 rows of this CTA's half.
    static constexpr int kOffRowsHalf = 0;
    static constexpr int kOffColsHalf = kHalf;
    static constexpr uint32_t kTmemCols = 512;
    static constexpr uint32_t kColS = 0;     // S^T, then P^T (bf16)
    static constexpr uint32_t kColDP = 128;  // dP^T, then dS^T (bf16), then dQ (fp32, 64 columns)
    static constexpr uint32_t kColDV = 256;
    static constexpr uint32_t kColDK = 384;
    // packed P^T / dS^T columns of K step kk (query rows 16 kk ..), as in the one-CTA kernel
    __host__ __device__ static constexpr uint32_t packed_col(int kk) { return 8 * kk + (kk >= 4 ? 32 : 0); }
    static constexpr uint32_t kIdescST = idesc_bf16(256, 128, false, false);  // pair, K-major x K-major
    static constexpr uint32_t kIdescAcc = idesc_bf16(256, D, false, true);    // pair, TMEM A x MN-major B
    static constexpr uint32_t kIdescDQ = idesc_bf16(128, D, true, true);      // pair M = 128, MN-major A and B
    static constexpr uint32_t kRegsLaunch = 128;
    static constexpr uint32_t kRegsGrad = 144, kRegsMisc = 88, kRegsDq = 136;
    static_assert(2 * kRegsGrad + kRegsMisc + kRegsDq <= 4 * kRegsLaunch, "register split exceeds the launch allocation");
};

// Suspend-time hint of the waits (ns).
constexpr uint32_t kPairHintNs = 1000;

// Waits and arrivals of the per-tile hand-offs between the pair's roles.  They
// publish TMEM contents (ordered by tcgen05.wait and the tcgen05 thread-sync
// fences) or the completion of the pair's own products, so they synchronise
// at CTA scope; a cluster-scope release made every hand-off about twice as
// slow.  The two that publish generic-proxy data across the pair -- the work
// queue ring and the dS rows written into the peer's shared memory -- use
// cluster scope (mbar_wait_cl, mbar_arrive_cl).
__device__ __forceinline__ bool pair_wait(uint64_t *bar, uint32_t parity, const Watchdog &wd) {
    return mbar_wait(bar, parity, wd);
}
__device__ __forceinline__ void pair_arrive_warp(uint32_t cl_addr) {
    __syncwarp();
    if ((threadIdx.x & 31u) == 0) mbar_arrive_cl_cta(cl_addr);
}

// ring consumers per CTA: rank 0 = MMA, 8 gradient, flush, row statistics,
// 4 dQ warps; rank 1 = producer and the same 14 others
constexpr uint32_t kPairRingConsumers = 30;

struct PairBars {
    uint64_t kv_full, kv_empty;        // kv_full: rank 0's, the loads of both CTAs
    uint64_t q_full[2], q_empty[2];    // q_full: rank 0's; q_empty: pair commit after dK
    uint64_t do_full[2], do_empty[2];  // do_full: rank 0's; do_empty: this CTA's flush
    uint64_t s_full, dp_full, dv_done, dq_full, acc_full;  // pair commits (both CTAs)
    uint64_t p_full, dst_full, ds_full, dq_empty, acc_empty;  // rank 0's: arrivals of both CTAs
    uint64_t stg_full;                 // this CTA's dQ staging is written
    uint64_t mma_done;
    uint64_t row_full[2], row_empty[2];
    uint64_t ring_full[4], ring_empty[4];  // ring_empty: rank 0's
    int32_t ring[4];
    uint32_t tmem_base;
    uint32_t abort_flag;
};
static_assert(sizeof(PairBars) <= PairCfg::kBarBytes, "barrier block exceeds its shared-memory reservation");

struct PairGeo {
    int32_t doc, g, jp, n_q, kv_off, doc_len, t_begin, t_end;
};

__device__ __forceinline__ PairGeo decode_pair(const PairParams &p, int32_t idx) {
    const BwdItem it = p.items[idx];
    PairGeo k;
    k.doc = it.doc;
    k.g = it.g;
    k.jp = it.kv_tile;
    k.n_q = it.n_q;
    k.kv_off = p.doc_info[2 * it.doc];
    k.doc_len = p.doc_info[2 * it.doc + 1];
    k.t_begin = p.doc_task_ptr[it.doc];
    k.t_end = p.doc_task_ptr[it.doc + 1];
    return k;
}

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

// Warp roles per CTA (512 threads), as in the one-CTA kernel: warps 0-7
// gradient warpgroups, 8 TMA producer, 9 MMA issuer (rank 0; TMEM owner in
// both), 10 dQ flush, 11 row statistics, 12-15 dQ readout.
__global__ void __launch_bounds__(512, 1)
    ca_bwd_pair_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_qn,
                       const __grid_constant__ CUtensorMap tm_do, const __grid_constant__ CUtensorMap tm_don,
                       const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                       const __grid_constant__ CUtensorMap tm_dq, const PairParams p) {
    using C = PairCfg;
    extern __shared__ __align__(1024) uint8_t smem[];
    if (smem_u32(smem) & 1023u) {  // the same in both CTAs: both leave before any cluster operation
        if (threadIdx.x == 0) atomicOr(p.ctl.err, kErrBounds);
        return;
    }
    uint8_t *sK = smem + C::kOffK;
    uint8_t *sV = smem + C::kOffV;
    uint8_t *sKD = smem + C::kOffKD;
    uint8_t *sQ = smem + C::kOffQ;
    uint8_t *sDO = smem + C::kOffDO;
    float *sLse = reinterpret_cast<float *>(smem + C::kOffRow);  // [2][128]
    float *sD = sLse + 256;                                        // [2][128]
    PairBars &bars = *reinterpret_cast<PairBars *>(smem + C::kOffBar);

    const uint32_t warp = warp_id();
    const uint32_t lane = lane_id();
    const uint32_t rank = cluster_ctarank();
    const int32_t half_tok = p.tpt / 2;  // query tokens of a CTA's 64 rows

    if (threadIdx.x == 0) {
        mbar_init(&bars.kv_full, 1);
        mbar_init(&bars.kv_empty, 1);
        for (int s = 0; s < 2; ++s) {
            mbar_init(&bars.q_full[s], 1);
            mbar_init(&bars.q_empty[s], 1);
            mbar_init(&bars.do_full[s], 1);
            mbar_init(&bars.do_empty[s], 1);
            mbar_init(&bars.row_full[s], 1);
            mbar_init(&bars.row_empty[s], 8);
        }
        mbar_init(&bars.s_full, 1);
        mbar_init(&bars.dp_full, 1);
        mbar_init(&bars.dv_done, 1);
        mbar_init(&bars.dq_full, 1);
        mbar_init(&bars.acc_full, 1);
        mbar_init(&bars.p_full, 16);    // one arrival per gradient warp of both CTAs
        mbar_init(&bars.dst_full, 16);
        mbar_init(&bars.ds_full, 16);
        mbar_init(&bars.dq_empty, 8);   // one per dQ warp of both CTAs
        mbar_init(&bars.acc_empty, 16);
        mbar_init(&bars.stg_full, 4);
        mbar_init(&bars.mma_done, 1);
        for (int r = 0; r < 4; ++r) {
            mbar_init(&bars.ring_full[r], 1);
            mbar_init(&bars.ring_empty[r], kPairRingConsumers);
            bars.ring[r] = -1;
        }
        bars.abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 9) {
        tmem_alloc_pair(&bars.tmem_base, C::kTmemCols);
        tmem_relinquish_pair();
    }
    if (warp == 8 && lane == 0) {
        tma_prefetch_desc(&tm_q);
        tma_prefetch_desc(&tm_qn);
        tma_prefetch_desc(&tm_do);
        tma_prefetch_desc(&tm_don);
        tma_prefetch_desc(&tm_k);
        tma_prefetch_desc(&tm_v);
        tma_prefetch_desc(&tm_dq);
    }
    tc_fence_before();
    cluster_sync();  // both CTAs' barriers initialised and the pair's TMEM allocated
    tc_fence_after();
    const uint32_t tmem = bars.tmem_base;
    const Watchdog wd{&p.ctl, &bars.abort_flag};
    // rank 0's barriers as cluster addresses
    auto lead = [&](uint64_t *bar) -> uint32_t { return mapa_shared(smem_u32(bar), 0); };

    // Every role enumerates the query tiles of an item in the same order.
    auto ring_take = [&](uint32_t r, bool &ok) -> int32_t {
        ok = mbar_wait_cl<kPairHintNs>(&bars.ring_full[r & 3], (r >> 2) & 1, wd);
        if (!ok) return -1;
        int32_t idx = *reinterpret_cast<volatile int32_t *>(&bars.ring[r & 3]);
        mbar_arrive_cl(lead(&bars.ring_empty[r & 3]));
        if (idx >= p.n_items) idx = -1;  // never index the item list out of range
        return idx;
    };

    if (warp >= 8 && warp < 12) {
        regs_set<C::kRegsMisc, C::kRegsLaunch>();
        if (warp == 8) {
            // ------------------------------------------------------------ producer (lane 0 issues)
            uint32_t act = 0, qt = 0;
            bool ok = true;
            const uint32_t kv_full_cl = lead(&bars.kv_full);
            for (uint32_t r = 0; ok; ++r) {
                int32_t idx = -1;
                if (lane == 0) {
                    if (rank == 0) {
                        // take the next item and publish it to both CTAs
                        ok = mbar_wait_cl<kPairHintNs>(&bars.ring_empty[r & 3], ((r >> 2) & 1) ^ 1, wd);
                        if (ok) idx = atomicAdd(p.sched, 1);
                        if (idx >= p.n_items) idx = -1;
                        bars.ring[r & 3] = idx;
                        st_cluster_b32(mapa_shared(smem_u32(&bars.ring[r & 3]), 1), static_cast<uint32_t>(idx));
                        mbar_arrive_cl(mapa_shared(smem_u32(&bars.ring_full[r & 3]), 0));
                        mbar_arrive_cl(mapa_shared(smem_u32(&bars.ring_full[r & 3]), 1));
                    } else {
                        idx = ring_take(r, ok);
                    }
                }
                ok = __shfl_sync(0xffffffffu, ok, 0);
                idx = __shfl_sync(0xffffffffu, idx, 0);
                if (!ok || idx < 0) break;
                const PairGeo kg = decode_pair(p, idx);
                if (kg.n_q == 0) continue;
                if (lane == 0) {
                    ok = pair_wait(&bars.kv_empty, (act & 1) ^ 1, wd);
                    if (ok) {
                        if (rank == 0) mbar_arrive_expect_tx(&bars.kv_full, 2 * 6 * C::kHalf);  // K, V, KD of both CTAs
                        const int32_t row_a = kg.kv_off + 2 * kg.jp * kTileKeys;  // key tile 2 jp
                        const int32_t row_own = row_a + static_cast<int32_t>(rank) * kTileKeys;
#pragma unroll
                        for (int h = 0; h < 2; ++h) {
                            tma_load_3d_pair(sK + h * C::kHalf, &tm_k, kv_full_cl, h * 64, kg.g, row_own);
                            tma_load_3d_pair(sV + h * C::kHalf, &tm_v, kv_full_cl, h * 64, kg.g, row_own);
                        }
                        tma_load_3d_pair(sKD, &tm_k, kv_full_cl, static_cast<int32_t>(rank) * 64, kg.g, row_a);
                        tma_load_3d_pair(sKD + C::kHalf, &tm_k, kv_full_cl, static_cast<int32_t>(rank) * 64, kg.g,
                                         row_a + kTileKeys);
                    }
                }
                ok = __shfl_sync(0xffffffffu, ok, 0);
                for (int32_t k = kg.t_begin; k < kg.t_end && ok; ++k) {
                    const DevTask t = p.tasks[p.doc_tasks[k]];
                    int32_t first, count;
                    key_pair_query_tiles(t, kg.jp, p.tpt, &first, &count);
                    for (int32_t tile = first; tile < first + count; ++tile, ++qt) {
                        const uint32_t st = qt & 1;
                        const int32_t qrow = t.row0 + tile * p.tpt;
                        const int32_t qrow_half = qrow + static_cast<int32_t>(rank) * half_tok;
                        if (lane == 0) {
                            ok = pair_wait(&bars.q_empty[st], ((qt >> 1) & 1) ^ 1, wd);
                            if (ok) {
                                const uint32_t full = lead(&bars.q_full[st]);
                                if (rank == 0) mbar_arrive_expect_tx(&bars.q_full[st], 2 * C::kStage);
                                uint8_t *dst = sQ + st * C::kStage;
                                tma_load_3d_pair(dst + C::kOffRowsHalf, &tm_qn, full, 0, kg.g * p.G, qrow_half);
                                tma_load_3d_pair(dst + C::kOffRowsHalf + C::kQuarter, &tm_qn, full, 64, kg.g * p.G,
                                                 qrow_half);
                                tma_load_3d_pair(dst + C::kOffColsHalf, &tm_q, full, static_cast<int32_t>(rank) * 64,
                                                 kg.g * p.G, qrow);
                            }
                            if (ok) ok = pair_wait(&bars.do_empty[st], ((qt >> 1) & 1) ^ 1, wd);
                            if (ok) {
                                const uint32_t full = lead(&bars.do_full[st]);
                                if (rank == 0) mbar_arrive_expect_tx(&bars.do_full[st], 2 * C::kStage);
                                uint8_t *dst = sDO + st * C::kStage;
                                tma_load_3d_pair(dst + C::kOffRowsHalf, &tm_don, full, 0, kg.g * p.G, qrow_half);
                                tma_load_3d_pair(dst + C::kOffRowsHalf + C::kQuarter, &tm_don, full, 64, kg.g * p.G,
                                                 qrow_half);
                                tma_load_3d_pair(dst + C::kOffColsHalf, &tm_do, full, static_cast<int32_t>(rank) * 64,
                                                 kg.g * p.G, qrow);
                            }
                        }
                        ok = __shfl_sync(0xffffffffu, ok, 0);
                        if (!ok) break;
                    }
                }
                ++act;
            }
            if (!ok && lane == 0) __nanosleep(1000000);  // let copies already in flight land before the CTA drains
        } else if (warp == 9) {
            // ------------------------------------------------------------ MMA issuer (rank 0, lane 0)
            if (rank == 0 && lane == 0) {
                uint32_t act = 0, qt = 0;
                bool ok = true;
                const uint32_t k_base = smem_u32(sK), v_base = smem_u32(sV), kd_base = smem_u32(sKD),
                               q_base = smem_u32(sQ), do_base = smem_u32(sDO);
                const uint32_t kd_k = sdesc_lo(k_base, 16), vd_k = sdesc_lo(v_base, 16),
                               kdd = sdesc_lo(kd_base, C::kHalf);
                // S^T = K Q^T of the query tile in stage slot qi % 2
                auto issue_st = [&](uint32_t qi) -> bool {
                    const uint32_t st = qi & 1;
                    if (!pair_wait(&bars.q_full[st], (qi >> 1) & 1, wd)) return false;
                    tc_fence_after();
                    const uint32_t qn = sdesc_lo(q_base + st * C::kStage + C::kOffRowsHalf, 16);
#pragma unroll
                    for (int kk = 0; kk < 8; ++kk)
                        umma_pair_ss(tmem + C::kColS, sdesc_at(kd_k, (kk / 4) * C::kHalf + (kk % 4) * 32),
                                     sdesc_at(qn, (kk / 4) * C::kQuarter + (kk % 4) * 32), C::kIdescST,
                                     kk > 0 ? 1u : 0u);
                    umma_pair_commit_both(&bars.s_full);
                    return true;
                };
                for (uint32_t r = 0; ok; ++r) {
                    const int32_t idx = ring_take(r, ok);
                    if (!ok || idx < 0) break;
                    const PairGeo kg = decode_pair(p, idx);
                    if (kg.n_q == 0) continue;
                    if (!(ok = pair_wait(&bars.kv_full, act & 1, wd))) break;
                    tc_fence_after();
                    if (!(ok = issue_st(qt))) break;
                    for (int32_t j = 0; j < kg.n_q && ok; ++j, ++qt) {
                        const uint32_t st = qt & 1;
                        const uint32_t stage_q = q_base + st * C::kStage, stage_do = do_base + st * C::kStage;
                        const uint32_t qd_mn = sdesc_lo(stage_q + C::kOffColsHalf, C::kHalf);
                        const uint32_t don = sdesc_lo(stage_do + C::kOffRowsHalf, 16);
                        const uint32_t dod_mn = sdesc_lo(stage_do + C::kOffColsHalf, C::kHalf);
                        // dP^T = V dO^T, once dQ of the previous tile has left the dP^T columns
                        if (!(ok = pair_wait(&bars.do_full[st], (qt >> 1) & 1, wd))) break;
                        if (!(ok = pair_wait(&bars.dq_empty, (qt & 1) ^ 1, wd))) break;
                        tc_fence_after();
#pragma unroll
                        for (int kk = 0; kk < 8; ++kk)
                            umma_pair_ss(tmem + C::kColDP, sdesc_at(vd_k, (kk / 4) * C::kHalf + (kk % 4) * 32),
                                         sdesc_at(don, (kk / 4) * C::kQuarter + (kk % 4) * 32), C::kIdescST,
                                         kk > 0 ? 1u : 0u);
                        umma_pair_commit_both(&bars.dp_full);
                        // dV += P^T dO
                        if (!(ok = pair_wait(&bars.p_full, qt & 1, wd))) break;
                        if (j == 0 && !(ok = pair_wait(&bars.acc_empty, (act & 1) ^ 1, wd))) break;
                        tc_fence_after();
#pragma unroll
                        for (int kk = 0; kk < 8; ++kk)
                            umma_pair_ts(tmem + C::kColDV, tmem + C::kColS + C::packed_col(kk),
                                         sdesc_at(dod_mn, kk * 2048), C::kIdescAcc, (j == 0 && kk == 0) ? 0u : 1u);
                        umma_pair_commit_both(&bars.dv_done);
                        // dK += dS^T Q as soon as dS^T is in TMEM; the Q stage then goes back
                        if (!(ok = pair_wait(&bars.dst_full, qt & 1, wd))) break;
                        tc_fence_after();
#pragma unroll
                        for (int kk = 0; kk < 8; ++kk)
                            umma_pair_ts(tmem + C::kColDK, tmem + C::kColDP + C::packed_col(kk),
                                         sdesc_at(qd_mn, kk * 2048), C::kIdescAcc, (j == 0 && kk == 0) ? 0u : 1u);
                        umma_pair_commit_both(&bars.q_empty[st]);
                        if (j + 1 == kg.n_q) umma_pair_commit_both(&bars.acc_full);
                        // S^T of the next query tile (the P^T columns were read by dV above)
                        if (j + 1 < kg.n_q && !(ok = issue_st(qt + 1))) break;
                        // dQ = dS K over both key tiles, once both CTAs' dS rows are in place
                        if (!(ok = mbar_wait_cl<kPairHintNs>(&bars.ds_full, qt & 1, wd))) break;
                        tc_fence_after();
                        const uint32_t dsd = sdesc_lo(stage_do, C::kHalf);
#pragma unroll
                        for (int kk = 0; kk < 16; ++kk)
                            umma_pair_ss(tmem + C::kColDP, sdesc_at(dsd, kk * 2048), sdesc_at(kdd, kk * 2048),
                                         C::kIdescDQ, kk > 0 ? 1u : 0u);
                        umma_pair_commit_both(&bars.dq_full);
                    }
                    if (!ok) break;
                    umma_pair_commit_both(&bars.kv_empty);
                    ++act;
                }
                umma_pair_commit(&bars.mma_done);
                const DevCtl drain{p.ctl.err, p.ctl.wait_limit_ns};
                uint32_t zero = 0;
                const Watchdog wd2{&drain, &zero};
                pair_wait(&bars.mma_done, 0, wd2);
            }
            __syncwarp();
        } else if (warp == 11) {
            // ------------------------------------------------------------ row statistics (all 128 rows)
            uint32_t qt = 0;
            bool ok = true;
            const float log2_scale = lg2(p.scale);
            for (uint32_t r = 0; ok; ++r) {
                int32_t idx = -1;
                if (lane == 0) idx = ring_take(r, ok);
                ok = __shfl_sync(0xffffffffu, ok, 0);
                idx = __shfl_sync(0xffffffffu, idx, 0);
                if (!ok || idx < 0) break;
                const PairGeo kg = decode_pair(p, idx);
                if (kg.n_q == 0) continue;
                for (int32_t k = kg.t_begin; k < kg.t_end && ok; ++k) {
                    const DevTask t = p.tasks[p.doc_tasks[k]];
                    int32_t first, count;
                    key_pair_query_tiles(t, kg.jp, p.tpt, &first, &count);
                    for (int32_t tile = first; tile < first + count; ++tile, ++qt) {
                        const uint32_t b = qt & 1;
                        ok = __all_sync(0xffffffffu, mbar_wait(&bars.row_empty[b], ((qt >> 1) & 1) ^ 1, wd));
                        if (!ok) break;
                        const int32_t tok0 = tile * p.tpt;
                        const int32_t qrow = t.row0 + tok0;
                        const int32_t ntok = min(p.tpt, t.q_len - tok0);
                        float l2[4], nd[4];
#pragma unroll
                        for (int j = 0; j < 4; ++j) {
                            const int32_t rr = static_cast<int32_t>(lane) + 32 * j;
                            const int32_t tok = rr / p.G;
                            l2[j] = INFINITY;
                            nd[j] = 0.f;
                            if (tok < ntok) {
                                const size_t ix = static_cast<size_t>(qrow + tok) * p.hq + kg.g * p.G + (rr % p.G);
                                const float l = __ldg(p.lse + ix);
                                l2[j] = (l == -INFINITY) ? INFINITY : l * 1.4426950408889634f - log2_scale;
                                nd[j] = -__ldg(p.Dvec + ix);
                            }
                        }
#pragma unroll
                        for (int j = 0; j < 4; ++j) {
                            sLse[b * 128 + lane + 32 * j] = l2[j];
                            sD[b * 128 + lane + 32 * j] = nd[j];
                        }
                        mbar_arrive_warp(&bars.row_full[b]);
                    }
                }
            }
        } else {
            // ------------------------------------------------------------ dQ flush (lane 0)
            // Adds this CTA's 64 staged dQ rows into the fp32 accumulator, then
            // releases the dO stage that held them.
            if (lane == 0) {
                uint32_t qt = 0;
                bool ok = true;
                for (uint32_t r = 0; ok; ++r) {
                    const int32_t idx = ring_take(r, ok);
                    if (!ok || idx < 0) break;
                    const PairGeo kg = decode_pair(p, idx);
                    if (kg.n_q == 0) continue;
                    for (int32_t k = kg.t_begin; k < kg.t_end && ok; ++k) {
                        const DevTask t = p.tasks[p.doc_tasks[k]];
                        int32_t first, count;
                        key_pair_query_tiles(t, kg.jp, p.tpt, &first, &count);
                        for (int32_t tile = first; tile < first + count; ++tile, ++qt) {
                            const uint32_t st = qt & 1;
                            if (!(ok = mbar_wait(&bars.stg_full, qt & 1, wd))) break;
                            const int32_t qrow_half = t.row0 + tile * p.tpt + static_cast<int32_t>(rank) * half_tok;
#pragma unroll
                            for (int b = 0; b < 4; ++b)
                                tma_reduce_add_3d(&tm_dq, sDO + st * C::kStage + b * C::kQuarter, b * 32, kg.g * p.G,
                                                  qrow_half);
                            bulk_commit_group();
                            bulk_wait_group_read0();
                            mbar_arrive(&bars.do_empty[st]);
                        }
                    }
                }
                bulk_wait_group0();  // every dQ reduction has completed before the CTA exits
            }
        }
    } else if (warp >= 12) {
        // ------------------------------------------------------------ dQ readout
        // TMEM lanes 0-63 hold this CTA's 64 query rows x head_dim 0..63, lanes
        // 64-127 the same rows x head_dim 64..127 (64 columns).  Warp q reads
        // 32 lanes (rows 32 (q & 1) .., half q >> 1) into registers, releases the
        // columns, then stages its rows into the dO stage of the tile (boxes of
        // 32 fp32 columns x 64 rows, 128-byte swizzle).
        regs_set<C::kRegsDq, C::kRegsLaunch>();
        const uint32_t quad = warp & 3u;
        const uint32_t row = (quad & 1u) * 32u + lane;  // 0..63
        const int dhalf = static_cast<int>(quad >> 1);
        const uint32_t lane_addr = (quad * 32u) << 16;
        const uint32_t dq_empty_cl = lead(&bars.dq_empty);
        uint32_t qt = 0;
        bool ok = true;
        for (uint32_t r = 0; ok; ++r) {
            int32_t idx = -1;
            if (lane == 0) idx = ring_take(r, ok);
            ok = __shfl_sync(0xffffffffu, ok, 0);
            idx = __shfl_sync(0xffffffffu, idx, 0);
            if (!ok || idx < 0) break;
            const PairGeo kg = decode_pair(p, idx);
            if (kg.n_q == 0) continue;
            for (int32_t k = kg.t_begin; k < kg.t_end && ok; ++k) {
                const DevTask t = p.tasks[p.doc_tasks[k]];
                int32_t first, count;
                key_pair_query_tiles(t, kg.jp, p.tpt, &first, &count);
                for (int32_t tile = first; tile < first + count; ++tile, ++qt) {
                    const uint32_t st = qt & 1;
                    const int32_t ntok = min(p.tpt, t.q_len - tile * p.tpt);
                    const bool row_ok = static_cast<int32_t>(rank) * half_tok + static_cast<int32_t>(row) / p.G < ntok;
                    ok = __all_sync(0xffffffffu, pair_wait(&bars.dq_full, qt & 1, wd));
                    if (!ok) break;
                    tc_fence_after();
                    uint32_t qr[2][32];
                    tmem_ld32(tmem + lane_addr + C::kColDP, qr[0]);
                    tmem_ld32(tmem + lane_addr + C::kColDP + 32, qr[1]);
                    tmem_ld_wait();
                    reg_fence(qr[0]);
                    reg_fence(qr[1]);
                    tc_fence_before();
                    pair_arrive_warp(dq_empty_cl);
#pragma unroll
                    for (int c = 0; c < 2; ++c) {
                        uint8_t *srow = sDO + st * C::kStage + (2 * dhalf + c) * C::kQuarter + row * 128;
#pragma unroll
                        for (int c8 = 0; c8 < 8; ++c8) {
                            const uint4 v = row_ok ? make_uint4(qr[c][4 * c8], qr[c][4 * c8 + 1], qr[c][4 * c8 + 2],
                                                                qr[c][4 * c8 + 3])
                                                   : make_uint4(0, 0, 0, 0);
                            *reinterpret_cast<uint4 *>(srow + ((c8 ^ (row & 7)) * 16)) = v;
                        }
                    }
                    fence_view_async_shared();
                    mbar_arrive_warp(&bars.stg_full);
                }
            }
        }
    } else {
        // ------------------------------------------------------------ gradient warpgroups
        // Warpgroup w owns S^T columns (query rows) 64 w .. 64 w + 63 of the
        // CTA's key tile and head_dim columns 64 w .. of its dK, dV epilogue.
        regs_set<C::kRegsGrad, C::kRegsLaunch>();
        const int wg = static_cast<int>(warp >> 2);
        const uint32_t i = threadIdx.x & 127u;  // key row of this CTA's tile
        const uint32_t lane_addr = ((warp & 3u) * 32u) << 16;
        const int c0 = 64 * wg;
        const float inv_scale = 1.f / p.scale;
        const float2 c2 = make_float2(p.scale_log2, p.scale_log2);
        const uint32_t p_full_cl = lead(&bars.p_full), dst_full_cl = lead(&bars.dst_full),
                       ds_full_cl = lead(&bars.ds_full), acc_empty_cl = lead(&bars.acc_empty);
        // this thread's dS row in the dS buffer of CTA wg (rows 128 rank .. of the 256 key rows)
        const uint32_t ds_row_off = C::kOffDO + (rank * 128u + i) * 128u;
        uint32_t qt = 0, act = 0;
        bool ok = true;
        for (uint32_t r = 0; ok; ++r) {
            int32_t idx = -1;
            if (lane == 0) idx = ring_take(r, ok);
            ok = __shfl_sync(0xffffffffu, ok, 0);
            idx = __shfl_sync(0xffffffffu, idx, 0);
            if (!ok || idx < 0) break;
            const PairGeo kg = decode_pair(p, idx);
            const int32_t kpos = (2 * kg.jp + static_cast<int32_t>(rank)) * kTileKeys + static_cast<int32_t>(i);
            const bool key_in_doc = kpos < kg.doc_len;
            const size_t key_out = (static_cast<size_t>(kg.kv_off) + kpos) * p.hkv + kg.g;
            if (kg.n_q == 0) {
                if (key_in_doc) {
                    uint4 *a = reinterpret_cast<uint4 *>(p.dk + key_out * C::D + wg * (C::D / 2));
                    uint4 *b = reinterpret_cast<uint4 *>(p.dv + key_out * C::D + wg * (C::D / 2));
#pragma unroll
                    for (int c = 0; c < C::D / 16; ++c) {
                        a[c] = make_uint4(0, 0, 0, 0);
                        b[c] = make_uint4(0, 0, 0, 0);
                    }
                }
                continue;
            }
            for (int32_t k = kg.t_begin; k < kg.t_end && ok; ++k) {
                const DevTask t = p.tasks[p.doc_tasks[k]];
                int32_t first, count;
                key_pair_query_tiles(t, kg.jp, p.tpt, &first, &count);
                const bool key_in_block = kpos >= t.kv_start && kpos < t.kv_start + t.kv_len &&
                                          (kpos < t.sink || kpos >= t.lo);
                const int64_t row_end = (kpos < t.sink || t.win == 0) ? int64_t(1) << 40 : int64_t(kpos) + t.win - 1;
                for (int32_t tile = first; tile < first + count; ++tile, ++qt) {
                    const uint32_t st = qt & 1;
                    const int32_t tok0 = tile * p.tpt;
                    const int32_t ntok = min(p.tpt, t.q_len - tok0);
                    const int32_t p_first = t.q_start + tok0;
                    const float *lse_b = sLse + st * 128;
                    const float *nd_b = sD + st * 128;
                    ok = __all_sync(0xffffffffu, mbar_wait(&bars.row_full[st], (qt >> 1) & 1, wd));
                    if (!ok) break;
                    const int32_t tok_hi = static_cast<int32_t>(
                        row_end - p_first + 1 < ntok ? (row_end - p_first + 1 > 0 ? row_end - p_first + 1 : 0) : ntok);
                    const int32_t r_hi = tok_hi * p.G;
                    const int32_t r_lo = key_in_block ? min(max(kpos - p_first, 0) * p.G, r_hi) : r_hi;
                    const bool edge = r_lo > c0 || r_hi < c0 + 64;
                    // ---- P'^T = scale P^T
                    ok = __all_sync(0xffffffffu, pair_wait(&bars.s_full, qt & 1, wd));
                    if (!ok) break;
                    tc_fence_after();
                    float pt[64];
                    const uint32_t s_addr = tmem + lane_addr + C::kColS;
                    {
                        uint32_t sr[2][32];
                        tmem_ld32(s_addr + c0, sr[0]);
                        tmem_ld32(s_addr + c0 + 32, sr[1]);
                        tmem_ld_wait();
                        reg_fence(sr[0]);
                        reg_fence(sr[1]);
                        const float2 *l2p = reinterpret_cast<const float2 *>(lse_b + c0);
#pragma unroll
                        for (int e = 0; e < 64; e += 2) {
                            const float2 s2 = make_float2(__uint_as_float(sr[e >> 5][e & 31]),
                                                          __uint_as_float(sr[e >> 5][(e & 31) + 1]));
                            const float2 nl = l2p[e / 2];
                            const float2 x = __ffma2_rn(s2, c2, make_float2(-nl.x, -nl.y));
                            pt[e] = ex2(x.x);
                            pt[e + 1] = ex2(x.y);
                        }
                        if (edge) {
#pragma unroll
                            for (int e = 0; e < 64; ++e) {
                                const int rr = c0 + e;
                                if (rr < r_lo || rr >= r_hi) pt[e] = 0.f;
                            }
                        }
                        uint32_t pk[32];
#pragma unroll
                        for (int w = 0; w < 32; ++w) pk[w] = pack_bf16(pt[2 * w], pt[2 * w + 1]);
                        tmem_st32(s_addr + c0, pk);
                    }
                    tmem_st_wait();
                    tc_fence_before();
                    pair_arrive_warp(p_full_cl);
                    // ---- dS'^T = P'^T (dP^T - D): to TMEM (A of dK), and its rows to
                    // the dS buffer of CTA wg (MN-major A of dQ, 128-byte swizzle)
                    ok = __all_sync(0xffffffffu, pair_wait(&bars.dp_full, qt & 1, wd));
                    if (!ok) break;
                    tc_fence_after();
                    {
                        const uint32_t dp_addr = tmem + lane_addr + C::kColDP;
                        const float2 *nd2 = reinterpret_cast<const float2 *>(nd_b + c0);
                        uint32_t dr[2][32];
                        tmem_ld32(dp_addr + c0, dr[0]);
                        tmem_ld32(dp_addr + c0 + 32, dr[1]);
                        tmem_ld_wait();
                        reg_fence(dr[0]);
                        reg_fence(dr[1]);
                        uint32_t pk[2][16];
#pragma unroll
                        for (int c = 0; c < 2; ++c) {
#pragma unroll
                            for (int e = 0; e < 32; e += 2) {
                                const float2 d2 = make_float2(__uint_as_float(dr[c][e]), __uint_as_float(dr[c][e + 1]));
                                const float2 x = __fmul2_rn(make_float2(pt[32 * c + e], pt[32 * c + e + 1]),
                                                            __fadd2_rn(d2, nd2[16 * c + e / 2]));
                                pk[c][e / 2] = pack_bf16(x.x, x.y);
                            }
                        }
                        tmem_st16(dp_addr + c0, pk[0]);
                        tmem_st16(dp_addr + c0 + 16, pk[1]);
                        tmem_st_wait();
                        tc_fence_before();
                        pair_arrive_warp(dst_full_cl);
                        // both CTAs' dO stages are free once the pair's dV has read them
                        ok = __all_sync(0xffffffffu, pair_wait(&bars.dv_done, qt & 1, wd));
                        if (ok) {
                            const uint32_t row_off = ds_row_off + st * C::kStage;
                            if (wg == static_cast<int>(rank)) {
                                uint8_t *rowp = smem + row_off;
#pragma unroll
                                for (int c8 = 0; c8 < 8; ++c8)
                                    *reinterpret_cast<uint4 *>(rowp + ((c8 ^ (i & 7)) * 16)) =
                                        make_uint4(pk[c8 >> 2][4 * (c8 & 3)], pk[c8 >> 2][4 * (c8 & 3) + 1],
                                                   pk[c8 >> 2][4 * (c8 & 3) + 2], pk[c8 >> 2][4 * (c8 & 3) + 3]);
                            } else {
                                const uint32_t rowc = mapa_shared(smem_u32(smem) + row_off, static_cast<uint32_t>(wg));
#pragma unroll
                                for (int c8 = 0; c8 < 8; ++c8)
                                    st_cluster_v4(rowc + ((c8 ^ (i & 7)) * 16),
                                                  make_uint4(pk[c8 >> 2][4 * (c8 & 3)], pk[c8 >> 2][4 * (c8 & 3) + 1],
                                                             pk[c8 >> 2][4 * (c8 & 3) + 2], pk[c8 >> 2][4 * (c8 & 3) + 3]));
                            }
                        }
                    }
                    if (!ok) break;
                    mbar_arrive_warp(&bars.row_empty[st]);
                    // the dS rows are read by the pair's dQ product (async proxy): rows
                    // written into the peer's shared memory are published at cluster
                    // scope, rows written here at CTA scope
                    if (wg == static_cast<int>(rank)) {
                        fence_view_async_shared();
                        pair_arrive_warp(ds_full_cl);
                    } else {
                        fence_view_async_cluster();
                        mbar_arrive_warp_cl(ds_full_cl);
                    }
                }
            }
            if (!ok) break;
            // ---- epilogue: dK, dV of this CTA's key tile once the item's last dK completed
            ok = __all_sync(0xffffffffu, pair_wait(&bars.acc_full, act & 1, wd));
            if (!ok) break;
            tc_fence_after();
            {
                const uint32_t dv_addr = tmem + lane_addr + C::kColDV + wg * (C::D / 2);
                const uint32_t dk_addr = tmem + lane_addr + C::kColDK + wg * (C::D / 2);
#pragma unroll
                for (int c = 0; c < C::D / 64; ++c) {
                    uint32_t a[32], b[32];
                    tmem_ld32(dv_addr + c * 32, a);
                    tmem_ld32(dk_addr + c * 32, b);
                    tmem_ld_wait();
                    reg_fence(a);
                    reg_fence(b);
                    if (key_in_doc) {
                        uint4 *va = reinterpret_cast<uint4 *>(p.dv + key_out * C::D + wg * (C::D / 2) + c * 32);
                        uint4 *kb = reinterpret_cast<uint4 *>(p.dk + key_out * C::D + wg * (C::D / 2) + c * 32);
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            va[e] = make_uint4(
                                pack_bf16(__uint_as_float(a[8 * e]) * inv_scale, __uint_as_float(a[8 * e + 1]) * inv_scale),
                                pack_bf16(__uint_as_float(a[8 * e + 2]) * inv_scale, __uint_as_float(a[8 * e + 3]) * inv_scale),
                                pack_bf16(__uint_as_float(a[8 * e + 4]) * inv_scale, __uint_as_float(a[8 * e + 5]) * inv_scale),
                                pack_bf16(__uint_as_float(a[8 * e + 6]) * inv_scale, __uint_as_float(a[8 * e + 7]) * inv_scale));
                            kb[e] = make_uint4(pack_bf16(__uint_as_float(b[8 * e]), __uint_as_float(b[8 * e + 1])),
                                               pack_bf16(__uint_as_float(b[8 * e + 2]), __uint_as_float(b[8 * e + 3])),
                                               pack_bf16(__uint_as_float(b[8 * e + 4]), __uint_as_float(b[8 * e + 5])),
                                               pack_bf16(__uint_as_float(b[8 * e + 6]), __uint_as_float(b[8 * e + 7])));
                        }
                    }
                }
                tc_fence_before();
                pair_arrive_warp(acc_empty_cl);
            }
            ++act;
        }
    }

    tc_fence_before();
    __syncthreads();
    cluster_sync();  // no CTA leaves while its peer may still touch its shared memory or TMEM
    if (warp == 9) {
        tc_fence_after();
        tmem_dealloc_pair(tmem, C::kTmemCols);
    }
}

}  // namespace

cudaError_t launch_bwd_main_pair(const ca_plan *pl, const void *q, const void *k, const void *v, const void *d_o,
                                 float *dq_acc, const float *lse, const float *Dvec, int32_t *sched, void *dk,
                                 void *dv, cudaStream_t stream) {
    using C = PairCfg;
    if (pl->d != C::D || 64 % pl->G != 0 || pl->n_bwd_pair <= 0) return cudaErrorInvalidValue;
    const int32_t half = pl->tpt / 2;
    CUtensorMap tq, tqn, tdo, tdon, tk, tv, tdq;
    if (make_tmap_3d(&tq, q, pl->total_q, pl->hq, pl->d, pl->G, pl->tpt) != CA_OK ||
        make_tmap_3d(&tqn, q, pl->total_q, pl->hq, pl->d, pl->G, half) != CA_OK ||
        make_tmap_3d(&tdo, d_o, pl->total_q, pl->hq, pl->d, pl->G, pl->tpt) != CA_OK ||
        make_tmap_3d(&tdon, d_o, pl->total_q, pl->hq, pl->d, pl->G, half) != CA_OK ||
        make_tmap_3d(&tk, k, pl->total_kv, pl->hkv, pl->d, 1, kTileKeys) != CA_OK ||
        make_tmap_3d(&tv, v, pl->total_kv, pl->hkv, pl->d, 1, kTileKeys) != CA_OK ||
        make_tmap_3d(&tdq, dq_acc, pl->total_q, pl->hq, pl->d, pl->G, half, true) != CA_OK)
        return cudaErrorInvalidValue;
    PairParams prm;
    prm.tasks = pl->d_tasks;
    prm.items = pl->d_bwd_pair;
    prm.doc_task_ptr = pl->d_doc_task_ptr;
    prm.doc_tasks = pl->d_doc_tasks;
    prm.doc_info = pl->d_doc_info;
    prm.n_items = static_cast<int32_t>(pl->n_bwd_pair);
    prm.hq = pl->hq;
    prm.hkv = pl->hkv;
    prm.G = pl->G;
    prm.tpt = pl->tpt;
    prm.scale = pl->scale;
    prm.scale_log2 = pl->scale * 1.4426950408889634f;
    prm.lse = lse;
    prm.Dvec = Dvec;
    prm.sched = sched;
    prm.dk = static_cast<__nv_bfloat16 *>(dk);
    prm.dv = static_cast<__nv_bfloat16 *>(dv);
    prm.ctl.err = pl->d_err;
    prm.ctl.wait_limit_ns = static_cast<unsigned long long>(pl->wait_limit_ns);

    auto kern = ca_bwd_pair_kernel;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
    if (e != cudaSuccess) return e;
    cudaFuncAttributes fa;
    if ((e = cudaFuncGetAttributes(&fa, kern)) != cudaSuccess) return e;
    if (fa.numRegs * 4 < static_cast<int>(2 * C::kRegsGrad + C::kRegsMisc + C::kRegsDq)) {
        set_error("pair backward kernel was built with " + std::to_string(fa.numRegs) +
                  " registers per thread, below its warpgroup register split");
        return cudaErrorInvalidConfiguration;
    }
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.blockDim = dim3(512, 1, 1);
    cfg.dynamicSmemBytes = C::kSmemBytes;
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cfg.gridDim = dim3(static_cast<unsigned>(pl->num_sms & ~1), 1, 1);
    int max_clusters = 0;
    if ((e = cudaOccupancyMaxActiveClusters(&max_clusters, kern, &cfg)) != cudaSuccess) return e;
    if (max_clusters < 1) {
        set_error("no CTA pair of the backward kernel fits on the device");
        return cudaErrorInvalidConfiguration;
    }
    const int64_t clusters = std::min<int64_t>(pl->n_bwd_pair, max_clusters);
    cfg.gridDim = dim3(static_cast<unsigned>(2 * clusters), 1, 1);
    e = cudaLaunchKernelEx(&cfg, kern, tq, tqn, tdo, tdon, tk, tv, tdq, prm);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

}  // namespace ca
