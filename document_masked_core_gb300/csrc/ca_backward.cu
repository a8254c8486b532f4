// Backward core attention over a rebatched pool of CA-tasks (sm_103a), with
// recompute: only LSE is kept from the forward (Efficient Long-context
// Language Model Training by Core Attention Disaggregation, §3.4
// "Property 1: Statelessness"; §3.2 "Information flow (backward pass)").
//
// Three launches:
//   1. preprocess   D_p = dO_p . O_p per (row, head); zero the fp32 dQ
//                   accumulator.  Memory-bound.
//   2. main         one persistent CTA per SM walks (document, kv head g,
//                   128-key tile) items, longest first.  K and V of the tile
//                   stay in shared memory; the CTA loops over every query tile
//                   (of every task of the document) that sees the key tile:
//                     S^T  = K Q^T          tcgen05, fp32 in TMEM
//                     dP^T = V dO^T         tcgen05, fp32 in TMEM
//                     P^T  = exp(scale S^T - LSE), dS^T = scale P^T (dP^T - D)
//                                           one thread per key row
//                     dV  += P^T dO         A = P^T (bf16) from TMEM
//                     dK  += dS^T Q         A = dS^T (bf16) from TMEM
//                     dQ   = dS K           A = dS (bf16, MN-major) in smem
//                   dK/dV accumulate in TMEM across all query tiles and all G
//                   heads of the group (no atomics); dQ of each pair goes from
//                   TMEM through shared memory into the fp32 accumulator by a
//                   TMA reduce-add.
//   3. finalize     fp32 dQ -> bf16.
#include <algorithm>
#include <cmath>

#include <cuda_bf16.h>

#include "ca_sm100.cuh"

namespace ca {
namespace {

using namespace dev;

// ------------------------------------------------------------------ preprocess
template <bool O_F32>
__global__ void __launch_bounds__(256) ca_bwd_pre_kernel(const void *o, const __nv_bfloat16 *d_o, float *D,
                                                          float *dq_acc, int64_t units, int32_t d,
                                                          int32_t *sched) {
    if (blockIdx.x == 0 && threadIdx.x == 0) *sched = 0;  // work queue of the main kernel
    const int32_t tpu = d / 8;  // 8 or 16 threads per (row, head), a power of two dividing 32
    const int64_t gtid = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    const int64_t unit = gtid / tpu;
    const int32_t part = static_cast<int32_t>(gtid % tpu);
    float acc = 0.f;
    if (unit < units) {
        const int64_t elem = unit * d + part * 8;
        const uint4 du = __ldg(reinterpret_cast<const uint4 *>(d_o + elem));
        const uint32_t dw[4] = {du.x, du.y, du.z, du.w};
        float ov[8];
        if (O_F32) {
            const float4 *src = reinterpret_cast<const float4 *>(static_cast<const float *>(o) + elem);
            const float4 a = __ldg(src), b = __ldg(src + 1);
            ov[0] = a.x; ov[1] = a.y; ov[2] = a.z; ov[3] = a.w;
            ov[4] = b.x; ov[5] = b.y; ov[6] = b.z; ov[7] = b.w;
        } else {
            const uint4 u = __ldg(reinterpret_cast<const uint4 *>(static_cast<const __nv_bfloat16 *>(o) + elem));
            const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                ov[2 * i] = __uint_as_float(w[i] << 16);
                ov[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
            }
        }
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            acc = fmaf(__uint_as_float(dw[i] << 16), ov[2 * i], acc);
            acc = fmaf(__uint_as_float(dw[i] & 0xFFFF0000u), ov[2 * i + 1], acc);
        }
        float4 *z = reinterpret_cast<float4 *>(dq_acc + elem);
        z[0] = make_float4(0.f, 0.f, 0.f, 0.f);
        z[1] = make_float4(0.f, 0.f, 0.f, 0.f);
    }
    for (int off = tpu / 2; off > 0; off >>= 1) acc += __shfl_down_sync(0xffffffffu, acc, off, tpu);
    if (unit < units && part == 0) D[unit] = acc;
}

// ------------------------------------------------------------------ finalize
__global__ void __launch_bounds__(256) ca_bwd_dq_kernel(const float *dq_acc, __nv_bfloat16 *dq, int64_t n8) {
    const int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    if (i >= n8) return;
    const float4 *src = reinterpret_cast<const float4 *>(dq_acc) + 2 * i;
    const float4 a = __ldg(src), b = __ldg(src + 1);
    uint4 w;
    w.x = pack_bf16(a.x, a.y);
    w.y = pack_bf16(a.z, a.w);
    w.z = pack_bf16(b.x, b.y);
    w.w = pack_bf16(b.z, b.w);
    reinterpret_cast<uint4 *>(dq)[i] = w;
}

// ------------------------------------------------------------------ main
struct BwdParams {
    const DevTask *tasks;
    const BwdItem *items;
    const int32_t *doc_task_ptr;
    const int32_t *doc_tasks;
    const int32_t *doc_info;  // {kv_off, doc_len} per document
    int32_t n_items;
    int32_t hq, hkv, G, tpt;
    float scale;       // softmax scale
    float scale_log2;  // softmax scale * log2(e)
    const float *lse;  // [total_q, hq]
    const float *Dvec; // [total_q, hq]
    int32_t *sched;    // work-queue counter (zeroed by the preprocess kernel)
    __nv_bfloat16 *dk, *dv;
    DevCtl ctl;
};

template <int D>
struct BwdCfg {
    static constexpr int kHalfBytes = 128 * 128;
    static constexpr int kTileBytes = (D / 64) * kHalfBytes;
    static constexpr int kQStages = 2;
    // dS (128 keys x 128 q rows bf16, 32 KB) lives in the dO tile of its query
    // tile once dV has read that tile, when the tile is large enough (D = 128);
    // otherwise in a buffer of its own.
    static constexpr bool kDsInDo = kTileBytes >= 2 * kHalfBytes;
    static constexpr int kOffK = 0;
    static constexpr int kOffV = kOffK + kTileBytes;
    static constexpr int kOffQ = kOffV + kTileBytes;
    static constexpr int kOffDO = kOffQ + kQStages * kTileBytes;
    static constexpr int kOffDS = kOffDO + kQStages * kTileBytes;    // own dS buffer (D = 64 only)
    static constexpr int kOffStg = kOffDS + (kDsInDo ? 0 : 2 * kHalfBytes);  // dQ staging, 2 boxes
    static constexpr int kOffRow = kOffStg + 2 * kHalfBytes;         // LSE2[2][128], D[2][128]
    static constexpr int kOffBar = kOffRow + 4 * 128 * 4;
    // No alignment slack: the dynamic shared window starts 1024-byte aligned
    // (checked at kernel entry).  At least 120 KB so one CTA runs per SM.
    static constexpr int kBarBytes = 512;  // BwdBars (checked below)
    static constexpr int kSmemRaw = kOffBar + kBarBytes;
    static constexpr int kSmemBytes = kSmemRaw > 122880 ? kSmemRaw : 122880;
    static_assert(kSmemBytes <= 232448, "backward tiles exceed 227 KB of shared memory");
    static constexpr uint32_t kTmemCols = 512;
    static constexpr uint32_t kColS = 0;     // S^T, then P^T (bf16)
    static constexpr uint32_t kColDP = 128;  // dP^T, then dS^T (bf16), then dQ (fp32, D columns)
    static constexpr uint32_t kColDV = 256;
    static constexpr uint32_t kColDK = 256 + D;
    // Packed bf16 P^T / dS^T: warpgroup w writes its 64 q rows (two per
    // column) to the first 32 of the 64 columns it read, so neither warpgroup
    // overwrites columns the other has yet to load.  K step kk (q rows
    // 16kk .. 16kk+15) of the dV / dK products starts at this column.
    __host__ __device__ static constexpr uint32_t packed_col(int kk) { return 8 * kk + (kk >= 4 ? 32 : 0); }
    static constexpr uint32_t kIdescST = idesc_bf16(128, 128, false, false);  // K-major x K-major
    static constexpr uint32_t kIdescAcc = idesc_bf16(128, D, false, true);    // TMEM A x MN-major B
    static constexpr uint32_t kIdescDQ = idesc_bf16(128, D, true, true);      // MN-major A x MN-major B
    // dQ staging for the TMA reduction: D/32 boxes of 32 fp32 columns x 128
    // rows (16 KB each, 128-byte swizzle).  With dS in the dO tile, boxes 0
    // and 1 go there too (dQ, the last reader of dS, has completed); the
    // others go to the staging buffer.  The Q tile is not used, so it returns
    // to the producer as soon as dK has read it.
    static constexpr int kDoBoxes = kDsInDo ? 2 : 0;
    static_assert(D / 32 - kDoBoxes == 2, "staging buffer holds two boxes");
    __device__ static uint32_t stage_box_off(int b, uint32_t st) {
        return b < kDoBoxes ? kOffDO + st * kTileBytes + b * kHalfBytes : kOffStg + (b - kDoBoxes) * kHalfBytes;
    }
    __device__ static uint32_t ds_off(uint32_t st) { return kDsInDo ? kOffDO + st * kTileBytes : kOffDS; }
    // Register split of the 512 threads (launch allocation 128 each):
    // gradient warpgroups, the warpgroup of single-warp roles, dQ warpgroup.
    static constexpr uint32_t kRegsLaunch = 128;  // 65536 / 512 threads
    static constexpr uint32_t kRegsGrad = 144, kRegsMisc = 88, kRegsDq = 136;
    static_assert(2 * kRegsGrad + kRegsMisc + kRegsDq <= 4 * kRegsLaunch, "register split exceeds the launch allocation");
};

// warps that read each ring entry: MMA, 8 gradient, flush, row statistics, 4 dQ
constexpr uint32_t kRingConsumers = 15;

struct BwdBars {
    uint64_t kv_full, kv_empty;
    uint64_t q_full[2], q_empty[2];    // Q tile of stage s (q_empty: committed after dK)
    uint64_t do_full[2], do_empty[2];  // dO tile of stage s (do_empty: its dQ staging was read)
    uint64_t s_full, dp_full, p_full, dq_full, dq_empty, stg_full, mma_done;
    uint64_t dst_full;      // dS^T of the current tile is in TMEM (dK may read it)
    uint64_t ds_full;       // dS of the current tile is in shared memory (dQ may read it)
    uint64_t acc_full;      // dK, dV of the item are complete (committed after its last dK)
    uint64_t acc_empty;     // the gradient warpgroups have read dK, dV out of TMEM
    uint64_t dv_done;       // dV of the current tile has read the dO tile (dS may overwrite it)
    uint64_t stg_empty;     // the staging buffer's boxes have been read by the reduction
    uint64_t row_full[2];   // row statistics of query tile t (buffer t % 2) are in shared memory
    uint64_t row_empty[2];  // the gradient warpgroups are done with buffer t % 2
    // work queue: the producer takes the next item from the global counter and
    // publishes it to the other roles through a 4-entry ring
    uint64_t ring_full[4], ring_empty[4];
    int32_t ring[4];
    uint32_t tmem_base;
    uint32_t abort_flag;
};

static_assert(sizeof(BwdBars) <= 512, "barrier block exceeds its shared-memory reservation");

struct KvGeo {
    int32_t doc, g, jt, n_q, kv_off, doc_len, t_begin, t_end;
};

__device__ __forceinline__ KvGeo decode_kv(const BwdParams &p, int32_t idx) {
    const BwdItem it = p.items[idx];
    KvGeo k;
    k.doc = it.doc;
    k.g = it.g;
    k.jt = it.kv_tile;
    k.n_q = it.n_q;
    k.kv_off = p.doc_info[2 * it.doc];
    k.doc_len = p.doc_info[2 * it.doc + 1];
    k.t_begin = p.doc_task_ptr[it.doc];
    k.t_end = p.doc_task_ptr[it.doc + 1];
    return k;
}

// Query tiles of task t that see key tile jt (same rule as the host plan):
// the rows of key_tile_rows inside the task.
__device__ __forceinline__ void task_tiles(const DevTask &t, int32_t jt, int32_t tpt, int32_t &first, int32_t &count) {
    first = 0;
    count = 0;
    int32_t pmin, pmax;
    key_tile_rows(t, jt * kTileKeys, &pmin, &pmax);
    const int32_t q0 = t.q_start, q1 = t.q_start + t.q_len - 1;
    const int32_t lo = max(pmin, q0), hi = min(pmax, q1);
    if (lo > hi) return;
    first = (lo - q0) / tpt;
    count = (hi - q0) / tpt - first + 1;
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

// Warp roles (512 threads, four warpgroups):
//   warps 0-7   gradient warpgroups (P^T, dS^T; dK/dV epilogue)
//   warp 8      TMA producer          warp 9   TMEM owner + MMA issuer
//   warp 10     dQ flush (TMA reduce) warp 11  row statistics (LSE, D)
//   warps 12-15 dQ readout: TMEM -> shared staging
// Per query tile t (in the order every role enumerates them):
//   MMA:      [dq_empty(t-1)] dP^T(t) | [p_full(t)] dV += P^T dO -> dv_done |
//             [dst_full(t)] dK += dS^T Q -> q_empty | S^T(t+1) when the item has a
//             next tile (S^T(first) at item start) | [ds_full(t)] dQ = dS K (into
//             the dP^T columns)
//   gradient: P^T(t) -> p_full | dS^T(t) to TMEM -> dst_full, then dS(t) into
//             the dO tile of t once dV has read it -> ds_full | P^T(t+1)
// The order keeps the dS stores beside a TS product (dK): an SS product reads
// 128 B of shared memory per clock and leaves other shared-memory traffic
// little bandwidth.
//   dQ warps: dQ(t) -> registers (all D columns) -> dq_empty -> staging in the
//             dO tile of t and the staging buffer -> stg_full
//   flush:    TMA reduce-adds of the staging into the fp32 accumulator; the
//             dO tile is released (do_empty) once its boxes have been read,
//             the staging buffer (stg_empty) once the others have.
template <int D>
__global__ void __launch_bounds__(512, 1)
    ca_bwd_main_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                       const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
                       const __grid_constant__ CUtensorMap tm_dq, const BwdParams p) {
    using C = BwdCfg<D>;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    if (smem_u32(smem_raw) & 1023u) {  // the swizzled tiles need 1024-byte alignment
        if (threadIdx.x == 0) atomicOr(p.ctl.err, kErrBounds);
        return;
    }
    uint8_t *smem = smem_raw;
    uint8_t *sK = smem + C::kOffK;
    uint8_t *sV = smem + C::kOffV;
    uint8_t *sQ = smem + C::kOffQ;
    uint8_t *sDO = smem + C::kOffDO;
    // row statistics of the query tile in each Q/dO stage, written by the
    // row-statistics warp: log2(e) LSE - log2(scale) (so exp2(scale log2(e) s
    // - that) = scale P) and -D
    float *sLse = reinterpret_cast<float *>(smem + C::kOffRow);  // [2][128]
    float *sD = sLse + 256;                                        // [2][128]
    BwdBars &bars = *reinterpret_cast<BwdBars *>(smem + C::kOffBar);

    const uint32_t warp = warp_id();
    const uint32_t lane = lane_id();

    if (threadIdx.x == 0) {
        mbar_init(&bars.kv_full, 1);
        mbar_init(&bars.kv_empty, 1);
        for (int s = 0; s < C::kQStages; ++s) {
            mbar_init(&bars.q_full[s], 1);
            mbar_init(&bars.q_empty[s], 1);
            mbar_init(&bars.do_full[s], 1);
            mbar_init(&bars.do_empty[s], 1);
        }
        mbar_init(&bars.s_full, 1);
        mbar_init(&bars.dp_full, 1);
        mbar_init(&bars.p_full, 8);  // one arrival per warp
        mbar_init(&bars.ds_full, 8);  // one arrival per warp
        mbar_init(&bars.dst_full, 8);  // one arrival per warp
        mbar_init(&bars.dq_full, 1);
        mbar_init(&bars.dq_empty, 4);  // one arrival per warp
        mbar_init(&bars.stg_full, 4);  // one arrival per warp
        mbar_init(&bars.mma_done, 1);
        mbar_init(&bars.acc_full, 1);
        mbar_init(&bars.acc_empty, 8);  // one arrival per warp
        mbar_init(&bars.dv_done, 1);
        mbar_init(&bars.stg_empty, 1);
        for (int b = 0; b < 2; ++b) {
            mbar_init(&bars.row_full[b], 1);   // one arrival per warp
            mbar_init(&bars.row_empty[b], 8);
        }
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
        tma_prefetch_desc(&tm_do);
        tma_prefetch_desc(&tm_dq);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = bars.tmem_base;
    const Watchdog wd{&p.ctl, &bars.abort_flag};

    if (warp >= 8 && warp < 12) {
        regs_set<C::kRegsMisc, C::kRegsLaunch>();
        if (warp == 8) {
            // ------------------------------------------------------------ producer (lane 0 issues)
            uint32_t act = 0, qt = 0;
            bool ok = true;
            for (uint32_t r = 0; ok; ++r) {
                // take the next item and publish it to the other roles
                int32_t idx = -1;
                if (lane == 0) {
                    ok = mbar_wait(&bars.ring_empty[r & 3], ((r >> 2) & 1) ^ 1, wd);
                    if (ok) idx = atomicAdd(p.sched, 1);
                    if (idx >= p.n_items) idx = -1;
                    bars.ring[r & 3] = idx;
                    mbar_arrive(&bars.ring_full[r & 3]);
                }
                ok = __shfl_sync(0xffffffffu, ok, 0);
                idx = __shfl_sync(0xffffffffu, idx, 0);
                if (!ok || idx < 0) break;
                const KvGeo kg = decode_kv(p, idx);
                if (kg.n_q == 0) continue;
                if (lane == 0) {
                    ok = mbar_wait(&bars.kv_empty, (act & 1) ^ 1, wd);
                    if (ok) {
                        const int32_t key_row = kg.kv_off + kg.jt * kTileKeys;
                        mbar_arrive_expect_tx(&bars.kv_full, 2 * C::kTileBytes);
#pragma unroll
                        for (int h = 0; h < D / 64; ++h) {
                            tma_load_3d(sK + h * C::kHalfBytes, &tm_k, &bars.kv_full, h * 64, kg.g, key_row);
                            tma_load_3d(sV + h * C::kHalfBytes, &tm_v, &bars.kv_full, h * 64, kg.g, key_row);
                        }
                    }
                }
                ok = __shfl_sync(0xffffffffu, ok, 0);
                for (int32_t k = kg.t_begin; k < kg.t_end && ok; ++k) {
                    const DevTask t = p.tasks[p.doc_tasks[k]];
                    int32_t first, count;
                    task_tiles(t, kg.jt, p.tpt, first, count);
                    for (int32_t tile = first; tile < first + count; ++tile, ++qt) {
                        const uint32_t st = qt % C::kQStages;
                        const int32_t qrow = t.row0 + tile * p.tpt;
                        if (lane == 0) {
                            ok = mbar_wait(&bars.q_empty[st], ((qt / C::kQStages) & 1) ^ 1, wd);
                            if (ok) {
                                mbar_arrive_expect_tx(&bars.q_full[st], C::kTileBytes);
#pragma unroll
                                for (int h = 0; h < D / 64; ++h)
                                    tma_load_3d(sQ + st * C::kTileBytes + h * C::kHalfBytes, &tm_q,
                                                &bars.q_full[st], h * 64, kg.g * p.G, qrow);
                            }
                            if (ok) ok = mbar_wait(&bars.do_empty[st], ((qt / C::kQStages) & 1) ^ 1, wd);
                            if (ok) {
                                mbar_arrive_expect_tx(&bars.do_full[st], C::kTileBytes);
#pragma unroll
                                for (int h = 0; h < D / 64; ++h)
                                    tma_load_3d(sDO + st * C::kTileBytes + h * C::kHalfBytes, &tm_do,
                                                &bars.do_full[st], h * 64, kg.g * p.G, qrow);
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
            // ------------------------------------------------------------ MMA issuer
            if (lane == 0) {
                uint32_t act = 0, qt = 0;
                bool ok = true;
                const uint32_t k_base = smem_u32(sK), v_base = smem_u32(sV), q_base = smem_u32(sQ),
                               do_base = smem_u32(sDO), smem_base = smem_u32(smem);
                // K and V tiles stay at fixed addresses: their descriptors (K-major for
                // S^T and dP^T, MN-major for dQ) are built once
                const uint32_t kd_k = sdesc_lo(k_base, 16), vd_k = sdesc_lo(v_base, 16),
                               kd_mn = sdesc_lo(k_base, C::kHalfBytes);
                // S^T = K Q^T of the query tile in ring slot qi
                auto issue_st = [&](uint32_t qi) -> bool {
                    const uint32_t st = qi % C::kQStages;
                    if (!mbar_wait(&bars.q_full[st], (qi / C::kQStages) & 1, wd)) return false;
                    tc_fence_after();
                    const uint32_t qd = sdesc_lo(q_base + st * C::kTileBytes, 16);
#pragma unroll
                    for (int kk = 0; kk < D / 16; ++kk) {
                        const uint32_t off = (kk / 4) * C::kHalfBytes + (kk % 4) * 32;
                        umma_ss(tmem + C::kColS, sdesc_at(kd_k, off), sdesc_at(qd, off), C::kIdescST,
                                kk > 0 ? 1u : 0u);
                    }
                    umma_commit(&bars.s_full);
                    return true;
                };
                for (uint32_t r = 0; ok; ++r) {
                    if (!(ok = mbar_wait(&bars.ring_full[r & 3], (r >> 2) & 1, wd))) break;
                    const int32_t idx = *reinterpret_cast<volatile int32_t *>(&bars.ring[r & 3]);
                    mbar_arrive(&bars.ring_empty[r & 3]);
                    if (idx < 0) break;
                    const KvGeo kg = decode_kv(p, idx);
                    if (kg.n_q == 0) continue;
                    if (!(ok = mbar_wait(&bars.kv_full, act & 1, wd))) break;
                    tc_fence_after();
                    if (!(ok = issue_st(qt))) break;
                    for (int32_t j = 0; j < kg.n_q && ok; ++j, ++qt) {
                        const uint32_t st = qt % C::kQStages;
                        const uint32_t qd_mn = sdesc_lo(q_base + st * C::kTileBytes, C::kHalfBytes);
                        const uint32_t dod = sdesc_lo(do_base + st * C::kTileBytes, 16);
                        const uint32_t dod_mn = sdesc_lo(do_base + st * C::kTileBytes, C::kHalfBytes);
                        // dP^T = V dO^T, once dQ of the previous tile has left the dP^T columns
                        if (!(ok = mbar_wait(&bars.do_full[st], (qt / C::kQStages) & 1, wd))) break;
                        if (!(ok = mbar_wait(&bars.dq_empty, (qt & 1) ^ 1, wd))) break;
                        tc_fence_after();
#pragma unroll
                        for (int kk = 0; kk < D / 16; ++kk) {
                            const uint32_t off = (kk / 4) * C::kHalfBytes + (kk % 4) * 32;
                            umma_ss(tmem + C::kColDP, sdesc_at(vd_k, off), sdesc_at(dod, off), C::kIdescST,
                                    kk > 0 ? 1u : 0u);
                        }
                        umma_commit(&bars.dp_full);
                        // dV += P^T dO
                        if (!(ok = mbar_wait(&bars.p_full, qt & 1, wd))) break;
                        if (j == 0 && !(ok = mbar_wait(&bars.acc_empty, (act & 1) ^ 1, wd))) break;
                        tc_fence_after();
#pragma unroll
                        for (int kk = 0; kk < 8; ++kk)
                            umma_ts(tmem + C::kColDV, tmem + C::kColS + C::packed_col(kk), sdesc_at(dod_mn, kk * 2048),
                                    C::kIdescAcc, (j == 0 && kk == 0) ? 0u : 1u);
                        if (C::kDsInDo) umma_commit(&bars.dv_done);
                        // dK += dS^T Q as soon as dS^T is in TMEM (a TS product: the gradient
                        // warpgroups' shared-memory stores of dS run beside it); the Q tile
                        // then goes back to the producer
                        if (!(ok = mbar_wait(&bars.dst_full, qt & 1, wd))) break;
                        tc_fence_after();
#pragma unroll
                        for (int kk = 0; kk < 8; ++kk)
                            umma_ts(tmem + C::kColDK, tmem + C::kColDP + C::packed_col(kk), sdesc_at(qd_mn, kk * 2048),
                                    C::kIdescAcc, (j == 0 && kk == 0) ? 0u : 1u);
                        umma_commit(&bars.q_empty[st]);
                        if (j + 1 == kg.n_q) umma_commit(&bars.acc_full);
                        // S^T of the next query tile of this key tile: the P^T columns
                        // are free once dV (issued above) has read them
                        if (j + 1 < kg.n_q && !(ok = issue_st(qt + 1))) break;
                        // dQ = dS K (into the dP^T columns, read by dK just before) once
                        // dS is in shared memory
                        if (!(ok = mbar_wait(&bars.ds_full, qt & 1, wd))) break;
                        tc_fence_after();
                        const uint32_t dsd = sdesc_lo(smem_base + C::ds_off(st), C::kHalfBytes);
#pragma unroll
                        for (int kk = 0; kk < 8; ++kk)
                            umma_ss(tmem + C::kColDP, sdesc_at(dsd, kk * 2048), sdesc_at(kd_mn, kk * 2048),
                                    C::kIdescDQ, kk > 0 ? 1u : 0u);
                        umma_commit(&bars.dq_full);
                    }
                    if (!ok) break;
                    umma_commit(&bars.kv_empty);
                    ++act;
                }
                umma_commit(&bars.mma_done);
                const DevCtl drain{p.ctl.err, p.ctl.wait_limit_ns};
                uint32_t zero = 0;
                const Watchdog wd2{&drain, &zero};
                mbar_wait(&bars.mma_done, 0, wd2);
            }
            __syncwarp();
        } else if (warp == 11) {
            // ------------------------------------------------------------ row statistics
            // All 32 lanes load LSE and D of each query tile's 128 rows from global
            // memory into a 2-entry buffer ring, ahead of the gradient warpgroups.
            uint32_t qt = 0;
            bool ok = true;
            const float log2_scale = lg2(p.scale);
            for (uint32_t r = 0; ok; ++r) {
                ok = __all_sync(0xffffffffu, mbar_wait(&bars.ring_full[r & 3], (r >> 2) & 1, wd));
                if (!ok) break;
                const int32_t idx = *reinterpret_cast<volatile int32_t *>(&bars.ring[r & 3]);
                __syncwarp();
                if (lane == 0) mbar_arrive(&bars.ring_empty[r & 3]);
                if (idx < 0) break;
                const KvGeo kg = decode_kv(p, idx);
                if (kg.n_q == 0) continue;
                for (int32_t k = kg.t_begin; k < kg.t_end && ok; ++k) {
                    const DevTask t = p.tasks[p.doc_tasks[k]];
                    int32_t first, count;
                    task_tiles(t, kg.jt, p.tpt, first, count);
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
                            const int32_t r = static_cast<int32_t>(lane) + 32 * j;
                            const int32_t tok = r / p.G;
                            l2[j] = INFINITY;
                            nd[j] = 0.f;
                            if (tok < ntok) {
                                const size_t ix = static_cast<size_t>(qrow + tok) * p.hq + kg.g * p.G + (r % p.G);
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
            // ------------------------------------------------------------ dQ flush
            // Lane 0: once the dQ warps have staged dQ of a query tile, add it
            // into the fp32 accumulator with TMA reduce-adds; release the dO
            // tile once its boxes have been read (the next dO load waits for
            // it), then the staging buffer.
            if (lane == 0) {
                uint32_t qt = 0;
                bool ok = true;
                for (uint32_t r = 0; ok; ++r) {
                    if (!(ok = mbar_wait(&bars.ring_full[r & 3], (r >> 2) & 1, wd))) break;
                    const int32_t idx = *reinterpret_cast<volatile int32_t *>(&bars.ring[r & 3]);
                    mbar_arrive(&bars.ring_empty[r & 3]);
                    if (idx < 0) break;
                    const KvGeo kg = decode_kv(p, idx);
                    if (kg.n_q == 0) continue;
                    for (int32_t k = kg.t_begin; k < kg.t_end && ok; ++k) {
                        const DevTask t = p.tasks[p.doc_tasks[k]];
                        int32_t first, count;
                        task_tiles(t, kg.jt, p.tpt, first, count);
                        for (int32_t tile = first; tile < first + count; ++tile, ++qt) {
                            const uint32_t st = qt % C::kQStages;
                            if (!(ok = mbar_wait(&bars.stg_full, qt & 1, wd))) break;
                            const int32_t qrow0 = t.row0 + tile * p.tpt;
#pragma unroll
                            for (int b = 0; b < C::kDoBoxes; ++b)
                                tma_reduce_add_3d(&tm_dq, smem + C::stage_box_off(b, st), b * 32, kg.g * p.G, qrow0);
                            bulk_commit_group();
#pragma unroll
                            for (int b = C::kDoBoxes; b < D / 32; ++b)
                                tma_reduce_add_3d(&tm_dq, smem + C::stage_box_off(b, st), b * 32, kg.g * p.G, qrow0);
                            bulk_commit_group();
                            bulk_wait_group_read1();
                            mbar_arrive(&bars.do_empty[st]);
                            bulk_wait_group_read0();
                            mbar_arrive(&bars.stg_empty);
                        }
                    }
                }
                bulk_wait_group0();  // every dQ reduction has completed before the CTA exits
            }
        }
    } else if (warp >= 12) {
        // ------------------------------------------------------------ dQ readout
        // Lane i = q row i of the tile: dQ (fp32, D columns of the dP^T region)
        // -> registers, all D columns before the TMEM columns are released (the
        // next dP^T waits for them) -> the staging boxes.
        regs_set<C::kRegsDq, C::kRegsLaunch>();
        const uint32_t i = threadIdx.x & 127u;
        const uint32_t lane_addr = ((warp & 3u) * 32u) << 16;
        uint32_t qt = 0;
        bool ok = true;
        for (uint32_t r = 0; ok; ++r) {
            ok = __all_sync(0xffffffffu, mbar_wait(&bars.ring_full[r & 3], (r >> 2) & 1, wd));
            if (!ok) break;
            const int32_t idx = *reinterpret_cast<volatile int32_t *>(&bars.ring[r & 3]);
            __syncwarp();
            if (lane == 0) mbar_arrive(&bars.ring_empty[r & 3]);
            if (idx < 0) break;
            const KvGeo kg = decode_kv(p, idx);
            if (kg.n_q == 0) continue;
            for (int32_t k = kg.t_begin; k < kg.t_end && ok; ++k) {
                const DevTask t = p.tasks[p.doc_tasks[k]];
                int32_t first, count;
                task_tiles(t, kg.jt, p.tpt, first, count);
                for (int32_t tile = first; tile < first + count; ++tile, ++qt) {
                    const uint32_t st = qt % C::kQStages;
                    const int32_t ntok = min(p.tpt, t.q_len - tile * p.tpt);
                    const bool row_ok = static_cast<int32_t>(i / p.G) < ntok;
                    ok = __all_sync(0xffffffffu, mbar_wait(&bars.dq_full, qt & 1, wd));
                    if (!ok) break;
                    tc_fence_after();
                    uint32_t qr[D / 32][32];
                    const uint32_t q_addr = tmem + lane_addr + C::kColDP;
#pragma unroll
                    for (int c = 0; c < D / 32; ++c) tmem_ld32(q_addr + 32 * c, qr[c]);
                    tmem_ld_wait();
#pragma unroll
                    for (int c = 0; c < D / 32; ++c) reg_fence(qr[c]);
                    tc_fence_before();
                    mbar_arrive_warp(&bars.dq_empty);
#pragma unroll
                    for (int b = 0; b < D / 32; ++b) {
                        if (b == C::kDoBoxes) {  // the remaining boxes go to the staging buffer
                            ok = __all_sync(0xffffffffu, mbar_wait(&bars.stg_empty, (qt & 1) ^ 1, wd));
                            if (!ok) break;
                        }
                        uint8_t *srow = smem + C::stage_box_off(b, st) + i * 128;
#pragma unroll
                        for (int c8 = 0; c8 < 8; ++c8) {
                            const uint4 v = row_ok ? make_uint4(qr[b][4 * c8], qr[b][4 * c8 + 1], qr[b][4 * c8 + 2],
                                                                qr[b][4 * c8 + 3])
                                                   : make_uint4(0, 0, 0, 0);
                            *reinterpret_cast<uint4 *>(srow + ((c8 ^ (i & 7)) * 16)) = v;
                        }
                    }
                    if (!ok) break;
                    fence_view_async_shared();
                    mbar_arrive_warp(&bars.stg_full);
                }
            }
        }
    } else {
        // ------------------------------------------------------------ gradient warpgroups
        // Warpgroup w (warps 4w .. 4w+3) owns query rows / S^T columns
        // 64w .. 64w+63 of every tile and head_dim columns D/2 w .. of dK, dV.
        regs_set<C::kRegsGrad, C::kRegsLaunch>();
        const int wg = static_cast<int>(warp >> 2);
        const uint32_t i = threadIdx.x & 127u;  // TMEM lane: key row of S^T, dP^T, dK, dV
        const uint32_t lane_addr = ((warp & 3u) * 32u) << 16;
        const int c0 = 64 * wg;
        const float inv_scale = 1.f / p.scale;
        const float2 c2 = make_float2(p.scale_log2, p.scale_log2);
        uint32_t qt = 0, act = 0;
        bool ok = true;
        for (uint32_t r = 0; ok; ++r) {
            ok = __all_sync(0xffffffffu, mbar_wait(&bars.ring_full[r & 3], (r >> 2) & 1, wd));
            if (!ok) break;
            const int32_t idx = *reinterpret_cast<volatile int32_t *>(&bars.ring[r & 3]);
            __syncwarp();
            if (lane == 0) mbar_arrive(&bars.ring_empty[r & 3]);
            if (idx < 0) break;
            const KvGeo kg = decode_kv(p, idx);
            const int32_t kpos = kg.jt * kTileKeys + static_cast<int32_t>(i);  // this thread's key
            const bool key_in_doc = kpos < kg.doc_len;
            const size_t key_out = (static_cast<size_t>(kg.kv_off) + kpos) * p.hkv + kg.g;
            if (kg.n_q == 0) {
                if (key_in_doc) {
                    uint4 *a = reinterpret_cast<uint4 *>(p.dk + key_out * D + wg * (D / 2));
                    uint4 *b = reinterpret_cast<uint4 *>(p.dv + key_out * D + wg * (D / 2));
#pragma unroll
                    for (int c = 0; c < D / 16; ++c) {
                        a[c] = make_uint4(0, 0, 0, 0);
                        b[c] = make_uint4(0, 0, 0, 0);
                    }
                }
                continue;
            }
            for (int32_t k = kg.t_begin; k < kg.t_end && ok; ++k) {
                const DevTask t = p.tasks[p.doc_tasks[k]];
                int32_t first, count;
                task_tiles(t, kg.jt, p.tpt, first, count);
                // rows that see this key: [kpos, row_end] (sink key: unbounded; window:
                // kpos + win - 1), none when the key is outside the block or below lo
                const bool key_in_block = kpos >= t.kv_start && kpos < t.kv_start + t.kv_len &&
                                          (kpos < t.sink || kpos >= t.lo);
                const int64_t row_end = (kpos < t.sink || t.win == 0) ? int64_t(1) << 40 : int64_t(kpos) + t.win - 1;
                for (int32_t tile = first; tile < first + count; ++tile, ++qt) {
                    const int32_t tok0 = tile * p.tpt;
                    const int32_t ntok = min(p.tpt, t.q_len - tok0);
                    const int32_t p_first = t.q_start + tok0;
                    const float *lse_b = sLse + (qt & 1) * 128;
                    const float *nd_b = sD + (qt & 1) * 128;
                    ok = __all_sync(0xffffffffu, mbar_wait(&bars.row_full[qt & 1], (qt >> 1) & 1, wd));
                    if (!ok) break;
                    // visible rows for this key: tile rows r (token r / G) with
                    // r_lo <= r < r_hi, i.e. kpos <= p <= row_end and the token inside the task
                    const int32_t tok_hi = static_cast<int32_t>(
                        row_end - p_first + 1 < ntok ? (row_end - p_first + 1 > 0 ? row_end - p_first + 1 : 0) : ntok);
                    const int32_t r_hi = tok_hi * p.G;
                    const int32_t r_lo = key_in_block ? min(max(kpos - p_first, 0) * p.G, r_hi) : r_hi;
                    const bool edge = r_lo > c0 || r_hi < c0 + 64;
                    // ---- P'^T = scale P^T = exp2(scale log2(e) S^T - log2(e) LSE + log2(scale))
                    ok = __all_sync(0xffffffffu, mbar_wait(&bars.s_full, qt & 1, wd));
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
                                const int r = c0 + e;
                                if (r < r_lo || r >= r_hi) pt[e] = 0.f;
                            }
                        }
                        uint32_t pk[32];
#pragma unroll
                        for (int w = 0; w < 32; ++w) pk[w] = pack_bf16(pt[2 * w], pt[2 * w + 1]);
                        tmem_st32(s_addr + c0, pk);  // q rows 64w.. packed two per column
                    }
                    tmem_st_wait();
                    tc_fence_before();
                    mbar_arrive_warp(&bars.p_full);
                    // ---- dS'^T = P'^T (dP^T - D) = scale dS^T: to TMEM (A of dK += dS^T Q) and
                    // to shared memory half w as the MN-major A of dQ = dS K (key row i
                    // holds q rows 64w .. 64w+63, 16-byte chunks swizzled by i % 8)
                    ok = __all_sync(0xffffffffu, mbar_wait(&bars.dp_full, qt & 1, wd));
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
                        for (int c = 0; c < 2; ++c) {  // q rows 64w + 32c ..
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
                        mbar_arrive_warp(&bars.dst_full);
                        // the dS buffer is free: dV has read the dO tile it shares, or
                        // the previous dQ has read the own buffer
                        ok = C::kDsInDo ? mbar_wait(&bars.dv_done, qt & 1, wd) : mbar_wait(&bars.dq_full, (qt & 1) ^ 1, wd);
                        ok = __all_sync(0xffffffffu, ok);
                        if (ok) {
                            uint8_t *row = smem + C::ds_off(qt % C::kQStages) + wg * C::kHalfBytes + i * 128;
#pragma unroll
                            for (int c8 = 0; c8 < 8; ++c8)  // 16-byte chunk: q rows 8 c8 .. 8 c8 + 7 of the half
                                *reinterpret_cast<uint4 *>(row + ((c8 ^ (i & 7)) * 16)) =
                                    make_uint4(pk[c8 >> 2][4 * (c8 & 3)], pk[c8 >> 2][4 * (c8 & 3) + 1],
                                               pk[c8 >> 2][4 * (c8 & 3) + 2], pk[c8 >> 2][4 * (c8 & 3) + 3]);
                        }
                    }
                    if (!ok) break;
                    mbar_arrive_warp(&bars.row_empty[qt & 1]);  // row statistics of this tile no longer read
                    fence_view_async_shared();
                    mbar_arrive_warp(&bars.ds_full);
                }
            }
            if (!ok) break;
            // ---- epilogue: dK, dV of this key tile (lane i = key i, columns D/2 w ..)
            // once the item's last dK has completed.  The dV accumulator holds
            // scale dV (it summed P' = scale P).
            ok = __all_sync(0xffffffffu, mbar_wait(&bars.acc_full, act & 1, wd));
            if (!ok) break;
            tc_fence_after();
            {
                const uint32_t dv_addr = tmem + lane_addr + C::kColDV + wg * (D / 2);
                const uint32_t dk_addr = tmem + lane_addr + C::kColDK + wg * (D / 2);
#pragma unroll
                for (int c = 0; c < D / 64; ++c) {
                    uint32_t a[32], b[32];
                    tmem_ld32(dv_addr + c * 32, a);
                    tmem_ld32(dk_addr + c * 32, b);
                    tmem_ld_wait();
                    reg_fence(a);
                    reg_fence(b);
                    if (key_in_doc) {
                        uint4 *va = reinterpret_cast<uint4 *>(p.dv + key_out * D + wg * (D / 2) + c * 32);
                        uint4 *kb = reinterpret_cast<uint4 *>(p.dk + key_out * D + wg * (D / 2) + c * 32);
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
                mbar_arrive_warp(&bars.acc_empty);
            }
            ++act;
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 9) {
        tc_fence_after();
        tmem_dealloc(tmem, C::kTmemCols);
    }
}

cudaError_t launch_dq_finalize(const ca_plan *pl, const float *dq_acc, void *dq, cudaStream_t stream) {
    const int64_t n8 = pl->total_q * pl->hq * pl->d / 8;
    const unsigned blocks = static_cast<unsigned>((n8 + 255) / 256);
    ca_bwd_dq_kernel<<<blocks, 256, 0, stream>>>(dq_acc, static_cast<__nv_bfloat16 *>(dq), n8);
    cudaError_t e = cudaGetLastError();
    if (e == cudaSuccess) e = mark(pl, 5, stream);
    return e;
}

template <int D>
cudaError_t launch_main_t(const ca_plan *pl, const CUtensorMap &tq, const CUtensorMap &tk, const CUtensorMap &tv,
                          const CUtensorMap &tdo, const CUtensorMap &tdq, const BwdParams &prm,
                          cudaStream_t stream) {
    using C = BwdCfg<D>;
    auto kern = ca_bwd_main_kernel<D>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
    if (e != cudaSuccess) return e;
    // The warpgroups' register increases draw on the CTA's launch allocation
    // (512 threads x registers per thread): refuse to launch a build whose
    // allocation could not cover the split, where an increase would block.
    cudaFuncAttributes fa;
    e = cudaFuncGetAttributes(&fa, kern);
    if (e != cudaSuccess) return e;
    if (fa.numRegs * 4 < static_cast<int>(2 * C::kRegsGrad + C::kRegsMisc + C::kRegsDq)) {
        set_error("backward main kernel was built with " + std::to_string(fa.numRegs) +
                  " registers per thread, below its warpgroup register split");
        return cudaErrorInvalidConfiguration;
    }
    const int grid = static_cast<int>(std::min<int64_t>(pl->n_bwd, pl->num_sms));
    if (grid <= 0) return cudaSuccess;
    kern<<<grid, 512, C::kSmemBytes, stream>>>(tq, tk, tv, tdo, tdq, prm);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_backward(const ca_plan *pl, const void *q, const void *k, const void *v, const void *o,
                            const float *lse, const void *d_o, void *dq, void *dk, void *dv, void *workspace,
                            cudaStream_t stream) {
    const int64_t units = pl->total_q * pl->hq;
    float *dq_acc = static_cast<float *>(workspace);
    float *Dvec = reinterpret_cast<float *>(static_cast<uint8_t *>(workspace) +
                                            (units * pl->d * 4 + 255) / 256 * 256);
    int32_t *sched = work_counters(pl, workspace);
    // 1. D = rowsum(dO * O), dQ accumulator = 0
    {
        cudaError_t e0 = mark(pl, 2, stream);
        if (e0 != cudaSuccess) return e0;
        const int64_t threads = units * (pl->d / 8);
        const unsigned blocks = static_cast<unsigned>((threads + 255) / 256);
        if (pl->o_dtype == CA_DTYPE_FP32)
            ca_bwd_pre_kernel<true><<<blocks, 256, 0, stream>>>(o, static_cast<const __nv_bfloat16 *>(d_o), Dvec,
                                                                dq_acc, units, pl->d, sched);
        else
            ca_bwd_pre_kernel<false><<<blocks, 256, 0, stream>>>(o, static_cast<const __nv_bfloat16 *>(d_o), Dvec,
                                                                 dq_acc, units, pl->d, sched);
        cudaError_t e = cudaGetLastError();
        if (e == cudaSuccess) e = mark(pl, 3, stream);
        if (e != cudaSuccess) return e;
    }
    // 2. main pass: on CTA pairs where the plan selects them
    if (use_bwd_pair(pl)) {
        cudaError_t e = launch_bwd_main_pair(pl, q, k, v, d_o, dq_acc, lse, Dvec, sched, dk, dv, stream);
        if (e == cudaSuccess) e = mark(pl, 4, stream);
        if (e != cudaSuccess) return e;
        return launch_dq_finalize(pl, dq_acc, dq, stream);
    }
    CUtensorMap tq, tk, tv, tdo, tdq;
    if (make_tmap_3d(&tq, q, pl->total_q, pl->hq, pl->d, pl->G, pl->tpt) != CA_OK ||
        make_tmap_3d(&tdq, dq_acc, pl->total_q, pl->hq, pl->d, pl->G, pl->tpt, true) != CA_OK ||
        make_tmap_3d(&tdo, d_o, pl->total_q, pl->hq, pl->d, pl->G, pl->tpt) != CA_OK ||
        make_tmap_3d(&tk, k, pl->total_kv, pl->hkv, pl->d, 1, kTileKeys) != CA_OK ||
        make_tmap_3d(&tv, v, pl->total_kv, pl->hkv, pl->d, 1, kTileKeys) != CA_OK)
        return cudaErrorInvalidValue;
    BwdParams prm;
    prm.tasks = pl->d_tasks;
    prm.items = pl->d_bwd;
    prm.doc_task_ptr = pl->d_doc_task_ptr;
    prm.doc_tasks = pl->d_doc_tasks;
    prm.doc_info = pl->d_doc_info;
    prm.n_items = static_cast<int32_t>(pl->n_bwd);
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
    cudaError_t e = pl->d == 128 ? launch_main_t<128>(pl, tq, tk, tv, tdo, tdq, prm, stream)
                                 : launch_main_t<64>(pl, tq, tk, tv, tdo, tdq, prm, stream);
    if (e == cudaSuccess) e = mark(pl, 4, stream);
    if (e != cudaSuccess) return e;
    // 3. dQ accumulator -> bf16
    return launch_dq_finalize(pl, dq_acc, dq, stream);
}

}  // namespace ca
