// Host side of the C ABI: argument validation, integer accounting, the
// forward/backward tile lists (longest first), device upload, tensor maps and
// the entry points declared in include/ca.h.
#include <algorithm>
#include <cmath>
#include <cstring>
#include <mutex>
#include <new>
#include <numeric>
#include <string>
#include <vector>

#include <cudaTypedefs.h>

#include "ca_internal.h"

namespace ca {

namespace {
thread_local std::string g_last_error;

// Pairs of one task: sum over rows p in [q0, q0 + ql) of
// |{j : a <= j < e, j <= p}|, by splitting the rows into the ramp
// a <= p < e - 1 (p - a + 1 keys) and the plateau p >= e - 1 (e - a keys).
int64_t task_pairs_closed_form(int64_t q0, int64_t ql, int64_t a, int64_t kl) {
    const int64_t e = a + kl;
    const int64_t q1 = q0 + ql;  // exclusive
    int64_t total = 0;
    const int64_t r0 = std::max(q0, a), r1 = std::min(q1, e - 1);
    if (r1 > r0) {
        // sum_{p=r0}^{r1-1} (p - a + 1)
        const int64_t first = r0 - a + 1, last = r1 - 1 - a + 1, n = r1 - r0;
        total += (first + last) * n / 2;
    }
    const int64_t s0 = std::max(q0, e - 1);
    if (q1 > s0) total += (q1 - s0) * kl;
    return total;
}

// Pairs of a masked task, row by row: |[a, r1) U [r2, hi)| for every row.
int64_t task_pairs_rows(const DevTask &t) {
    int64_t total = 0;
    for (int32_t p = t.q_start; p < t.q_start + t.q_len; ++p) {
        const RowKeys k = row_keys(t, p);
        const int64_t c1 = std::max(0, k.r1 - k.a);
        const int64_t lo2 = std::max(k.r2, k.a);
        const int64_t c2 = std::max<int64_t>(0, k.hi - lo2);
        const int64_t ov = std::max<int64_t>(0, std::min<int64_t>(k.r1, k.hi) - lo2);
        total += c1 + c2 - ov;
    }
    return total;
}

// Query tiles of task t that see key tile jt (mirrored by the backward
// kernel): the rows of key_tile_rows inside the task.  Returns the first tile
// and the count.
void bwd_task_tiles(const DevTask &t, int32_t jt, int32_t tpt, int32_t *first, int32_t *count) {
    *first = 0;
    *count = 0;
    int32_t pmin, pmax;
    key_tile_rows(t, jt * kTileKeys, &pmin, &pmax);
    const int32_t q0 = t.q_start, q1 = t.q_start + t.q_len - 1;  // inclusive
    const int32_t lo = std::max(pmin, q0), hi = std::min(pmax, q1);
    if (lo > hi) return;
    *first = (lo - q0) / tpt;
    *count = (hi - q0) / tpt - *first + 1;
}

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;

}  // namespace

void set_error(const std::string &msg) { g_last_error = msg; }

ca_status_t fail(ca_status_t st, const std::string &msg) {
    g_last_error = msg;
    return st;
}

ca_status_t cuda_fail(cudaError_t e, const char *what) {
    g_last_error = std::string(what) + ": " + cudaGetErrorString(e);
    return CA_ERR_CUDA;
}

ca_status_t check_plan_device(const ca_plan *p) {
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    if (dev != p->device)
        return fail(CA_ERR_INVALID_ARG, "the plan was created on device " + std::to_string(p->device) +
                                            " but device " + std::to_string(dev) + " is current");
    return CA_OK;
}

ca_status_t check_backward_args(const ca_plan *p, const void *q, const void *k, const void *v, const void *o,
                                const void *lse, const void *d_o, const void *dq, const void *dk, const void *dv,
                                const void *scratch, int64_t scratch_bytes) {
    const void *in[] = {q, k, v, o, lse, d_o};
    const void *out[] = {dq, dk, dv, scratch};
    for (const void *x : in)
        if (!x) return fail(CA_ERR_INVALID_ARG, "NULL pointer");
    for (const void *x : out)
        if (!x) return fail(CA_ERR_INVALID_ARG, "NULL pointer");
    for (const void *x : in)
        if (reinterpret_cast<uintptr_t>(x) & 15u) return fail(CA_ERR_INVALID_ARG, "pointers must be 16-byte aligned");
    for (const void *x : out)
        if (reinterpret_cast<uintptr_t>(x) & 15u) return fail(CA_ERR_INVALID_ARG, "pointers must be 16-byte aligned");
    const int64_t q_b = p->total_q * p->hq * p->d * 2, kv_b = p->total_kv * p->hkv * p->d * 2;
    const int64_t o_b = p->total_q * p->hq * p->d * (p->o_dtype == CA_DTYPE_FP32 ? 4 : 2);
    const int64_t lse_b = p->total_q * p->hq * 4;
    const int64_t in_n[] = {q_b, kv_b, kv_b, o_b, lse_b, q_b};
    const int64_t out_n[] = {q_b, kv_b, kv_b, scratch_bytes};
    auto overlaps = [](const void *a, int64_t na, const void *b, int64_t nb) {
        const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
        return na > 0 && nb > 0 && x < y + static_cast<uintptr_t>(nb) && y < x + static_cast<uintptr_t>(na);
    };
    // outputs (dq, dk, dv, the scratch) must not share a byte with each other or with an input
    for (int i = 0; i < 4; ++i) {
        for (int j = i + 1; j < 4; ++j)
            if (overlaps(out[i], out_n[i], out[j], out_n[j]))
                return fail(CA_ERR_INVALID_ARG, "output buffers overlap");
        for (int j = 0; j < 6; ++j)
            if (overlaps(out[i], out_n[i], in[j], in_n[j]))
                return fail(CA_ERR_INVALID_ARG, "an output buffer overlaps an input");
    }
    return CA_OK;
}

ca_status_t make_tmap_3d(CUtensorMap *map, const void *base, int64_t rows, int32_t heads, int32_t dim,
                         int32_t box_heads, int32_t box_rows, bool fp32) {
    std::call_once(g_encode_once, [] {
        cudaDriverEntryPointQueryResult q{};
        void *fn = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    });
    if (!g_encode) return fail(CA_ERR_CUDA, "cuTensorMapEncodeTiled is unavailable");
    cuuint64_t gdim[3] = {static_cast<cuuint64_t>(dim), static_cast<cuuint64_t>(heads),
                          static_cast<cuuint64_t>(std::max<int64_t>(rows, 1))};
    const cuuint64_t esz = fp32 ? 4 : 2;
    cuuint64_t gstride[2] = {static_cast<cuuint64_t>(dim) * esz, static_cast<cuuint64_t>(heads) * dim * esz};
    // the box's inner extent is one 128-byte swizzle row: 64 bf16 or 32 fp32
    cuuint32_t box[3] = {fp32 ? 32u : 64u, static_cast<cuuint32_t>(box_heads), static_cast<cuuint32_t>(box_rows)};
    cuuint32_t estride[3] = {1, 1, 1};
    CUresult r = g_encode(map, fp32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3,
                          const_cast<void *>(base), gdim, gstride, box,
                          estride, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return fail(CA_ERR_CUDA, "cuTensorMapEncodeTiled failed (" + std::to_string(r) + ")");
    return CA_OK;
}

}  // namespace ca

using namespace ca;

namespace {

template <typename T>
cudaError_t upload(T **dst, const std::vector<T> &src, cudaStream_t s) {
    *dst = nullptr;
    if (src.empty()) return cudaSuccess;
    cudaError_t e = cudaMalloc(reinterpret_cast<void **>(dst), src.size() * sizeof(T));
    if (e != cudaSuccess) return e;
    return cudaMemcpyAsync(*dst, src.data(), src.size() * sizeof(T), cudaMemcpyHostToDevice, s);
}

void free_device(ca_plan *p) {
    cudaFree(p->d_tasks);
    cudaFree(p->d_fwd);
    cudaFree(p->d_bwd);
    cudaFree(p->d_bwd_pair);
    cudaFree(p->d_doc_task_ptr);
    cudaFree(p->d_doc_tasks);
    cudaFree(p->d_doc_info);
    cudaFree(p->d_err);
    p->d_tasks = nullptr;
    p->d_fwd = nullptr;
    p->d_bwd = nullptr;
    p->d_bwd_pair = nullptr;
    p->d_doc_task_ptr = nullptr;
    p->d_doc_tasks = nullptr;
    p->d_doc_info = nullptr;
    p->d_err = nullptr;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

constexpr int64_t kI32Max = 2147483647LL;
constexpr int32_t kMaxQHeads = 4096;  // keeps every per-row index product far inside int64
constexpr int32_t kDryRunSms = 152;   // SM count assumed without a device (a GB300)

// Whether byte ranges [a, a + na) and [b, b + nb) share a byte.
bool overlap(const void *a, int64_t na, const void *b, int64_t nb) {
    const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
    if (na <= 0 || nb <= 0) return false;
    return x < y + static_cast<uintptr_t>(nb) && y < x + static_cast<uintptr_t>(na);
}

// Byte sizes of a plan's tensors (every count is bounded far inside int64 by
// the planning limits).
struct BufferSizes {
    int64_t q, kv, o, lse;
};
BufferSizes buffer_sizes(const ca_plan *p) {
    BufferSizes b;
    b.q = p->total_q * p->hq * p->d * 2;
    b.kv = p->total_kv * p->hkv * p->d * 2;
    b.o = p->total_q * p->hq * p->d * (p->o_dtype == CA_DTYPE_FP32 ? 4 : 2);
    b.lse = p->total_q * p->hq * 4;
    return b;
}

}  // namespace

extern "C" {

int32_t ca_version(void) { return (1 << 16) | 0; }

const char *ca_status_string(ca_status_t s) {
    switch (s) {
        case CA_OK: return "ok";
        case CA_ERR_INVALID_ARG: return "invalid argument";
        case CA_ERR_UNSUPPORTED: return "unsupported configuration";
        case CA_ERR_CUDA: return "CUDA error";
        case CA_ERR_DEVICE_TIMEOUT: return "device wait limit exceeded";
        case CA_ERR_DEVICE_BOUNDS: return "device index check failed";
        case CA_ERR_NO_DEVICE: return "no sm_103 device";
    }
    return "unknown status";
}

const char *ca_last_error(void) { return g_last_error.c_str(); }

namespace {

// Workspace: fp32 dQ accumulator + fp32 D, each 256-byte aligned, 256 bytes
// of work-queue counters, then the split-KV forward scratch (split_scratch).
void set_workspace_bytes(ca_plan *p) {
    const int64_t rows_heads = p->total_q * p->hq;
    const int64_t dq_bytes = (rows_heads * p->d * 4 + 255) / 256 * 256;
    const int64_t d_bytes = (rows_heads * 4 + 255) / 256 * 256;
    p->split_ws_off = dq_bytes + d_bytes + 256;
    const int64_t split_bytes = (p->n_slots * 256 * (p->d + 1) * 4 + p->n_split * 256 * 4 + 255) / 256 * 256;
    p->workspace_bytes = p->split_ws_off + split_bytes;
}

// Forward items: (task, kv head, pair of consecutive query tiles 2t, 2t+1).
// The second tile is absent past the task's last tile.  The pair visits the
// key tiles of key_tile_ranges over both tiles' rows (each tile a prefix of
// that sequence).  A pair with more visits than the split size is cut into
// nparts balanced items over [i0, i1) of its sequence.  Split size:
// kv_split > 0 as given; kv_split < 0 never; kv_split = 0 (automatic) only
// when the launch has fewer than 4 waves of items on num_sms SMs: then total
// visits / num_sms clamped to [64, 128] key tiles per part (measured on
// decode batches of 1 to 32 sequences of 128K tokens).
//
// Order: items of one (document, kv head) are consecutive, so the CTAs that
// run at the same time read the same K/V prefix and it stays in L2; groups
// with the most key-tile visits first, longest items first inside a group,
// so the launch still ends on the shortest items.
struct FwdList {
    std::vector<FwdItem> items;
    int64_t n_split = 0, n_slots = 0, fwd_tile_pairs = 0;
};

void build_fwd_items(const ca_plan *p, int32_t kv_split, int32_t num_sms, FwdList *out) {
    std::vector<FwdItem> &fwd = out->items;
    fwd.clear();
    out->n_split = out->n_slots = out->fwd_tile_pairs = 0;
    struct Pair {
        int32_t t, tile, na, nb, n;
    };
    std::vector<Pair> pairs;
    int64_t total_visits = 0;
    for (int32_t t = 0; t < p->n_tasks; ++t) {
        const DevTask &d = p->h_tasks[t];
        const int32_t ntiles = (d.q_len + p->tpt - 1) / p->tpt;
        for (int32_t tile = 0; tile < ntiles; tile += 2) {
            const int32_t p0 = d.q_start + tile * p->tpt;
            const int32_t end0 = std::min(p0 + p->tpt, d.q_start + d.q_len) - 1;
            const bool has_b = tile + 1 < ntiles;
            const int32_t end1 = has_b ? std::min(p0 + 2 * p->tpt, d.q_start + d.q_len) - 1 : end0;
            const KeyTileRanges r = key_tile_ranges(d, p0, end1);
            const int32_t na = visits_upto(r, d, p0, end0);
            const int32_t nb = has_b ? visits_upto(r, d, end0 + 1, end1) : 0;
            pairs.push_back({t, tile, na, nb, std::max(na, nb)});
            total_visits += static_cast<int64_t>(std::max(na, nb)) * p->hkv;
            out->fwd_tile_pairs += static_cast<int64_t>(na + nb) * p->hkv;
        }
    }
    const int64_t sms = std::max<int32_t>(1, num_sms);
    int64_t chunk = 0;  // 0 = no split
    if (kv_split > 0) {
        chunk = kv_split;
    } else if (kv_split == 0 && static_cast<int64_t>(pairs.size()) * p->hkv < 4 * sms) {
        chunk = std::min<int64_t>(128, std::max<int64_t>(64, (total_visits + sms - 1) / sms));
    }
    for (const Pair &pr : pairs) {
        const int32_t nparts = (chunk > 0 && pr.n > chunk) ? static_cast<int32_t>((pr.n + chunk - 1) / chunk) : 1;
        for (int32_t g = 0; g < p->hkv; ++g) {
            int32_t split = -1, slot0 = 0;
            if (nparts > 1) {
                split = static_cast<int32_t>(out->n_split++);
                slot0 = static_cast<int32_t>(out->n_slots);
                out->n_slots += nparts;
            }
            for (int32_t part = 0; part < nparts; ++part) {
                const int32_t i0 = static_cast<int32_t>(static_cast<int64_t>(pr.n) * part / nparts);
                const int32_t i1 = static_cast<int32_t>(static_cast<int64_t>(pr.n) * (part + 1) / nparts);
                fwd.push_back({pr.t, g, pr.tile, i1 - i0, i0, i1, part, nparts, split, slot0});
            }
        }
    }
    std::vector<int64_t> group_work(static_cast<size_t>(p->n_docs) * p->hkv, 0);
    auto group = [&](const FwdItem &a) {
        return static_cast<size_t>(p->h_tasks[a.task].doc) * p->hkv + a.g;
    };
    for (const FwdItem &a : fwd) group_work[group(a)] += a.n_kv;
    std::stable_sort(fwd.begin(), fwd.end(), [&](const FwdItem &a, const FwdItem &b) {
        const size_t ga = group(a), gb = group(b);
        if (ga != gb) {
            if (group_work[ga] != group_work[gb]) return group_work[ga] > group_work[gb];
            return ga < gb;
        }
        return a.n_kv > b.n_kv;
    });
}

// Installs a forward list's counts in the plan (the items go to the device
// separately).
void apply_fwd_counts(ca_plan *p, const FwdList &f) {
    p->n_fwd = static_cast<int64_t>(f.items.size());
    p->n_split = f.n_split;
    p->n_slots = f.n_slots;
    p->fwd_tile_pairs = f.fwd_tile_pairs;
}

struct HostPlan {
    ca_plan *p = nullptr;
    FwdList fwd;
    std::vector<BwdItem> bwd;
    std::vector<BwdItem> bwd_pair;  // items of the CTA-pair backward (head_dim 128, G divides 64)
    std::vector<int32_t> ptr, dtasks, doc_info;
};

// Validation and all integer work of a plan; touches no device.
ca_status_t build_host_plan(const ca_task_t *tasks, const ca_mask_t *masks, int32_t n_tasks, const int64_t *doc_len,
                            const int64_t *doc_kv_offset, int32_t n_docs, const ca_shape_t *shape, int32_t num_sms,
                            HostPlan *hp) {
    if (!tasks || !doc_len || !doc_kv_offset || !shape) return fail(CA_ERR_INVALID_ARG, "NULL argument");
    if (n_tasks < 1) return fail(CA_ERR_INVALID_ARG, "n_tasks must be >= 1");
    if (n_docs < 1) return fail(CA_ERR_INVALID_ARG, "n_docs must be >= 1");
    const ca_shape_t sh = *shape;
    if (sh.num_q_heads < 1 || sh.num_kv_heads < 1 || sh.num_q_heads % sh.num_kv_heads != 0)
        return fail(CA_ERR_INVALID_ARG, "num_q_heads must be a positive multiple of num_kv_heads");
    if (sh.num_q_heads > kMaxQHeads) return fail(CA_ERR_UNSUPPORTED, "num_q_heads must be at most 4096");
    if (!(sh.softmax_scale > 0.f) || !std::isfinite(sh.softmax_scale))
        return fail(CA_ERR_INVALID_ARG, "softmax_scale must be positive and finite");
    if (sh.o_dtype != CA_DTYPE_BF16 && sh.o_dtype != CA_DTYPE_FP32)
        return fail(CA_ERR_INVALID_ARG, "o_dtype must be CA_DTYPE_BF16 or CA_DTYPE_FP32");
    if (sh.head_dim != 64 && sh.head_dim != 128) return fail(CA_ERR_UNSUPPORTED, "head_dim must be 64 or 128");
    const int32_t G = sh.num_q_heads / sh.num_kv_heads;
    if (G > kTileRows || kTileRows % G != 0)
        return fail(CA_ERR_UNSUPPORTED, "num_q_heads / num_kv_heads must divide 128");

    // documents: non-negative, non-overlapping KV ranges
    std::vector<std::pair<int64_t, int64_t>> ranges(n_docs);
    int64_t total_kv = 0;
    for (int32_t i = 0; i < n_docs; ++i) {
        if (doc_len[i] < 1 || doc_kv_offset[i] < 0)
            return fail(CA_ERR_INVALID_ARG, "document " + std::to_string(i) + " has a bad length or offset");
        if (doc_len[i] > kI32Max || doc_kv_offset[i] > kI32Max - doc_len[i])  // no int64 overflow
            return fail(CA_ERR_INVALID_ARG, "document rows must stay below 2^31");
        ranges[i] = {doc_kv_offset[i], doc_kv_offset[i] + doc_len[i]};
        total_kv = std::max(total_kv, doc_kv_offset[i] + doc_len[i]);
    }
    std::sort(ranges.begin(), ranges.end());
    for (int32_t i = 1; i < n_docs; ++i)
        if (ranges[i].first < ranges[i - 1].second) return fail(CA_ERR_INVALID_ARG, "document KV ranges overlap");

    ca_plan *p = new (std::nothrow) ca_plan();
    if (!p) return fail(CA_ERR_INVALID_ARG, "out of host memory");
    hp->p = p;
    p->n_tasks = n_tasks;
    p->n_docs = n_docs;
    p->hq = sh.num_q_heads;
    p->hkv = sh.num_kv_heads;
    p->d = sh.head_dim;
    p->G = G;
    p->tpt = kTileRows / G;
    p->scale = sh.softmax_scale;
    p->o_dtype = sh.o_dtype;
    p->total_kv = total_kv;
    p->task_pairs.resize(n_tasks);
    p->h_tasks.resize(n_tasks);

    int64_t row0 = 0;
    for (int32_t t = 0; t < n_tasks; ++t) {
        const ca_task_t &T = tasks[t];
        const std::string tn = "task " + std::to_string(t) + ": ";
        if (T.reserved != 0) return fail(CA_ERR_INVALID_ARG, tn + "reserved field must be 0");
        if (T.doc_id < 0 || T.doc_id >= n_docs) return fail(CA_ERR_INVALID_ARG, tn + "unknown doc_id");
        const int64_t L = doc_len[T.doc_id];
        if (T.q_len < 1 || T.kv_len < 1) return fail(CA_ERR_INVALID_ARG, tn + "q_len and kv_len must be >= 1");
        if (T.q_start < 0 || T.kv_start < 0) return fail(CA_ERR_INVALID_ARG, tn + "negative start");
        // written as L - len so that no int64 sum can overflow (L <= 2^31 - 1, len >= 1)
        if (T.q_start > L - T.q_len) return fail(CA_ERR_INVALID_ARG, tn + "query shard runs past the document");
        if (T.kv_start > L - T.kv_len) return fail(CA_ERR_INVALID_ARG, tn + "KV block runs past the document");
        if (row0 + T.q_len > kI32Max) return fail(CA_ERR_INVALID_ARG, "total query rows must stay below 2^31");
        DevTask &d = p->h_tasks[t];
        d.row0 = static_cast<int32_t>(row0);
        d.q_start = static_cast<int32_t>(T.q_start);
        d.q_len = static_cast<int32_t>(T.q_len);
        d.kv_start = static_cast<int32_t>(T.kv_start);
        d.kv_len = static_cast<int32_t>(T.kv_len);
        d.doc = T.doc_id;
        d.kv_off = static_cast<int32_t>(doc_kv_offset[T.doc_id]);
        d.doc_len = static_cast<int32_t>(L);
        d.sink = d.lo = d.win = 0;
        if (masks) {
            const ca_mask_t &M = masks[t];
            if (M.sink < 0 || M.lo < 0 || M.window < 0 || M.sink > L || M.lo > L || M.window > L)
                return fail(CA_ERR_INVALID_ARG, tn + "mask fields must lie in [0, document length]");
            d.sink = static_cast<int32_t>(M.sink);
            d.lo = static_cast<int32_t>(M.lo);
            d.win = static_cast<int32_t>(M.window);
        }
        const bool plain = d.sink == 0 && d.lo == 0 && d.win == 0;
        p->task_pairs[t] = plain ? task_pairs_closed_form(T.q_start, T.q_len, T.kv_start, T.kv_len)
                                 : task_pairs_rows(d);
        p->pairs += p->task_pairs[t];
        row0 += T.q_len;
    }
    p->total_q = row0;

    p->num_sms = num_sms;
    build_fwd_items(p, p->kv_split, num_sms, &hp->fwd);
    apply_fwd_counts(p, hp->fwd);
    if (p->n_fwd > kI32Max) return fail(CA_ERR_UNSUPPORTED, "the forward work list exceeds 2^31 items");

    // documents -> tasks (CSR), and backward tiles: (document, kv head, key tile)
    std::vector<int32_t> &ptr = hp->ptr, &dtasks = hp->dtasks, &doc_info = hp->doc_info;
    ptr.assign(n_docs + 1, 0);
    dtasks.assign(n_tasks, 0);
    for (int32_t t = 0; t < n_tasks; ++t) ptr[tasks[t].doc_id + 1]++;
    for (int32_t i = 0; i < n_docs; ++i) ptr[i + 1] += ptr[i];
    {
        std::vector<int32_t> fill(ptr.begin(), ptr.end() - 1);
        for (int32_t t = 0; t < n_tasks; ++t) dtasks[fill[tasks[t].doc_id]++] = t;
    }
    std::vector<BwdItem> &bwd = hp->bwd;
    doc_info.assign(2 * n_docs, 0);
    for (int32_t i = 0; i < n_docs; ++i) {
        doc_info[2 * i] = static_cast<int32_t>(doc_kv_offset[i]);
        doc_info[2 * i + 1] = static_cast<int32_t>(doc_len[i]);
        const int32_t nkt = static_cast<int32_t>((doc_len[i] + kTileKeys - 1) / kTileKeys);
        for (int32_t jt = 0; jt < nkt; ++jt) {
            int32_t nq = 0;
            for (int32_t k = ptr[i]; k < ptr[i + 1]; ++k) {
                int32_t f, c;
                bwd_task_tiles(p->h_tasks[dtasks[k]], jt, p->tpt, &f, &c);
                nq += c;
            }
            for (int32_t g = 0; g < p->hkv; ++g) bwd.push_back({i, g, jt, nq});
            p->bwd_tile_pairs += static_cast<int64_t>(nq) * p->hkv;
        }
    }
    // The CTA-pair kernel's items: pairs of key tiles (2 jp, 2 jp + 1), the
    // second past the document's end when it has an odd number of tiles.
    std::vector<BwdItem> &bwd_pair = hp->bwd_pair;
    if (p->d == 128 && 64 % p->G == 0) {
        for (int32_t i = 0; i < n_docs; ++i) {
            const int32_t nkt = static_cast<int32_t>((doc_len[i] + kTileKeys - 1) / kTileKeys);
            for (int32_t jp = 0; 2 * jp < nkt; ++jp) {
                int32_t nq = 0;
                for (int32_t k = ptr[i]; k < ptr[i + 1]; ++k) {
                    int32_t f, c;
                    key_pair_query_tiles(p->h_tasks[dtasks[k]], jp, p->tpt, &f, &c);
                    nq += c;
                }
                for (int32_t g = 0; g < p->hkv; ++g) bwd_pair.push_back({i, g, jp, nq});
            }
        }
    }
    // Group the items of one (document, kv head): CTAs that run at the same
    // time then add into the same rows of the fp32 dQ accumulator, which keeps
    // that working set (document length x G x head_dim x 4 bytes) in L2.
    // Groups with the most work first; longest items first inside a group.
    for (std::vector<BwdItem> *list : {&bwd, &bwd_pair}) {
        std::vector<int64_t> group_work(static_cast<size_t>(n_docs) * p->hkv, 0);
        for (const BwdItem &b : *list) group_work[static_cast<size_t>(b.doc) * p->hkv + b.g] += b.n_q;
        std::stable_sort(list->begin(), list->end(), [&](const BwdItem &a, const BwdItem &b) {
            const int64_t wa = group_work[static_cast<size_t>(a.doc) * p->hkv + a.g];
            const int64_t wb = group_work[static_cast<size_t>(b.doc) * p->hkv + b.g];
            if (wa != wb) return wa > wb;
            if (a.doc != b.doc) return a.doc < b.doc;
            if (a.g != b.g) return a.g < b.g;
            return a.n_q > b.n_q;
        });
    }
    p->n_bwd = static_cast<int64_t>(bwd.size());
    p->n_bwd_pair = static_cast<int64_t>(bwd_pair.size());
    if (p->n_bwd > kI32Max || p->n_bwd_pair > kI32Max)
        return fail(CA_ERR_UNSUPPORTED, "the backward work list exceeds 2^31 items");

    set_workspace_bytes(p);
    return CA_OK;
}

// build_host_plan behind the C boundary: a failed host allocation becomes a
// status instead of an exception leaving an extern "C" function.
ca_status_t build_host_plan_guarded(const ca_task_t *tasks, const ca_mask_t *masks, int32_t n_tasks,
                                    const int64_t *doc_len, const int64_t *doc_kv_offset, int32_t n_docs,
                                    const ca_shape_t *shape, int32_t num_sms, HostPlan *hp) {
    try {
        return build_host_plan(tasks, masks, n_tasks, doc_len, doc_kv_offset, n_docs, shape, num_sms, hp);
    } catch (const std::bad_alloc &) {
        return fail(CA_ERR_INVALID_ARG, "host memory exhausted while planning");
    }
}

}  // namespace

namespace {

ca_status_t set_kv_split_impl(ca_plan *p, int32_t visits_per_part) {
    // everything is built and uploaded to a new list first; the plan changes
    // only once that has succeeded
    FwdList fwd;
    build_fwd_items(p, visits_per_part, p->num_sms, &fwd);
    if (static_cast<int64_t>(fwd.items.size()) > kI32Max)
        return fail(CA_ERR_UNSUPPORTED, "the forward work list exceeds 2^31 items");
    FwdItem *d_new = nullptr;
    cudaError_t e = upload(&d_new, fwd.items, nullptr);
    if (e == cudaSuccess) e = cudaDeviceSynchronize();  // upload done; no launch still reads the old list
    if (e != cudaSuccess) {
        cudaFree(d_new);
        return cuda_fail(e, "forward item upload");
    }
    cudaFree(p->d_fwd);
    p->d_fwd = d_new;
    p->kv_split = visits_per_part;
    apply_fwd_counts(p, fwd);
    set_workspace_bytes(p);
    return CA_OK;
}

}  // namespace

// Re-cut the forward items with a new split size (see build_fwd_items) and
// upload them; the workspace size may change.
extern "C" ca_status_t ca_plan_set_kv_split(ca_plan_t *p, int32_t visits_per_part) {
    if (!p) return fail(CA_ERR_INVALID_ARG, "plan is NULL");
    const ca_status_t st = check_plan_device(p);
    if (st != CA_OK) return st;
    try {
        return set_kv_split_impl(p, visits_per_part);
    } catch (const std::bad_alloc &) {
        return fail(CA_ERR_INVALID_ARG, "host memory exhausted while re-cutting the forward items");
    }
}

namespace {

void fill_info(const ca_plan *p, ca_plan_info_t *o) {
    o->total_q = p->total_q;
    o->total_kv = p->total_kv;
    o->n_tasks = p->n_tasks;
    o->n_docs = p->n_docs;
    o->causal_pairs = p->pairs;
    o->flops_fwd = 4LL * p->d * p->hq * p->pairs;
    o->flops_bwd = 8LL * p->d * p->hq * p->pairs;
    o->workspace_bytes = p->workspace_bytes;
    o->n_fwd_items = p->n_fwd;
    o->n_bwd_items = p->n_bwd;
    o->fwd_tile_pairs = p->fwd_tile_pairs;
    o->bwd_tile_pairs = p->bwd_tile_pairs;
}

}  // namespace

ca_status_t ca_plan_dry_run_masked(const ca_task_t *tasks, const ca_mask_t *masks, int32_t n_tasks,
                                   const int64_t *doc_len, const int64_t *doc_kv_offset, int32_t n_docs,
                                   const ca_shape_t *shape, ca_plan_info_t *info, int64_t *task_pairs) {
    if (!info) return fail(CA_ERR_INVALID_ARG, "info is NULL");
    HostPlan hp;
    ca_status_t st = build_host_plan_guarded(tasks, masks, n_tasks, doc_len, doc_kv_offset, n_docs, shape,
                                             kDryRunSms, &hp);
    if (st == CA_OK) {
        fill_info(hp.p, info);
        if (task_pairs) std::copy(hp.p->task_pairs.begin(), hp.p->task_pairs.end(), task_pairs);
    }
    delete hp.p;
    return st;
}

ca_status_t ca_plan_dry_run(const ca_task_t *tasks, int32_t n_tasks, const int64_t *doc_len,
                            const int64_t *doc_kv_offset, int32_t n_docs, const ca_shape_t *shape,
                            ca_plan_info_t *info, int64_t *task_pairs) {
    return ca_plan_dry_run_masked(tasks, nullptr, n_tasks, doc_len, doc_kv_offset, n_docs, shape, info, task_pairs);
}

ca_status_t ca_plan_create(const ca_task_t *tasks, int32_t n_tasks, const int64_t *doc_len,
                           const int64_t *doc_kv_offset, int32_t n_docs, const ca_shape_t *shape,
                           void *upload_stream, ca_plan_t **out) {
    return ca_plan_create_masked(tasks, nullptr, n_tasks, doc_len, doc_kv_offset, n_docs, shape, upload_stream, out);
}

ca_status_t ca_plan_create_masked(const ca_task_t *tasks, const ca_mask_t *masks, int32_t n_tasks,
                                  const int64_t *doc_len, const int64_t *doc_kv_offset, int32_t n_docs,
                                  const ca_shape_t *shape, void *upload_stream, ca_plan_t **out) {
    if (!out) return fail(CA_ERR_INVALID_ARG, "out is NULL");
    *out = nullptr;
    // The device's SM count sizes the forward split; argument errors are
    // still reported before device errors.
    int device = -1;
    cudaDeviceProp prop;
    cudaError_t e = cudaGetDevice(&device);
    const char *what = "cudaGetDevice";
    if (e == cudaSuccess) {
        e = cudaGetDeviceProperties(&prop, device);
        what = "cudaGetDeviceProperties";
    }
    const int32_t num_sms = e == cudaSuccess ? prop.multiProcessorCount : kDryRunSms;
    HostPlan hp;
    ca_status_t st =
        build_host_plan_guarded(tasks, masks, n_tasks, doc_len, doc_kv_offset, n_docs, shape, num_sms, &hp);
    if (st != CA_OK) {
        delete hp.p;
        return st;
    }
    ca_plan *p = hp.p;
    if (e != cudaSuccess) { delete p; return cuda_fail(e, what); }
    p->device = device;
    if (prop.major != 10 || prop.minor != 3) {
        delete p;
        return fail(CA_ERR_NO_DEVICE, "current device is sm_" + std::to_string(prop.major) +
                                          std::to_string(prop.minor) + ", the kernels are built for sm_103a");
    }
    cudaStream_t s = static_cast<cudaStream_t>(upload_stream);
    if ((e = upload(&p->d_tasks, p->h_tasks, s)) != cudaSuccess ||
        (e = upload(&p->d_fwd, hp.fwd.items, s)) != cudaSuccess || (e = upload(&p->d_bwd, hp.bwd, s)) != cudaSuccess ||
        (e = upload(&p->d_bwd_pair, hp.bwd_pair, s)) != cudaSuccess ||
        (e = upload(&p->d_doc_task_ptr, hp.ptr, s)) != cudaSuccess ||
        (e = upload(&p->d_doc_tasks, hp.dtasks, s)) != cudaSuccess ||
        (e = upload(&p->d_doc_info, hp.doc_info, s)) != cudaSuccess ||
        (e = cudaMalloc(reinterpret_cast<void **>(&p->d_err), 16)) != cudaSuccess ||
        (e = cudaMemsetAsync(p->d_err, 0, 16, s)) != cudaSuccess || (e = cudaStreamSynchronize(s)) != cudaSuccess) {
        free_device(p);
        delete p;
        return cuda_fail(e, "plan upload");
    }
    *out = p;
    return CA_OK;
}

ca_status_t ca_plan_info(const ca_plan_t *p, ca_plan_info_t *o) {
    if (!p || !o) return fail(CA_ERR_INVALID_ARG, "NULL argument");
    fill_info(p, o);
    return CA_OK;
}

ca_status_t ca_plan_task_pairs(const ca_plan_t *p, int64_t *out) {
    if (!p || !out) return fail(CA_ERR_INVALID_ARG, "NULL argument");
    std::copy(p->task_pairs.begin(), p->task_pairs.end(), out);
    return CA_OK;
}

void ca_plan_destroy(ca_plan_t *p) {
    if (!p) return;
    // free on the plan's device, whichever device the caller has current
    int cur = -1;
    const bool switched = cudaGetDevice(&cur) == cudaSuccess && cur != p->device &&
                          cudaSetDevice(p->device) == cudaSuccess;
    cudaDeviceSynchronize();
    free_device(p);
    if (switched) cudaSetDevice(cur);
    delete p;
}

ca_status_t ca_plan_set_backward_kernel(ca_plan_t *p, int32_t kind) {
    if (!p) return fail(CA_ERR_INVALID_ARG, "plan is NULL");
    if (kind != CA_BWD_KERNEL_AUTO && kind != CA_BWD_KERNEL_SINGLE && kind != CA_BWD_KERNEL_PAIR)
        return fail(CA_ERR_INVALID_ARG, "unknown backward kernel kind " + std::to_string(kind));
    p->bwd_kernel = kind;
    return CA_OK;
}

ca_status_t ca_plan_set_wait_limit(ca_plan_t *p, int64_t ns) {
    if (!p || ns < 0) return fail(CA_ERR_INVALID_ARG, "bad plan or limit");
    p->wait_limit_ns = ns;
    return CA_OK;
}

ca_status_t ca_plan_set_timing_events(ca_plan_t *p, void *const *events, int32_t n_events) {
    if (!p) return fail(CA_ERR_INVALID_ARG, "plan is NULL");
    if (events && n_events < 6) return fail(CA_ERR_INVALID_ARG, "need 6 events");
    if (events)
        for (int32_t i = 0; i < 6; ++i)
            if (!events[i]) return fail(CA_ERR_INVALID_ARG, "NULL event");
    p->timing_events = events;
    return CA_OK;
}

ca_status_t ca_forward(const ca_plan_t *p, const void *q, const void *k, const void *v, void *o, float *lse,
                       void *workspace, void *stream) {
    if (!p) return fail(CA_ERR_INVALID_ARG, "plan is NULL");
    if (!q || !k || !v || !o || !lse || !workspace) return fail(CA_ERR_INVALID_ARG, "NULL pointer");
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(lse) || !aligned16(workspace))
        return fail(CA_ERR_INVALID_ARG, "pointers must be 16-byte aligned");
    const BufferSizes b = buffer_sizes(p);
    // outputs (o, lse, the workspace) must not share a byte with each other or with an input
    const void *out[] = {o, lse, workspace};
    const int64_t out_n[] = {b.o, b.lse, p->workspace_bytes};
    const void *in[] = {q, k, v};
    const int64_t in_n[] = {b.q, b.kv, b.kv};
    for (int i = 0; i < 3; ++i) {
        for (int j = i + 1; j < 3; ++j)
            if (overlap(out[i], out_n[i], out[j], out_n[j])) return fail(CA_ERR_INVALID_ARG, "output buffers overlap");
        for (int j = 0; j < 3; ++j)
            if (overlap(out[i], out_n[i], in[j], in_n[j]))
                return fail(CA_ERR_INVALID_ARG, "an output buffer overlaps an input");
    }
    const ca_status_t st = check_plan_device(p);
    if (st != CA_OK) return st;
    cudaError_t e = launch_forward(p, q, k, v, o, lse, workspace, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "forward launch");
    return CA_OK;
}

ca_status_t ca_backward(const ca_plan_t *p, const void *q, const void *k, const void *v, const void *o,
                        const float *lse, const void *d_o, void *dq, void *dk, void *dv, void *workspace,
                        void *stream) {
    if (!p) return fail(CA_ERR_INVALID_ARG, "plan is NULL");
    if (!workspace) return fail(CA_ERR_INVALID_ARG, "NULL pointer");
    ca_status_t st = check_backward_args(p, q, k, v, o, lse, d_o, dq, dk, dv, workspace, p->workspace_bytes);
    if (st != CA_OK) return st;
    if ((st = check_plan_device(p)) != CA_OK) return st;
    cudaError_t e = launch_backward(p, q, k, v, o, lse, d_o, dq, dk, dv, workspace, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "backward launch");
    return CA_OK;
}

ca_status_t ca_merge(int32_t n_parts, const void *const *o_parts, const float *const *lse_parts, int32_t parts_dtype,
                     int64_t rows, int32_t heads, int32_t head_dim, void *o_out, int32_t out_dtype, float *lse_out,
                     void *stream) {
    if (n_parts < 1 || n_parts > kMaxMergeParts) return fail(CA_ERR_INVALID_ARG, "n_parts must be in [1, 64]");
    if (!o_parts || !lse_parts || !o_out) return fail(CA_ERR_INVALID_ARG, "NULL pointer");
    if (rows < 0 || heads < 1 || head_dim < 8 || head_dim > 256 || head_dim % 8 != 0)
        return fail(CA_ERR_INVALID_ARG, "bad rows / heads / head_dim");
    if (rows > (int64_t(1) << 50) / (int64_t(heads) * head_dim))  // the launch sizes in int64
        return fail(CA_ERR_INVALID_ARG, "rows * heads * head_dim exceeds 2^50 elements");
    if ((parts_dtype != CA_DTYPE_BF16 && parts_dtype != CA_DTYPE_FP32) ||
        (out_dtype != CA_DTYPE_BF16 && out_dtype != CA_DTYPE_FP32))
        return fail(CA_ERR_INVALID_ARG, "bad dtype");
    for (int32_t s = 0; s < n_parts; ++s) {
        if (!o_parts[s] || !lse_parts[s]) return fail(CA_ERR_INVALID_ARG, "NULL part pointer");
        if (!aligned16(o_parts[s]) || !aligned16(lse_parts[s]))
            return fail(CA_ERR_INVALID_ARG, "part pointers must be 16-byte aligned");
    }
    if (!aligned16(o_out) || (lse_out && !aligned16(lse_out)))
        return fail(CA_ERR_INVALID_ARG, "output pointers must be 16-byte aligned");
    if (rows == 0) return CA_OK;
    cudaError_t e = launch_merge(n_parts, o_parts, lse_parts, parts_dtype, rows, heads, head_dim, o_out, out_dtype,
                                 lse_out, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "merge launch");
    return CA_OK;
}

ca_status_t ca_device_status(const ca_plan_t *p, void *stream) {
    if (!p) return fail(CA_ERR_INVALID_ARG, "plan is NULL");
    const ca_status_t st = check_plan_device(p);
    if (st != CA_OK) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    uint32_t word = 0;
    cudaError_t e = cudaMemcpyAsync(&word, p->d_err, sizeof(word), cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return cuda_fail(e, "device status");
    if (word == 0) return CA_OK;
    e = cudaMemsetAsync(p->d_err, 0, sizeof(word), s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return cuda_fail(e, "device status clear");
    if (word & kErrTimeout) return fail(CA_ERR_DEVICE_TIMEOUT, "a kernel wait ran out of its limit");
    return fail(CA_ERR_DEVICE_BOUNDS, "a kernel index check failed");
}

ca_status_t ca_watchdog_selftest(const ca_plan_t *p, int64_t limit_ns, void *stream) {
    if (!p || limit_ns < 0) return fail(CA_ERR_INVALID_ARG, "bad plan or limit");
    const ca_status_t st = check_plan_device(p);
    if (st != CA_OK) return st;
    cudaError_t e = launch_watchdog_selftest(p, limit_ns, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "watchdog self-test launch");
    return CA_OK;
}

}  // extern "C"
