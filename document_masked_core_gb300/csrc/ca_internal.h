// Internal declarations shared by the host plan code and the kernels.
#pragma once

#include <cstdint>
#include <string>
#include <vector>

#include <cuda.h>
#include <cuda_runtime.h>

#include "../../include/ca.h"

namespace ca {

constexpr int kTileRows = 128;   // query-tile rows = (128 / G tokens) x G heads
constexpr int kTileKeys = 128;   // keys per KV tile
constexpr int kMaxMergeParts = 64;

// One CA-task as the kernels see it (token units, int32; element offsets are
// formed in 64-bit inside the kernels).
struct DevTask {
    int32_t row0;      // first packed query row
    int32_t q_start;   // document position of the first query row
    int32_t q_len;
    int32_t kv_start;  // visible key block [kv_start, kv_start + kv_len)
    int32_t kv_len;
    int32_t doc;
    int32_t kv_off;    // first K/V row of the document
    int32_t doc_len;
    int32_t sink, lo, win;  // sparse visibility (ca_mask_t); 0, 0, 0 = plain
};

// Visible keys of row p: [kv_start, min(kv_end, p + 1)) intersected with
// [0, sink) U [max(lo, p - win + 1), inf)  (win = 0: [lo, inf)).  As two
// intervals [a, r1) U [r2, hi) (either may be empty; they may overlap).
struct RowKeys {
    int32_t a, r1, r2, hi;
};

__host__ __device__ inline RowKeys row_keys(const DevTask &t, int32_t p) {
    RowKeys k;
    k.a = t.kv_start;
    k.hi = p + 1 < t.kv_start + t.kv_len ? p + 1 : t.kv_start + t.kv_len;
    k.r1 = t.sink < k.hi ? t.sink : k.hi;
    int32_t lo = t.lo;
    if (t.win > 0 && p - t.win + 1 > lo) lo = p - t.win + 1;
    k.r2 = lo > t.kv_start ? lo : t.kv_start;
    return k;
}

// Key tiles (of 128) a query tile with rows p in [p0, p1] visits: the sink
// range [sa, sb) and the window range [wa, wb) of key-tile indices, merged
// into one range (sb = sa) when they touch or overlap.  Row p0 has the
// smallest window start and p1 the largest end.
struct KeyTileRanges {
    int32_t sa, sb, wa, wb;
    __host__ __device__ int32_t count() const { return (sb - sa) + (wb - wa); }
    // key tile of the i-th visit (i < count())
    __host__ __device__ int32_t tile(int32_t i) const { return i < sb - sa ? sa + i : wa + (i - (sb - sa)); }
};

__host__ __device__ inline KeyTileRanges key_tile_ranges(const DevTask &t, int32_t p0, int32_t p1) {
    KeyTileRanges r;
    const RowKeys k0 = row_keys(t, p0), k1 = row_keys(t, p1);
    // sink part: keys [a, min(sink, hi(p1)))
    const int32_t s_end = k1.r1;
    // window part: keys [r2(p0), hi(p1))
    const int32_t w_beg = k0.r2, w_end = k1.hi;
    r.sa = k0.a / 128;
    r.sb = s_end > k0.a ? (s_end - 1) / 128 + 1 : r.sa;
    if (w_end > w_beg) {
        r.wa = w_beg / 128;
        r.wb = (w_end - 1) / 128 + 1;
    } else {
        r.wa = r.wb = 0;
    }
    if (r.sb > r.sa && r.wb > r.wa && r.wa <= r.sb) {  // touching or overlapping: one range
        r.wa = r.sa < r.wa ? r.sa : r.wa;
        r.wb = r.sb > r.wb ? r.sb : r.wb;
        r.sb = r.sa;
    }
    return r;
}

// Number of visits (in the order of key_tile_ranges over rows [p0, p1]) up
// to and including the furthest key tile any row of [q0x, q1x] sees: the
// prefix of the item's sequence a query tile with those rows needs.  The
// furthest key is not always the last row's: a row's window part [r2, hi) is
// non-empty exactly for rows max(lo, kv_start) <= p <= kv_end + window - 2
// (no upper end when window = 0; none at all when lo >= kv_end), and hi grows
// with p, so the furthest window key is that of the last such row in the
// tile; the sink part's end r1 grows with p, so its furthest key is the last
// row's.
__host__ __device__ inline int32_t visits_upto(const KeyTileRanges &r, const DevTask &t, int32_t q0x,
                                               int32_t q1x) {
    int32_t last = -1;  // furthest visible key of the rows
    const int64_t e = static_cast<int64_t>(t.kv_start) + t.kv_len;
    if (t.lo < e) {
        const int64_t first_w = t.lo > t.kv_start ? t.lo : t.kv_start;
        const int64_t last_w = t.win > 0 ? e + t.win - 2 : int64_t(q1x);
        const int64_t pw = last_w < q1x ? last_w : int64_t(q1x);
        if (pw >= q0x && pw >= first_w) last = row_keys(t, static_cast<int32_t>(pw)).hi - 1;
    }
    const RowKeys k = row_keys(t, q1x);
    if (k.r1 > k.a && k.r1 - 1 > last) last = k.r1 - 1;
    if (last < 0) return 0;
    const int32_t lt = last / 128;
    int32_t n = 0;
    if (lt >= r.sa && r.sb > r.sa) n += (lt < r.sb ? lt + 1 : r.sb) - r.sa;
    if (r.wb > r.wa && lt >= r.wa) n += (lt < r.wb ? lt + 1 : r.wb) - r.wa;
    return n;
}

// Query rows that see at least one key of key tile [k0, k0 + 128): a
// contiguous range [pmin, pmax] (pmax = INT32_MAX: unbounded); empty when
// pmin > pmax.  A key j is seen by rows p >= j when j < sink, by rows
// j <= p <= j + win - 1 when j >= lo (any p >= j when win = 0).
__host__ __device__ inline void key_tile_rows(const DevTask &t, int32_t k0, int32_t *pmin, int32_t *pmax) {
    const int32_t j0 = k0 > t.kv_start ? k0 : t.kv_start;
    const int32_t j1 = (k0 + 128 < t.kv_start + t.kv_len ? k0 + 128 : t.kv_start + t.kv_len) - 1;  // inclusive
    *pmin = 2147483647;
    *pmax = -1;
    if (j1 < j0) return;
    if (j0 < t.sink) {  // sink keys: every later row
        *pmin = j0;
        *pmax = 2147483647;
    }
    const int32_t jl = j0 > t.lo ? j0 : t.lo;  // first key past lo
    if (jl <= j1) {
        if (jl < *pmin) *pmin = jl;
        const int64_t hi = t.win > 0 ? static_cast<int64_t>(j1) + t.win - 1 : int64_t(2147483647);
        const int32_t hi32 = hi < 2147483647 ? static_cast<int32_t>(hi) : 2147483647;
        if (hi32 > *pmax) *pmax = hi32;
    }
}

// Query tiles (of tpt tokens) of task t whose rows see key tile jt: the rows
// of key_tile_rows inside the task, as a first tile and a count (0: none).
__host__ __device__ inline void key_tile_query_tiles(const DevTask &t, int32_t jt, int32_t tpt, int32_t *first,
                                                     int32_t *count) {
    *first = 0;
    *count = 0;
    int32_t pmin, pmax;
    key_tile_rows(t, jt * 128, &pmin, &pmax);
    const int32_t q0 = t.q_start, q1 = t.q_start + t.q_len - 1;  // inclusive
    const int32_t lo = pmin > q0 ? pmin : q0, hi = pmax < q1 ? pmax : q1;
    if (lo > hi) return;
    *first = (lo - q0) / tpt;
    *count = (hi - q0) / tpt - *first + 1;
}

// The same for the pair of key tiles 2 jp and 2 jp + 1 that a CTA pair
// processes together: one range covering both tiles' ranges (a query tile in
// between that sees neither gets all-zero probabilities and adds nothing).
__host__ __device__ inline void key_pair_query_tiles(const DevTask &t, int32_t jp, int32_t tpt, int32_t *first,
                                                     int32_t *count) {
    int32_t fa, ca, fb, cb;
    key_tile_query_tiles(t, 2 * jp, tpt, &fa, &ca);
    key_tile_query_tiles(t, 2 * jp + 1, tpt, &fb, &cb);
    if (cb == 0) {
        *first = fa;
        *count = ca;
    } else if (ca == 0) {
        *first = fb;
        *count = cb;
    } else {
        const int32_t lo = fa < fb ? fa : fb, hi = fa + ca > fb + cb ? fa + ca : fb + cb;
        *first = lo;
        *count = hi - lo;
    }
}

// Forward item: query tiles `tile` and `tile + 1` (tile even; tokens
// [tile*T, tile*T+2T) of the task, T = 128 / G) of kv head g, processed
// together by one CTA, over visits [i0, i1) of the pair's key-tile sequence
// (n_kv = i1 - i0).  A pair split into nparts > 1 items writes partial
// (O, LSE) rows to slots slot0 + part of the workspace; the last part to
// finish a row merges the parts (per-row counters of split pair `split`).
struct FwdItem {
    int32_t task, g, tile, n_kv;
    int32_t i0, i1, part, nparts;
    int32_t split, slot0;
};

// Backward tile: key tile kv_tile of document doc, kv head g; n_q = number of
// query tiles (over all tasks of the document) that see it.  In the list of
// the CTA-pair kernel, kv_tile is the pair index jp (key tiles 2 jp, 2 jp + 1)
// and n_q counts the query tiles of key_pair_query_tiles.
struct BwdItem {
    int32_t doc, g, kv_tile, n_q;
};

// Device-side error word values (bit flags).
enum : uint32_t { kErrTimeout = 1u, kErrBounds = 2u };

// Kernel-side control shared by all launches of a plan.
struct DevCtl {
    uint32_t *err;          // device error word
    unsigned long long wait_limit_ns;
};

}  // namespace ca

struct ca_plan {
    int32_t n_tasks = 0, n_docs = 0;
    int32_t hq = 0, hkv = 0, d = 0, G = 0, tpt = 0;  // tpt = query tokens per tile
    float scale = 0.f;
    int32_t o_dtype = CA_DTYPE_BF16;
    int64_t total_q = 0, total_kv = 0;
    int64_t pairs = 0;
    int64_t fwd_tile_pairs = 0, bwd_tile_pairs = 0;
    std::vector<int64_t> task_pairs;
    std::vector<ca::DevTask> h_tasks;
    int64_t n_fwd = 0, n_bwd = 0;
    int64_t n_bwd_pair = 0;               // items of the CTA-pair backward (0: not applicable)
    int32_t bwd_kernel = 0;               // CA_BWD_KERNEL_*: which backward main kernel runs
    int64_t workspace_bytes = 0;
    int32_t kv_split = 0;                 // 0: automatic, < 0: never split, > 0: visits per part
    int64_t n_split = 0, n_slots = 0;     // split pairs, partial slots (256 rows each)
    int64_t split_ws_off = 0;             // workspace offset of the partial O / LSE / counters
    int64_t wait_limit_ns = 2000000000LL;
    void *const *timing_events = nullptr;  // optional cudaEvent_t[6], see ca_plan_set_timing_events
    int device = 0, num_sms = 0;
    // device metadata (owned)
    ca::DevTask *d_tasks = nullptr;
    ca::FwdItem *d_fwd = nullptr;
    ca::BwdItem *d_bwd = nullptr;
    ca::BwdItem *d_bwd_pair = nullptr;
    int32_t *d_doc_task_ptr = nullptr;  // [n_docs + 1] CSR into d_doc_tasks
    int32_t *d_doc_tasks = nullptr;     // task ids grouped by document
    int32_t *d_doc_info = nullptr;      // [n_docs][2] = {kv_off, doc_len}
    uint32_t *d_err = nullptr;
};

namespace ca {

void set_error(const std::string &msg);
ca_status_t fail(ca_status_t st, const std::string &msg);
ca_status_t cuda_fail(cudaError_t e, const char *what);

// CA_ERR_INVALID_ARG unless the plan's device is current (its tables, error
// word and the tensor maps of a launch live there).
ca_status_t check_plan_device(const ca_plan *p);

// Backward argument checks shared by ca_backward and ca_backward_noalloc:
// non-NULL, 16-byte aligned, and no output (dq, dk, dv, the scratch of
// scratch_bytes) sharing a byte with another output or with an input.
ca_status_t check_backward_args(const ca_plan *p, const void *q, const void *k, const void *v, const void *o,
                                const void *lse, const void *d_o, const void *dq, const void *dk, const void *dv,
                                const void *scratch, int64_t scratch_bytes);

// Builds a 3D tensor map over a [rows, heads, dim] token-major bf16 (or fp32)
// tensor with a box of (128 bytes of dim, box_heads, box_rows) and 128-byte
// swizzle.
ca_status_t make_tmap_3d(CUtensorMap *map, const void *base, int64_t rows, int32_t heads, int32_t dim,
                         int32_t box_heads, int32_t box_rows, bool fp32 = false);

// Records the plan's timing event `slot` on stream when timing is enabled.
inline cudaError_t mark(const ca_plan *p, int slot, cudaStream_t stream) {
    if (!p->timing_events) return cudaSuccess;
    return cudaEventRecord(static_cast<cudaEvent_t>(p->timing_events[slot]), stream);
}

// Work-queue counters (256 bytes after the fp32 dQ accumulator and the D
// vector): [0] backward main kernel, [1] forward.
inline int32_t *work_counters(const ca_plan *p, void *workspace) {
    const int64_t units = p->total_q * p->hq;
    const int64_t off = (units * p->d * 4 + 255) / 256 * 256 + (units * 4 + 255) / 256 * 256;
    return reinterpret_cast<int32_t *>(static_cast<uint8_t *>(workspace) + off);
}

// Split-KV forward scratch after the counters: partial O [n_slots][256][d]
// fp32, partial LSE [n_slots][256] fp32, row counters [n_split][256] int32.
struct SplitScratch {
    float *o, *lse;
    int32_t *cnt;
};
inline SplitScratch split_scratch(const ca_plan *p, void *workspace) {
    uint8_t *base = static_cast<uint8_t *>(workspace) + p->split_ws_off;
    SplitScratch s;
    s.o = reinterpret_cast<float *>(base);
    s.lse = reinterpret_cast<float *>(base + p->n_slots * 256 * p->d * 4);
    s.cnt = reinterpret_cast<int32_t *>(base + p->n_slots * 256 * (p->d + 1) * 4);
    return s;
}

cudaError_t launch_forward(const ca_plan *p, const void *q, const void *k, const void *v, void *o,
                           float *lse, void *workspace, cudaStream_t stream);
cudaError_t launch_backward(const ca_plan *p, const void *q, const void *k, const void *v, const void *o,
                            const float *lse, const void *d_o, void *dq, void *dk, void *dv,
                            void *workspace, cudaStream_t stream);
// Backward main pass on CTA pairs (head_dim 128, G dividing 64): see ca_backward_pair.cu.
cudaError_t launch_bwd_main_pair(const ca_plan *p, const void *q, const void *k, const void *v, const void *d_o,
                                 float *dq_acc, const float *lse, const float *Dvec, int32_t *sched, void *dk,
                                 void *dv, cudaStream_t stream);
// Whether the plan's backward runs the CTA-pair main kernel (selected and applicable).
inline bool use_bwd_pair(const ca_plan *p) { return p->n_bwd_pair > 0 && p->bwd_kernel == CA_BWD_KERNEL_PAIR; }
cudaError_t launch_merge(int32_t n_parts, const void *const *o_parts, const float *const *lse_parts,
                         int32_t parts_dtype, int64_t rows, int32_t heads, int32_t head_dim, void *o_out,
                         int32_t out_dtype, float *lse_out, cudaStream_t stream);
cudaError_t launch_watchdog_selftest(const ca_plan *p, int64_t limit_ns, cudaStream_t stream);

}  // namespace ca
