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
};

// Forward item: query tiles `tile` and `tile + 1` (tile even; tokens
// [tile*T, tile*T+2T) of the task, T = 128 / G) of kv head g, processed
// together by one CTA; n_kv = visible 128-key tiles of the later tile.
struct FwdItem {
    int32_t task, g, tile, n_kv;
};

// Backward tile: key tile kv_tile of document doc, kv head g; n_q = number of
// query tiles (over all tasks of the document) that see it.
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
    int64_t workspace_bytes = 0;
    int64_t wait_limit_ns = 2000000000LL;
    void *const *timing_events = nullptr;  // optional cudaEvent_t[6], see ca_plan_set_timing_events
    int device = 0, num_sms = 0;
    // device metadata (owned)
    ca::DevTask *d_tasks = nullptr;
    ca::FwdItem *d_fwd = nullptr;
    ca::BwdItem *d_bwd = nullptr;
    int32_t *d_doc_task_ptr = nullptr;  // [n_docs + 1] CSR into d_doc_tasks
    int32_t *d_doc_tasks = nullptr;     // task ids grouped by document
    int32_t *d_doc_info = nullptr;      // [n_docs][2] = {kv_off, doc_len}
    uint32_t *d_err = nullptr;
};

namespace ca {

void set_error(const std::string &msg);
ca_status_t fail(ca_status_t st, const std::string &msg);
ca_status_t cuda_fail(cudaError_t e, const char *what);

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

// Work-queue counters at the end of the workspace (256 bytes after the fp32
// dQ accumulator and the D vector): [0] backward main kernel, [1] forward.
inline int32_t *work_counters(const ca_plan *p, void *workspace) {
    const int64_t units = p->total_q * p->hq;
    const int64_t off = (units * p->d * 4 + 255) / 256 * 256 + (units * 4 + 255) / 256 * 256;
    return reinterpret_cast<int32_t *>(static_cast<uint8_t *>(workspace) + off);
}

cudaError_t launch_forward(const ca_plan *p, const void *q, const void *k, const void *v, void *o,
                           float *lse, void *workspace, cudaStream_t stream);
cudaError_t launch_backward(const ca_plan *p, const void *q, const void *k, const void *v, const void *o,
                            const float *lse, const void *d_o, void *dq, void *dk, void *dv,
                            void *workspace, cudaStream_t stream);
cudaError_t launch_merge(int32_t n_parts, const void *const *o_parts, const float *const *lse_parts,
                         int32_t parts_dtype, int64_t rows, int32_t heads, int32_t head_dim, void *o_out,
                         int32_t out_dtype, float *lse_out, cudaStream_t stream);
cudaError_t launch_watchdog_selftest(const ca_plan *p, int64_t limit_ns, cudaStream_t stream);

}  // namespace ca
