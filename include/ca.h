/*
 * ca.h -- C ABI of the document-masked core-attention library (libca.so).
 *
 * Core attention (CA) is softmax(Q K^T / sqrt(d)) V, the parameter-free step
 * between the QKV and O projections ("Core Attention Disaggregation", CMU CSD
 * blog, Figure 2; Efficient Long-context Language Model Training by Core
 * Attention Disaggregation, §2 "How This Paper Positions Itself").  The
 * library runs it as one launch over a rebatched pool of CA-tasks: query
 * shards of packed documents, each with the keys/values it attends to under a
 * causal per-document mask (same paper, §3.4 "The CA-Task Abstraction" and
 * "Property 2: Composability").
 *
 * Every call takes plain device pointers owned by the caller.  Nothing here
 * allocates device memory except ca_plan_create (the plan's own metadata) and
 * ca_plan_set_kv_split (the plan's re-cut forward list).  All argument errors
 * are detected on the host before any launch and returned as a status; the
 * library never aborts the process.  Functions are safe to call from several
 * host threads on distinct plans; one plan may be used concurrently on
 * several streams if each call has its own workspace.  Four calls change a
 * plan -- ca_plan_set_kv_split, ca_plan_set_backward_kernel,
 * ca_plan_set_wait_limit and ca_plan_set_timing_events -- and must not race
 * with any other call on the same plan from another host thread.  Every call that takes a plan needs
 * the device the plan was created on to be current (CA_ERR_INVALID_ARG
 * otherwise, before any launch).
 *
 * Layouts (all token-major, row-major, densely packed):
 *   q, o, dq, d_o : [total_q, num_q_heads, head_dim]   -- the query rows of
 *                   all tasks packed in task order (task t owns rows
 *                   [row0(t), row0(t) + q_len(t)), row0 = prefix sum of q_len)
 *   k, v, dk, dv  : [total_kv, num_kv_heads, head_dim] -- document i owns rows
 *                   [doc_kv_offset[i], doc_kv_offset[i] + doc_len[i])
 *   lse           : [total_q, num_q_heads] float32
 *   q, k, v, d_o, dq, dk, dv are bf16; o is bf16 or float32 (ca_shape_t.o_dtype).
 * Every pointer must be 16-byte aligned.
 */
#ifndef CA_H_
#define CA_H_

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    CA_OK = 0,
    CA_ERR_INVALID_ARG = 1,     /* a descriptor, size or pointer is invalid */
    CA_ERR_UNSUPPORTED = 2,     /* valid but outside what the kernels handle (head_dim, G) */
    CA_ERR_CUDA = 3,            /* a CUDA runtime/driver call failed */
    CA_ERR_DEVICE_TIMEOUT = 4,  /* a kernel's bounded wait ran out (see ca_device_status) */
    CA_ERR_DEVICE_BOUNDS = 5,   /* a kernel's index check failed (see ca_device_status) */
    CA_ERR_NO_DEVICE = 6        /* no sm_103 device is current */
} ca_status_t;

enum { CA_DTYPE_BF16 = 0, CA_DTYPE_FP32 = 1 };

/*
 * One CA-task.  Query positions q_start .. q_start+q_len-1 of document doc_id
 * attend to key positions j with kv_start <= j < kv_start+kv_len and j <= p
 * (positions are inside the document, the causal diagonal included: "up to
 * and including the last token in q(t)", §3.4 of the disaggregation paper).
 * The prefix CA-task of the paper is kv_start = 0, kv_len = q_start + q_len;
 * kv_start > 0 expresses one KV block of a split context, whose partial
 * (O, LSE) ca_merge combines (Context Parallelism for Scalable Million-Token
 * Inference, §3.5.2 pass-KV and Appendix B).  A row whose visible set is
 * empty gets O = 0, LSE = -inf and no gradient.
 */
typedef struct {
    int32_t doc_id;
    int32_t reserved;   /* must be 0 */
    int64_t q_start;
    int64_t q_len;      /* >= 1 */
    int64_t kv_start;
    int64_t kv_len;     /* >= 1 */
} ca_task_t;

typedef struct {
    int32_t num_q_heads;   /* H_q; query head h uses kv head h / (H_q / H_kv) */
    int32_t num_kv_heads;  /* H_kv; H_q % H_kv == 0, H_q / H_kv divides 128 */
    int32_t head_dim;      /* 64 or 128 */
    float softmax_scale;   /* usually 1/sqrt(head_dim) */
    int32_t o_dtype;       /* CA_DTYPE_BF16 or CA_DTYPE_FP32: dtype of o */
} ca_shape_t;

typedef struct ca_plan ca_plan_t;

typedef struct {
    int64_t total_q;          /* sum of q_len */
    int64_t total_kv;         /* max over documents of doc_kv_offset + doc_len */
    int64_t n_tasks, n_docs;
    int64_t causal_pairs;     /* sum over tasks and rows of |visible set|, per head */
    int64_t flops_fwd;        /* 4 * head_dim * num_q_heads * causal_pairs */
    int64_t flops_bwd;        /* 8 * head_dim * num_q_heads * causal_pairs */
    int64_t workspace_bytes;  /* device workspace that ca_forward/ca_backward need */
    int64_t n_fwd_items;      /* forward items (task, kv head, two 128-row query tiles) */
    int64_t n_bwd_items;      /* backward tiles (document, kv head, 128-key tile) */
    int64_t fwd_tile_pairs;   /* (query tile, key tile) pairs the forward computes */
    int64_t bwd_tile_pairs;   /* (key tile, query tile) pairs the backward computes */
} ca_plan_info_t;

/*
 * Validate the tasks and documents and build the plan: per-task pair counts,
 * the forward tile list (fully masked key tiles never appear) and the
 * backward tile list, both grouped per (document, kv head) with the groups
 * of most work first and the longest items first inside a group, uploaded to
 * the current device on upload_stream (a cudaStream_t; NULL = default
 * stream).  The
 * upload is synchronised before return.  The host arrays are only read.
 * Errors: CA_ERR_INVALID_ARG for n_tasks < 1, n_docs < 1, q_len < 1,
 * kv_len < 1, q_start < 0, kv_start < 0, q_start + q_len > doc_len,
 * kv_start + kv_len > doc_len, unknown doc_id, overlapping document ranges,
 * H_q % H_kv != 0, non-positive or non-finite scale, token counts >= 2^31,
 * host memory exhausted while planning; CA_ERR_UNSUPPORTED for head_dim not
 * in {64, 128}, H_q / H_kv not a divisor of 128, H_q > 4096, or a work list
 * of 2^31 items or more.  *out is set only on CA_OK; free with
 * ca_plan_destroy.
 */
ca_status_t ca_plan_create(const ca_task_t *tasks, int32_t n_tasks,
                           const int64_t *doc_len, const int64_t *doc_kv_offset, int32_t n_docs,
                           const ca_shape_t *shape, void *upload_stream, ca_plan_t **out);

/*
 * The same validation and integer accounting as ca_plan_create, without a
 * device: fills *info (every field ca_plan_info reports) and, when task_pairs
 * is not NULL, the causal pairs of every task (task_pairs[n_tasks]).  Used by
 * host-side schedulers to size CA-task pools.  Same error codes as
 * ca_plan_create except CA_ERR_CUDA / CA_ERR_NO_DEVICE.
 */
ca_status_t ca_plan_dry_run(const ca_task_t *tasks, int32_t n_tasks,
                            const int64_t *doc_len, const int64_t *doc_kv_offset, int32_t n_docs,
                            const ca_shape_t *shape, ca_plan_info_t *info, int64_t *task_pairs);

/*
 * Sparse visibility of one task ("DCP: Addressing Input Dynamism In
 * Long-Context Training via Dynamic Context Parallelism", §2.4 and Figure 6:
 * lambda-shaped sink + sliding window, causal blockwise, shared question
 * masks).  Row p of the
 * task sees key j iff the plain rule holds (kv_start <= j < kv_start+kv_len,
 * j <= p) AND
 *     j < sink  OR  j >= max(lo, p - window + 1)        (window = 0: j >= lo)
 * The three families map onto it as:
 *   lambda:           sink = S, lo = 0, window = W         (one task per shard)
 *   causal blockwise: per block of B tokens, a task of its rows with
 *                     sink = (sink blocks) * B, lo = (first visible block) * B,
 *                     window = 0; the final (test) block a plain task
 *   shared question:  the question a plain task; answer i a task of its rows
 *                     with sink = question length, lo = start of answer i
 * {0, 0, 0} is the plain rule.  All three fields >= 0 and <= the document
 * length.
 */
typedef struct {
    int64_t sink;
    int64_t lo;
    int64_t window;
} ca_mask_t;

/*
 * ca_plan_create / ca_plan_dry_run with a mask per task (masks[n_tasks];
 * NULL = every task plain).  The pair counts, FLOPs and tile lists count only
 * visible pairs and tiles with at least one visible pair.  Extra errors:
 * CA_ERR_INVALID_ARG for a negative mask field or one above the document
 * length.
 */
ca_status_t ca_plan_create_masked(const ca_task_t *tasks, const ca_mask_t *masks, int32_t n_tasks,
                                  const int64_t *doc_len, const int64_t *doc_kv_offset, int32_t n_docs,
                                  const ca_shape_t *shape, void *upload_stream, ca_plan_t **out);
ca_status_t ca_plan_dry_run_masked(const ca_task_t *tasks, const ca_mask_t *masks, int32_t n_tasks,
                                   const int64_t *doc_len, const int64_t *doc_kv_offset, int32_t n_docs,
                                   const ca_shape_t *shape, ca_plan_info_t *info, int64_t *task_pairs);

/*
 * Split-KV inside the forward launch (the pass-KV merge of "Context
 * Parallelism for Scalable Million-Token Inference", §3.5.2 and Appendix B,
 * Eq. 4, done in the same launch): a forward item (two query tiles of one
 * task and kv head) whose key-tile sequence is longer than visits_per_part
 * tiles is cut into ceil(n / visits_per_part) balanced parts that run on
 * different SMs; each part writes its rows' partial (O, LSE) to the
 * workspace and the last part to finish a row merges the parts.  This serves
 * decode and pass-Q shapes (few query rows, long contexts) and the tail of
 * very long rows.  visits_per_part > 0: that size; < 0: never split; 0
 * (the default of every plan): split only when the launch has fewer than 4
 * waves of items (4 x the device's SM count: 608 on a 152-SM GB300), into
 * parts of (total key-tile visits / SM count) clamped to [64, 128] tiles.
 * Builds and uploads a new forward list (a device allocation), synchronises
 * the device so that no enqueued launch still reads the old list, then
 * swaps it in; the workspace size in ca_plan_info may change.  On any error
 * the plan is left as it was.  It changes the plan: no other host thread
 * may use the plan meanwhile.
 */
ca_status_t ca_plan_set_kv_split(ca_plan_t *plan, int32_t visits_per_part);

/*
 * Which backward main kernel a plan's ca_backward / ca_backward_noalloc run.
 * CA_BWD_KERNEL_AUTO (every plan's default) and CA_BWD_KERNEL_SINGLE: the
 * one-CTA kernel (one SM per 128-key tile).  CA_BWD_KERNEL_PAIR: where it
 * applies (head_dim 128 and a number of query heads per kv head that divides
 * 64), the CTA-pair kernel, which processes two neighbouring key tiles of a
 * document on the two SMs of a cluster with tcgen05 pair products (each SM
 * reads half of every product's shared-memory B operand and reduces half of
 * each query tile's dQ) and exchanges dS rows between the two SMs; elsewhere
 * the one-CTA kernel.  On a GB300 the pair kernel is the slower of the two
 * (about 1.5x on the 64K packed chunk), which is why AUTO does not select it.
 * Both compute the same definition (Efficient Long-context Language Model
 * Training by Core Attention Disaggregation, §3.2 "Information flow (backward
 * pass)"); dK and dV are equal bit for bit, dQ to fp32 summation order.  It
 * changes the plan: no other host thread may use the plan meanwhile.
 * CA_ERR_INVALID_ARG for an unknown kind.
 */
enum { CA_BWD_KERNEL_AUTO = 0, CA_BWD_KERNEL_SINGLE = 1, CA_BWD_KERNEL_PAIR = 2 };
ca_status_t ca_plan_set_backward_kernel(ca_plan_t *plan, int32_t kind);

/* Sizes and integer accounting of a plan (all exact, int64). */
ca_status_t ca_plan_info(const ca_plan_t *plan, ca_plan_info_t *out);

/* Causal pairs of every task (per head), out[n_tasks]. */
ca_status_t ca_plan_task_pairs(const ca_plan_t *plan, int64_t *out);

/* Free the plan and its device metadata (synchronises the plan's device
 * first; the caller's current device is restored).  NULL is ignored. */
void ca_plan_destroy(ca_plan_t *plan);

/*
 * Forward: O and LSE of every task row and query head.
 *   LSE_p = ln sum_{j visible} exp(scale q_p . k_j)  (natural log of the
 *   scaled scores, as in the merge appendix of the million-token paper);
 *   O_p = sum_j exp(scale q_p . k_j - LSE_p) v_j.
 * workspace: ca_plan_info().workspace_bytes bytes of device memory (the
 * forward uses a work-queue counter in it).  Asynchronous on stream; launch
 * failures return CA_ERR_CUDA.  Device-side watchdog/bounds failures are
 * reported by ca_device_status.  CA_ERR_INVALID_ARG before any launch for
 * NULL or unaligned pointers, an output (o, lse, workspace) that shares a
 * byte with another output or with q, k or v (sizes from the plan), or a
 * current device other than the plan's.
 */
ca_status_t ca_forward(const ca_plan_t *plan, const void *q, const void *k, const void *v,
                       void *o, float *lse, void *workspace, void *stream);

/*
 * Backward with recompute (only LSE kept from the forward; §3.4
 * "Statelessness" of the disaggregation paper):
 *   D_p = dO_p . O_p,  dS_pj = P_pj (dO_p . v_j - D_p),
 *   dQ_p = scale sum_j dS_pj k_j,
 *   dK_j = scale sum dS_pj q_p,  dV_j = sum P_pj dO_p
 * where dK/dV sum over every task of the document and every query head of
 * the kv head's group.  dk and dv are overwritten for every row of every
 * document (0 where no task sees the key); rows outside all documents are not
 * written.  o and lse are the forward's outputs (o in the plan's o_dtype).
 * workspace: ca_plan_info().workspace_bytes bytes (fp32 dQ accumulator and
 * the D vector).  CA_ERR_INVALID_ARG before any launch for NULL or unaligned
 * pointers, an output (dq, dk, dv, workspace) that shares a byte with another
 * output or with an input (q, k, v, o, lse, d_o), or a current device other
 * than the plan's.
 */
ca_status_t ca_backward(const ca_plan_t *plan, const void *q, const void *k, const void *v,
                        const void *o, const float *lse, const void *d_o,
                        void *dq, void *dk, void *dv, void *workspace, void *stream);

/*
 * ca_backward without a workspace argument, for callers that cannot allocate
 * device memory: code inside a host framework that owns every device
 * allocation (a fixed arena or caching allocator it may not bypass), or
 * plug-in code handed only its input and output buffers.  The papers have no
 * counterpart to this entry point; it exists for such callers only.
 *
 * The scratch (fp32 dQ accumulator, D vector and work-queue counters:
 * total_q * num_q_heads * (head_dim + 1) * 4 bytes, each part rounded up to
 * 256, plus 256) lives in one file-scope device array of 16 MiB that every
 * GPU loading libca.so holds until the process exits.  Plans whose backward
 * scratch exceeds 16 MiB are rejected with CA_ERR_UNSUPPORTED before any
 * launch (the split-KV scratch of the forward, also counted in
 * ca_plan_info().workspace_bytes, is not needed here).  The entry point calls
 * no cudaMalloc, cudaFree or other allocating routine.  A call made outside a
 * stream capture looks up the array's device address (cudaGetSymbolAddress)
 * with the plan's device current; a call inside a capture reuses the address
 * of the last call outside one, so make the first call on a device before
 * any stream capture.
 * All calls on a device share the array: calls that overlap on the GPU (on
 * different streams, or from several threads) race and give wrong results,
 * so serialise them.  The array keeps the last call's contents; every call
 * clears what must start at zero itself.  Arguments and results are those of
 * ca_backward.
 */
ca_status_t ca_backward_noalloc(const ca_plan_t *plan, const void *q, const void *k, const void *v,
                                const void *o, const float *lse, const void *d_o,
                                void *dq, void *dk, void *dv, void *stream);

/*
 * Merge of partial results over KV blocks (million-token paper, Appendix B,
 * Eq. 4): for every (row, head), with M = max_s LSE_s and w_s = exp(LSE_s - M),
 *   O = sum_s w_s O_s / sum_s w_s,   LSE = M + ln sum_s w_s.
 * Parts with LSE = -inf get weight 0; if all parts are empty, O = 0 and
 * LSE = -inf.  o_parts / lse_parts are HOST arrays of n_parts device
 * pointers (1 <= n_parts <= 64); each o part is [rows, heads, head_dim] of
 * parts_dtype, each lse part [rows, heads] float32.  o_out is
 * [rows, heads, head_dim] of out_dtype; lse_out may be NULL.  head_dim must
 * be a multiple of 8 and at most 256, and rows * heads * head_dim at most
 * 2^50; other sizes, NULL or unaligned pointers give CA_ERR_INVALID_ARG
 * before anything is launched.
 */
ca_status_t ca_merge(int32_t n_parts, const void *const *o_parts, const float *const *lse_parts,
                     int32_t parts_dtype, int64_t rows, int32_t heads, int32_t head_dim,
                     void *o_out, int32_t out_dtype, float *lse_out, void *stream);

/*
 * Synchronise stream and read the plan's device error word, which every
 * kernel of the plan sets when a bounded wait runs out or an index check
 * fails.  Returns CA_OK, CA_ERR_DEVICE_TIMEOUT or CA_ERR_DEVICE_BOUNDS (and
 * clears the word), or CA_ERR_CUDA if the stream itself reports an error.
 */
ca_status_t ca_device_status(const ca_plan_t *plan, void *stream);

/* Set the bounded-wait limit (nanoseconds, default 2e9) of the plan's
 * kernels.  Used by tests to exercise the watchdog path.  It changes the
 * plan: no other host thread may use the plan meanwhile. */
ca_status_t ca_plan_set_wait_limit(ca_plan_t *plan, int64_t ns);

/*
 * Self-test of the device watchdog: launches one CTA that waits on an
 * mbarrier nothing ever arrives on, with a wait limit of limit_ns.  The wait
 * runs out, the kernel records CA_ERR_DEVICE_TIMEOUT in the plan's error
 * word and returns; the context stays usable.  Read the result with
 * ca_device_status.
 */
ca_status_t ca_watchdog_selftest(const ca_plan_t *plan, int64_t limit_ns, void *stream);

/*
 * Optional per-launch timing for profiling harnesses: when events is not
 * NULL, ca_forward records events[0] before and events[1] after its kernel,
 * and ca_backward records events[2] before its preprocess kernel, events[3]
 * after it, events[4] after the main kernel and events[5] after the dQ
 * finalize kernel, all on the call's stream.  events is a host array of
 * n_events (>= 6) cudaEvent_t handles owned by the caller; pass NULL to stop.
 * The plan keeps the pointer, not a copy of the array.  It changes the plan:
 * no other host thread may use the plan meanwhile.
 */
ca_status_t ca_plan_set_timing_events(ca_plan_t *plan, void *const *events, int32_t n_events);

/* Static description of a status code. */
const char *ca_status_string(ca_status_t status);

/* Detail of the last failing call on this host thread ("" if none). */
const char *ca_last_error(void);

/* Library version, (major << 16) | minor. */
int32_t ca_version(void);

#ifdef __cplusplus
}
#endif

#endif /* CA_H_ */
