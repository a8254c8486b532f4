/*
 * ca_sched.h -- host-side planning of CA-tasks across attention servers
 * (part of libca.so; no GPU is touched by anything declared here).
 *
 * Three pieces, all from "Efficient Long-context Language Model Training by
 * Core Attention Disaggregation":
 *
 *   - the profiler cost model ("The Profiler and Cost Model"): measured
 *     fwd+bwd times on a grid of (query length, context length) CA-task
 *     shapes, bilinear interpolation inside the grid, FLOPs / peak measured
 *     throughput in the saturation region beyond it;
 *   - the optimal shard dimensions of a split ("Appendix B: Optimal Shard
 *     Dimension Computation"): the query length n_q and context length n_kv
 *     of a sub-shard that carries a fraction alpha of an Item's attention
 *     work with the least communication n_q*sizeof(q) + n_kv*sizeof(kv);
 *   - the communication-aware greedy scheduler ("The Communication-Aware
 *     Greedy Scheduler", steps 1-4): documents start on the devices that hold
 *     their tokens, and Items (whole or split) migrate from surplus to
 *     deficit attention servers in order of transferred work per byte.
 *
 * Units.  Attention work is counted in causal (query, key) pairs of one head
 * (int64, exact): a query shard [a, b) of a document with the prefix context
 * [0, b) has b(b+1)/2 - a(a+1)/2 pairs.  FLOPs are 4*head_dim*H_q per pair
 * forward and 8*head_dim*H_q backward; a common factor, so the scheduler
 * balances pairs.  Communication is in bytes.
 *
 * Every function validates its arguments and returns CA_ERR_INVALID_ARG
 * without side effects when they are wrong; none aborts the process.
 */
#ifndef CA_SCHED_H_
#define CA_SCHED_H_

#include <stdint.h>

#include "ca.h"

#ifdef __cplusplus
extern "C" {
#endif

/* ------------------------------------------------------------------ profiler */

typedef struct ca_profile ca_profile_t;

/*
 * Builds a cost model from a measured grid.  nq_grid[0..n_nq) and
 * nkv_grid[0..n_nkv) are strictly increasing positive token counts;
 * seconds[i * n_nkv + j] is the measured fwd+bwd time of one CA-task with
 * query length nq_grid[i] and context length nkv_grid[j] (a query shard that
 * ends at the end of its context; where nq_grid[i] > nkv_grid[j] the entry
 * is the time of the task with n_q = n_kv).  Every entry must be > 0.
 * flops_per_pair is the FLOPs credited to one causal pair (12*d*H_q for
 * fwd+bwd).  The peak throughput of the saturation region is the largest
 * flops / seconds over the grid.  The profile copies its inputs; the caller
 * keeps ownership of the arrays.
 */
ca_status_t ca_profile_create(const int64_t *nq_grid, int32_t n_nq, const int64_t *nkv_grid, int32_t n_nkv,
                              const double *seconds, double flops_per_pair, ca_profile_t **out);

/*
 * Predicted seconds of a CA-task with query length n_q and context length
 * n_kv (1 <= n_q <= n_kv).  Inside the grid's box [nq_grid[0], max] x
 * [nkv_grid[0], max]: bilinear interpolation between the four grid points of
 * the enclosing cell (coordinates below the first grid point are clamped to
 * it).  Beyond the largest grid value on either axis: pairs * flops_per_pair
 * / peak throughput.
 */
ca_status_t ca_profile_predict(const ca_profile_t *prof, int64_t n_q, int64_t n_kv, double *seconds);

/* Peak measured throughput (FLOP/s) of the profile. */
ca_status_t ca_profile_peak(const ca_profile_t *prof, double *flops_per_s);

void ca_profile_destroy(ca_profile_t *prof);

/* ------------------------------------------------------------------ optimal shard (App. B) */

/*
 * Sub-shard of an Item with query length L_q and context length L_kv (its
 * queries are the last L_q positions of the prefix [0, L_kv)) carrying the
 * fraction alpha (0 < alpha <= 1) of the Item's work with the least
 * communication, bytes_q per query token and bytes_kv per context token.
 *
 * Continuous optimum (the appendix's closed form, beta = bytes_kv/bytes_q):
 *   n_q* = sqrt(alpha beta L_q (2 L_kv - L_q) / (beta + 2)),
 * projected onto the feasible range where n_kv = (A / n_q + n_q) / 2 with
 * A = alpha L_q (2 L_kv - L_q) satisfies n_q + L_kv - L_q <= n_kv <= L_kv
 * and n_q <= L_q (the communication is convex in n_q, so the constrained
 * optimum is the projection).
 *
 * Integer shard: n_q = the nearest integer to that optimum (halves round
 * up), in [1, L_q];
 * then n_kv = the integer in [n_q + L_kv - L_q, L_kv] whose exact pair count
 * n_q n_kv - n_q (n_q - 1) / 2 is nearest to target_pairs (ties to the
 * smaller n_kv).  *n_q_out, *n_kv_out receive the integer shard,
 * *nq_real_out (may be NULL) the projected continuous optimum.
 */
ca_status_t ca_optimal_shard(int64_t L_q, int64_t L_kv, double alpha, int64_t target_pairs, double bytes_q,
                             double bytes_kv, int64_t *n_q_out, int64_t *n_kv_out, double *nq_real_out);

/* ------------------------------------------------------------------ greedy scheduler */

typedef struct {
    int32_t n_servers;        /* k >= 1 attention servers (= devices) */
    double tolerance;         /* epsilon >= 0: stop once every deficit is <= epsilon * target */
    double min_score;         /* stop a server when the best E = pairs / byte is <= this (>= 0) */
    double bytes_q;           /* bytes sent per query token (> 0) */
    double bytes_kv;          /* bytes sent per context token (> 0) */
    int64_t min_shard_tokens; /* 0 = any split; else splits whose shard or remaining pieces
                                 are shorter than this many query tokens are not considered */
} ca_sched_params_t;

/* One scheduled CA-task: a query shard of a document with its prefix context. */
typedef struct {
    int32_t server;     /* attention server that computes it */
    int32_t home;       /* device that holds its tokens (where the shard started) */
    int32_t doc_id;
    int32_t reserved;   /* 0 */
    int64_t q_start;    /* query positions [q_start, q_start + q_len) */
    int64_t q_len;
    int64_t kv_len;     /* context [0, kv_len), kv_len = q_start + q_len */
    int64_t pairs;      /* causal pairs of the shard (per head) */
} ca_sched_task_t;

typedef struct {
    int64_t target_pairs_x1000; /* 1000 * total pairs / k, rounded down (reporting only) */
    int64_t max_load, min_load; /* pairs on the most / least loaded server after scheduling */
    int64_t n_tasks;            /* tasks written */
    int64_t n_migrations;       /* whole Items moved */
    int64_t n_splits;           /* Items split */
    double comm_bytes;          /* bytes of every migration (q and context of moved shards) */
} ca_sched_result_t;

/*
 * Schedules documents doc_len[0..n_docs) (doc_id = index) onto
 * params->n_servers attention servers.
 *
 * Initial placement (the "Problem formulation" paragraph): the documents are
 * laid out in order and device s holds tokens [s T, (s+1) T) of the stream,
 * T = ceil(total / k); a document crossing a boundary is split there, each
 * piece an Item on the device holding it (its context is the document prefix).
 * Step 1: target = total pairs / k.  Step 2: deficit servers in descending
 * order of deficit; for each, repeatedly pick over every Item t on a surplus
 * server s the largest E = dF / bytes, dF = min(pairs(t), surplus(s),
 * deficit), bytes = the whole Item's q and context bytes when dF = pairs(t),
 * else those of the ca_optimal_shard split with alpha = dF / pairs(t) and
 * target = dF rounded to the nearest integer (ties: the earliest Item in
 * creation order).  Step 3: move the Item, or cut the shard out of it (the
 * remainder stays as up to two Items on the source).  Step 4: a server is done
 * when its deficit is <= tolerance * target or no candidate has E > min_score.
 *
 * tasks_out has room for max_tasks entries; the tasks are written grouped by
 * server, and within a server by (doc_id, q_start).  Returns
 * CA_ERR_INVALID_ARG if max_tasks is too small (result->n_tasks then holds the
 * number needed).
 */
ca_status_t ca_schedule(const int64_t *doc_len, int32_t n_docs, const ca_sched_params_t *params,
                        ca_sched_task_t *tasks_out, int64_t max_tasks, ca_sched_result_t *result);

/* ------------------------------------------------------------------ 2N-chunk sharding */

/*
 * Load-balanced sharding of every document over n_ranks ranks ("Context
 * Parallelism for Scalable Million-Token Inference", §3.5.1 "Load-Balanced
 * Sharding of Input Sequences"; the head-tail shards of "Efficient
 * Long-context Language Model Training by Core Attention Disaggregation",
 * "The role of head-tail sharding in practice"): each document is cut into
 * 2N chunks C_0 .. C_{2N-1} and rank i takes C_i and C_{2N-1-i}.  Padding is
 * not materialised: chunk size c = ceil(L / 2N), chunk j covers positions
 * [j c, min((j+1) c, L)), and empty chunks are omitted.  Each chunk becomes
 * one CA-task with its prefix context (server = home = rank).  Tasks are
 * written grouped by rank, then by (doc_id, q_start); *n_tasks_out receives
 * the count (also when max_tasks is too small, which returns
 * CA_ERR_INVALID_ARG).
 */
ca_status_t ca_shard_2n(const int64_t *doc_len, int32_t n_docs, int32_t n_ranks, ca_sched_task_t *tasks_out,
                        int64_t max_tasks, int64_t *n_tasks_out);

#ifdef __cplusplus
}
#endif

#endif /* CA_SCHED_H_ */
