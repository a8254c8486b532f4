/*
 * ca_oracle.c -- plain fp64 CPU oracle for document-masked core attention.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may link, load or
 * call this file: only the tests, the package's smoke check and the
 * benchmark's CPU-baseline leg use it.  It shares no code, header, table or
 * helper with the CUDA library; the two meet only in the seeded workload
 * generator, which holds none of the arithmetic below.
 *
 * What it computes (core attention, softmax(Q K^T) V, between the QKV and O
 * projections -- "Core Attention Disaggregation" blog, Figure 2; Efficient
 * Long-context Language Model Training by Core Attention Disaggregation, §2):
 *
 *   A CA-task t (same paper, §3.4 "The CA-Task Abstraction") is a query shard
 *   of document doc(t): positions p in [q_start, q_start + q_len).  Row p
 *   sees the key positions
 *       V(p) = { j : kv_start <= j < kv_start + kv_len  and  j <= p }
 *   (causal mask including the diagonal: "up to and including the last token
 *   in q(t)").  kv_start/kv_len express one KV block of a split context
 *   (Context Parallelism for Scalable Million-Token Inference, §3.5.2
 *   pass-KV); the prefix task is kv_start = 0, kv_len = q_start + q_len.
 *   A task may carry a sparse mask (sink, lo, window) ("DCP: Addressing
 *   Input Dynamism In Long-Context Training via Dynamic Context
 *   Parallelism", §2.4, Figure 6: attention sink + sliding window, causal
 *   blockwise, shared question): j in V(p) additionally needs
 *       j < sink  or  j >= max(lo, p - window + 1)    (window 0: j >= lo).
 *
 *   For query head h the kv head is g = floor(h / G), G = H_q / H_kv
 *   (contiguous GQA grouping).  With s_pj = scale * q_p . k_j:
 *       LSE_p = m_p + ln sum_{j in V(p)} exp(s_pj - m_p),  m_p = max_j s_pj
 *       P_pj  = exp(s_pj - LSE_p),     O_p = sum_j P_pj v_j
 *   (LSE is the natural log-sum-exp of the *scaled* scores, as in the merge
 *   appendix of the million-token paper, Appendix B.)  Backward (recompute,
 *   nothing but the row statistics kept -- §3.4 "Statelessness"):
 *       D_p   = dO_p . O_p,   dP_pj = dO_p . v_j,   dS_pj = P_pj (dP_pj - D_p)
 *       dQ_p  = scale sum_j dS_pj k_j
 *       dK_j  = scale sum_{(p,h) seeing j} dS_pj q_p
 *       dV_j  = sum_{(p,h) seeing j} P_pj dO_p
 *   dK/dV sum over every task of the document and every head of the group.
 *   An empty V(p) gives LSE = -inf, O = 0 and no gradient.
 *
 *   Merge of partial results over KV splits (million-token paper, Appendix B,
 *   Eq. 4):  M = max_s LSE_s,  w_s = exp(LSE_s - M),
 *       O = sum_s w_s O_s / sum_s w_s,   LSE = M + ln sum_s w_s.
 *   (The merged LSE is the log-sum-exp over the union of the blocks, which is
 *   what the LSE definition above gives for the unsplit row.)
 *
 * Inputs are the exact bf16 bit patterns widened to double; all arithmetic
 * is double.  Loops follow the definitions above one row / one column at a
 * time; OpenMP only spreads independent rows/columns over cores.
 *
 * Parity pins (tests/test_oracle_pins.py): numpy brute force of the masked
 * score matrix with scipy's logsumexp, torch fp64 autograd, central finite
 * differences, the Q = 0 closed forms, constant V, first-token identity,
 * composability of shards, and the merge identity.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

typedef struct {
    int32_t n_tasks;
    const int32_t *t_doc;
    const int64_t *t_q_start, *t_q_len, *t_kv_start, *t_kv_len;
    const int64_t *t_row0; /* first packed query row of each task */
    const int64_t *t_sink, *t_lo, *t_win; /* per-task sparse mask; NULL = none */
    int32_t n_docs;
    const int64_t *doc_len, *doc_kv_offset;
    int32_t hq, hkv, d;
    double scale;
    const uint16_t *q, *k, *v, *dout; /* bf16 bit patterns, token-major */
} orc_problem;

static double bf(uint16_t x) {
    union { uint32_t u; float f; } c;
    c.u = ((uint32_t)x) << 16;
    return (double)c.f;
}

int orc_version(void) { return 1; }

int orc_num_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* |V(p)| written out from the definition of the visible set. */
int64_t orc_visible_count(int64_t p, int64_t kv_start, int64_t kv_len) {
    int64_t hi = kv_start + kv_len - 1; /* last key of the block */
    if (p < hi) hi = p;                 /* causal: j <= p */
    return hi >= kv_start ? hi - kv_start + 1 : 0;
}

/* The sparse part of the visibility rule for key j of row p. */
static int mask_allows(int64_t p, int64_t j, int64_t sink, int64_t lo, int64_t window) {
    if (j < sink) return 1;
    if (j < lo) return 0;
    return window == 0 || j >= p - window + 1;
}

/* |V(p)| of a masked task: every key of the block up to p, tested one by one. */
int64_t orc_visible_count_masked(int64_t p, int64_t kv_start, int64_t kv_len, int64_t sink, int64_t lo,
                                 int64_t window) {
    int64_t n = 0;
    for (int64_t j = kv_start; j < kv_start + kv_len && j <= p; ++j) n += mask_allows(p, j, sink, lo, window);
    return n;
}

/* Whether row p of task t sees key j. */
static int sees(const orc_problem *pb, int32_t t, int64_t p, int64_t j) {
    if (j < pb->t_kv_start[t] || j >= pb->t_kv_start[t] + pb->t_kv_len[t] || j > p) return 0;
    if (!pb->t_sink) return 1;
    return mask_allows(p, j, pb->t_sink[t], pb->t_lo[t], pb->t_win[t]);
}

/* Causal pairs of every task: sum over its rows of |V(p)|. */
void orc_task_pairs(int32_t n_tasks, const int64_t *q_start, const int64_t *q_len,
                    const int64_t *kv_start, const int64_t *kv_len, int64_t *out) {
    for (int32_t t = 0; t < n_tasks; ++t) {
        int64_t acc = 0;
        for (int64_t p = q_start[t]; p < q_start[t] + q_len[t]; ++p)
            acc += orc_visible_count(p, kv_start[t], kv_len[t]);
        out[t] = acc;
    }
}

/* Locate the task owning packed query row r (tasks are packed in order). */
static int32_t task_of_row(const orc_problem *pb, int64_t r) {
    int32_t lo = 0, hi = pb->n_tasks - 1;
    while (lo < hi) {
        int32_t mid = (lo + hi + 1) / 2;
        if (pb->t_row0[mid] <= r) lo = mid; else hi = mid - 1;
    }
    return lo;
}

static const uint16_t *qrow(const orc_problem *pb, const uint16_t *base, int64_t r, int32_t h) {
    return base + ((size_t)r * pb->hq + h) * pb->d;
}
static const uint16_t *kvrow(const orc_problem *pb, const uint16_t *base, int64_t row, int32_t g) {
    return base + ((size_t)row * pb->hkv + g) * pb->d;
}

/* Row statistics of packed row r, head h: LSE, O (length d) and, when
 * D != NULL, D = dO . O.  Returns |V(p)|. */
static int64_t row_forward(const orc_problem *pb, int64_t r, int32_t h,
                           double *lse, double *o, double *D, double *qv) {
    const int32_t t = task_of_row(pb, r);
    const int64_t p = pb->t_q_start[t] + (r - pb->t_row0[t]);
    const int32_t doc = pb->t_doc[t];
    const int64_t base = pb->doc_kv_offset[doc];
    const int32_t G = pb->hq / pb->hkv, g = h / G, d = pb->d;
    const int64_t j0 = pb->t_kv_start[t];
    const int64_t j1 = j0 + orc_visible_count(p, j0, pb->t_kv_len[t]); /* keys [j0, j1) pass the block and causal tests */
    int64_t n = 0;
    for (int64_t j = j0; j < j1; ++j) n += sees(pb, t, p, j);
    const uint16_t *qr = qrow(pb, pb->q, r, h);
    for (int c = 0; c < d; ++c) { qv[c] = bf(qr[c]); o[c] = 0.0; }
    if (n == 0) {
        *lse = -INFINITY;
        if (D) *D = 0.0;
        return 0;
    }
    /* pass 1: max of the scaled scores */
    double m = -INFINITY;
    for (int64_t j = j0; j < j1; ++j) {
        if (!sees(pb, t, p, j)) continue;
        const uint16_t *kr = kvrow(pb, pb->k, base + j, g);
        double s = 0.0;
        for (int c = 0; c < d; ++c) s += qv[c] * bf(kr[c]);
        s *= pb->scale;
        if (s > m) m = s;
    }
    /* pass 2: normaliser */
    double sum = 0.0;
    for (int64_t j = j0; j < j1; ++j) {
        if (!sees(pb, t, p, j)) continue;
        const uint16_t *kr = kvrow(pb, pb->k, base + j, g);
        double s = 0.0;
        for (int c = 0; c < d; ++c) s += qv[c] * bf(kr[c]);
        sum += exp(s * pb->scale - m);
    }
    const double L = m + log(sum);
    /* pass 3: O = sum_j P_pj v_j with P_pj = exp(s_pj - LSE) */
    for (int64_t j = j0; j < j1; ++j) {
        if (!sees(pb, t, p, j)) continue;
        const uint16_t *kr = kvrow(pb, pb->k, base + j, g);
        const uint16_t *vr = kvrow(pb, pb->v, base + j, g);
        double s = 0.0;
        for (int c = 0; c < d; ++c) s += qv[c] * bf(kr[c]);
        const double P = exp(s * pb->scale - L);
        for (int c = 0; c < d; ++c) o[c] += P * bf(vr[c]);
    }
    *lse = L;
    if (D) {
        const uint16_t *dor = qrow(pb, pb->dout, r, h);
        double acc = 0.0;
        for (int c = 0; c < d; ++c) acc += bf(dor[c]) * o[c];
        *D = acc;
    }
    return n;
}

/* Forward of selected (row, head) pairs: o_out [n, d], lse_out [n]. */
int orc_forward_rows(const orc_problem *pb, int64_t n_rows, const int64_t *rows,
                     const int32_t *heads, double *o_out, double *lse_out) {
    int err = 0;
#pragma omp parallel
    {
        double *qv = (double *)malloc(sizeof(double) * pb->d);
        if (!qv) {
#pragma omp atomic write
            err = 1;
        } else {
#pragma omp for schedule(dynamic, 1)
            for (int64_t i = 0; i < n_rows; ++i)
                row_forward(pb, rows[i], heads[i], &lse_out[i], &o_out[(size_t)i * pb->d], NULL, qv);
            free(qv);
        }
    }
    return err;
}

/* Forward of every row: o_out [total_q, hq, d], lse_out [total_q, hq]. */
int orc_forward_all(const orc_problem *pb, int64_t total_q, double *o_out, double *lse_out) {
    int err = 0;
#pragma omp parallel
    {
        double *qv = (double *)malloc(sizeof(double) * pb->d);
        if (!qv) {
#pragma omp atomic write
            err = 1;
        } else {
#pragma omp for schedule(dynamic, 4)
            for (int64_t i = 0; i < total_q * pb->hq; ++i)
                row_forward(pb, i / pb->hq, (int32_t)(i % pb->hq), &lse_out[i],
                            &o_out[(size_t)i * pb->d], NULL, qv);
            free(qv);
        }
    }
    return err;
}

/* dQ of selected (row, head) pairs: dq_out [n, d].  Recomputes LSE, O, D. */
int orc_dq_rows(const orc_problem *pb, int64_t n_rows, const int64_t *rows,
                const int32_t *heads, double *dq_out) {
    int err = 0;
    const int d = pb->d;
#pragma omp parallel
    {
        double *qv = (double *)malloc(sizeof(double) * d);
        double *o = (double *)malloc(sizeof(double) * d);
        double *dov = (double *)malloc(sizeof(double) * d);
        if (!qv || !o || !dov) {
#pragma omp atomic write
            err = 1;
        } else {
#pragma omp for schedule(dynamic, 1)
            for (int64_t i = 0; i < n_rows; ++i) {
                const int64_t r = rows[i];
                const int32_t h = heads[i];
                double L, D;
                double *dq = &dq_out[(size_t)i * d];
                for (int c = 0; c < d; ++c) dq[c] = 0.0;
                const int64_t n = row_forward(pb, r, h, &L, o, &D, qv);
                if (n == 0) continue;
                const int32_t t = task_of_row(pb, r);
                const int64_t base = pb->doc_kv_offset[pb->t_doc[t]];
                const int32_t g = h / (pb->hq / pb->hkv);
                const uint16_t *dor = qrow(pb, pb->dout, r, h);
                for (int c = 0; c < d; ++c) dov[c] = bf(dor[c]);
                const int64_t p = pb->t_q_start[t] + (r - pb->t_row0[t]);
                for (int64_t j = pb->t_kv_start[t]; j <= p && j < pb->t_kv_start[t] + pb->t_kv_len[t]; ++j) {
                    if (!sees(pb, t, p, j)) continue;
                    const uint16_t *kr = kvrow(pb, pb->k, base + j, g);
                    const uint16_t *vr = kvrow(pb, pb->v, base + j, g);
                    double s = 0.0, dP = 0.0;
                    for (int c = 0; c < d; ++c) { s += qv[c] * bf(kr[c]); dP += dov[c] * bf(vr[c]); }
                    const double P = exp(s * pb->scale - L);
                    const double dS = P * (dP - D);
                    for (int c = 0; c < d; ++c) dq[c] += pb->scale * dS * bf(kr[c]);
                }
            }
        }
        free(qv); free(o); free(dov);
    }
    return err;
}

/*
 * dK, dV of selected key columns (kv row, kv head).  A column at document
 * position j of document doc collects, over every task of doc whose KV block
 * holds j, every row p >= j of the task and every query head of the group:
 *   dK_j += scale dS_pj q_p,  dV_j += P_pj dO_p.
 * Row statistics (LSE_p, D_p) come from rs_lse / rs_D, indexed by
 * [packed row * hq + head]; rows the columns depend on must have been filled
 * by orc_row_stats first (the caller marks and computes them).
 */
static void dkdv_column(const orc_problem *pb, int32_t doc, int64_t j, int32_t g,
                        const double *rs_lse, const double *rs_D,
                        double *dk, double *dv, double *kv_k, double *kv_v) {
    const int d = pb->d, G = pb->hq / pb->hkv;
    const int64_t base = pb->doc_kv_offset[doc];
    const uint16_t *kr = kvrow(pb, pb->k, base + j, g);
    const uint16_t *vr = kvrow(pb, pb->v, base + j, g);
    for (int c = 0; c < d; ++c) { kv_k[c] = bf(kr[c]); kv_v[c] = bf(vr[c]); dk[c] = 0.0; dv[c] = 0.0; }
    for (int32_t t = 0; t < pb->n_tasks; ++t) {
        if (pb->t_doc[t] != doc) continue;
        if (j < pb->t_kv_start[t] || j >= pb->t_kv_start[t] + pb->t_kv_len[t]) continue;
        for (int64_t i = 0; i < pb->t_q_len[t]; ++i) {
            const int64_t p = pb->t_q_start[t] + i;
            if (!sees(pb, t, p, j)) continue;
            const int64_t r = pb->t_row0[t] + i;
            for (int32_t h = g * G; h < (g + 1) * G; ++h) {
                const size_t ix = (size_t)r * pb->hq + h;
                const uint16_t *qr = qrow(pb, pb->q, r, h);
                const uint16_t *dor = qrow(pb, pb->dout, r, h);
                double s = 0.0, dP = 0.0;
                for (int c = 0; c < d; ++c) { s += bf(qr[c]) * kv_k[c]; dP += bf(dor[c]) * kv_v[c]; }
                const double P = exp(s * pb->scale - rs_lse[ix]);
                const double dS = P * (dP - rs_D[ix]);
                for (int c = 0; c < d; ++c) {
                    dk[c] += pb->scale * dS * bf(qr[c]);
                    dv[c] += P * bf(dor[c]);
                }
            }
        }
    }
}

/* Row statistics (LSE, D) of the (row, head) pairs with mark[row*hq+head]
 * != 0, written to lse/D at the same index. */
int orc_row_stats(const orc_problem *pb, int64_t total_q, const uint8_t *mark,
                  double *lse, double *D) {
    int err = 0;
#pragma omp parallel
    {
        double *qv = (double *)malloc(sizeof(double) * pb->d);
        double *o = (double *)malloc(sizeof(double) * pb->d);
        if (!qv || !o) {
#pragma omp atomic write
            err = 1;
        } else {
#pragma omp for schedule(dynamic, 4)
            for (int64_t i = 0; i < total_q * pb->hq; ++i) {
                if (!mark[i]) continue;
                row_forward(pb, i / pb->hq, (int32_t)(i % pb->hq), &lse[i], o, &D[i], qv);
            }
        }
        free(qv); free(o);
    }
    return err;
}

/* dK, dV of selected columns: col_doc, col_pos (document position), col_g.
 * dk_out, dv_out [n, d]. */
int orc_dkdv_cols(const orc_problem *pb, int64_t n_cols, const int32_t *col_doc,
                  const int64_t *col_pos, const int32_t *col_g,
                  const double *rs_lse, const double *rs_D, double *dk_out, double *dv_out) {
    int err = 0;
#pragma omp parallel
    {
        double *a = (double *)malloc(sizeof(double) * pb->d);
        double *b = (double *)malloc(sizeof(double) * pb->d);
        if (!a || !b) {
#pragma omp atomic write
            err = 1;
        } else {
#pragma omp for schedule(dynamic, 1)
            for (int64_t i = 0; i < n_cols; ++i)
                dkdv_column(pb, col_doc[i], col_pos[i], col_g[i], rs_lse, rs_D,
                            &dk_out[(size_t)i * pb->d], &dv_out[(size_t)i * pb->d], a, b);
        }
        free(a); free(b);
    }
    return err;
}

/* Merge of n_parts partial results (million-token paper, Appendix B, Eq. 4).
 * o_parts [n_parts, rows, d], lse_parts [n_parts, rows] -> o [rows, d], lse [rows]. */
void orc_merge(int32_t n_parts, int64_t rows, int32_t d, const double *o_parts,
               const double *lse_parts, double *o, double *lse) {
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < rows; ++r) {
        double M = -INFINITY;
        for (int32_t s = 0; s < n_parts; ++s)
            if (lse_parts[(size_t)s * rows + r] > M) M = lse_parts[(size_t)s * rows + r];
        double *out = &o[(size_t)r * d];
        for (int c = 0; c < d; ++c) out[c] = 0.0;
        if (M == -INFINITY) { lse[r] = -INFINITY; continue; }
        double wsum = 0.0;
        for (int32_t s = 0; s < n_parts; ++s) {
            const double w = exp(lse_parts[(size_t)s * rows + r] - M);
            wsum += w;
            const double *os = &o_parts[((size_t)s * rows + r) * d];
            for (int c = 0; c < d; ++c) out[c] += w * os[c];
        }
        for (int c = 0; c < d; ++c) out[c] /= wsum;
        lse[r] = M + log(wsum);
    }
}
