// Host-side planning of CA-tasks across attention servers: profiler cost
// model, optimal split dimensions and the communication-aware greedy
// scheduler of "Efficient Long-context Language Model Training by Core
// Attention Disaggregation" ("The Profiler and Cost Model", "The
// Communication-Aware Greedy Scheduler", "Appendix B: Optimal Shard Dimension
// Computation").  Plain C++; the declarations and the exact rules are in
// include/ca_sched.h.
#include <algorithm>
#include <cmath>
#include <new>
#include <string>
#include <vector>

#include "../../include/ca_sched.h"
#include "ca_internal.h"

namespace {

// Causal pairs of a query shard of n_q tokens ending at context length n_kv.
inline int64_t shard_pairs(int64_t n_q, int64_t n_kv) { return n_q * n_kv - n_q * (n_q - 1) / 2; }

// Causal pairs of query positions [a, b) with prefix context.
inline int64_t range_pairs(int64_t a, int64_t b) { return b * (b + 1) / 2 - a * (a + 1) / 2; }

}  // namespace

struct ca_profile {
    std::vector<int64_t> nq, nkv;
    std::vector<double> sec;
    double flops_per_pair = 0.0;
    double peak = 0.0;  // FLOP/s
};

extern "C" {

static ca_status_t profile_create_impl(const int64_t *nq_grid, int32_t n_nq, const int64_t *nkv_grid, int32_t n_nkv,
                                      const double *seconds, double flops_per_pair, ca_profile_t **out) {
    using ca::fail;
    if (!out) return fail(CA_ERR_INVALID_ARG, "ca_profile_create: out is NULL");
    *out = nullptr;
    if (!nq_grid || !nkv_grid || !seconds || n_nq < 1 || n_nkv < 1)
        return fail(CA_ERR_INVALID_ARG, "ca_profile_create: empty grid");
    if (!(flops_per_pair > 0.0)) return fail(CA_ERR_INVALID_ARG, "ca_profile_create: flops_per_pair must be > 0");
    for (int32_t i = 0; i < n_nq; ++i)
        if (nq_grid[i] < 1 || (i > 0 && nq_grid[i] <= nq_grid[i - 1]))
            return fail(CA_ERR_INVALID_ARG, "ca_profile_create: nq_grid must be positive and strictly increasing");
    for (int32_t j = 0; j < n_nkv; ++j)
        if (nkv_grid[j] < 1 || (j > 0 && nkv_grid[j] <= nkv_grid[j - 1]))
            return fail(CA_ERR_INVALID_ARG, "ca_profile_create: nkv_grid must be positive and strictly increasing");
    auto *p = new ca_profile;
    p->nq.assign(nq_grid, nq_grid + n_nq);
    p->nkv.assign(nkv_grid, nkv_grid + n_nkv);
    p->sec.assign(seconds, seconds + static_cast<size_t>(n_nq) * n_nkv);
    p->flops_per_pair = flops_per_pair;
    for (int32_t i = 0; i < n_nq; ++i)
        for (int32_t j = 0; j < n_nkv; ++j) {
            const double s = p->sec[static_cast<size_t>(i) * n_nkv + j];
            if (!(s > 0.0) || !std::isfinite(s)) {
                delete p;
                return fail(CA_ERR_INVALID_ARG, "ca_profile_create: every measured time must be > 0");
            }
            const int64_t q = std::min(p->nq[i], p->nkv[j]);
            p->peak = std::max(p->peak, static_cast<double>(shard_pairs(q, p->nkv[j])) * flops_per_pair / s);
        }
    *out = p;
    return CA_OK;
}

// Each entry point that builds host containers returns a failed allocation
// as a status instead of letting the exception leave an extern "C" function.
ca_status_t ca_profile_create(const int64_t *nq_grid, int32_t n_nq, const int64_t *nkv_grid, int32_t n_nkv,
                              const double *seconds, double flops_per_pair, ca_profile_t **out) {
    try {
        return profile_create_impl(nq_grid, n_nq, nkv_grid, n_nkv, seconds, flops_per_pair, out);
    } catch (const std::bad_alloc &) {
        return ca::fail(CA_ERR_INVALID_ARG, "ca_profile_create: host memory exhausted");
    }
}

ca_status_t ca_profile_predict(const ca_profile_t *prof, int64_t n_q, int64_t n_kv, double *seconds) {
    using ca::fail;
    if (!prof || !seconds) return fail(CA_ERR_INVALID_ARG, "ca_profile_predict: NULL argument");
    if (n_q < 1 || n_kv < n_q) return fail(CA_ERR_INVALID_ARG, "ca_profile_predict: need 1 <= n_q <= n_kv");
    if (n_q > prof->nq.back() || n_kv > prof->nkv.back()) {  // saturation region
        *seconds = static_cast<double>(shard_pairs(n_q, n_kv)) * prof->flops_per_pair / prof->peak;
        return CA_OK;
    }
    // enclosing cell and the position inside it along one axis
    auto locate = [](const std::vector<int64_t> &g, int64_t x, size_t &i, double &t) {
        if (g.size() == 1 || x <= g[0]) {
            i = 0;
            t = 0.0;
            return;
        }
        i = static_cast<size_t>(std::upper_bound(g.begin(), g.end(), x) - g.begin()) - 1;
        if (i >= g.size() - 1) i = g.size() - 2;
        t = static_cast<double>(x - g[i]) / static_cast<double>(g[i + 1] - g[i]);
    };
    size_t i, j;
    double tq, tk;
    locate(prof->nq, n_q, i, tq);
    locate(prof->nkv, n_kv, j, tk);
    const size_t w = prof->nkv.size();
    const size_t i1 = std::min(i + 1, prof->nq.size() - 1), j1 = std::min(j + 1, w - 1);
    const double s00 = prof->sec[i * w + j], s01 = prof->sec[i * w + j1];
    const double s10 = prof->sec[i1 * w + j], s11 = prof->sec[i1 * w + j1];
    *seconds = (1.0 - tq) * ((1.0 - tk) * s00 + tk * s01) + tq * ((1.0 - tk) * s10 + tk * s11);
    return CA_OK;
}

ca_status_t ca_profile_peak(const ca_profile_t *prof, double *flops_per_s) {
    if (!prof || !flops_per_s) return ca::fail(CA_ERR_INVALID_ARG, "ca_profile_peak: NULL argument");
    *flops_per_s = prof->peak;
    return CA_OK;
}

void ca_profile_destroy(ca_profile_t *prof) { delete prof; }

ca_status_t ca_optimal_shard(int64_t L_q, int64_t L_kv, double alpha, int64_t target_pairs, double bytes_q,
                             double bytes_kv, int64_t *n_q_out, int64_t *n_kv_out, double *nq_real_out) {
    using ca::fail;
    if (!n_q_out || !n_kv_out) return fail(CA_ERR_INVALID_ARG, "ca_optimal_shard: NULL output");
    if (L_q < 1 || L_kv < L_q) return fail(CA_ERR_INVALID_ARG, "ca_optimal_shard: need 1 <= L_q <= L_kv");
    if (!(alpha > 0.0 && alpha <= 1.0)) return fail(CA_ERR_INVALID_ARG, "ca_optimal_shard: need 0 < alpha <= 1");
    if (!(bytes_q > 0.0 && bytes_kv > 0.0)) return fail(CA_ERR_INVALID_ARG, "ca_optimal_shard: bytes must be > 0");
    if (target_pairs < 1) return fail(CA_ERR_INVALID_ARG, "ca_optimal_shard: target_pairs must be >= 1");
    const double lq = static_cast<double>(L_q), lkv = static_cast<double>(L_kv);
    const double beta = bytes_kv / bytes_q;
    const double A = alpha * lq * (2.0 * lkv - lq);
    const double n_opt = std::sqrt(alpha * beta * lq * (2.0 * lkv - lq) / (beta + 2.0));
    // feasible n_q: n_kv(n_q) = (A / n_q + n_q) / 2 <= L_kv  and  n_kv - n_q >= L_kv - L_q, n_q <= L_q
    const double c = lkv - lq;
    const double lo = A / (lkv + std::sqrt(std::max(lkv * lkv - A, 0.0)));
    const double hi = std::min(lq, A / (std::sqrt(c * c + A) + c));
    const double n_real = std::min(std::max(n_opt, lo), std::max(hi, lo));
    int64_t n_q = static_cast<int64_t>(std::floor(n_real + 0.5));
    n_q = std::min(std::max<int64_t>(n_q, 1), L_q);
    // n_kv with the exact pair count nearest to the target (ties: the smaller)
    const int64_t num = target_pairs + n_q * (n_q - 1) / 2;
    int64_t n_kv = num / n_q;
    if (2 * (num - n_kv * n_q) > n_q) ++n_kv;
    n_kv = std::min(std::max(n_kv, n_q + L_kv - L_q), L_kv);
    *n_q_out = n_q;
    *n_kv_out = n_kv;
    if (nq_real_out) *nq_real_out = n_real;
    return CA_OK;
}

}  // extern "C"

namespace {

struct Item {
    int32_t doc;
    int64_t q0, q1;  // query positions [q0, q1), context [0, q1)
    int32_t server, home;
    bool alive;
};

}  // namespace

static ca_status_t schedule_impl(const int64_t *doc_len, int32_t n_docs, const ca_sched_params_t *params,
                                 ca_sched_task_t *tasks_out, int64_t max_tasks, ca_sched_result_t *result) {
    using ca::fail;
    if (!doc_len || !params || !result || n_docs < 1) return fail(CA_ERR_INVALID_ARG, "ca_schedule: NULL or empty input");
    const ca_sched_params_t &P = *params;
    if (P.n_servers < 1) return fail(CA_ERR_INVALID_ARG, "ca_schedule: n_servers must be >= 1");
    if (!(P.tolerance >= 0.0) || !(P.min_score >= 0.0))
        return fail(CA_ERR_INVALID_ARG, "ca_schedule: tolerance and min_score must be >= 0");
    if (!(P.bytes_q > 0.0) || !(P.bytes_kv > 0.0)) return fail(CA_ERR_INVALID_ARG, "ca_schedule: bytes must be > 0");
    if (P.min_shard_tokens < 0) return fail(CA_ERR_INVALID_ARG, "ca_schedule: min_shard_tokens must be >= 0");
    int64_t total = 0;
    for (int32_t d = 0; d < n_docs; ++d) {
        if (doc_len[d] < 1 || doc_len[d] > (int64_t(1) << 31))
            return fail(CA_ERR_INVALID_ARG, "ca_schedule: document " + std::to_string(d) + " has an invalid length");
        total += doc_len[d];
    }
    const int32_t k = P.n_servers;
    *result = ca_sched_result_t{};

    // initial placement: device s holds tokens [s T, (s+1) T) of the stream
    const int64_t T = (total + k - 1) / k;
    std::vector<Item> items;
    std::vector<int64_t> load(k, 0);
    int64_t off = 0;
    for (int32_t d = 0; d < n_docs; ++d) {
        int64_t pos = off;
        const int64_t end = off + doc_len[d];
        while (pos < end) {
            const int32_t s = static_cast<int32_t>(std::min<int64_t>(pos / T, k - 1));
            const int64_t stop = std::min(end, (s + 1) * T);
            Item it{d, pos - off, stop - off, s, s, true};
            load[s] += range_pairs(it.q0, it.q1);
            items.push_back(it);
            pos = stop;
        }
        off = end;
    }
    int64_t total_pairs = 0;
    for (int32_t s = 0; s < k; ++s) total_pairs += load[s];
    const double target = static_cast<double>(total_pairs) / k;

    // step 2: deficit servers, largest deficit first (ties: lower index)
    std::vector<int32_t> deficit;
    for (int32_t s = 0; s < k; ++s)
        if (static_cast<double>(load[s]) < target) deficit.push_back(s);
    std::stable_sort(deficit.begin(), deficit.end(),
                     [&](int32_t a, int32_t b) { return load[a] < load[b]; });

    int64_t steps = 0;
    for (const int32_t dst : deficit) {
        while (target - static_cast<double>(load[dst]) > P.tolerance * target) {
            if (++steps > 4 * static_cast<int64_t>(n_docs) * k + 1000000)
                return fail(CA_ERR_INVALID_ARG, "ca_schedule: no convergence");
            const double D = target - static_cast<double>(load[dst]);
            double best_e = -1.0;
            size_t best = 0;
            bool best_split = false;
            int64_t best_nq = 0, best_nkv = 0;
            double best_bytes = 0.0;
            for (size_t t = 0; t < items.size(); ++t) {
                const Item &it = items[t];
                if (!it.alive || it.server == dst) continue;
                const double S = static_cast<double>(load[it.server]) - target;
                if (!(S > 0.0)) continue;
                const int64_t f = range_pairs(it.q0, it.q1);
                const double dF = std::min(std::min(static_cast<double>(f), S), D);
                bool split = dF < static_cast<double>(f);
                int64_t nq = it.q1 - it.q0, nkv = it.q1;
                if (split) {
                    const int64_t tgt = std::max<int64_t>(1, static_cast<int64_t>(std::floor(dF + 0.5)));
                    if (ca_optimal_shard(it.q1 - it.q0, it.q1, dF / static_cast<double>(f), tgt, P.bytes_q, P.bytes_kv,
                                         &nq, &nkv, nullptr) != CA_OK)
                        continue;
                    if (nq == it.q1 - it.q0 && nkv == it.q1) {
                        split = false;  // the optimum is the whole Item
                    } else if (P.min_shard_tokens > 0) {
                        const int64_t left = (nkv - nq) - it.q0, right = it.q1 - nkv;
                        if (nq < P.min_shard_tokens || (left > 0 && left < P.min_shard_tokens) ||
                            (right > 0 && right < P.min_shard_tokens))
                            continue;
                    }
                }
                const double bytes = static_cast<double>(nq) * P.bytes_q + static_cast<double>(nkv) * P.bytes_kv;
                const double e = dF / bytes;
                if (e > best_e) {
                    best_e = e;
                    best = t;
                    best_split = split;
                    best_nq = nq;
                    best_nkv = nkv;
                    best_bytes = bytes;
                }
            }
            if (best_e < 0.0 || !(best_e > P.min_score)) break;
            Item it = items[best];
            const int32_t src = it.server;
            result->comm_bytes += best_bytes;
            if (!best_split) {
                const int64_t f = range_pairs(it.q0, it.q1);
                load[src] -= f;
                load[dst] += f;
                items[best].server = dst;
                ++result->n_migrations;
            } else {
                const int64_t a = best_nkv - best_nq, b = best_nkv;
                const int64_t moved = range_pairs(a, b);
                load[src] -= moved;
                load[dst] += moved;
                items[best].alive = false;
                if (a > it.q0) items.push_back(Item{it.doc, it.q0, a, src, it.home, true});
                items.push_back(Item{it.doc, a, b, dst, it.home, true});
                if (it.q1 > b) items.push_back(Item{it.doc, b, it.q1, src, it.home, true});
                ++result->n_splits;
            }
        }
    }

    // output: grouped by server, then (doc, q_start)
    std::vector<const Item *> live;
    for (const Item &it : items)
        if (it.alive) live.push_back(&it);
    std::sort(live.begin(), live.end(), [](const Item *a, const Item *b) {
        if (a->server != b->server) return a->server < b->server;
        if (a->doc != b->doc) return a->doc < b->doc;
        return a->q0 < b->q0;
    });
    result->n_tasks = static_cast<int64_t>(live.size());
    result->target_pairs_x1000 = static_cast<int64_t>(std::floor(target * 1000.0));
    result->max_load = *std::max_element(load.begin(), load.end());
    result->min_load = *std::min_element(load.begin(), load.end());
    if (!tasks_out || max_tasks < result->n_tasks)
        return fail(CA_ERR_INVALID_ARG, "ca_schedule: task buffer too small (" + std::to_string(result->n_tasks) +
                                            " needed)");
    for (size_t i = 0; i < live.size(); ++i) {
        const Item &it = *live[i];
        ca_sched_task_t &o = tasks_out[i];
        o.server = it.server;
        o.home = it.home;
        o.doc_id = it.doc;
        o.reserved = 0;
        o.q_start = it.q0;
        o.q_len = it.q1 - it.q0;
        o.kv_len = it.q1;
        o.pairs = range_pairs(it.q0, it.q1);
    }
    return CA_OK;
}

extern "C" ca_status_t ca_schedule(const int64_t *doc_len, int32_t n_docs, const ca_sched_params_t *params,
                                   ca_sched_task_t *tasks_out, int64_t max_tasks, ca_sched_result_t *result) {
    try {
        return schedule_impl(doc_len, n_docs, params, tasks_out, max_tasks, result);
    } catch (const std::bad_alloc &) {
        return ca::fail(CA_ERR_INVALID_ARG, "ca_schedule: host memory exhausted");
    }
}

static ca_status_t shard_2n_impl(const int64_t *doc_len, int32_t n_docs, int32_t n_ranks, ca_sched_task_t *tasks_out,
                                 int64_t max_tasks, int64_t *n_tasks_out) {
    using ca::fail;
    if (!doc_len || !n_tasks_out || n_docs < 1) return fail(CA_ERR_INVALID_ARG, "ca_shard_2n: NULL or empty input");
    if (n_ranks < 1) return fail(CA_ERR_INVALID_ARG, "ca_shard_2n: n_ranks must be >= 1");
    for (int32_t d = 0; d < n_docs; ++d)
        if (doc_len[d] < 1 || doc_len[d] > (int64_t(1) << 31))
            return fail(CA_ERR_INVALID_ARG, "ca_shard_2n: document " + std::to_string(d) + " has an invalid length");
    std::vector<ca_sched_task_t> out;
    const int64_t two_n = 2 * static_cast<int64_t>(n_ranks);
    for (int32_t r = 0; r < n_ranks; ++r)
        for (int32_t d = 0; d < n_docs; ++d) {
            const int64_t L = doc_len[d], c = (L + two_n - 1) / two_n;
            const int64_t chunks[2] = {r, two_n - 1 - r};
            for (int64_t j : chunks) {  // ascending q_start: j = r first, then 2N-1-r
                const int64_t a = j * c, b = std::min((j + 1) * c, L);
                if (a >= b) continue;
                ca_sched_task_t t{};
                t.server = r;
                t.home = r;
                t.doc_id = d;
                t.q_start = a;
                t.q_len = b - a;
                t.kv_len = b;
                t.pairs = range_pairs(a, b);
                out.push_back(t);
            }
        }
    *n_tasks_out = static_cast<int64_t>(out.size());
    if (!tasks_out || max_tasks < *n_tasks_out)
        return fail(CA_ERR_INVALID_ARG, "ca_shard_2n: task buffer too small (" + std::to_string(*n_tasks_out) + " needed)");
    std::copy(out.begin(), out.end(), tasks_out);
    return CA_OK;
}

extern "C" ca_status_t ca_shard_2n(const int64_t *doc_len, int32_t n_docs, int32_t n_ranks, ca_sched_task_t *tasks_out,
                                   int64_t max_tasks, int64_t *n_tasks_out) {
    try {
        return shard_2n_impl(doc_len, n_docs, n_ranks, tasks_out, max_tasks, n_tasks_out);
    } catch (const std::bad_alloc &) {
        return ca::fail(CA_ERR_INVALID_ARG, "ca_shard_2n: host memory exhausted");
    }
}
