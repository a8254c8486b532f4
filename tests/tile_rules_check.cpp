// Host-side check of the key-tile rules that the plan and the kernels share
// (document_masked_core_gb300/csrc/ca_internal.h) against brute-force
// enumeration of the visibility rule of include/ca.h (ca_task_t and
// ca_mask_t), on random tasks:
//   rows:     row_keys' two key intervals hold exactly the keys a row sees;
//   forward:  for every pair of query tiles (an item), key_tile_ranges gives
//             an increasing sequence of key tiles and visits_upto a prefix of
//             it for each tile; the prefix holds every key tile a row of the
//             tile sees and ends on the furthest one (0 when no row sees a key);
//   backward: key_tile_rows gives exactly the rows that see some key of the
//             key tile (they form one range), key_tile_query_tiles exactly the
//             query tiles holding such a row, key_pair_query_tiles a range
//             covering both tiles of a pair.
// Usage: tile_rules_check <n_tasks> <seed>; prints "ok ..." and exits 0, or
// prints the first failure and exits 1.
#include <cstdio>
#include <cstdlib>
#include <cstdint>
#include <random>
#include <vector>

#include "../document_masked_core_gb300/csrc/ca_internal.h"

using ca::DevTask;

static bool visible(const DevTask &t, int64_t p, int64_t j) {
    if (j < t.kv_start || j >= static_cast<int64_t>(t.kv_start) + t.kv_len || j > p) return false;
    if (t.sink == 0 && t.lo == 0 && t.win == 0) return true;
    if (j < t.sink) return true;
    return j >= t.lo && (t.win == 0 || j >= p - t.win + 1);
}

static int fail(const DevTask &t, int tpt, const char *what, long a, long b) {
    std::printf("FAIL %s (%ld vs %ld): q_start %d q_len %d kv_start %d kv_len %d doc_len %d sink %d lo %d win %d tpt %d\n",
                what, a, b, t.q_start, t.q_len, t.kv_start, t.kv_len, t.doc_len, t.sink, t.lo, t.win, tpt);
    return 1;
}

int main(int argc, char **argv) {
    const long n_tasks = argc > 1 ? std::atol(argv[1]) : 2000;
    std::mt19937_64 rng(argc > 2 ? std::strtoull(argv[2], nullptr, 10) : 1);
    auto uni = [&](int64_t lo, int64_t hi) {  // inclusive
        return static_cast<int32_t>(lo + static_cast<int64_t>(rng() % static_cast<uint64_t>(hi - lo + 1)));
    };
    long items = 0, key_tiles = 0;
    for (long n = 0; n < n_tasks; ++n) {
        DevTask t{};
        t.doc_len = uni(1, n % 4 == 0 ? 1500 : 500);
        const int32_t L = t.doc_len;
        t.q_start = uni(0, L - 1);
        t.q_len = uni(1, L - t.q_start);
        t.kv_start = rng() % 3 == 0 ? uni(0, L - 1) : 0;
        t.kv_len = rng() % 3 == 0 ? uni(1, L - t.kv_start) : L - t.kv_start;
        if (rng() % 2) {
            auto field = [&]() { return rng() % 3 == 0 ? 0 : uni(0, L); };
            t.sink = field();
            t.lo = field();
            t.win = field();
        }
        const int tpt = 1 << uni(0, 7);
        const int32_t q_end = t.q_start + t.q_len;  // one past the last row
        const int32_t n_keytiles = (L + 127) / 128;
        // brute force: bit jt of seen[p] is set when row p sees some key of key tile jt;
        // row_keys' two intervals [a, r1) U [r2, hi) hold exactly the keys row p sees
        std::vector<uint32_t> seen(L, 0);
        for (int32_t p = 0; p < L; ++p) {
            const ca::RowKeys k = ca::row_keys(t, p);
            for (int32_t j = 0; j < L; ++j) {
                const bool vis = visible(t, p, j);
                if (vis != (j >= k.a && (j < k.r1 || (j >= k.r2 && j < k.hi))))
                    return fail(t, 1, "row_keys intervals", p, j);
                if (vis) seen[p] |= 1u << (j / 128);
            }
        }
        auto furthest = [&](int32_t p0, int32_t p1) {  // furthest key tile rows [p0, p1] see, -1: none
            int32_t f = -1;
            for (int32_t p = p0; p <= p1; ++p)
                for (int32_t jt = n_keytiles - 1; jt > f; --jt)
                    if (seen[p] >> jt & 1u) {
                        f = jt;
                        break;
                    }
            return f;
        };
        auto sees_tile = [&](int32_t p0, int32_t p1, int32_t jt) {
            for (int32_t p = p0; p <= p1; ++p)
                if (seen[p] >> jt & 1u) return true;
            return false;
        };
        // forward items: query tiles (2i, 2i + 1)
        const int32_t ntiles = (t.q_len + tpt - 1) / tpt;
        for (int32_t tile = 0; tile < ntiles; tile += 2) {
            const int32_t p0 = t.q_start + tile * tpt;
            const int32_t end0 = (p0 + tpt < q_end ? p0 + tpt : q_end) - 1;
            const bool has_b = tile + 1 < ntiles;
            const int32_t end1 = has_b ? (p0 + 2 * tpt < q_end ? p0 + 2 * tpt : q_end) - 1 : end0;
            const ca::KeyTileRanges r = ca::key_tile_ranges(t, p0, end1);
            for (int32_t i = 1; i < r.count(); ++i)
                if (r.tile(i) <= r.tile(i - 1)) return fail(t, tpt, "key tile sequence not increasing", r.tile(i - 1), r.tile(i));
            const int32_t spans[2][2] = {{p0, end0}, {end0 + 1, end1}};
            for (int x = 0; x < (has_b ? 2 : 1); ++x) {
                const int32_t a = spans[x][0], b = spans[x][1];
                const int32_t nv = ca::visits_upto(r, t, a, b);
                const int32_t f = furthest(a, b);
                if (nv < 0 || nv > r.count()) return fail(t, tpt, "prefix longer than the sequence", nv, r.count());
                if ((f < 0) != (nv == 0)) return fail(t, tpt, "empty prefix iff no visible key", nv, f);
                if (nv > 0 && r.tile(nv - 1) != f) return fail(t, tpt, "prefix ends on the furthest key tile", r.tile(nv - 1), f);
                for (int32_t jt = 0; jt < n_keytiles; ++jt) {
                    if (!sees_tile(a, b, jt)) continue;
                    bool in = false;
                    for (int32_t i = 0; i < nv; ++i) in |= r.tile(i) == jt;
                    if (!in) return fail(t, tpt, "visible key tile missing from the prefix", jt, nv);
                }
                ++items;
            }
        }
        // backward: rows and query tiles of every key tile
        for (int32_t jt = 0; jt < n_keytiles; ++jt) {
            int32_t pmin, pmax;
            ca::key_tile_rows(t, jt * 128, &pmin, &pmax);
            int32_t bmin = INT32_MAX, bmax = -1;
            for (int32_t p = 0; p < L; ++p)
                if (sees_tile(p, p, jt)) {
                    if (p < bmin) bmin = p;
                    if (p > bmax) bmax = p;
                }
            for (int32_t p = bmin; bmax >= 0 && p <= bmax; ++p)
                if (!sees_tile(p, p, jt)) return fail(t, tpt, "rows seeing a key tile are not one range", jt, p);
            const int32_t cmax = pmax < L - 1 ? pmax : L - 1;
            if (bmax < 0 ? (pmin <= cmax) : (pmin != bmin || cmax != bmax))
                return fail(t, tpt, "key_tile_rows", static_cast<long>(pmin) * 100000 + cmax,
                            static_cast<long>(bmin) * 100000 + bmax);
            int32_t first, count;
            ca::key_tile_query_tiles(t, jt, tpt, &first, &count);
            for (int32_t qt = 0; qt < ntiles; ++qt) {
                const int32_t a = t.q_start + qt * tpt, b = (a + tpt < q_end ? a + tpt : q_end) - 1;
                const bool want = sees_tile(a, b, jt), got = qt >= first && qt < first + count;
                if (want != got) return fail(t, tpt, "key_tile_query_tiles", qt, want);
            }
            if (jt % 2 == 0) {
                int32_t pf, pc;
                ca::key_pair_query_tiles(t, jt / 2, tpt, &pf, &pc);
                for (int32_t qt = 0; qt < ntiles; ++qt) {
                    const int32_t a = t.q_start + qt * tpt, b = (a + tpt < q_end ? a + tpt : q_end) - 1;
                    const bool want = sees_tile(a, b, jt) || (jt + 1 < n_keytiles && sees_tile(a, b, jt + 1));
                    if (want && !(qt >= pf && qt < pf + pc)) return fail(t, tpt, "key_pair_query_tiles misses a tile", qt, jt);
                }
            }
            ++key_tiles;
        }
    }
    std::printf("ok %ld tasks, %ld query tiles, %ld key tiles\n", n_tasks, items, key_tiles);
    return 0;
}
