// ra_stats.cpp -- host-only analysis of the ring plans (no GPU): what the
// tensor-core passes visit for a packing, for the planner's coverage tests
// and for reports.  Uses the planner and the tile classifier the drivers
// and kernels use.
#include <algorithm>
#include <cstdint>
#include <functional>
#include <queue>
#include <vector>

#include "ra_internal.h"
#include "ra_kernels.h"

using namespace ra;

// Walks each tensor-core pass's work items over their ring-step ranges the
// way the kernels do (forward and dQ: rank r at step t reads the key tiles
// of rank (r - t) mod cp; dK/dV: the key tile of rank s meets the query
// tiles of rank (s + t) mod cp) and counts what they visit.  key_lo /
// key_hi: an interval mask (then causal and window are not used).
static ra_status plan_stats_impl(const int32_t *cu, int B, int cp, int mode, int G, int Hkv, int causal, int window,
                                 int sched, int exact, int n_sm, int64_t *stats, const int32_t *key_lo,
                                 const int32_t *key_hi) {
    if (!stats) return fail(RA_ERR_INVALID_ARG, "stats is NULL");
    if (n_sm < 1) return fail(RA_ERR_INVALID_ARG, "n_sm must be >= 1");
    if (cp < 1 || cp > kMaxMergeParts) return fail(RA_ERR_INVALID_ARG, "cp must be in [1, 64]");
    if (mode != RA_ZZ_GLOBAL && mode != RA_ZZ_PER_DOC) return fail(RA_ERR_INVALID_ARG, "unknown zigzag mode");
    if (sched != RA_SCHED_FUSED && sched != RA_SCHED_STEPWISE && sched != RA_SCHED_ALLGATHER)
        return fail(RA_ERR_INVALID_ARG, "unknown schedule");
    if (G < 1 || G > kBM || (G & (G - 1)) || Hkv < 1) return fail(RA_ERR_INVALID_ARG, "bad head grouping");
    ra_status st = validate_cu(cu, B, -1);
    if (st) return st;
    const int64_t T = cu[B];
    if (window >= T) window = -1;
    if (window < -1) window = -1;
    if (key_lo || key_hi) {
        causal = 0;
        window = -1;
    }
    auto plan = get_ring_plan(cu, B, cp, mode, G, Hkv, causal ? 1 : 0, window, true,
                              sched == RA_SCHED_ALLGATHER, &st, key_lo, key_hi);
    if (!plan) return st;
    const TilePlan &tp = plan->tiles;
    for (int i = 0; i < RA_PLAN_STATS_N; ++i) stats[i] = 0;
    stats[0] = (int64_t)tp.qtiles.size();
    stats[1] = (int64_t)tp.kvtiles.size();
    stats[2] = (int64_t)tp.items.size();
    stats[3] = (int64_t)tp.bitems.size();
    stats[4] = (int64_t)tp.qitems.size();
    const uint8_t *blob = plan->dev.blob.data();
    for (int64_t i = 0; i < T; ++i) {
        stats[7] += blob[plan->dev.o_qmask + i];
        stats[8] += blob[plan->dev.o_kvmask + i];
    }
    auto pos_of = [](const Tile &t, int i) { return i < t.split ? (int64_t)t.pos0 + i : (int64_t)t.pos1 + (i - t.split); };
    // allowed (query token, key) pairs of one tile pair; `bad` counts the
    // disallowed ones among the valid rows and keys
    auto count = [&](const Tile &q, const Tile &k, int64_t *bad) {
        int64_t ok = 0;
        for (int i = 0; i < q.len; ++i) {
            const int64_t qp = pos_of(q, i);
            for (int j = 0; j < k.len; ++j) {
                const int64_t kp = pos_of(k, j);
                const bool allowed = key_lo ? (kp >= key_lo[qp] && kp <= key_hi[qp])
                                            : (!causal || kp <= qp) && (window < 0 || kp >= qp - window);
                if (allowed)
                    ++ok;
                else if (bad)
                    ++*bad;
            }
        }
        return ok;
    };
    const int q_tokens = tp.q_tokens;
    auto seg = [&](int r, int b) { return (size_t)r * (B + 1) + b; };
    // visited tile pairs of each item (its cost in the scheduling model);
    // the coverage counts come from the items of KV head 0 (the others repeat
    // them for their own head)
    std::vector<int64_t> c_fwd, c_kv, c_q;
    c_fwd.reserve(tp.items.size());
    for (const WorkItem &w : tp.items) {
        int64_t n = 0;
        for (int t = w.t0; t < w.t1; ++t) {
            const int s = ((w.r - t) % cp + cp) % cp;
            for (int j = tp.kv_off[seg(s, w.b)]; j < tp.kv_off[seg(s, w.b) + 1]; ++j) {
                if (w.g == 0 && (tp.pair_class(w.qt0, j, causal, window) != kSkip ||
                                 (w.qt1 >= 0 && tp.pair_class(w.qt1, j, causal, window) != kSkip)))
                    ++stats[19];
                for (int qt : {w.qt0, w.qt1}) {
                    if (qt < 0) continue;
                    const int c = tp.pair_class(qt, j, causal, window);
                    if (c == kSkip) continue;
                    ++n;
                    if (w.g != 0) continue;
                    ++stats[5];
                    stats[9] += (int64_t)q_tokens * kBN;
                    if (c == kFull) ++stats[6];
                    if (exact) stats[10] += count(tp.qtiles[qt], tp.kvtiles[j], c == kFull ? &stats[11] : nullptr);
                }
            }
        }
        c_fwd.push_back(n);
    }
    c_kv.reserve(tp.bitems.size());
    for (const WorkItem &w : tp.bitems) {
        int64_t n = 0;
        for (int t = w.t0; t < w.t1; ++t) {
            const int r = (w.r + t) % cp;
            for (int i = tp.q_off[seg(r, w.b)]; i < tp.q_off[seg(r, w.b) + 1]; ++i) {
                if (tp.pair_class(i, w.qt0, causal, window) == kSkip) continue;
                ++n;
                if (w.g != 0) continue;
                ++stats[14];
                if (exact) stats[12] += count(tp.qtiles[i], tp.kvtiles[w.qt0], nullptr);
            }
        }
        c_kv.push_back(n);
    }
    c_q.reserve(tp.qitems.size());
    for (const WorkItem &w : tp.qitems) {
        int64_t n = 0;
        for (int t = w.t0; t < w.t1; ++t) {
            const int s = ((w.r - t) % cp + cp) % cp;
            for (int j = tp.kv_off[seg(s, w.b)]; j < tp.kv_off[seg(s, w.b) + 1]; ++j) {
                if (tp.pair_class(w.qt0, j, causal, window) == kSkip) continue;
                ++n;
                if (w.g != 0) continue;
                ++stats[15];
                if (exact) stats[13] += count(tp.qtiles[w.qt0], tp.kvtiles[j], nullptr);
            }
        }
        c_q.push_back(n);
    }
    if (!exact) stats[10] = stats[11] = stats[12] = stats[13] = -1;
    // Scheduling model, in tile visits: the forward's persistent CTAs claim
    // items in list order from a counter, and the key-side grid (one CTA per
    // item) is dispatched in block order as SMs free up -- both greedy list
    // scheduling over n_sm workers; the dQ grid takes items with a static
    // stride (CTA c runs items c, c + n_sm, ...).
    auto greedy = [n_sm](const std::vector<int64_t> &cost) {
        std::priority_queue<int64_t, std::vector<int64_t>, std::greater<int64_t>> free_at;
        for (int i = 0; i < n_sm; ++i) free_at.push(0);
        int64_t end = 0;
        for (int64_t c : cost) {
            const int64_t t = free_at.top() + c;
            free_at.pop();
            free_at.push(t);
            end = std::max(end, t);
        }
        return end;
    };
    auto strided = [n_sm](const std::vector<int64_t> &cost) {
        std::vector<int64_t> load((size_t)n_sm, 0);
        for (size_t i = 0; i < cost.size(); ++i) load[i % (size_t)n_sm] += cost[i];
        return load.empty() ? (int64_t)0 : *std::max_element(load.begin(), load.end());
    };
    stats[16] = greedy(c_fwd);
    stats[17] = greedy(c_kv);
    stats[18] = strided(c_q);
    return RA_OK;
}

extern "C" {

ra_status ra_ring_plan_stats(const int32_t *cu, int B, int cp, int mode, int G, int Hkv, int causal, int window,
                             int sched, int exact, int n_sm, int64_t *stats) {
    return plan_stats_impl(cu, B, cp, mode, G, Hkv, causal, window, sched, exact, n_sm, stats, nullptr, nullptr);
}

ra_status ra_ring_plan_stats_masked(const int32_t *cu, int B, int cp, int mode, int G, int Hkv,
                                    const int32_t *key_lo, const int32_t *key_hi, int sched, int exact, int n_sm,
                                    int64_t *stats) {
    if (!key_lo || !key_hi) return fail(RA_ERR_INVALID_ARG, "key_lo / key_hi is NULL");
    if (sched == RA_SCHED_STEPWISE) return fail(RA_ERR_UNSUPPORTED, "interval masks run in the fused and all-gather schedules");
    return plan_stats_impl(cu, B, cp, mode, G, Hkv, 0, -1, sched, exact, n_sm, stats, key_lo, key_hi);
}

}  // extern "C"
