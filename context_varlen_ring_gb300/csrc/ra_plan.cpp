// ra_plan.cpp -- host planner: zigzag plan, tile tables, work lists.
//
// Zigzag ("Zigzag attention support?", ring-attention-pytorch #20, the
// extract_local snippet; maxtext PR #1133, review comment on reordering):
// a stream of L tokens is cut into n = 2*cp chunks and rank r keeps chunks
// r and n-1-r.  Here the chunk bounds are floor(c*L/n), which is the same
// split as chunking into equal pieces when n divides L and stays defined
// when it does not.  Per-document mode applies the rule to each document
// ("Question about varlen ring attention", MiniMax-01 #6, on zigzag under
// packing).
//
// The planner works on ranges: rank r's part of a stream is two ranges of
// consecutive tokens, appended in increasing order.
#include <algorithm>
#include <cstring>
#include <map>
#include <mutex>

#include "ra_internal.h"

namespace ra {

ra_status validate_cu(const int32_t *cu, int B, int64_t T) {
    if (!cu) return fail(RA_ERR_INVALID_ARG, "cu_seqlens is NULL");
    if (B < 1) return fail(RA_ERR_INVALID_ARG, "B must be >= 1");
    if (cu[0] != 0) return fail(RA_ERR_INVALID_ARG, "cu_seqlens[0] != 0");
    for (int b = 0; b < B; ++b)
        if (cu[b + 1] < cu[b]) return fail(RA_ERR_INVALID_ARG, "cu_seqlens not non-decreasing at " + std::to_string(b));
    if (T >= 0 && (int64_t)cu[B] != T)
        return fail(RA_ERR_INVALID_ARG, "cu_seqlens[B] != T");
    return RA_OK;
}

static inline int64_t bound(int64_t c, int64_t L, int64_t n) { return c * L / n; }

ra_status build_zigzag(const int32_t *cu, int B, int cp, int mode, ZigzagPlan &zp) {
    ra_status st = validate_cu(cu, B, -1);
    if (st) return st;
    if (cp < 1 || cp > 4096) return fail(RA_ERR_INVALID_ARG, "cp must be in [1, 4096]");
    if (mode != RA_ZZ_GLOBAL && mode != RA_ZZ_PER_DOC) return fail(RA_ERR_INVALID_ARG, "unknown zigzag mode");
    const int64_t T = cu[B];
    const int64_t n = 2 * (int64_t)cp;
    zp.T = T;
    zp.B = B;
    zp.cp = cp;
    zp.mode = mode;
    zp.cu.assign(cu, cu + B + 1);
    zp.perm.resize((size_t)T);
    zp.off.assign((size_t)cp + 1, 0);
    zp.cu_local.assign((size_t)cp * (B + 1), 0);
    int64_t p = 0;
    for (int r = 0; r < cp; ++r) {
        zp.off[r] = (int32_t)p;
        int32_t *cl = zp.cu_local.data() + (size_t)r * (B + 1);
        // the two ranges of rank r, per stream
        auto emit = [&](int64_t a, int64_t e) {
            for (int64_t i = a; i < e; ++i) zp.perm[(size_t)p++] = (int32_t)i;
        };
        if (mode == RA_ZZ_GLOBAL) {
            const int64_t a0 = bound(r, T, n), e0 = bound(r + 1, T, n);
            const int64_t a1 = bound(n - 1 - r, T, n), e1 = bound(n - r, T, n);
            emit(a0, e0);
            emit(a1, e1);
            // local documents: intersect each document with the two ranges
            for (int b = 0; b < B; ++b) {
                auto inter = [&](int64_t a, int64_t e) {
                    int64_t lo = std::max<int64_t>(a, cu[b]), hi = std::min<int64_t>(e, cu[b + 1]);
                    return hi > lo ? hi - lo : 0;
                };
                cl[b + 1] = cl[b] + (int32_t)(inter(a0, e0) + inter(a1, e1));
            }
        } else {
            for (int b = 0; b < B; ++b) {
                const int64_t L = (int64_t)cu[b + 1] - cu[b], base = cu[b];
                const int64_t a0 = base + bound(r, L, n), e0 = base + bound(r + 1, L, n);
                const int64_t a1 = base + bound(n - 1 - r, L, n), e1 = base + bound(n - r, L, n);
                emit(a0, e0);
                emit(a1, e1);
                cl[b + 1] = cl[b] + (int32_t)((e0 - a0) + (e1 - a1));
            }
        }
    }
    zp.off[cp] = (int32_t)p;
    if (p != T) return fail(RA_ERR_INVALID_ARG, "internal: zigzag plan does not cover all tokens");
    return RA_OK;
}

void append_tiles(std::vector<Tile> &out, const int32_t *pos, int64_t lo, int64_t hi, int tile_rows, int seg,
                  int max_runs) {
    int64_t i = lo;
    while (i < hi) {
        const int64_t start = i;
        const int32_t p0 = pos ? pos[i] : (int32_t)i;
        auto P = [&](int64_t x) { return pos ? pos[x] : (int32_t)x; };
        ++i;
        while (i < hi && i - start < tile_rows && P(i) == P(i - 1) + 1) ++i;
        const int32_t split = (int32_t)(i - start);
        int32_t p1 = p0 + split;
        bool two = false;
        if (max_runs > 1 && i < hi && i - start < tile_rows) {
            p1 = P(i);
            two = true;
            ++i;
            while (i < hi && i - start < tile_rows && P(i) == P(i - 1) + 1) ++i;
        }
        const int32_t len = (int32_t)(i - start);
        Tile t;
        t.row0 = (int32_t)start;
        t.len = len;
        t.split = split;
        t.pos0 = p0;
        t.pos1 = p1;
        t.pmin = two ? std::min(p0, p1) : p0;
        t.pmax = two ? std::max(p0 + split - 1, p1 + (len - split) - 1) : p0 + len - 1;
        t.seg = seg;
        out.push_back(t);
    }
}

// Forward items: pairs of query tiles of one document, replicated over KV
// heads; backward items: one per KV tile and KV head.
//
// A forward item walks the union of its two query tiles' KV tiles, and a
// KV tile that only one of them needs costs the item about as much time as
// one that both need (the kernel's loop is set by the latency of each query
// tile's S -> softmax -> PV chain, and the two tiles cover each other's
// softmax only when both have products).  So the query tiles of a document
// are paired in order of their visit counts, from the most visits down,
// across the simulated ranks: tiles with the same KV needs share items, and
// when the count is odd the tile left alone is the one with the fewest
// visits.  An item walks the ring steps of its first tile's rank; the
// second tile, possibly of another rank, meets its own KV tiles in that
// order (the same tiles: each rank's steps run over every rank's shard),
// which changes its result only in the order of the online softmax's
// floating-point accumulation.
static void build_items(TilePlan &tp, int Hkv, int causal, int window) {
    const int cp = tp.cp, B = tp.B;
    tp.items.clear();
    tp.bitems.clear();
    tp.qitems.clear();
    tp.fwd_tile_pairs = 0;
    auto seg_idx = [&](int r, int b) { return r * (B + 1) + b; };
    const bool bounds = !tp.qbounds.empty();
    // vis[qi * cp + s]: the KV tiles of rank s's share of query tile qi's
    // document that qi visits
    std::vector<int32_t> vis(tp.qtiles.size() * (size_t)cp, 0);
    for (int b = 0; b < B; ++b)
        for (int r = 0; r < cp; ++r) {
            const int qa = tp.q_off[seg_idx(r, b)], qe = tp.q_off[seg_idx(r, b) + 1];
            for (int s = 0; s < cp && qe > qa; ++s) {
                const int ka = tp.kv_off[seg_idx(s, b)], ke = tp.kv_off[seg_idx(s, b) + 1];
                kv_tiles_visited_each(tp.qtiles.data() + qa, bounds ? tp.qbounds.data() + qa : nullptr, qe - qa,
                                      tp.kvtiles.data() + ka, ke - ka, causal, window, vis.data() + (size_t)qa * cp + s,
                                      cp);
            }
        }
    auto kv_visits = [&](int qi, int s) -> int64_t { return vis[(size_t)qi * cp + s]; };
    // visited KV tiles of query tile qi over the ring steps, and the step
    // range [tf, tl) that holds them
    auto q_visits = [&](int qi, int r, int *tf, int *tl) {
        int64_t c = 0;
        *tf = cp;
        *tl = 0;
        for (int t = 0; t < cp; ++t) {
            const int s = ((r - t) % cp + cp) % cp;
            const int64_t c_t = kv_visits(qi, s);
            if (c_t) {
                *tf = std::min(*tf, t);
                *tl = t + 1;
            }
            c += c_t;
        }
        if (*tf > *tl) *tf = *tl = 0;
        return c;
    };
    struct QEntry {
        int qi, r;
        int64_t cnt;
    };
    std::vector<QEntry> qs;
    // One record per tile or tile pair (KV head 0); each pass's item list is
    // its records sorted and then repeated for every KV head (no cost
    // depends on the head).
    std::vector<WorkItem> fwd1, dq1, kv1;
    fwd1.reserve((tp.qtiles.size() + (size_t)B) / 2 + 1);
    dq1.reserve(tp.qtiles.size());
    kv1.reserve(tp.kvtiles.size());
    for (int b = 0; b < B; ++b) {
        // the query tiles of document b on every rank, with their visits
        qs.clear();
        for (int r = 0; r < cp; ++r) {
            for (int qi = tp.q_off[seg_idx(r, b)]; qi < tp.q_off[seg_idx(r, b) + 1]; ++qi) {
                int tf, tl;
                const int64_t c = q_visits(qi, r, &tf, &tl);
                qs.push_back(QEntry{qi, r, c});
                // per-query-tile items of the dQ pass (the tile's own ring order)
                dq1.push_back(WorkItem{qi, -1, 0, r, b, tf, tl, (int32_t)std::min<int64_t>(c, INT32_MAX)});
            }
        }
        // Forward items pair the document's query tiles in order of their
        // visits, from the most down, across ranks: the item walks the KV
        // tiles in the ring order of its first tile's rank (every rank's
        // shards, so the second tile meets all of its own as well), and two
        // tiles with the same visits share (nearly) every KV step.
        std::stable_sort(qs.begin(), qs.end(), [&](const QEntry &x, const QEntry &y) {
            if (x.cnt != y.cnt) return x.cnt > y.cnt;
            return tp.qtiles[x.qi].pmax > tp.qtiles[y.qi].pmax;
        });
        const int n = (int)qs.size();
        for (int j = 0; j < n; j += 2) {
            const QEntry &x = qs[(size_t)j];
            const int q1 = j + 1 < n ? qs[(size_t)j + 1].qi : -1;
            const int r = x.r, i = x.qi;
            // the steps [tf, tl) of rank r's ring order that hold a KV tile
            // either query tile visits; the cost is their visits
            int64_t cost = 0;
            int tf = cp, tl = 0;
            for (int t = 0; t < cp; ++t) {
                const int sr = ((r - t) % cp + cp) % cp;
                const int64_t c_t = kv_visits(i, sr) + (q1 >= 0 ? kv_visits(q1, sr) : 0);
                if (c_t) {
                    tf = std::min(tf, t);
                    tl = t + 1;
                }
                cost += c_t;
            }
            if (tf >= tl) tf = tl = 0;
            fwd1.push_back(WorkItem{i, q1, 0, r, b, tf, tl, (int32_t)std::min<int64_t>(cost, INT32_MAX)});
            tp.fwd_tile_pairs += cost * Hkv;
        }
    }
    for (int s = 0; s < cp; ++s) {
        for (int b = 0; b < B; ++b) {
            const int ka = tp.kv_off[seg_idx(s, b)], ke = tp.kv_off[seg_idx(s, b) + 1];
            for (int j = ka; j < ke; ++j) {
                int64_t cost = 0;
                int tf = cp, tl = 0;
                for (int t = 0; t < cp; ++t) {
                    const int r = (s + t) % cp;
                    const int qa = tp.q_off[seg_idx(r, b)], qe = tp.q_off[seg_idx(r, b) + 1];
                    const int64_t c_t = q_tiles_visiting(tp.qtiles.data() + qa, bounds ? tp.qbounds.data() + qa : nullptr,
                                                         qe - qa, tp.kvtiles[(size_t)j], causal, window);
                    if (c_t) {
                        tf = std::min(tf, t);
                        tl = t + 1;
                    }
                    cost += c_t;
                }
                if (tf > tl) tf = tl = 0;
                kv1.push_back(WorkItem{j, -1, 0, s, b, tf, tl, (int32_t)std::min<int64_t>(cost, INT32_MAX)});
            }
        }
    }
    // KV head major, then longest-processing-time first within a head: the
    // CTAs resident at any moment read the K/V of one or two heads (tens of
    // MB), which stays in L2, and the launch ends on short items.
    auto per_head = [&](std::vector<WorkItem> &one, std::vector<WorkItem> &all) {
        std::stable_sort(one.begin(), one.end(), [](const WorkItem &a, const WorkItem &b) { return a.cost > b.cost; });
        all.reserve(one.size() * (size_t)Hkv);
        for (int g = 0; g < Hkv; ++g)
            for (WorkItem w : one) {
                w.g = g;
                all.push_back(w);
            }
    };
    per_head(fwd1, tp.items);
    per_head(dq1, tp.qitems);
    // Key-side items: document major (heaviest document first), then KV
    // head, then longest first.  A long document's first KV tile sees every
    // query tile of the document, more work than one head's share of an SM,
    // so under the head-major order the last head's heaviest items start
    // late and leave the other SMs idle at the end; here they start in the
    // first waves and the launch ends on the shortest documents.  The CTAs
    // resident at once read the Q and dO of one or two (document, head)
    // pairs, a smaller set than one head of every document.
    std::vector<int32_t> doc_max(B, 0);
    for (const WorkItem &w : kv1) doc_max[w.b] = std::max(doc_max[w.b], w.cost);
    std::stable_sort(kv1.begin(), kv1.end(), [&](const WorkItem &a, const WorkItem &b) {
        if (doc_max[a.b] != doc_max[b.b]) return doc_max[a.b] > doc_max[b.b];
        if (a.b != b.b) return a.b < b.b;
        return a.cost > b.cost;
    });
    tp.bitems.reserve(kv1.size() * (size_t)Hkv);
    for (size_t a = 0; a < kv1.size();) {
        size_t e = a;
        while (e < kv1.size() && kv1[e].b == kv1[a].b) ++e;
        for (int g = 0; g < Hkv; ++g)
            for (size_t i = a; i < e; ++i) {
                WorkItem w = kv1[i];
                w.g = g;
                tp.bitems.push_back(w);
            }
        a = e;
    }
}

ra_status build_ring_tiles(const ZigzagPlan &zp, int G, int Hkv, int causal, int window, bool allgather,
                           TilePlan &tp, const int32_t *key_lo, const int32_t *key_hi, int kv_runs) {
    if (G < 1 || kBM % G != 0) return fail(RA_ERR_UNSUPPORTED, "GQA group must divide 128");
    if ((key_lo == nullptr) != (key_hi == nullptr)) return fail(RA_ERR_INVALID_ARG, "key_lo and key_hi go together");
    if (key_lo) {
        // the key-side backward inverts each row's interval with a binary
        // search, which needs bounds that never decrease inside a document
        for (int b = 0; b < zp.B; ++b)
            for (int64_t i = (int64_t)zp.cu[b] + 1; i < zp.cu[b + 1]; ++i)
                if (key_lo[i] < key_lo[i - 1] || key_hi[i] < key_hi[i - 1])
                    return fail(RA_ERR_INVALID_ARG, "key_lo and key_hi must be non-decreasing inside each document "
                                                    "(token " + std::to_string(i) + ")");
    }
    tp = TilePlan();
    tp.cp = zp.cp;
    tp.B = zp.B;
    tp.q_tokens = kBM / G;
    const int B = zp.B;
    tp.q_off.assign((size_t)zp.cp * (B + 1) + 1, 0);
    tp.kv_off.assign((size_t)zp.cp * (B + 1) + 1, 0);
    auto seg_rows = [&](int r, int b, int64_t *lo, int64_t *hi) {
        const size_t idx = (size_t)r * (B + 1) + b;
        *lo = zp.off[r] + zp.cu_local[idx];
        *hi = zp.off[r] + zp.cu_local[idx + 1];
    };
    for (int r = 0; r < zp.cp; ++r) {
        for (int b = 0; b <= B; ++b) {
            tp.q_off[(size_t)r * (B + 1) + b] = (int32_t)tp.qtiles.size();
            if (b == B) break;
            int64_t lo, hi;
            seg_rows(r, b, &lo, &hi);
            append_tiles(tp.qtiles, zp.perm.data(), lo, hi, tp.q_tokens, b);
        }
    }
    tp.q_off.back() = (int32_t)tp.qtiles.size();
    if (key_lo) {
        const int64_t T = (int64_t)zp.perm.size();
        tp.key_lo.assign(key_lo, key_lo + T);
        tp.key_hi.assign(key_hi, key_hi + T);
        tp.qbounds.resize(tp.qtiles.size());
        for (size_t i = 0; i < tp.qtiles.size(); ++i) {
            const Tile &t = tp.qtiles[i];
            QBounds qb{INT32_MAX, INT32_MIN, INT32_MAX, INT32_MIN};
            for (int c = 0; c < t.len; ++c) {
                const int64_t pos = c < t.split ? (int64_t)t.pos0 + c : (int64_t)t.pos1 + (c - t.split);
                qb.lo_min = std::min(qb.lo_min, key_lo[pos]);
                qb.lo_max = std::max(qb.lo_max, key_lo[pos]);
                qb.hi_min = std::min(qb.hi_min, key_hi[pos]);
                qb.hi_max = std::max(qb.hi_max, key_hi[pos]);
            }
            tp.qbounds[i] = qb;
        }
    }
    // KV tiles.  A ring KV tile may join the tail of a rank's early zigzag
    // chunk and the head of its late one.  Under the causal mask that saves
    // visits (one tile instead of two short ones once both runs are needed);
    // under a sliding window or an interval mask the two runs, far apart,
    // are often not both needed, and tiles of one run are visited less.  So
    // each rank's KV tiles of a segment are built both ways and the way with
    // fewer forward visits (tile pairs with any allowed pair, over every
    // query tile of the segment's document) is kept (kv_runs = 1 or 2 forces
    // one way).
    std::vector<Tile> cand[2];
    for (int r = 0; r < zp.cp; ++r) {
        for (int b = 0; b <= B; ++b) {
            tp.kv_off[(size_t)r * (B + 1) + b] = (int32_t)tp.kvtiles.size();
            if (b == B) break;
            if (allgather) {
                if (r == 0)  // the whole document, original rows = positions
                    append_tiles(tp.kvtiles, nullptr, zp.cu[b], zp.cu[b + 1], kBN, b);
                continue;
            }
            int64_t lo, hi;
            seg_rows(r, b, &lo, &hi);
            int runs = kv_runs == 1 ? 1 : 2;
            if (kv_runs == 0) {
                int64_t vis[2] = {0, 0};
                for (int w = 0; w < 2; ++w) {
                    cand[w].clear();
                    append_tiles(cand[w], zp.perm.data(), lo, hi, kBN, b, w + 1);
                }
                // (the same number of tiles can still cut the runs differently)
                for (int w = 0; w < 2; ++w)
                    for (int rq = 0; rq < zp.cp; ++rq) {
                        const size_t qi = (size_t)rq * (B + 1) + b;
                        const int qa = tp.q_off[qi], qe = tp.q_off[qi + 1];
                        vis[w] += kv_tiles_visited_each(tp.qtiles.data() + qa,
                                                        tp.qbounds.empty() ? nullptr : tp.qbounds.data() + qa, qe - qa,
                                                        cand[w].data(), (int)cand[w].size(), causal, window, nullptr, 1);
                    }
                if (vis[0] < vis[1]) runs = 1;
            }
            append_tiles(tp.kvtiles, zp.perm.data(), lo, hi, kBN, b, runs);
        }
    }
    tp.kv_off.back() = (int32_t)tp.kvtiles.size();
    build_items(tp, Hkv, causal, window);
    return RA_OK;
}

ra_status build_partial_tiles(const int32_t *cu_q, const int32_t *cu_k, int nseg,
                              const int32_t *q_pos, const int32_t *k_pos, int64_t Tq, int64_t Tk,
                              int G, int Hkv, int causal, int window, TilePlan &tp) {
    if (G < 1 || kBM % G != 0) return fail(RA_ERR_UNSUPPORTED, "GQA group must divide 128");
    ra_status st = validate_cu(cu_q, nseg, Tq);
    if (st) return st;
    st = validate_cu(cu_k, nseg, Tk);
    if (st) return st;
    tp = TilePlan();
    tp.cp = 1;
    tp.B = nseg;
    tp.q_tokens = kBM / G;
    tp.q_off.assign((size_t)nseg + 2, 0);
    tp.kv_off.assign((size_t)nseg + 2, 0);
    for (int b = 0; b <= nseg; ++b) {
        tp.q_off[b] = (int32_t)tp.qtiles.size();
        tp.kv_off[b] = (int32_t)tp.kvtiles.size();
        if (b == nseg) break;
        append_tiles(tp.qtiles, q_pos, cu_q[b], cu_q[b + 1], tp.q_tokens, b);
        append_tiles(tp.kvtiles, k_pos, cu_k[b], cu_k[b + 1], kBN, b);
    }
    tp.q_off.back() = (int32_t)tp.qtiles.size();
    tp.kv_off.back() = (int32_t)tp.kvtiles.size();
    build_items(tp, Hkv, causal, window);
    return RA_OK;
}

size_t layout_tables(const TableCounts &n, DeviceTables &dt) {
    size_t o = 0;
    auto take = [&](size_t bytes) {
        size_t at = o;
        o = align_up(o + bytes, 256);
        return at;
    };
    dt.o_perm = take(n.T * 4);
    dt.o_qt = take(n.qt * sizeof(Tile));
    dt.o_kt = take(n.kt * sizeof(Tile));
    dt.o_qoff = take(n.qoff * 4);
    dt.o_kvoff = take(n.kvoff * 4);
    dt.o_items = take(n.items * sizeof(WorkItem));
    dt.o_bitems = take(n.bitems * sizeof(WorkItem));
    dt.o_qitems = take(n.qitems * sizeof(WorkItem));
    dt.o_cul = take(n.cul * 4);
    dt.o_off = take(n.off * 4);
    dt.o_sched = take(64);
    dt.o_qmask = take(n.tiles ? n.T : 0);
    dt.o_kvmask = take(n.tiles ? n.T : 0);
    dt.bounds = n.qb > 0;
    dt.o_qb = take(n.qb * sizeof(QBounds));
    dt.o_klo = take(n.klo * 4);
    dt.o_khi = take(n.khi * 4);
    return o;
}

void pack_tables(const ZigzagPlan *zp, const TilePlan *tp, DeviceTables &dt) {
    TableCounts n;
    if (zp) {
        n.T = zp->perm.size();
        n.cul = zp->cu_local.size();
        n.off = zp->off.size();
    }
    if (tp) {
        n.tiles = zp != nullptr;
        n.qt = tp->qtiles.size();
        n.kt = tp->kvtiles.size();
        n.qoff = tp->q_off.size();
        n.kvoff = tp->kv_off.size();
        n.items = tp->items.size();
        n.bitems = tp->bitems.size();
        n.qitems = tp->qitems.size();
        if (!tp->qbounds.empty()) {
            n.qb = tp->qbounds.size();
            n.klo = tp->key_lo.size();
            n.khi = tp->key_hi.size();
        }
    }
    dt.blob.assign(layout_tables(n, dt), 0);
    auto put = [&](size_t at, const void *src, size_t bytes) {
        if (bytes) std::memcpy(dt.blob.data() + at, src, bytes);
    };
    if (zp) {
        put(dt.o_perm, zp->perm.data(), zp->perm.size() * 4);
        put(dt.o_cul, zp->cu_local.data(), zp->cu_local.size() * 4);
        put(dt.o_off, zp->off.data(), zp->off.size() * 4);
    }
    if (tp) {
        put(dt.o_qt, tp->qtiles.data(), tp->qtiles.size() * sizeof(Tile));
        put(dt.o_kt, tp->kvtiles.data(), tp->kvtiles.size() * sizeof(Tile));
        put(dt.o_qoff, tp->q_off.data(), tp->q_off.size() * 4);
        put(dt.o_kvoff, tp->kv_off.data(), tp->kv_off.size() * 4);
        put(dt.o_items, tp->items.data(), tp->items.size() * sizeof(WorkItem));
        put(dt.o_bitems, tp->bitems.data(), tp->bitems.size() * sizeof(WorkItem));
        put(dt.o_qitems, tp->qitems.data(), tp->qitems.size() * sizeof(WorkItem));
        if (dt.bounds) {
            put(dt.o_qb, tp->qbounds.data(), tp->qbounds.size() * sizeof(QBounds));
            put(dt.o_klo, tp->key_lo.data(), tp->key_lo.size() * 4);
            put(dt.o_khi, tp->key_hi.data(), tp->key_hi.size() * 4);
        }
        dt.n_items = (int)tp->items.size();
        dt.n_bitems = (int)tp->bitems.size();
        dt.n_qitems = (int)tp->qitems.size();
    }
    if (zp && tp) {
        // the whole box a kernel copies for a two-run tile (q_tokens rows,
        // padding included), so that its padding rows hold finite values
        // like every other row a tile reads (the key-side backward sums
        // over a tile's padded rows with zero weight)
        const int64_t T = (int64_t)zp->perm.size();
        auto mark = [&](size_t at, const std::vector<Tile> &tiles, int box) {
            uint8_t *mask = dt.blob.data() + at;
            for (const Tile &t : tiles)
                if (t.split < t.len)
                    for (int64_t i = t.row0; i < (int64_t)t.row0 + box && i < T; ++i) mask[i] = 1;
        };
        mark(dt.o_qmask, tp->qtiles, tp->q_tokens);
        mark(dt.o_kvmask, tp->kvtiles, kBN);
    }
}

ra_status ring_tables_bound(const int32_t *cu, int B, int cp, int mode, int G, int Hkv, bool want_tiles,
                            bool allgather, size_t *blob_bytes, size_t *n_qtiles) {
    ra_status st = validate_cu(cu, B, -1);
    if (st) return st;
    ZigzagPlan zp;
    if ((st = build_zigzag(cu, B, cp, mode, zp))) return st;
    TableCounts n;
    n.T = zp.perm.size();
    n.cul = zp.cu_local.size();
    n.off = zp.off.size();
    *n_qtiles = 0;
    if (want_tiles) {
        if (G < 1 || kBM % G != 0) return fail(RA_ERR_UNSUPPORTED, "GQA group must divide 128");
        std::vector<Tile> scratch;
        std::vector<size_t> q_doc((size_t)B, 0);
        for (int r = 0; r < cp; ++r) {
            for (int b = 0; b < B; ++b) {
                const size_t idx = (size_t)r * (B + 1) + b;
                const int64_t lo = zp.off[r] + zp.cu_local[idx], hi = zp.off[r] + zp.cu_local[idx + 1];
                scratch.clear();
                append_tiles(scratch, zp.perm.data(), lo, hi, kBM / G, b);
                n.qt += scratch.size();
                q_doc[(size_t)b] += scratch.size();
                scratch.clear();
                if (allgather) {
                    if (r == 0) append_tiles(scratch, nullptr, zp.cu[b], zp.cu[b + 1], kBN, b);
                } else {
                    append_tiles(scratch, zp.perm.data(), lo, hi, kBN, b, 1);
                }
                n.kt += scratch.size();
            }
        }
        n.tiles = true;
        n.qoff = n.kvoff = (size_t)cp * (B + 1) + 1;
        for (size_t q : q_doc) n.items += (q + 1) / 2;  // pairs of a document's query tiles
        n.items *= (size_t)Hkv;
        n.bitems = n.kt * (size_t)Hkv;
        n.qitems = n.qt * (size_t)Hkv;
        *n_qtiles = n.qt;
    }
    DeviceTables dt;
    *blob_bytes = layout_tables(n, dt);
    return RA_OK;
}

std::shared_ptr<RingPlan> get_ring_plan(const int32_t *cu, int B, int cp, int mode, int G, int Hkv,
                                        int causal, int window, bool want_tiles, bool allgather, ra_status *st,
                                        const int32_t *key_lo, const int32_t *key_hi, int kv_runs) {
    static std::mutex mu;
    static std::map<std::string, std::shared_ptr<RingPlan>> cache;
    static std::vector<std::string> order;
    *st = validate_cu(cu, B, -1);
    if (*st) return nullptr;
    std::string key;
    key.append(reinterpret_cast<const char *>(cu), sizeof(int32_t) * (size_t)(B + 1));
    const bool bounds = key_lo != nullptr || key_hi != nullptr;
    if (bounds && (!key_lo || !key_hi || !want_tiles)) {
        *st = fail(RA_ERR_INVALID_ARG, "interval masks need both bounds and the tensor-core path");
        return nullptr;
    }
    int32_t tail[11] = {B,      cp, mode, G, Hkv, causal, window, want_tiles ? 1 : 0, allgather ? 1 : 0,
                        bounds ? 1 : 0, kv_runs};
    key.append(reinterpret_cast<const char *>(tail), sizeof(tail));
    if (bounds) {  // the plan depends on every token's bounds
        const size_t T = (size_t)cu[B];
        key.append(reinterpret_cast<const char *>(key_lo), T * sizeof(int32_t));
        key.append(reinterpret_cast<const char *>(key_hi), T * sizeof(int32_t));
    }
    {
        std::lock_guard<std::mutex> lk(mu);
        auto it = cache.find(key);
        if (it != cache.end()) return it->second;
    }
    auto plan = std::make_shared<RingPlan>();
    *st = build_zigzag(cu, B, cp, mode, plan->zz);
    if (*st) return nullptr;
    if (want_tiles) {
        *st = build_ring_tiles(plan->zz, G, Hkv, causal, window, allgather, plan->tiles, key_lo, key_hi, kv_runs);
        if (*st) return nullptr;
        plan->has_tiles = true;
    }
    pack_tables(&plan->zz, want_tiles ? &plan->tiles : nullptr, plan->dev);
    std::lock_guard<std::mutex> lk(mu);
    cache[key] = plan;
    order.push_back(key);
    if (order.size() > 16) {
        cache.erase(order.front());
        order.erase(order.begin());
    }
    return plan;
}

}  // namespace ra
