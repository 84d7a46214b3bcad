// ra_internal.h -- host-side structures shared by the library's translation
// units (planner, drivers, kernel launchers).  Not part of the public ABI.
#pragma once

#include <algorithm>
#include <cstddef>
#include <cstdint>
#include <memory>
#include <mutex>
#include <string>
#include <vector>

#include "../../include/ra.h"

namespace ra {

// Sets the thread-local detail message and returns the status.
ra_status fail(ra_status s, const std::string &msg);

// Tile geometry of the tensor-core kernels: 128 MMA rows (query tokens x
// GQA heads packed together), 128-key KV tiles, head dim 128.
constexpr int kBM = 128;
constexpr int kBN = 128;
constexpr int kHeadDim = 128;

// A tile is up to `rows` consecutive local rows of one segment whose
// positions form at most two runs of consecutive integers:
//   row c < split       -> pos0 + c
//   split <= c < len    -> pos1 + (c - split)
// Two int4 per tile on the device: {row0, len, split, pos0}, {pos1, pmin, pmax, seg}.
struct Tile {
    int32_t row0, len, split, pos0;
    int32_t pos1, pmin, pmax, seg;
};
static_assert(sizeof(Tile) == 32, "tile record is two int4");

// A work item of the tensor-core kernels.  Forward: two query tiles
// (qt1 = -1 when absent) of one (rank r, segment b), one KV head g, and the
// ring steps [t0, t1) whose KV tiles it visits.  Backward: qt0 is a KV
// tile, qt1 unused, and the steps name the query ranks visited.
struct WorkItem {
    int32_t qt0, qt1, g, r;
    int32_t b, t0, t1, cost;
};
static_assert(sizeof(WorkItem) == 32, "work item is two int4");

// Zigzag plan (host): see ra_zigzag_plan in ra.h.
struct ZigzagPlan {
    int64_t T = 0;
    int B = 0, cp = 0, mode = 0;
    std::vector<int32_t> cu;        // [B+1]
    std::vector<int32_t> perm;      // [T]
    std::vector<int32_t> off;       // [cp+1]
    std::vector<int32_t> cu_local;  // [cp*(B+1)]
};

ra_status validate_cu(const int32_t *cu, int B, int64_t T);
ra_status build_zigzag(const int32_t *cu, int B, int cp, int mode, ZigzagPlan &zp);

// Tile-pair class used by both the host cost model and the kernels: skip
// when no pair is allowed (every key after every query under the causal
// mask, or further behind every query than the window), full when every
// pair of a 128-key tile is allowed.  window < 0: no window.
enum { kSkip = 0, kFull = 1, kPartial = 2 };
inline int classify(const Tile &q, const Tile &k, int causal, int window) {
    if (q.len <= 0 || k.len <= 0) return kSkip;
    if (causal && q.pmax < k.pmin) return kSkip;
    if (window >= 0 && (int64_t)q.pmin - window > k.pmax) return kSkip;
    if (k.len == kBN && (!causal || q.pmin >= k.pmax) && (window < 0 || (int64_t)q.pmax - window <= k.pmin))
        return kFull;
    return kPartial;
}

// Interval masks: query token i sees key j of its own document iff
// lo[i] <= j <= hi[i] (original token indices).  Per query tile the planner
// keeps the extremes of its rows' bounds, from which a tile pair is
// classified: skip when every row's interval misses the KV tile's positions
// (hi_max < kpmin or lo_min > kpmax), full when every row's interval covers
// a complete KV tile (lo_max <= kpmin and hi_min >= kpmax), else partial.
struct QBounds {
    int32_t lo_min, lo_max, hi_min, hi_max;
};
static_assert(sizeof(QBounds) == 16, "query tile bounds are one int4");
inline int classify_bounds(const Tile &q, const QBounds &b, const Tile &k) {
    if (q.len <= 0 || k.len <= 0) return kSkip;
    if (b.hi_max < k.pmin || b.lo_min > k.pmax) return kSkip;
    if (k.len == kBN && b.lo_max <= k.pmin && b.hi_min >= k.pmax) return kFull;
    return kPartial;
}

// Counting visits without walking every tile pair.  The tiles of one
// segment cover consecutive rows whose positions increase, so along them
// both pmin and pmax increase, and under the interval masks (bounds that
// never decrease inside a document) so do a query tile's lo_min and hi_max.
// A tile pair is skipped above exactly when one of two monotone tests
// fails, so the tiles of a segment that a fixed partner visits form one
// index range: two binary searches find it, and for a whole segment of
// partners in order two pointers that only move forward.
//
// For every query tile q[0, nq) of one segment (bounds qb[0, nq) under
// interval masks, else null), the KV tiles of k[0, nk) (one segment) that
// it visits (classify or classify_bounds other than kSkip): a tile pair is
// visited iff k.pmin <= hi and k.pmax >= lo, with hi and lo from the query
// tile, and along the query tiles both move forward, so two pointers walk
// each list once.  Writes the counts to out[i * stride] when out is not
// null; returns their sum.
inline int64_t kv_tiles_visited_each(const Tile *q, const QBounds *qb, int nq, const Tile *k, int nk, int causal,
                                     int window, int32_t *out, int stride) {
    int64_t sum = 0;
    int b = 0, e = 0;
    for (int i = 0; i < nq; ++i) {
        int64_t hi = INT64_MAX, lo = INT64_MIN;
        if (qb) {
            hi = qb[i].hi_max;
            lo = qb[i].lo_min;
        } else {
            if (causal) hi = q[i].pmax;
            if (window >= 0) lo = (int64_t)q[i].pmin - window;
        }
        while (e < nk && (int64_t)k[e].pmin <= hi) ++e;
        while (b < nk && (int64_t)k[b].pmax < lo) ++b;
        const int c = (q[i].len > 0 && e > b) ? e - b : 0;
        if (out) out[(size_t)i * stride] = c;
        sum += c;
    }
    return sum;
}

// Query tiles q[0, n) of one segment (with their bounds qb[0, n) under
// interval masks, else null) that visit KV tile k.
inline int64_t q_tiles_visiting(const Tile *q, const QBounds *qb, int n, const Tile &k, int causal, int window) {
    if (k.len <= 0 || n <= 0) return 0;
    int b = 0, e = n;
    if (qb) {  // visited iff hi_max >= k.pmin and lo_min <= k.pmax
        b = (int)(std::lower_bound(qb, qb + n, k.pmin, [](const QBounds &x, int32_t v) { return x.hi_max < v; }) - qb);
        e = (int)(std::upper_bound(qb, qb + n, k.pmax, [](int32_t v, const QBounds &x) { return v < x.lo_min; }) - qb);
    } else {  // visited iff q.pmax >= k.pmin (causal) and q.pmin - window <= k.pmax (window)
        if (causal)
            b = (int)(std::lower_bound(q, q + n, k.pmin, [](const Tile &t, int32_t v) { return t.pmax < v; }) - q);
        if (window >= 0) {
            const int64_t lim = (int64_t)k.pmax + window;
            e = (int)(std::upper_bound(q, q + n, lim, [](int64_t v, const Tile &t) { return v < (int64_t)t.pmin; }) - q);
        }
    }
    return e > b ? e - b : 0;
}

// Tile tables for one query side and one key side.  Tiles of segment b of
// rank r are [q_off[r*(B+1)+b], q_off[r*(B+1)+b+1]) (same for kv_off).
struct TilePlan {
    int cp = 1, B = 0;
    int q_tokens = 0;                    // tokens per query tile (128 / G)
    std::vector<Tile> qtiles, kvtiles;
    std::vector<int32_t> q_off, kv_off;  // [cp*(B+1)+1]
    std::vector<WorkItem> items;         // forward items, LPT order
    std::vector<WorkItem> bitems;        // backward dK/dV items (one per KV tile x head)
    std::vector<WorkItem> qitems;        // backward dQ items (one per query tile x head)
    int64_t fwd_tile_pairs = 0;          // non-skipped (query tile, KV tile) visits
    // interval masks only: bounds extremes per query tile, and the per-token
    // bounds [T] the kernels read at a row's original position
    std::vector<QBounds> qbounds;
    std::vector<int32_t> key_lo, key_hi;
    // tile-pair class under the plan's mask
    int pair_class(int qi, int kj, int causal, int window) const {
        return qbounds.empty() ? classify(qtiles[qi], kvtiles[kj], causal, window)
                               : classify_bounds(qtiles[qi], qbounds[qi], kvtiles[kj]);
    }
};

// Builds tiles over rows [lo, hi) with positions pos[row] (at most
// max_runs, 1 or 2, consecutive-position runs per tile) and appends them.
void append_tiles(std::vector<Tile> &out, const int32_t *pos, int64_t lo, int64_t hi,
                  int tile_rows, int seg, int max_runs = 2);

// Ring tile plan: query side = key side = the permuted buffer.
// allgather: the key side is every document's K/V in original order (the
// all-gather schedule), held as the segments of rank 0; otherwise each
// rank's zigzag shard, as the ring passes it.
// key_lo / key_hi (NULL = none): an interval mask (then causal and window
// are ignored), checked for non-decreasing bounds inside every document.
// kv_runs: 0 = the KV tiling with fewer forward visits (tiles of at most two
// position runs, or of one), 1 or 2 = that tiling.
ra_status build_ring_tiles(const ZigzagPlan &zp, int G, int Hkv, int causal, int window, bool allgather,
                           TilePlan &tp, const int32_t *key_lo = nullptr, const int32_t *key_hi = nullptr,
                           int kv_runs = 0);

// Generic partial's tile plan: one "rank", separate Q and K sides.
ra_status build_partial_tiles(const int32_t *cu_q, const int32_t *cu_k, int nseg,
                              const int32_t *q_pos, const int32_t *k_pos, int64_t Tq, int64_t Tk,
                              int G, int Hkv, int causal, int window, TilePlan &tp);

// Host image of the device tables, uploaded into the workspace each call.
struct DeviceTables {
    std::vector<uint8_t> blob;
    size_t o_perm = 0, o_qt = 0, o_kt = 0, o_qoff = 0, o_kvoff = 0, o_items = 0,
           o_bitems = 0, o_qitems = 0, o_cul = 0, o_off = 0;
    // One byte per rank-ordered row: 1 where the row belongs to a query tile
    // of two position runs (the tensor-core kernels read such tiles from the
    // rank-ordered copy; single-run tiles straight from the caller's tensor).
    size_t o_qmask = 0;
    size_t o_kvmask = 0;  // likewise for KV tiles (the K and V copies)
    // Work counters of the persistent kernels (uploaded as zeros; a kernel
    // returns its counter to zero when it finishes): [0, 2) forward.
    size_t o_sched = 0;
    // interval masks: QBounds per query tile, key_lo and key_hi [T]
    size_t o_qb = 0, o_klo = 0, o_khi = 0;
    bool bounds = false;
    int n_items = 0, n_bitems = 0, n_qitems = 0;
};
void pack_tables(const ZigzagPlan *zp, const TilePlan *tp, DeviceTables &dt);

// Record counts that fix the size and the offsets of the device tables.
struct TableCounts {
    size_t T = 0, cul = 0, off = 0;  // zigzag: perm [T], cu_local, off (all 0 without a zigzag plan)
    bool tiles = false;              // tile tables present (with the two-run row masks [T] each)
    size_t qt = 0, kt = 0, qoff = 0, kvoff = 0, items = 0, bitems = 0, qitems = 0;
    size_t qb = 0, klo = 0, khi = 0;  // interval masks: bounds per query tile, key_lo and key_hi
};
// Sets dt's offsets for tables with these counts; returns their total bytes.
size_t layout_tables(const TableCounts &n, DeviceTables &dt);

// Table bytes and query-tile count of the ring plan with the most KV tiles
// for this packing (every KV tile of one position run; a rank's share of a
// document cut at its chunk boundary never has fewer tiles than joined across
// it), found from the tiles alone, without work items.  No mask or per-share
// tiling choice gives a plan with larger tables.
ra_status ring_tables_bound(const int32_t *cu, int B, int cp, int mode, int G, int Hkv, bool want_tiles,
                            bool allgather, size_t *blob_bytes, size_t *n_qtiles);

struct RingPlan {
    ZigzagPlan zz;
    TilePlan tiles;
    bool has_tiles = false;
    DeviceTables dev;
    // Page-locked copy of dev.blob, made on the first upload outside stream
    // capture, so that the per-call table upload is an asynchronous copy that
    // never blocks the host.  Page-locked buffers are recycled through a
    // process-wide pool when plans leave the cache (no free, so no implicit
    // device synchronisation); a buffer that a captured graph copies from is
    // kept for the process lifetime.
    void *pinned = nullptr;
    size_t pinned_bytes = 0;
    void *uploaded = nullptr;          // cudaEvent_t of the last upload from `pinned`
    void *upload_stream = nullptr;     // its stream
    bool multi_stream = false;         // uploads went to more than one stream
    bool in_graph = false;             // an upload was captured into a graph
    std::mutex pin_mu;
    ~RingPlan();
};
// Enqueues the copy of plan.dev.blob into the workspace tables at `dst` on
// `stream` (a cudaStream_t).  Under stream capture the plan must already
// have its page-locked copy (an earlier call outside capture made it).
ra_status upload_plan_tables(RingPlan &plan, void *dst, void *stream);
// Cached plans keyed by content (cu_seqlens, cp, mode, G, Hkv, causal, window,
// and the interval bounds when given).
std::shared_ptr<RingPlan> get_ring_plan(const int32_t *cu, int B, int cp, int mode, int G, int Hkv,
                                        int causal, int window, bool want_tiles, bool allgather, ra_status *st,
                                        const int32_t *key_lo = nullptr, const int32_t *key_hi = nullptr,
                                        int kv_runs = 0);

inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

}  // namespace ra
