// ra_tc_bwd.cu -- tensor-core key-side backward (dK, dV) of packed causal
// varlen ring attention (bf16 in, fp32 accumulation, head dim 128) for
// sm_103a.
//
// What it computes: from the saved log-sum-exp and D = rowsum(dO o O),
//   P  = exp(scale * Q K^T - lse)   over allowed pairs (same document,
//                                    causal, and inside the sliding window)
//   dV = P^T dO,   dS = P o (dO V^T - D),   dK = scale * dS^T Q
// with GQA sums over the query heads of each KV head (the key side of the
// backward_impl of FlagScale PR #910's RingAttention; the query side, dQ, is
// ra_tc_dq.cu).  In the ring the K/V shard of rank s meets the queries of
// rank r = (s + t) mod cp at step t; one CTA owns one KV tile and walks the
// query tiles of its document over the ring steps, so dK and dV accumulate
// in fp32 in TMEM across all steps and are written once.
//
// GB300 design:
//  * CTA = one KV tile (128 keys of one KV head); K and V stay in shared
//    memory.  Visited query tiles (128 rows = 128/G tokens x G heads) and
//    their dO tiles stream through two TMA stages together with the tile's
//    128 LSE and D values (pre-gathered per tile, one bulk copy).
//  * Per tile S^T = K Q^T and dP^T = V dO^T are SS-MMAs, dV += P^T dO and
//    dK += dS^T Q are TS-MMAs with P^T and dS^T read from TMEM, so shared
//    memory only streams Q and dO (the SS products at N = 128 already use
//    most of the shared-memory read port).
//  * Each query tile is processed as two 64-column halves h (query rows
//    [64h, 64h+64)), and compute group h owns half h: S^T_h is an N=64
//    product into that group's TMEM columns, so group 0's exponentials
//    start while S^T_1 is still in the pipe and the groups stay staggered;
//    dP^T is one N=128 product (an SS product at N=64 reads 6 KB per 32
//    tensor cycles, above the 128 B/cycle of the shared-memory port, so it
//    runs at two thirds of the tensor rate); dV and dK take the matching
//    64-row slice of the contraction per group.
//  * Two warps issue, one per TMEM reuse chain: warp 1 dV_h(i) then
//    S^T_h(i+1) (which overwrites P^T_h(i)), warp 3 dK_0(i), dK_1(i) then
//    dP^T(i+1) (which overwrites both dS^T halves); each chain is ordered
//    by the tensor pipe's in-order execution of one issuer's products.
//    Each issuer warp runs converged and one elected lane issues: from one
//    lane of a divergent branch an MMA costs 45-60 cycles to issue.
//  * TMEM: dK [0,128), dV [128,256), S^T then P^T [256,384), dP^T then dS^T
//    [384,512).  Two compute warpgroups split the 128 query columns; each
//    packs its P^T / dS^T (bf16) over the first 32 of its own 64 columns.
//  * Every wait is bounded (2 s); a wait that runs out records
//    RA_ERR_TIMEOUT and the CTA drains its copies and returns.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <cmath>
#include <cstring>
#include <mutex>

#include "ra_dev.cuh"
#include "ra_internal.h"
#include "ra_kernels.h"

namespace ra {

namespace {

using namespace dev;

constexpr int kThreads = 384;
constexpr uint32_t kHalf = 16384;                 // 128 rows x 128 B
constexpr uint32_t kTile = 2 * kHalf;
constexpr uint32_t kOffK = 0;
constexpr uint32_t kOffV = kTile;
constexpr uint32_t kOffQ = 2 * kTile;             // [2] stages
constexpr uint32_t kOffDO = 4 * kTile;            // [2] stages
constexpr uint32_t kOffInfo = 6 * kTile;          // [2] x {lse[128], D[128], descriptor}
constexpr uint32_t kInfoBytes = 1024 + 64;
constexpr uint32_t kOffBar = kOffInfo + 2 * kInfoBytes;
constexpr uint32_t kSmemBytes = kOffBar + 128;    // 16 barrier words; base must be 1024-aligned (checked)

struct BwdParams {
    CUtensorMap tmQ, tmK, tmV, tmDO;
    CUtensorMap tmQo, tmDOo;  // Q and dO in original order (valid when qdo_direct)
    CUtensorMap tmKo, tmVo;   // K and V in original order (valid when kv_direct)
    const int4 *qtiles, *kvtiles, *items;
    const int *q_off;
    int qdo_direct;  // single-run query tiles: Q and dO read at their first position
    int kv_direct;   // single-run KV tiles: K and V likewise
    int n_items, cp, B, G, log2G, Hq, Hkv;
    int t0, t1, causal, window, out_mode;          // 0 bf16 store, 1 fp32 store, 2 fp32 +=
    const int4 *qbounds;         // interval masks: QBounds per query tile
    const int *key_lo, *key_hi;  // and each token's key bounds at its original position
    float scale, scale_log2;
    const float *tile_ld;
    void *dk, *dv;
    int *status;
    unsigned long long budget_ns;
};

struct QInfo {
    int len, pmin, pmax;
    int lo_min, lo_max, hi_min, hi_max;  // interval masks only
};

// The host's classify_bounds (interval masks), on device.
__device__ __forceinline__ int classify_b(const QInfo &q, int klen, int kpmin, int kpmax) {
    if (q.len <= 0 || klen <= 0) return kSkip;
    if (q.hi_max < kpmin || q.lo_min > kpmax) return kSkip;
    if (klen == kBN && q.lo_max <= kpmin && q.hi_min >= kpmax) return kFull;
    return kPartial;
}

__device__ __forceinline__ int classify_pair(const QInfo &q, int klen, int kpmin, int kpmax, int causal,
                                             int window) {
    if (q.len <= 0 || klen <= 0) return kSkip;
    if (causal && q.pmax < kpmin) return kSkip;
    if (window >= 0 && q.pmin - window > kpmax) return kSkip;
    if (klen == kBN && (!causal || q.pmin >= kpmax) && (window < 0 || q.pmax - window <= kpmin)) return kFull;
    return kPartial;
}

__device__ __forceinline__ uint32_t range_bits(int a, int b, int base) {
    const int lo = min(max(a - base, 0), 32), hi = min(max(b - base, 0), 32);
    return (uint32_t)(((1ull << hi) - 1ull) & ~((1ull << lo) - 1ull));
}

// kMask: 0 causal (or none), 1 with the sliding-window mask (p.window >= 0),
// 2 interval masks (per-token key bounds).
template <int kMask>
__global__ void __launch_bounds__(kThreads, 1) tc_dkdv_kernel(const __grid_constant__ BwdParams p) {
    constexpr bool kWindow = kMask == 1, kBounds = kMask == 2;
    extern __shared__ __align__(1024) uint8_t smem[];
    const uint32_t base_s = smem_u32(smem);
    if (base_s & 1023u) {  // the layout has no slack for realignment
        if (threadIdx.x == 0) record_status(p.status, RA_ERR_DEVICE_BOUNDS);
        return;
    }
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + kOffBar);
    uint64_t *kv_full = bars + 0;
    uint64_t *st_full = bars + 1;    // [2] Q, dO, lse, D of a stage (TMA + bulk copies)
    uint64_t *st_empty = bars + 3;   // [2]
    uint64_t *s_full = bars + 5;     // [2] S^T half h done
    uint64_t *dp_full = bars + 7;    // [2] dP^T half h done
    uint64_t *p_ready = bars + 9;    // [2] P^T half h in TMEM (128 arrivals)
    uint64_t *ds_ready = bars + 11;  // [2] dS^T half h in TMEM (128 arrivals)
    uint64_t *mma_done = bars + 13;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + 14);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(bars + 15);
    auto info = [&](uint32_t st) -> uint8_t * { return smem + kOffInfo + st * kInfoBytes; };

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int4 ia = __ldg(p.items + 2 * blockIdx.x), ib = __ldg(p.items + 2 * blockIdx.x + 1);
    const int kt = ia.x, g = ia.z, s = ia.w, b = ib.x;
    const int t0 = p.t0 >= 0 ? p.t0 : ib.y;
    const int t1 = p.t0 >= 0 ? p.t1 : ib.z;
    const int4 ka = __ldg(p.kvtiles + 2 * kt), kb = __ldg(p.kvtiles + 2 * kt + 1);
    // KV tile: row0 ka.x, len ka.y, split ka.z, pos0 ka.w, pos1 kb.x, pmin kb.y, pmax kb.z
    const int G = p.G;

    if (threadIdx.x == 0) {
        *abort_flag = 0;
        mbar_init(kv_full, 1);
        for (int i = 0; i < 2; ++i) {
            mbar_init(st_full + i, 1);
            mbar_init(st_empty + i, 2);  // one commit from each issuer
        }
        for (int h = 0; h < 2; ++h) {
            mbar_init(s_full + h, 1);
            mbar_init(dp_full + h, 1);
            mbar_init(p_ready + h, 128);
            mbar_init(ds_ready + h, 128);
        }
        mbar_init(mma_done, 2);  // one commit from each issuer
        fence_mbar_init();
    }
    if (warp == 2) {
        tmem_alloc(tmem_slot, 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const WaitCtl wc{abort_flag, p.status, p.budget_ns};
    const uint32_t tDK = tmem, tDV = tmem + 128, tS = tmem + 256, tDP = tmem + 384;

    if (warp == 0) {
        // ------------------------------------------------ producer
        if (lane == 0) {
            tma_prefetch_desc(&p.tmQ);
            tma_prefetch_desc(&p.tmK);
            tma_prefetch_desc(&p.tmV);
            tma_prefetch_desc(&p.tmDO);
            if (p.qdo_direct) {
                tma_prefetch_desc(&p.tmQo);
                tma_prefetch_desc(&p.tmDOo);
            }
            // one position run (split == len): the original rows
            const bool kdir = p.kv_direct && ka.z == ka.y;
            const CUtensorMap *mk = kdir ? &p.tmKo : &p.tmK, *mv = kdir ? &p.tmVo : &p.tmV;
            const int krow = kdir ? ka.w : ka.x;
            mbar_arrive_expect_tx(kv_full, 2 * kTile);
            tma_load_3d(smem + kOffK, mk, kv_full, 0, g, krow);
            tma_load_3d(smem + kOffK + kHalf, mk, kv_full, 64, g, krow);
            tma_load_3d(smem + kOffV, mv, kv_full, 0, g, krow);
            tma_load_3d(smem + kOffV + kHalf, mv, kv_full, 64, g, krow);
        }
        uint32_t n = 0;  // tiles published
        int ok = 1;
        // lane 0 publishes a query tile: descriptor, Q and dO by TMA, its 128
        // LSE and D values (pre-gathered per tile) by bulk copy, one barrier
        auto publish = [&](const int4 &d0, const int4 &d1, int qt, bool end) {
            const uint32_t st = n & 1u;
            if (lane == 0) {
                if (!mbar_wait(st_empty + st, ((n >> 1) & 1u) ^ 1u, wc)) {
                    ok = 0;
                } else {
                    int4 *desc = reinterpret_cast<int4 *>(info(st) + 1024);
                    desc[0] = d0;
                    desc[1] = end ? make_int4(0, 1, 0, 0) : d1;
                    if (!end) {
                        mbar_arrive_expect_tx(st_full + st, 2 * kTile + 1024);
                        const int hq0 = g * G;
                        // one position run (split == len): the original rows
                        const bool dir = p.qdo_direct && d0.z == d0.y;
                        const CUtensorMap *mq = dir ? &p.tmQo : &p.tmQ, *mdo = dir ? &p.tmDOo : &p.tmDO;
                        const int row = dir ? d0.w : d0.x;
                        tma_load_3d(smem + kOffQ + st * kTile, mq, st_full + st, 0, hq0, row);
                        tma_load_3d(smem + kOffQ + st * kTile + kHalf, mq, st_full + st, 64, hq0, row);
                        tma_load_3d(smem + kOffDO + st * kTile, mdo, st_full + st, 0, hq0, row);
                        tma_load_3d(smem + kOffDO + st * kTile + kHalf, mdo, st_full + st, 64, hq0, row);
                        bulk_load(info(st), p.tile_ld + ((long long)qt * p.Hkv + g) * 256, 1024, st_full + st);
                    } else {
                        mbar_arrive(st_full + st);
                    }
                }
            }
            ok = __shfl_sync(0xffffffffu, ok, 0);
            ++n;
        };
        for (int t = t0; t < t1 && ok; ++t) {
            const int r = (s + t) % p.cp;
            const int o = r * (p.B + 1) + b;
            const int lo = __ldg(p.q_off + o), hi = __ldg(p.q_off + o + 1);
            for (int bi = lo; bi < hi && ok; bi += 32) {
                const int idx = bi + lane;
                int4 qa = make_int4(0, 0, 0, 0), qb = make_int4(0, 0, 0, 0);
                int cls = kSkip;
                if (idx < hi) {
                    qa = __ldg(p.qtiles + 2 * idx);
                    qb = __ldg(p.qtiles + 2 * idx + 1);
                    if (kBounds) {
                        const int4 bb = __ldg(p.qbounds + idx);
                        cls = classify_b(QInfo{qa.y, qb.y, qb.z, bb.x, bb.y, bb.z, bb.w}, ka.y, kb.y, kb.z);
                    } else {
                        cls = classify_pair(QInfo{qa.y, qb.y, qb.z, 0, 0, 0, 0}, ka.y, kb.y, kb.z, p.causal,
                                            kWindow ? p.window : -1);
                    }
                }
                uint32_t vis = __ballot_sync(0xffffffffu, cls != kSkip);
                while (vis && ok) {
                    const int src = __ffs(vis) - 1;
                    vis &= vis - 1;
                    int4 d0, d1;
                    d0.x = __shfl_sync(0xffffffffu, qa.x, src);
                    d0.y = __shfl_sync(0xffffffffu, qa.y, src);
                    d0.z = __shfl_sync(0xffffffffu, qa.z, src);
                    d0.w = __shfl_sync(0xffffffffu, qa.w, src);
                    d1.x = __shfl_sync(0xffffffffu, qb.x, src);
                    d1.y = __shfl_sync(0xffffffffu, cls, src) << 1;  // flags: class << 1, bit 0 = end
                    d1.z = 0;
                    d1.w = 0;
                    publish(d0, d1, bi + src, false);
                }
            }
        }
        if (ok) publish(make_int4(0, 0, 0, 0), make_int4(0, 1, 0, 0), 0, true);
        if (lane == 0) {
            volatile int local_abort = 0;
            const WaitCtl drain{&local_abort, p.status, p.budget_ns};
            (void)mbar_wait(kv_full, 0, drain);
            for (uint32_t x = (n > 2 ? n - 2 : 0); x < n; ++x)
                (void)mbar_wait(st_full + (x & 1u), (x >> 1) & 1u, drain);
        }
    } else if (warp == 1 || warp == 3) {
        // ------------------------------------------------ MMA issuers
        // Each issuer warp runs converged; one elected lane issues (_w helpers).
        const uint32_t id_n64 = idesc_bf16_f32(128, 64, 0, 0);  // A, B K-major, N = 64 queries
        const uint32_t id_n128 = idesc_bf16_f32(128, 128, 0, 0);
        const uint32_t id_ts = idesc_bf16_f32(128, 128, 0, 1);  // A in TMEM, B MN-major
        auto is_end = [&](uint32_t st) {
            return (reinterpret_cast<const int4 *>(info(st) + 1024)[1].y & 1) != 0;
        };
        auto kstep = [](int ks) -> uint32_t { return (((ks >> 2) * kHalf + (ks & 3) * 32u) >> 4); };
        // warp 1: S^T_h and dV; warp 3: dP^T_h and dK
        const bool pchain = warp == 1;
        const uint32_t chain_d = pchain ? tS : tDP;                          // S^T / dP^T
        const uint64_t chain_a = sdesc_sw128(base_s + (pchain ? kOffK : kOffV), 16, 1024);
        const uint32_t chain_b = base_s + (pchain ? kOffQ : kOffDO);        // Q / dO stages
        const uint32_t grad_d = pchain ? tDV : tDK;                          // dV / dK
        const uint32_t grad_b = base_s + (pchain ? kOffDO : kOffQ);         // dO / Q stages
        uint64_t *chain_full = pchain ? s_full : dp_full;
        uint64_t *ready = pchain ? p_ready : ds_ready;
        // S^T_h / dP^T_h of stage st: 128 keys x query rows [64h, 64h+64)
        auto chain_mma = [&](int h, uint32_t st) {
            const uint64_t b0 = sdesc_sw128(chain_b + st * kTile + 8192u * h, 16, 1024);
#pragma unroll
            for (int ks = 0; ks < 8; ++ks)
                tc_mma_ss_w(chain_d + 64u * h, chain_a + kstep(ks), b0 + kstep(ks), id_n64, ks > 0);
            tc_commit_w(chain_full + h);
        };
        // dP^T of stage st as one N=128 product (both groups' barriers)
        auto chain_full_mma = [&](uint32_t st) {
            const uint64_t b0 = sdesc_sw128(chain_b + st * kTile, 16, 1024);
#pragma unroll
            for (int ks = 0; ks < 8; ++ks)
                tc_mma_ss_w(chain_d, chain_a + kstep(ks), b0 + kstep(ks), id_n128, ks > 0);
            tc_commit_w(chain_full + 0);
            tc_commit_w(chain_full + 1);
        };
        // dV / dK += P^T_h / dS^T_h (TMEM, group h's columns) x rows [64h, 64h+64)
        // of dO / Q (MN-major: d contiguous)
        auto grad_mma = [&](int h, uint32_t st, bool acc) {
            const uint64_t b0 = sdesc_sw128(grad_b + st * kTile + 8192u * h, kHalf, 1024);
#pragma unroll
            for (int k = 0; k < 4; ++k)
                tc_mma_ts_w(grad_d, chain_d + 64u * h + 8u * k, b0 + ((2048u * k) >> 4), id_ts, (acc || k > 0));
        };
        bool ok = mbar_wait_warp(kv_full, 0, wc) && mbar_wait_warp(st_full + 0, 0, wc);
        tc_fence_after();
        const bool have = ok && !is_end(0);
        if (have && pchain) {
            // S^T as two N=64 halves, so group 0's exponentials start while
            // half 1 is still in the pipe (the groups stay staggered)
            chain_mma(0, 0);
            chain_mma(1, 0);
            for (uint32_t i = 0; ok; ++i) {
                const uint32_t st = i & 1u, nst = (i + 1) & 1u;
                if (!mbar_wait_warp(ready + 0, i & 1u, wc)) break;
                tc_fence_after();
                grad_mma(0, st, i > 0);
                if (!mbar_wait_warp(st_full + nst, ((i + 1) >> 1) & 1u, wc)) break;
                tc_fence_after();
                const bool next_end = is_end(nst);
                // half 0 of the next tile overwrites P^T_0 after the product above (in order)
                if (!next_end) chain_mma(0, nst);
                if (!mbar_wait_warp(ready + 1, i & 1u, wc)) break;
                tc_fence_after();
                grad_mma(1, st, true);
                tc_commit_w(st_empty + st);  // this issuer no longer reads the stage
                if (next_end) break;
                chain_mma(1, nst);
            }
        } else if (have) {
            // dP^T as one N=128 product: the N=64 halves of an SS product
            // read 6 KB per 32 tensor cycles, above the 128 B/cycle of the
            // shared-memory port, and the dS work needs no staggering
            chain_full_mma(0);
            for (uint32_t i = 0; ok; ++i) {
                const uint32_t st = i & 1u, nst = (i + 1) & 1u;
                if (!mbar_wait_warp(ready + 0, i & 1u, wc)) break;
                tc_fence_after();
                grad_mma(0, st, i > 0);
                if (!mbar_wait_warp(ready + 1, i & 1u, wc)) break;
                tc_fence_after();
                grad_mma(1, st, true);
                tc_commit_w(st_empty + st);  // this issuer no longer reads the stage
                if (!mbar_wait_warp(st_full + nst, ((i + 1) >> 1) & 1u, wc)) break;
                tc_fence_after();
                if (is_end(nst)) break;
                // the next dP^T overwrites both dS^T halves after the two products above
                chain_full_mma(nst);
            }
        }
        tc_commit_w(mma_done);
        volatile int local_abort = 0;
        const WaitCtl drain{&local_abort, p.status, p.budget_ns};
        (void)mbar_wait_warp(mma_done, 0, drain);
    } else if (warp >= 4) {
        // ------------------------------------------------ compute warpgroups
        // Group h (warps 4-7: 0, warps 8-11: 1) owns columns [64h, 64h+64) of
        // S^T and dP^T and d columns [64h, 64h+64) of dK and dV; thread j owns
        // TMEM lane j (one key row).
        const int h = (warp >= 8) ? 1 : 0;
        const int j = (threadIdx.x - 128) & 127;
        const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
        const bool kvalid = j < ka.y;
        const int kpos = j < ka.z ? ka.w + j : kb.x + (j - ka.z);
        bool ok = true;
        uint32_t nt = 0;
        for (uint32_t i = 0;; ++i) {
            const uint32_t st = i & 1u;
            if (!mbar_wait(st_full + st, (i >> 1) & 1u, wc)) {
                ok = false;
                break;
            }
            const uint8_t *I = info(st);
            const int4 d0 = reinterpret_cast<const int4 *>(I + 1024)[0];
            const int4 d1 = reinterpret_cast<const int4 *>(I + 1024)[1];
            if (d1.y & 1) break;
            const int cls = d1.y >> 1;
            // ---- P^T = exp2(S^T * scale * log2e - lse * log2e), masked
            if (!mbar_wait(s_full + h, i & 1u, wc)) {
                ok = false;
                break;
            }
            tc_fence_after();
            uint32_t v[64];
            tmem_ld64(tS + lane_base + 64u * h, v);
            uint32_t wm[2] = {~0u, ~0u};
            if (cls == kPartial) {
                int a1 = 0, e1 = 0, a2 = 0, e2 = 0;
                if (kvalid && kBounds) {
                    // the tokens t of the query tile whose key interval holds
                    // kpos, [a1, e1): both bounds are non-decreasing along the
                    // tile (its two runs lie in one document, in position
                    // order), so each end is a binary search
                    const int qlen = d0.y, split = d0.z, pos0 = d0.w, pos1 = d1.x;
                    int lo_ = 0, hi_ = qlen;
                    while (lo_ < hi_) {  // first t with key_hi >= kpos
                        const int mid = (lo_ + hi_) >> 1;
                        const int pm = mid < split ? pos0 + mid : pos1 + (mid - split);
                        if (__ldg(p.key_hi + pm) >= kpos) hi_ = mid; else lo_ = mid + 1;
                    }
                    a1 = lo_;
                    lo_ = 0;
                    hi_ = qlen;
                    while (lo_ < hi_) {  // first t with key_lo > kpos
                        const int mid = (lo_ + hi_) >> 1;
                        const int pm = mid < split ? pos0 + mid : pos1 + (mid - split);
                        if (__ldg(p.key_lo + pm) > kpos) hi_ = mid; else lo_ = mid + 1;
                    }
                    e1 = lo_;
                } else if (kvalid) {
                    const int qlen = d0.y, split = d0.z, pos0 = d0.w, pos1 = d1.x;
                    if (p.causal) {
                        a1 = min(max(kpos - pos0, 0), split);
                        a2 = min(max(kpos - pos1 + split, split), qlen);
                    } else {
                        a1 = 0;
                        a2 = split;
                    }
                    e1 = split;
                    e2 = qlen;
                    if (kWindow) {  // queries at most `window` ahead of this key
                        e1 = min(max(kpos + p.window - pos0 + 1, 0), split);
                        e2 = min(max(kpos + p.window - pos1 + split + 1, split), qlen);
                    }
                }
#pragma unroll
                for (int ch = 0; ch < 2; ++ch) {
                    const int cb = 64 * h + 32 * ch;
                    wm[ch] = range_bits(a1 * G, e1 * G, cb) | range_bits(a2 * G, e2 * G, cb);
                }
            }
            // per query column: -lse * log2(e) at [0, 128), -D * scale at [128, 256)
            const float4 *l4 = reinterpret_cast<const float4 *>(I) + 16 * h;
            const float2 sl2 = make_float2(p.scale_log2, p.scale_log2);
            float P[64];
#pragma unroll
            for (int c4 = 0; c4 < 16; ++c4) {
                const float4 l = l4[c4];
                const int c = 4 * c4;
                const float2 x0 = fma2(make_float2(__uint_as_float(v[c]), __uint_as_float(v[c + 1])), sl2,
                                       make_float2(l.x, l.y));
                const float2 x1 = fma2(make_float2(__uint_as_float(v[c + 2]), __uint_as_float(v[c + 3])), sl2,
                                       make_float2(l.z, l.w));
                P[c] = ex2_approx(x0.x);
                P[c + 1] = ex2_approx(x0.y);
                P[c + 2] = ex2_approx(x1.x);
                P[c + 3] = ex2_approx(x1.y);
            }
            if (cls == kPartial) {
#pragma unroll
                for (int c = 0; c < 64; ++c) P[c] = ((wm[c >> 5] >> (c & 31)) & 1u) ? P[c] : 0.f;
            }
            {
                uint32_t pk[32];
#pragma unroll
                for (int c2 = 0; c2 < 32; ++c2) pk[c2] = pack_bf16x2(P[2 * c2], P[2 * c2 + 1]);
                tmem_st32(tS + lane_base + 64u * h, pk);
            }
            tc_fence_before();
            mbar_arrive(p_ready + h);
            // ---- dS^T = (dP^T * scale - D * scale) o P^T, bf16 over this group's dP^T columns
            if (!mbar_wait(dp_full + h, i & 1u, wc)) {
                ok = false;
                break;
            }
            tc_fence_after();
            tmem_ld64(tDP + lane_base + 64u * h, v);
            const float4 *d4 = reinterpret_cast<const float4 *>(I + 512) + 16 * h;
            const float2 sc2 = make_float2(p.scale, p.scale);
            uint32_t pk[32];
#pragma unroll
            for (int c4 = 0; c4 < 16; ++c4) {
                const float4 dd = d4[c4];
                const int c = 4 * c4;
                const float2 s0 = fma_mul2(make_float2(__uint_as_float(v[c]), __uint_as_float(v[c + 1])), sc2,
                                           make_float2(dd.x, dd.y), make_float2(P[c], P[c + 1]));
                const float2 s1 = fma_mul2(make_float2(__uint_as_float(v[c + 2]), __uint_as_float(v[c + 3])), sc2,
                                           make_float2(dd.z, dd.w), make_float2(P[c + 2], P[c + 3]));
                pk[2 * c4] = pack_bf16x2(s0.x, s0.y);
                pk[2 * c4 + 1] = pack_bf16x2(s1.x, s1.y);
            }
            tmem_st32(tDP + lane_base + 64u * h, pk);
            tc_fence_before();
            mbar_arrive(ds_ready + h);
            ++nt;
        }
        // ---------------------------------------------- epilogue: dK, dV rows
        if (ok && nt > 0) {
            ok = mbar_wait(mma_done, 0, wc);
            tc_fence_after();
        }
        const bool has_acc = ok && nt > 0;
        const long long rowoff = ((long long)kpos * p.Hkv + g) * 128 + 64 * h;
#pragma unroll 1
        for (int which = 0; which < 2; ++which) {
            uint32_t v[64];
            if (has_acc) {
                tmem_ld64((which ? tDV : tDK) + lane_base + 64u * h, v);
            } else {
#pragma unroll
                for (int e = 0; e < 64; ++e) v[e] = 0u;
            }
            if (!kvalid) continue;
            void *outp = which ? p.dv : p.dk;
            if (p.out_mode == 0) {
                // 128 contiguous bytes per thread as four 32-byte stores
                __nv_bfloat16 *dst = static_cast<__nv_bfloat16 *>(outp) + rowoff;
#pragma unroll
                for (int q8 = 0; q8 < 4; ++q8) {
                    uint32_t w[8];
#pragma unroll
                    for (int e = 0; e < 8; ++e)
                        w[e] = pack_bf16x2(__uint_as_float(v[16 * q8 + 2 * e]), __uint_as_float(v[16 * q8 + 2 * e + 1]));
                    st_global_v8(dst + 16 * q8, w);
                }
            } else {
                float4 *d4 = reinterpret_cast<float4 *>(static_cast<float *>(outp) + rowoff);
#pragma unroll
                for (int q4 = 0; q4 < 16; ++q4) {
                    float4 x = make_float4(__uint_as_float(v[4 * q4]), __uint_as_float(v[4 * q4 + 1]),
                                           __uint_as_float(v[4 * q4 + 2]), __uint_as_float(v[4 * q4 + 3]));
                    if (p.out_mode == 2) {
                        const float4 o = d4[q4];
                        x.x += o.x;
                        x.y += o.y;
                        x.z += o.z;
                        x.w += o.w;
                    }
                    d4[q4] = x;
                }
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 2) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
    });
    return fn;
}

bool make_map(CUtensorMap *m, const void *ptr, int64_t T, int H, int box_h, int box_t) {
    auto fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[3] = {128, (cuuint64_t)H, (cuuint64_t)(T > 0 ? T : 1)};
    cuuint64_t strides[2] = {128 * 2, (cuuint64_t)H * 128 * 2};
    cuuint32_t box[3] = {64, (cuuint32_t)box_h, (cuuint32_t)box_t};
    cuuint32_t es[3] = {1, 1, 1};
    CUresult rc = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(ptr), dims, strides, box, es,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return rc == CUDA_SUCCESS;
}

}  // namespace

cudaError_t launch_tc_bwd(const TcBwdArgs &a, cudaStream_t st) {
    if (a.n_items <= 0) return cudaSuccess;
    BwdParams p;
    memset(&p, 0, sizeof(p));
    const int G = a.G;
    if (!make_map(&p.tmQ, a.q, a.T, a.Hq, G, kBM / G) || !make_map(&p.tmDO, a.dout, a.T, a.Hq, G, kBM / G) ||
        !make_map(&p.tmK, a.k, a.T, a.Hkv, 1, kBN) || !make_map(&p.tmV, a.v, a.T, a.Hkv, 1, kBN))
        return cudaErrorInvalidValue;
    if ((a.q_orig != nullptr) != (a.dout_orig != nullptr)) return cudaErrorInvalidValue;
    if (a.q_orig) {
        if (!make_map(&p.tmQo, a.q_orig, a.T, a.Hq, G, kBM / G) || !make_map(&p.tmDOo, a.dout_orig, a.T, a.Hq, G, kBM / G))
            return cudaErrorInvalidValue;
        p.qdo_direct = 1;
    }
    if ((a.k_orig != nullptr) != (a.v_orig != nullptr)) return cudaErrorInvalidValue;
    if (a.k_orig) {
        if (!make_map(&p.tmKo, a.k_orig, a.T, a.Hkv, 1, kBN) || !make_map(&p.tmVo, a.v_orig, a.T, a.Hkv, 1, kBN))
            return cudaErrorInvalidValue;
        p.kv_direct = 1;
    }
    p.qtiles = static_cast<const int4 *>(a.qtiles);
    p.kvtiles = static_cast<const int4 *>(a.kvtiles);
    p.items = static_cast<const int4 *>(a.items);
    p.q_off = a.q_off;
    p.n_items = a.n_items;
    p.cp = a.cp;
    p.B = a.B;
    p.G = G;
    int lg = 0;
    while ((1 << lg) < G) ++lg;
    p.log2G = lg;
    p.Hq = a.Hq;
    p.Hkv = a.Hkv;
    p.t0 = a.t0;
    p.t1 = a.t1;
    p.causal = a.causal;
    p.window = a.window;
    if ((a.qbounds != nullptr) != (a.key_lo != nullptr) || (a.key_lo != nullptr) != (a.key_hi != nullptr))
        return cudaErrorInvalidValue;
    p.qbounds = static_cast<const int4 *>(a.qbounds);
    p.key_lo = a.key_lo;
    p.key_hi = a.key_hi;
    p.out_mode = a.out_mode;
    p.scale = a.scale;
    p.scale_log2 = a.scale * 1.4426950408889634f;
    p.tile_ld = a.tile_ld;
    p.dk = a.dk;
    p.dv = a.dv;
    p.status = device_status_ptr();
    p.budget_ns = wait_budget_ns();
    static bool attr_set[128] = {};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev >= 0 && dev < 128 && !attr_set[dev]) {
        for (const void *fn : {(const void *)tc_dkdv_kernel<0>, (const void *)tc_dkdv_kernel<1>,
                               (const void *)tc_dkdv_kernel<2>}) {
            cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
            if (e != cudaSuccess) return e;
        }
        attr_set[dev] = true;
    }
    if (p.qbounds)
        tc_dkdv_kernel<2><<<a.n_items, kThreads, kSmemBytes, st>>>(p);
    else if (p.window >= 0)
        tc_dkdv_kernel<1><<<a.n_items, kThreads, kSmemBytes, st>>>(p);
    else
        tc_dkdv_kernel<0><<<a.n_items, kThreads, kSmemBytes, st>>>(p);
    return cudaGetLastError();
}

}  // namespace ra
