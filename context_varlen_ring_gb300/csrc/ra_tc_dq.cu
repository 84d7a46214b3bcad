// ra_tc_dq.cu -- tensor-core dQ pass of the packed causal varlen ring
// backward (bf16 in, fp32 accumulation, head dim 128) for sm_103a.
//
// What it computes: for each query row, from the saved log-sum-exp and
// D = rowsum(dO o O),
//   P = exp(scale * q K^T - lse),  dS = P o (dO V^T - D),  dQ = scale * dS K
// over the keys of its document that pass the causal test, visiting the
// KV shards in ring order (rank r at step t reads the shard of rank
// s = (r - t) mod cp).  This is the query-side half of the backward of
// FlagScale PR #910's RingAttention (backward_impl); the key side (dK, dV)
// is ra_tc_bwd.cu run without dQ.  Splitting the two sides costs one extra
// S and dP product per tile pair but removes all fp32 atomics on dQ, whose
// reduction bandwidth into L2 (about 3 TB/s) would otherwise bound the
// backward.
//
// GB300 design: one CTA per query tile (128 MMA rows = 128/G tokens x G
// heads of one KV head).  Q and dO arrive by TMA once; Q is copied into
// TMEM by the compute warpgroups (S = Q K^T is a TS-MMA) and its staging
// area becomes a sixth slot of the K/V ring, while dO stays in shared
// memory as the A operand of dP = dO V^T.  K/V tiles are fed by a producer
// warp that publishes each visited KV tile (class and positions) through a
// shared-memory ring.  TMEM: dQ [0,128), S [128,256), dP [256,384), Q
// (bf16) [384,448), dS (bf16) [448,512).  Two compute warpgroups split the
// 128 key columns.
//
// dS has its own TMEM buffer, so dP(j+1) may start as soon as the compute
// groups have loaded dP(j), and the only loop left between products is
// dQ(j) -> (dS buffer free) -> store dS(j+1) -> dQ(j+1).  One thread issues
// a tcgen05.mma only about every 45-60 cycles, close to the 64 cycles an
// M=128 N=128 K=16 product runs, so three warps issue: warp 1 the S
// products, warp 2 dP and warp 3 dQ.
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
constexpr int kSlots = 6;  // slots 0-4 after the Q/dO staging, slot 5 reuses the Q staging
constexpr int kRing = 8;
constexpr uint32_t kHalf = 16384;
constexpr uint32_t kTile = 2 * kHalf;
constexpr uint32_t kOffQ = 0;
constexpr uint32_t kOffDO = kTile;
constexpr uint32_t kOffKV = 2 * kTile;
constexpr uint32_t kOffBar = kOffKV + 5 * kTile;
constexpr uint32_t kSmemBytes = kOffBar + 512 + 1024;

struct DqParams {
    CUtensorMap tmQ, tmK, tmV, tmDO;
    const int4 *qtiles, *kvtiles, *items;
    const int *kv_off;
    int n_items, cp, B, G, log2G, Hq;
    int t0, t1, causal, out_mode;  // out_mode: 0 bf16 store, 1 fp32 store, 2 fp32 +=
    float scale, scale_log2, log2_scale;
    const float *lse, *D;
    long long lse_T;
    void *dq;
    int *status;
    unsigned long long budget_ns;
};

struct QInfo {
    int len, pmin, pmax;
};

__device__ __forceinline__ int classify_q(const QInfo &q, int klen, int kpmin, int kpmax, int causal) {
    if (q.len <= 0 || klen <= 0) return kSkip;
    if (causal && q.pmax < kpmin) return kSkip;
    if (klen == kBN && (!causal || q.pmin >= kpmax)) return kFull;
    return kPartial;
}

__device__ __forceinline__ uint32_t range_bits(int a, int b, int base) {
    const int lo = min(max(a - base, 0), 32), hi = min(max(b - base, 0), 32);
    return (uint32_t)(((1ull << hi) - 1ull) & ~((1ull << lo) - 1ull));
}

__device__ __forceinline__ uint32_t slot_off(uint32_t s) { return s < 5 ? kOffKV + s * kTile : kOffQ; }

__global__ void __launch_bounds__(kThreads, 1) tc_dq_kernel(const __grid_constant__ DqParams p) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_s = smem_u32(smem_raw);
    const uint32_t base_s = (raw_s + 1023u) & ~1023u;
    uint8_t *base = smem_raw + (base_s - raw_s);

    uint64_t *bars = reinterpret_cast<uint64_t *>(base + kOffBar);
    uint64_t *q_full = bars + 0;
    uint64_t *kv_full = bars + 1;      // [kSlots]
    uint64_t *kv_empty = bars + 7;     // [kSlots]
    uint64_t *s_full = bars + 13;      // S done
    uint64_t *s_free = bars + 14;      // S read by both compute groups (256 arrivals)
    uint64_t *dp_full = bars + 15;     // dP done
    uint64_t *dp_free = bars + 16;     // dP read by both compute groups (256 arrivals)
    uint64_t *ds_ready = bars + 17;    // [2] dS half h in TMEM (128 arrivals each)
    uint64_t *dq_done = bars + 19;     // dQ(j) done: dS buffer free
    uint64_t *qc_ready = bars + 20;    // Q copied into TMEM (256 arrivals)
    uint64_t *mma_done = bars + 21;    // all dQ products done
    uint64_t *a_done = bars + 22;      // S issuer drained
    uint64_t *b_done = bars + 41;      // dP issuer drained
    uint64_t *info_full = bars + 23;   // [kRing]
    uint64_t *info_empty = bars + 31;  // [kRing]
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + 39);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(bars + 40);
    int4 *ring = reinterpret_cast<int4 *>(bars + 42);  // [kRing] (bars 42-57)

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int4 ia = __ldg(p.items + 2 * blockIdx.x), ib = __ldg(p.items + 2 * blockIdx.x + 1);
    const int qt = ia.x, g = ia.z, r = ia.w, b = ib.x;
    const int t0 = p.t0 >= 0 ? p.t0 : ib.y;
    const int t1 = p.t0 >= 0 ? p.t1 : ib.z;
    const int4 qa = __ldg(p.qtiles + 2 * qt), qb = __ldg(p.qtiles + 2 * qt + 1);
    // query tile: row0 qa.x, len qa.y, split qa.z, pos0 qa.w, pos1 qb.x, pmin qb.y, pmax qb.z

    if (threadIdx.x == 0) {
        *abort_flag = 0;
        mbar_init(q_full, 1);
        for (int i = 0; i < kSlots; ++i) {
            mbar_init(kv_full + i, 1);
            mbar_init(kv_empty + i, 1);
        }
        mbar_init(s_full, 1);
        mbar_init(s_free, 256);
        mbar_init(dp_full, 1);
        mbar_init(dp_free, 256);
        mbar_init(ds_ready + 0, 128);
        mbar_init(ds_ready + 1, 128);
        mbar_init(dq_done, 1);
        mbar_init(qc_ready, 256);
        mbar_init(mma_done, 1);
        mbar_init(a_done, 1);
        mbar_init(b_done, 1);
        for (int i = 0; i < kRing; ++i) {
            mbar_init(info_full + i, 1);
            mbar_init(info_empty + i, 3 + 256);
        }
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
    const uint32_t tDQ = tmem, tS = tmem + 128, tDP = tmem + 256, tQ = tmem + 384, tDS = tmem + 448;

    auto read_info = [&](uint32_t jt, int4 &e) -> bool {
        const uint32_t slot = jt % kRing;
        if (!mbar_wait(info_full + slot, (jt / kRing) & 1u, wc)) return false;
        e = ring[slot];
        mbar_arrive(info_empty + slot);
        return true;
    };

    if (warp < 4) {
        asm volatile("setmaxnreg.dec.sync.aligned.u32 56;\n" ::: "memory");
        if (warp == 0) {
            // -------------------------------------------- producer
            const QInfo q{qa.y, qb.y, qb.z};
            if (lane == 0) {
                tma_prefetch_desc(&p.tmQ);
                tma_prefetch_desc(&p.tmDO);
                tma_prefetch_desc(&p.tmK);
                tma_prefetch_desc(&p.tmV);
                const int hq0 = g * p.G;
                mbar_arrive_expect_tx(q_full, 2 * kTile);
                tma_load_3d(base + kOffQ, &p.tmQ, q_full, 0, hq0, qa.x);
                tma_load_3d(base + kOffQ + kHalf, &p.tmQ, q_full, 64, hq0, qa.x);
                tma_load_3d(base + kOffDO, &p.tmDO, q_full, 0, hq0, qa.x);
                tma_load_3d(base + kOffDO + kHalf, &p.tmDO, q_full, 64, hq0, qa.x);
            }
            uint32_t u = 0, jt = 0;
            int ok = 1;
            for (int t = t0; t < t1 && ok; ++t) {
                int s = (r - t) % p.cp;
                if (s < 0) s += p.cp;
                const int o = s * (p.B + 1) + b;
                const int lo = __ldg(p.kv_off + o), hi = __ldg(p.kv_off + o + 1);
                for (int bi = lo; bi < hi && ok; bi += 32) {
                    const int idx = bi + lane;
                    int4 ka = make_int4(0, 0, 0, 0), kb = make_int4(0, 0, 0, 0);
                    int c = kSkip;
                    if (idx < hi) {
                        ka = __ldg(p.kvtiles + 2 * idx);
                        kb = __ldg(p.kvtiles + 2 * idx + 1);
                        c = classify_q(q, ka.y, kb.y, kb.z, p.causal);
                    }
                    uint32_t vis = __ballot_sync(0xffffffffu, c != kSkip);
                    while (vis && ok) {
                        const int src = __ffs(vis) - 1;
                        vis &= vis - 1;
                        const int row0 = __shfl_sync(0xffffffffu, ka.x, src);
                        const int len = __shfl_sync(0xffffffffu, ka.y, src);
                        const int split = __shfl_sync(0xffffffffu, ka.z, src);
                        const int pos0 = __shfl_sync(0xffffffffu, ka.w, src);
                        const int pos1 = __shfl_sync(0xffffffffu, kb.x, src);
                        const int cc = __shfl_sync(0xffffffffu, c, src);
                        if (lane == 0) {
                            const uint32_t e = jt % kRing;
                            if (!mbar_wait(info_empty + e, ((jt / kRing) & 1u) ^ 1u, wc)) ok = 0;
                            if (ok) {
                                ring[e] = make_int4(cc, len | (split << 16), pos0, pos1);
                                mbar_arrive(info_full + e);
                            }
                            for (int kv = 0; kv < 2 && ok; ++kv, ++u) {
                                const uint32_t slot = u % kSlots, ph = (u / kSlots) & 1u;
                                if (!mbar_wait(kv_empty + slot, ph ^ 1u, wc)) {
                                    ok = 0;
                                    break;
                                }
                                // slot 5 is the Q staging: free once Q is copied into TMEM
                                if (u == 5 && !mbar_wait(qc_ready, 0, wc)) {
                                    ok = 0;
                                    break;
                                }
                                uint8_t *dst = base + slot_off(slot);
                                const CUtensorMap *m = kv ? &p.tmV : &p.tmK;
                                mbar_arrive_expect_tx(kv_full + slot, kTile);
                                tma_load_3d(dst, m, kv_full + slot, 0, g, row0);
                                tma_load_3d(dst + kHalf, m, kv_full + slot, 64, g, row0);
                            }
                        }
                        ok = __shfl_sync(0xffffffffu, ok, 0);
                        ++jt;
                    }
                }
            }
            if (lane == 0) {
                if (ok) {
                    const uint32_t e = jt % kRing;
                    if (mbar_wait(info_empty + e, ((jt / kRing) & 1u) ^ 1u, wc)) {
                        ring[e] = make_int4(1 << 4, 0, 0, 0);
                        mbar_arrive(info_full + e);
                    }
                }
                volatile int local_abort = 0;
                const WaitCtl drain{&local_abort, p.status, p.budget_ns};
                (void)mbar_wait(q_full, 0, drain);
                for (uint32_t x = (u > kSlots ? u - kSlots : 0); x < u; ++x)
                    (void)mbar_wait(kv_full + (x % kSlots), (x / kSlots) & 1u, drain);
            }
        } else if (lane == 0) {
            // -------------------------------------------- MMA issuers (warps 1-3)
            constexpr uint32_t id_s = idesc_bf16_f32(128, 128, 0, 0);  // S, dP: A and B K-major
            constexpr uint32_t id_q = idesc_bf16_f32(128, 128, 0, 1);  // dQ: B MN-major
            // K-major SW128 operand: 16-element k-step ks at (ks / 4) * kHalf + (ks % 4) * 32
            auto kstep = [](int ks) -> uint32_t { return (((ks >> 2) * kHalf + (ks & 3) * 32u) >> 4); };
            auto kv_par = [](uint32_t u) { return (u / kSlots) & 1u; };
            auto wait = [&](uint64_t *bar, uint32_t par) -> bool {
                const bool r = mbar_wait(bar, par, wc);
                tc_fence_after();
                return r;
            };
            uint64_t *drain_bar = warp == 1 ? a_done : (warp == 2 ? b_done : mma_done);
            if (warp == 1) {
                // S(j) = Q K(j)^T (Q from TMEM) once both groups have read S(j-1)
                bool ok = wait(qc_ready, 0);
                for (uint32_t j = 0; ok; ++j) {
                    int4 e;
                    if (!read_info(j, e) || (e.x & 16)) break;
                    if (j > 0 && !wait(s_free, (j - 1) & 1u)) break;
                    const uint32_t ku = 2 * j;
                    if (!wait(kv_full + ku % kSlots, kv_par(ku))) break;
                    const uint64_t d0 = sdesc_sw128(base_s + slot_off(ku % kSlots), 16, 1024);
#pragma unroll
                    for (int ks = 0; ks < 8; ++ks) tc_mma_ts(tS, tQ + 8u * ks, d0 + kstep(ks), id_s, ks > 0);
                    tc_commit(s_full);
                }
            } else if (warp == 2) {
                // dP(j) = dO V(j)^T (dO from shared memory) once dP(j-1) was read
                const uint64_t a0 = sdesc_sw128(base_s + kOffDO, 16, 1024);
                bool ok = wait(q_full, 0);
                for (uint32_t j = 0; ok; ++j) {
                    int4 e;
                    if (!read_info(j, e) || (e.x & 16)) break;
                    if (j > 0 && !wait(dp_free, (j - 1) & 1u)) break;
                    const uint32_t vu = 2 * j + 1;
                    if (!wait(kv_full + vu % kSlots, kv_par(vu))) break;
                    const uint64_t d0 = sdesc_sw128(base_s + slot_off(vu % kSlots), 16, 1024);
#pragma unroll
                    for (int ks = 0; ks < 8; ++ks) tc_mma_ss(tDP, a0 + kstep(ks), d0 + kstep(ks), id_s, ks > 0);
                    tc_commit(dp_full);
                    tc_commit(kv_empty + vu % kSlots);  // V only feeds dP
                }
            } else {
                // dQ += dS_h(j) K(j)_h: keys [64h, 64h + 64) = K rows (MN-major: d
                // contiguous), A = group h's dS at dS columns [32h, 32h + 32)
                for (uint32_t j = 0;; ++j) {
                    int4 e;
                    if (!read_info(j, e) || (e.x & 16)) break;
                    const uint32_t kslot = (2 * j) % kSlots;
                    const uint64_t d0 = sdesc_sw128(base_s + slot_off(kslot), kHalf, 1024);
                    bool okh = true;
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        if (!wait(ds_ready + h, j & 1u)) {
                            okh = false;
                            break;
                        }
#pragma unroll
                        for (int k = 0; k < 4; ++k)
                            tc_mma_ts(tDQ, tDS + 32u * h + 8u * k, d0 + ((8192u * h + 2048u * k) >> 4), id_q,
                                      (j > 0 || h > 0 || k > 0));
                    }
                    if (!okh) break;
                    tc_commit(dq_done);
                    tc_commit(kv_empty + kslot);  // K(j) done (S(j) finished before dS(j))
                }
            }
            tc_commit(drain_bar);
            volatile int local_abort = 0;
            const WaitCtl drain{&local_abort, p.status, p.budget_ns};
            (void)mbar_wait(drain_bar, 0, drain);
        }
    } else {
        asm volatile("setmaxnreg.inc.sync.aligned.u32 224;\n" ::: "memory");
        // ------------------------------------------------ compute warpgroups
        // Warpgroup h owns key columns [64h, 64h + 64) of S and dP and output
        // columns [64h, 64h + 64) of dQ; thread m owns query row m.
        const int h = (warp >= 8) ? 1 : 0;
        const int m = (threadIdx.x - 128) & 127;
        const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
        const int G = p.G;
        const int tok = m >> p.log2G, head = g * G + (m & (G - 1));
        const bool valid = tok < qa.y;
        const int qpos = tok < qa.z ? qa.w + tok : qb.x + (tok - qa.z);
        // P' = scale * P = exp2(s * scale * log2(e) + bias), bias = log2(scale) - lse * log2(e)
        float bias = -INFINITY, Dm = 0.f;
        if (valid) {
            const float l = __ldg(p.lse + (long long)head * p.lse_T + qpos);
            bias = (l == -INFINITY) ? -INFINITY : p.log2_scale - l * 1.4426950408889634f;
            Dm = __ldg(p.D + (long long)head * p.lse_T + qpos);
        }
        bool ok = mbar_wait(q_full, 0, wc);
        if (ok) {
            // copy this group's d half of the Q row into TMEM (bf16 pairs);
            // swizzled 128-byte rows: chunk c of row m at (c ^ (m & 7)) * 16
            const uint8_t *qrow = base + kOffQ + h * kHalf + (m >> 3) * 1024 + (m & 7) * 128;
#pragma unroll
            for (int part = 0; part < 2; ++part) {
                uint32_t w[16];
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    const int ch = 4 * part + c;
                    const uint4 x = *reinterpret_cast<const uint4 *>(qrow + ((ch ^ (m & 7)) << 4));
                    w[4 * c] = x.x;
                    w[4 * c + 1] = x.y;
                    w[4 * c + 2] = x.z;
                    w[4 * c + 3] = x.w;
                }
                tmem_st16(tQ + lane_base + 32u * h + 16u * part, w);
            }
        }
        tc_fence_before();
        mbar_arrive(qc_ready);
        uint32_t nd = 0;
        for (uint32_t jt = 0; ok; ++jt) {
            int4 e;
            if (!read_info(jt, e)) {
                ok = false;
                break;
            }
            if (e.x & 16) break;
            const int cls = e.x & 3;
            if (!mbar_wait(s_full, jt & 1u, wc)) {
                ok = false;
                break;
            }
            tc_fence_after();
            uint32_t v[64];
            tmem_ld64(tS + lane_base + 64u * h, v);
            tc_fence_before();
            mbar_arrive(s_free);
            float P[64];
#pragma unroll
            for (int c = 0; c < 64; c += 2) {
                const float2 x = fma2(make_float2(__uint_as_float(v[c]), __uint_as_float(v[c + 1])),
                                      make_float2(p.scale_log2, p.scale_log2), make_float2(bias, bias));
                P[c] = ex2_approx(x.x);
                P[c + 1] = ex2_approx(x.y);
            }
            if (cls == kPartial) {
                const int kt_len = e.y & 0xffff, kt_split = e.y >> 16, kt_pos0 = e.z, kt_pos1 = e.w;
                int lim1, lim2;
                if (p.causal) {
                    lim1 = min(max(qpos - kt_pos0 + 1, 0), kt_split);
                    lim2 = min(max(qpos - kt_pos1 + kt_split + 1, kt_split), kt_len);
                } else {
                    lim1 = kt_split;
                    lim2 = kt_len;
                }
                uint32_t wm[2];
#pragma unroll
                for (int ch = 0; ch < 2; ++ch) {
                    const int cb = 64 * h + 32 * ch;
                    wm[ch] = range_bits(0, lim1, cb) | range_bits(kt_split, lim2, cb);
                }
#pragma unroll
                for (int c = 0; c < 64; ++c) P[c] = ((wm[c >> 5] >> (c & 31)) & 1u) ? P[c] : 0.f;
            }
            if (!mbar_wait(dp_full, jt & 1u, wc)) {
                ok = false;
                break;
            }
            tc_fence_after();
            tmem_ld64(tDP + lane_base + 64u * h, v);
            tc_fence_before();
            mbar_arrive(dp_free);
            uint32_t pk[32];
#pragma unroll
            for (int c2 = 0; c2 < 32; ++c2) {
                const float2 d = sub_mul2(make_float2(__uint_as_float(v[2 * c2]), __uint_as_float(v[2 * c2 + 1])),
                                          make_float2(Dm, Dm), make_float2(P[2 * c2], P[2 * c2 + 1]));
                pk[c2] = pack_bf16x2(d.x, d.y);
            }
            // the dS buffer is free once dQ(jt - 1) has completed
            if (jt > 0 && !mbar_wait(dq_done, (jt - 1) & 1u, wc)) {
                ok = false;
                break;
            }
            tc_fence_after();
            tmem_st32(tDS + lane_base + 32u * h, pk);
            tc_fence_before();
            mbar_arrive(ds_ready + h);
            ++nd;
        }
        // ------------------------------------------------ epilogue
        // the MMA thread's final commit covers every dQ MMA
        if (ok && nd > 0) {
            ok = mbar_wait(mma_done, 0, wc);
            tc_fence_after();
        }
        uint32_t v[64];
        if (ok && nd > 0) {
            tmem_ld64(tDQ + lane_base + 64u * h, v);
        } else {
#pragma unroll
            for (int c = 0; c < 64; ++c) v[c] = 0u;
        }
        if (valid) {
            const long long e0 = ((long long)qpos * p.Hq + head) * 128 + 64 * h;
            if (p.out_mode == 0) {
                uint4 *dst = reinterpret_cast<uint4 *>(static_cast<__nv_bfloat16 *>(p.dq) + e0);
#pragma unroll
                for (int q4 = 0; q4 < 8; ++q4) {
                    uint4 w;
                    w.x = pack_bf16x2(__uint_as_float(v[8 * q4 + 0]), __uint_as_float(v[8 * q4 + 1]));
                    w.y = pack_bf16x2(__uint_as_float(v[8 * q4 + 2]), __uint_as_float(v[8 * q4 + 3]));
                    w.z = pack_bf16x2(__uint_as_float(v[8 * q4 + 4]), __uint_as_float(v[8 * q4 + 5]));
                    w.w = pack_bf16x2(__uint_as_float(v[8 * q4 + 6]), __uint_as_float(v[8 * q4 + 7]));
                    dst[q4] = w;
                }
            } else {
                float4 *dst = reinterpret_cast<float4 *>(static_cast<float *>(p.dq) + e0);
#pragma unroll
                for (int q4 = 0; q4 < 16; ++q4) {
                    float4 x = make_float4(__uint_as_float(v[4 * q4]), __uint_as_float(v[4 * q4 + 1]),
                                           __uint_as_float(v[4 * q4 + 2]), __uint_as_float(v[4 * q4 + 3]));
                    if (p.out_mode == 2) {
                        const float4 o = dst[q4];
                        x.x += o.x;
                        x.y += o.y;
                        x.z += o.z;
                        x.w += o.w;
                    }
                    dst[q4] = x;
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

cudaError_t launch_tc_dq(const TcDqArgs &a, cudaStream_t st) {
    if (a.n_items <= 0) return cudaSuccess;
    DqParams p;
    memset(&p, 0, sizeof(p));
    const int G = a.G;
    if (!make_map(&p.tmQ, a.q, a.T, a.Hq, G, kBM / G) || !make_map(&p.tmDO, a.dout, a.T, a.Hq, G, kBM / G) ||
        !make_map(&p.tmK, a.k, a.T, a.Hkv, 1, kBN) || !make_map(&p.tmV, a.v, a.T, a.Hkv, 1, kBN))
        return cudaErrorInvalidValue;
    p.qtiles = static_cast<const int4 *>(a.qtiles);
    p.kvtiles = static_cast<const int4 *>(a.kvtiles);
    p.items = static_cast<const int4 *>(a.items);
    p.kv_off = a.kv_off;
    p.n_items = a.n_items;
    p.cp = a.cp;
    p.B = a.B;
    p.G = G;
    int lg = 0;
    while ((1 << lg) < G) ++lg;
    p.log2G = lg;
    p.Hq = a.Hq;
    p.t0 = a.t0;
    p.t1 = a.t1;
    p.causal = a.causal;
    p.out_mode = a.out_mode;
    p.scale = a.scale;
    p.scale_log2 = a.scale * 1.4426950408889634f;
    p.log2_scale = std::log2(a.scale);
    p.lse = a.lse;
    p.D = a.D;
    p.lse_T = a.lse_T;
    p.dq = a.dq;
    p.status = device_status_ptr();
    p.budget_ns = wait_budget_ns();
    static bool attr_set[128] = {};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev >= 0 && dev < 128 && !attr_set[dev]) {
        cudaError_t e = cudaFuncSetAttribute(tc_dq_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
        if (e != cudaSuccess) return e;
        cudaFuncAttributes fa;
        e = cudaFuncGetAttributes(&fa, tc_dq_kernel);
        if (e != cudaSuccess) return e;
        if (fa.numRegs < 168) return cudaErrorInvalidConfiguration;  // setmaxnreg split needs 168
        attr_set[dev] = true;
    }
    tc_dq_kernel<<<a.n_items, kThreads, kSmemBytes, st>>>(p);
    return cudaGetLastError();
}

}  // namespace ra
