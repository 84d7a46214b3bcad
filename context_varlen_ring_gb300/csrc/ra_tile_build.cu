// ra_tile_build.cu -- the tile tables of one partial-attention call built on
// the device, from DEVICE segment boundaries and positions, so that a ring
// step whose positions live on the GPU needs no host round trip (and the
// call can be captured in a CUDA graph).
//
// The tiling is the host planner's, row for row: a tile is up to R
// consecutive rows of one segment whose positions form at most two runs of
// consecutive integers, taken greedily from the segment start (the first
// run as long as it lasts, then a second run, until R rows).  Work items
// pair consecutive query tiles of a segment, replicated over the KV heads,
// in KV-head-major order.
//
// One CTA of 1024 threads: warp w walks segments w, w + 32, ... (pass 1
// counts each segment's tiles, pass 2 writes them at offsets from a block
// scan over the segments).  The walk of a tile takes one ballot per 32 rows
// to find the position breaks.
#include <cuda_runtime.h>

#include <cstdint>

#include "ra_dev.cuh"
#include "ra_internal.h"
#include "ra_kernels.h"

namespace ra {

namespace {

constexpr int kBuildThreads = 1024;

__device__ __forceinline__ int posv(const int32_t *pos, int64_t i) { return pos ? pos[i] : (int)i; }

// The greedy tile starting at row s of a segment ending at hi: its length and
// the length of its first run (split == len for a one-run tile).  Warp-wide;
// every lane returns the same values.
__device__ __forceinline__ void walk_tile(const int32_t *pos, int64_t s, int64_t hi, int R, int lane, int &len,
                                          int &split) {
    const int64_t lim = s + R < hi ? s + R : hi;
    int64_t first = lim, second = lim;
    for (int64_t base = s + 1; base < lim && second == lim; base += 32) {
        const int64_t i = base + lane;
        const bool brk = i < lim && posv(pos, i) != posv(pos, i - 1) + 1;
        uint32_t m = __ballot_sync(0xffffffffu, brk);
        while (m && second == lim) {
            const int64_t j = base + __ffs(m) - 1;
            m &= m - 1;
            if (first == lim)
                first = j;
            else
                second = j;
        }
    }
    len = (int)(second - s);
    split = (int)(first - s < len ? first - s : len);
}

struct Side {
    const int32_t *cu, *pos;
    int64_t T;
    int R;
    Tile *tiles;
    int32_t *off;  // [nseg + 2]
    int32_t *cnt;  // [nseg] scratch
};

__global__ void __launch_bounds__(kBuildThreads) tile_build_kernel(Side qs, Side ks, int nseg, int Hkv,
                                                                    int check_pos, WorkItem *items, int *n_items,
                                                                    int *sched, int32_t *pair_off, int *status) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nw = blockDim.x >> 5;
    __shared__ int bad;
    __shared__ int64_t partial[kBuildThreads / 32];
    if (threadIdx.x == 0) bad = 0;
    __syncthreads();
    // segment boundaries must start at 0, never decrease and end at T
    for (int side = 0; side < 2; ++side) {
        const Side &S = side ? ks : qs;
        for (int b = threadIdx.x; b <= nseg; b += blockDim.x) {
            const int c = S.cu[b];
            if ((b == 0 && c != 0) || (b > 0 && c < S.cu[b - 1]) || (b == nseg && c != S.T)) bad = 1;
        }
        // with a sliding window the kernels add the window to positions in
        // 32-bit arithmetic: positions must lie in [0, 2^30)
        if (check_pos && S.pos)
            for (int64_t i = threadIdx.x; i < S.T; i += blockDim.x)
                if (S.pos[i] < 0 || S.pos[i] >= (1 << 30)) bad = 1;
    }
    __syncthreads();
    if (bad) {
        // no work: the count and the work counter the forward claims from
        // are still written, so that it finds nothing to do
        if (threadIdx.x == 0) {
            *n_items = 0;
            sched[0] = 0;
            sched[1] = 0;
            dev::record_status(status, RA_ERR_DEVICE_BOUNDS);
        }
        return;
    }
    // pass 1: tiles per segment
    for (int side = 0; side < 2; ++side) {
        const Side &S = side ? ks : qs;
        for (int b = warp; b < nseg; b += nw) {
            int n = 0;
            for (int64_t s = S.cu[b]; s < S.cu[b + 1];) {
                int len, split;
                walk_tile(S.pos, s, S.cu[b + 1], S.R, lane, len, split);
                s += len;
                ++n;
            }
            if (lane == 0) S.cnt[b] = n;
        }
    }
    __syncthreads();
    // exclusive scans over the segments: tile offsets of both sides and the
    // offsets of the query-tile pairs (one thread per chunk of segments)
    auto scan = [&](const int32_t *in, int32_t *out, bool pairs) {
        const int per = (nseg + blockDim.x - 1) / blockDim.x;
        const int a = threadIdx.x * per, e = min(nseg, a + per);
        int64_t local = 0;
        for (int b = a; b < e; ++b) local += pairs ? (in[b] + 1) / 2 : in[b];
        // block-wide exclusive scan of the per-thread sums (warp shuffles, then the warp totals)
        int64_t x = local;
        for (int o = 1; o < 32; o <<= 1) {
            const int64_t y = __shfl_up_sync(0xffffffffu, x, o);
            if (lane >= o) x += y;
        }
        if (lane == 31) partial[warp] = x;
        __syncthreads();
        if (warp == 0) {
            int64_t w = lane < nw ? partial[lane] : 0;
            for (int o = 1; o < 32; o <<= 1) {
                const int64_t y = __shfl_up_sync(0xffffffffu, w, o);
                if (lane >= o) w += y;
            }
            if (lane < nw) partial[lane] = w;
        }
        __syncthreads();
        int64_t run = x - local + (warp > 0 ? partial[warp - 1] : 0);
        for (int b = a; b < e; ++b) {
            out[b] = (int32_t)run;
            run += pairs ? (in[b] + 1) / 2 : in[b];
        }
        if (threadIdx.x == blockDim.x - 1) {
            out[nseg] = (int32_t)run;
            if (!pairs) out[nseg + 1] = (int32_t)run;
        }
        __syncthreads();
    };
    scan(qs.cnt, qs.off, false);
    scan(ks.cnt, ks.off, false);
    scan(qs.cnt, pair_off, true);
    const int n_pairs = pair_off[nseg];
    // pass 2: write the tiles, then the items
    for (int side = 0; side < 2; ++side) {
        const Side &S = side ? ks : qs;
        for (int b = warp; b < nseg; b += nw) {
            int idx = S.off[b];
            for (int64_t s = S.cu[b]; s < S.cu[b + 1];) {
                int len, split;
                walk_tile(S.pos, s, S.cu[b + 1], S.R, lane, len, split);
                if (lane == 0) {
                    const int p0 = posv(S.pos, s);
                    const bool two = split < len;
                    const int p1 = two ? posv(S.pos, s + split) : p0 + split;
                    Tile t;
                    t.row0 = (int32_t)s;
                    t.len = len;
                    t.split = split;
                    t.pos0 = p0;
                    t.pos1 = p1;
                    t.pmin = two ? min(p0, p1) : p0;
                    t.pmax = two ? max(p0 + split - 1, p1 + (len - split) - 1) : p0 + len - 1;
                    t.seg = b;
                    S.tiles[idx] = t;
                }
                ++idx;
                s += len;
            }
        }
    }
    for (int b = warp; b < nseg; b += nw) {
        const int qa = qs.off[b], qe = qs.off[b + 1], po = pair_off[b];
        for (int i = qa + 2 * lane; i < qe; i += 64) {
            const int pr = po + (i - qa) / 2;
            for (int g = 0; g < Hkv; ++g)
                items[(int64_t)g * n_pairs + pr] = WorkItem{i, i + 1 < qe ? i + 1 : -1, g, 0, b, 0, 1, 0};
        }
    }
    if (threadIdx.x == 0) {
        *n_items = n_pairs * Hkv;
        sched[0] = 0;
        sched[1] = 0;
    }
}

}  // namespace

cudaError_t launch_tile_build(const DevTileArgs &a, cudaStream_t st) {
    Side q{a.cu_q, a.q_pos, a.Tq, a.q_rows, static_cast<Tile *>(a.qtiles), a.q_off, a.q_cnt};
    Side k{a.cu_k, a.k_pos, a.Tk, kBN, static_cast<Tile *>(a.kvtiles), a.kv_off, a.k_cnt};
    tile_build_kernel<<<1, kBuildThreads, 0, st>>>(q, k, a.nseg, a.Hkv, a.check_pos, static_cast<WorkItem *>(a.items),
                                                   a.n_items, a.sched, a.pair_off, device_status_ptr());
    return cudaGetLastError();
}

}  // namespace ra
