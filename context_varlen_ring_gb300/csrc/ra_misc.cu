// ra_misc.cu -- bandwidth-bound kernels: zigzag permute / unpermute (the
// reordering the maxtext PR #1133 review asks the framework to do around
// load-balanced CP attention), the n-way LSE merge of ring partials, the
// backward's row-dot preprocess and fp32 -> output casts; plus the device
// status word and the wait-guard self-test.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <algorithm>

#include <cmath>
#include <cstdint>

#include "ra_dev.cuh"
#include "ra_kernels.h"

namespace ra {

__device__ int g_ra_status;

int *device_status_ptr() {
    static int *ptrs[128] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 128) return nullptr;
    if (!ptrs[dev]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_ra_status) != cudaSuccess) return nullptr;
        ptrs[dev] = static_cast<int *>(p);
    }
    return ptrs[dev];
}

uint64_t wait_budget_ns() { return 2000000000ull; }

static inline int num_sms() {
    static int sms[128] = {};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 0 || dev >= 128) return 148;
    if (!sms[dev]) {
        int v = 0;
        cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev);
        sms[dev] = v > 0 ? v : 148;
    }
    return sms[dev];
}

// ------------------------------------------------------------------ permute
struct PermJobs {
    PermJob j[4];
    int n;
};

// One warp per row; each lane moves vectors of type V (16 B when every row
// and pointer allows it), four in flight per lane before the stores.
template <typename V>
__global__ void __launch_bounds__(256) permute_kernel(PermJobs jobs, const int32_t *__restrict__ perm, int64_t T,
                                                       int inverse, int *status) {
    const int lane = threadIdx.x & 31;
    const int64_t warp = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    const int64_t nwarps = (int64_t)gridDim.x * (blockDim.x >> 5);
    for (int64_t i = warp; i < T; i += nwarps) {
        const int32_t p = __ldg(perm + i);
        if (p < 0 || (int64_t)p >= T) {
            if (lane == 0) dev::record_status(status, RA_ERR_DEVICE_BOUNDS);
            continue;
        }
        const int64_t srow = inverse ? i : (int64_t)p;
        const int64_t drow = inverse ? (int64_t)p : i;
        for (int jb = 0; jb < jobs.n; ++jb) {
            if (jobs.j[jb].only && !__ldg(jobs.j[jb].only + i)) continue;
            const int64_t nvec = jobs.j[jb].row_bytes / (int64_t)sizeof(V);
            const V *__restrict__ src = reinterpret_cast<const V *>(jobs.j[jb].src) + srow * nvec;
            V *__restrict__ dst = reinterpret_cast<V *>(jobs.j[jb].dst) + drow * nvec;
            for (int64_t c0 = lane; c0 < nvec; c0 += 128) {
                V tmp[4];
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    const int64_t c = c0 + u * 32;
                    if (c < nvec) tmp[u] = src[c];
                }
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    const int64_t c = c0 + u * 32;
                    if (c < nvec) dst[c] = tmp[u];
                }
            }
        }
    }
}

cudaError_t launch_permute(const PermJob *jobs, int njobs, const int32_t *perm, int64_t T, int inverse,
                           cudaStream_t st) {
    if (T <= 0 || njobs <= 0) return cudaSuccess;
    if (njobs > 4) return cudaErrorInvalidValue;
    PermJobs pj{};
    pj.n = njobs;
    int vec = 16;
    for (int i = 0; i < njobs; ++i) {
        pj.j[i] = jobs[i];
        auto al = [](const void *p, int64_t rb, int a) {
            return (reinterpret_cast<uintptr_t>(p) % a) == 0 && (rb % a) == 0;
        };
        while (vec > 1 && !(al(jobs[i].src, jobs[i].row_bytes, vec) && al(jobs[i].dst, jobs[i].row_bytes, vec)))
            vec >>= 2;
    }
    const int64_t want = (T + 7) / 8;
    const int blocks = (int)std::min<int64_t>(want, (int64_t)num_sms() * 8);
    int *status = device_status_ptr();
    if (vec == 16)
        permute_kernel<uint4><<<blocks, 256, 0, st>>>(pj, perm, T, inverse, status);
    else if (vec == 4)
        permute_kernel<uint32_t><<<blocks, 256, 0, st>>>(pj, perm, T, inverse, status);
    else
        permute_kernel<uint8_t><<<blocks, 256, 0, st>>>(pj, perm, T, inverse, status);
    return cudaGetLastError();
}

__global__ void unpermute_cols_kernel(const float *__restrict__ y, float *__restrict__ x,
                                      const int32_t *__restrict__ perm, int64_t T, int H, int *status) {
    const int64_t n = T * H;
    for (int64_t w = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; w < n; w += (int64_t)gridDim.x * blockDim.x) {
        const int64_t h = w / T, i = w % T;
        const int32_t p = __ldg(perm + i);
        if (p < 0 || (int64_t)p >= T) {
            dev::record_status(status, RA_ERR_DEVICE_BOUNDS);
            continue;
        }
        x[h * T + p] = y[w];
    }
}

cudaError_t launch_unpermute_cols(const float *y, float *x, const int32_t *perm, int64_t T, int H,
                                  cudaStream_t st) {
    if (T <= 0 || H <= 0) return cudaSuccess;
    const int64_t n = T * H;
    const int blocks = (int)std::min<int64_t>((n + 255) / 256, (int64_t)num_sms() * 8);
    unpermute_cols_kernel<<<blocks, 256, 0, st>>>(y, x, perm, T, H, device_status_ptr());
    return cudaGetLastError();
}

// ------------------------------------------------------------------ merge
struct MergePtrs {
    const float *o[kMaxMergeParts];
    const float *l[kMaxMergeParts];
};

// One warp per (token, head) row.  M = max lse_p, L = M + log sum exp(lse_p - M),
// out = sum_p exp(lse_p - L) out_p.  Lane p holds the weight of part p (and
// p + 32); every lane runs the same loops (the weights are broadcast with
// full-warp shuffles), and a lane whose 4 elements lie past d only skips its
// loads and stores.  Parts are read four at a time so that each warp keeps
// several 16-byte loads in flight.
template <typename TOut>
__global__ void __launch_bounds__(256) merge_kernel(MergePtrs P, int n, int64_t Tq, int Hq, int d, TOut *out,
                                                     float *lse_out) {
    const int lane = threadIdx.x & 31;
    const int64_t rows = Tq * Hq;
    const int64_t nw = (int64_t)gridDim.x * (blockDim.x >> 5);
    for (int64_t w = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); w < rows; w += nw) {
        const int64_t t = w / Hq;
        const int h = (int)(w % Hq);
        const int64_t li = (int64_t)h * Tq + t;
        float la = lane < n ? P.l[lane][li] : -INFINITY;
        float lb = lane + 32 < n ? P.l[lane + 32][li] : -INFINITY;
        float M = fmaxf(la, lb);
#pragma unroll
        for (int s = 16; s; s >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, s));
        float L = -INFINITY;
        if (M != -INFINITY) {
            float sm = (la == -INFINITY ? 0.f : expf(la - M)) + (lb == -INFINITY ? 0.f : expf(lb - M));
#pragma unroll
            for (int s = 16; s; s >>= 1) sm += __shfl_xor_sync(0xffffffffu, sm, s);
            L = M + logf(sm);
        }
        const float wa = (M == -INFINITY || la == -INFINITY) ? 0.f : expf(la - L);
        const float wb = (M == -INFINITY || lb == -INFINITY) ? 0.f : expf(lb - L);
        for (int c0 = 0; c0 < d; c0 += 128) {
            const int c = c0 + lane * 4;
            const bool act = c < d;
            float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
            for (int p0 = 0; p0 < n; p0 += 4) {
                float wq[4];
                float4 x[4];
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    const int p = p0 + u;
                    const float src = p < 32 ? wa : wb;
                    wq[u] = __shfl_sync(0xffffffffu, src, p & 31);
                    if (p >= n) wq[u] = 0.f;
                    x[u] = (act && wq[u] != 0.f) ? *reinterpret_cast<const float4 *>(P.o[p] + w * d + c)
                                                 : make_float4(0.f, 0.f, 0.f, 0.f);
                }
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    acc.x += wq[u] * x[u].x;
                    acc.y += wq[u] * x[u].y;
                    acc.z += wq[u] * x[u].z;
                    acc.w += wq[u] * x[u].w;
                }
            }
            if (act) {
                if constexpr (sizeof(TOut) == 4) {
                    *reinterpret_cast<float4 *>(reinterpret_cast<float *>(out) + w * d + c) = acc;
                } else {
                    uint2 pk;
                    pk.x = dev::pack_bf16x2(acc.x, acc.y);
                    pk.y = dev::pack_bf16x2(acc.z, acc.w);
                    *reinterpret_cast<uint2 *>(reinterpret_cast<__nv_bfloat16 *>(out) + w * d + c) = pk;
                }
            }
        }
        if (lse_out && lane == 0) lse_out[li] = L;
    }
}

cudaError_t launch_merge(int n, const float *const *outs, const float *const *lses, int64_t Tq, int Hq, int d,
                         void *out, int out_dtype, float *lse_out, cudaStream_t st) {
    if (Tq <= 0) return cudaSuccess;
    MergePtrs P{};
    for (int p = 0; p < n; ++p) {
        P.o[p] = outs[p];
        P.l[p] = lses[p];
    }
    const int64_t rows = Tq * Hq;
    const int blocks = (int)std::min<int64_t>((rows + 7) / 8, (int64_t)num_sms() * 16);
    if (out_dtype == RA_FP32)
        merge_kernel<float><<<blocks, 256, 0, st>>>(P, n, Tq, Hq, d, static_cast<float *>(out), lse_out);
    else
        merge_kernel<__nv_bfloat16><<<blocks, 256, 0, st>>>(P, n, Tq, Hq, d, static_cast<__nv_bfloat16 *>(out),
                                                            lse_out);
    return cudaGetLastError();
}

// ------------------------------------------------------------------ permute + rowdot
// Backward preprocess in one pass over the rows (bf16, head dim 128): the
// jobs (Q, K, V) are permuted as in permute_kernel, dO is permuted too, and
// D[h, p] = sum_c dO[p, h, c] * O[p, h, c] (fp32, exact bf16 products) is
// taken from the same dO reads at the original row p.  A head is 16 vectors
// of 8 elements, so each 16-lane half-warp holds one head per step and the
// dot product is a 4-step shuffle reduction inside the half.
__device__ __forceinline__ float dot8_bf16(const uint4 &a, const uint4 &b) {
    const __nv_bfloat162 *x = reinterpret_cast<const __nv_bfloat162 *>(&a);
    const __nv_bfloat162 *y = reinterpret_cast<const __nv_bfloat162 *>(&b);
    float s = 0.f;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const float2 u = __bfloat1622float2(x[k]), v = __bfloat1622float2(y[k]);
        s = fmaf(u.x, v.x, s);
        s = fmaf(u.y, v.y, s);
    }
    return s;
}

__global__ void __launch_bounds__(256) permute_rowdot_kernel(PermJobs jobs, const uint4 *__restrict__ dout,
                                                              uint4 *__restrict__ dout_p, const uint4 *__restrict__ out,
                                                              float *__restrict__ D, const int32_t *__restrict__ perm,
                                                              int64_t T, int Hq, const uint8_t *__restrict__ dout_only,
                                                              int *status) {
    const int lane = threadIdx.x & 31;
    const int64_t warp = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    const int64_t nwarps = (int64_t)gridDim.x * (blockDim.x >> 5);
    const int64_t nvo = (int64_t)Hq * 16;  // 16-byte vectors per dO / O row
    for (int64_t i = warp; i < T; i += nwarps) {
        const int32_t p = __ldg(perm + i);
        if (p < 0 || (int64_t)p >= T) {
            if (lane == 0) dev::record_status(status, RA_ERR_DEVICE_BOUNDS);
            continue;
        }
        for (int jb = 0; jb < jobs.n; ++jb) {
            if (jobs.j[jb].only && !__ldg(jobs.j[jb].only + i)) continue;
            const int64_t nvec = jobs.j[jb].row_bytes / 16;
            const uint4 *__restrict__ src = reinterpret_cast<const uint4 *>(jobs.j[jb].src) + (int64_t)p * nvec;
            uint4 *__restrict__ dst = reinterpret_cast<uint4 *>(jobs.j[jb].dst) + i * nvec;
            for (int64_t c0 = lane; c0 < nvec; c0 += 128) {
                uint4 tmp[4];
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    const int64_t c = c0 + u * 32;
                    if (c < nvec) tmp[u] = src[c];
                }
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    const int64_t c = c0 + u * 32;
                    if (c < nvec) dst[c] = tmp[u];
                }
            }
        }
        const uint4 *__restrict__ a = dout + (int64_t)p * nvo;
        const uint4 *__restrict__ b = out + (int64_t)p * nvo;
        uint4 *__restrict__ dst = dout_p + i * nvo;
        const bool keep = !dout_only || __ldg(dout_only + i);
        for (int64_t c0 = lane; c0 < nvo; c0 += 128) {
            uint4 x[4], y[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int64_t c = c0 + u * 32;
                if (c < nvo) {
                    x[u] = a[c];
                    y[u] = b[c];
                }
            }
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int64_t c = c0 + u * 32;
                if (c < nvo && keep) dst[c] = x[u];
            }
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int64_t c = c0 + u * 32;  // nvo is a multiple of 16: a half-warp is all in or all out
                float sum = c < nvo ? dot8_bf16(x[u], y[u]) : 0.f;
#pragma unroll
                for (int sh = 8; sh; sh >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, sh);
                if (c < nvo && (lane & 15) == 0) D[(c >> 4) * T + p] = sum;
            }
        }
    }
}

cudaError_t launch_permute_rowdot(const PermJob *jobs, int njobs, const void *dout, void *dout_p, const void *out,
                                  float *D, const int32_t *perm, int64_t T, int Hq, cudaStream_t st,
                                  const uint8_t *dout_only) {
    if (T <= 0) return cudaSuccess;
    if (njobs < 0 || njobs > 4) return cudaErrorInvalidValue;
    PermJobs pj{};
    pj.n = njobs;
    auto al = [](const void *q, int64_t rb) { return (reinterpret_cast<uintptr_t>(q) % 16) == 0 && (rb % 16) == 0; };
    for (int i = 0; i < njobs; ++i) {
        if (!al(jobs[i].src, jobs[i].row_bytes) || !al(jobs[i].dst, jobs[i].row_bytes)) return cudaErrorInvalidValue;
        pj.j[i] = jobs[i];
    }
    if (!al(dout, 16) || !al(dout_p, 16) || !al(out, 16)) return cudaErrorInvalidValue;
    const int64_t want = (T + 7) / 8;
    const int blocks = (int)std::min<int64_t>(want, (int64_t)num_sms() * 8);
    permute_rowdot_kernel<<<blocks, 256, 0, st>>>(pj, static_cast<const uint4 *>(dout), static_cast<uint4 *>(dout_p),
                                                  static_cast<const uint4 *>(out), D, perm, T, Hq, dout_only,
                                                  device_status_ptr());
    return cudaGetLastError();
}

// ------------------------------------------------------------------ rowdot
template <typename TIn>
__global__ void __launch_bounds__(256) rowdot_kernel(const TIn *a, const TIn *b, int64_t T, int H, int d,
                                                      float *D) {
    const int lane = threadIdx.x & 31;
    const int64_t rows = T * H;
    const int64_t nw = (int64_t)gridDim.x * (blockDim.x >> 5);
    for (int64_t w = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); w < rows; w += nw) {
        float acc = 0.f;
        for (int c = lane; c < d; c += 32) acc += (float)a[w * d + c] * (float)b[w * d + c];
#pragma unroll
        for (int s = 16; s; s >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, s);
        if (lane == 0) {
            const int64_t t = w / H;
            const int h = (int)(w % H);
            D[(int64_t)h * T + t] = acc;
        }
    }
}

cudaError_t launch_rowdot(const void *a, const void *b, int dtype, int64_t T, int H, int d, float *D,
                          cudaStream_t st) {
    if (T <= 0) return cudaSuccess;
    const int64_t rows = T * H;
    const int blocks = (int)std::min<int64_t>((rows + 7) / 8, (int64_t)num_sms() * 16);
    if (dtype == RA_FP32)
        rowdot_kernel<float><<<blocks, 256, 0, st>>>(static_cast<const float *>(a), static_cast<const float *>(b),
                                                     T, H, d, D);
    else
        rowdot_kernel<__nv_bfloat16><<<blocks, 256, 0, st>>>(static_cast<const __nv_bfloat16 *>(a),
                                                             static_cast<const __nv_bfloat16 *>(b), T, H, d, D);
    return cudaGetLastError();
}

// ------------------------------------------------------------------ tile LSE / D
// For every (query tile, KV head) the 128 MMA columns (token, head) get
// lse * log2(e) (+inf where the column has no token or lse is -inf) and D
// (0 where no token), stored contiguously: out[((tile * Hkv + g) * 2 + w) * 128 + c].
__global__ void tile_lse_d_kernel(const int4 *__restrict__ qtiles, int n_qtiles, int Hkv, int G, int log2G,
                                  const float *__restrict__ lse, const float *__restrict__ D, long long lse_T,
                                  float scale, float *__restrict__ out) {
    const long long total = (long long)n_qtiles * Hkv * 128;
    for (long long w = (long long)blockIdx.x * blockDim.x + threadIdx.x; w < total;
         w += (long long)gridDim.x * blockDim.x) {
        const int c = (int)(w & 127);
        const long long tg = w >> 7;
        const int g = (int)(tg % Hkv);
        const int qt = (int)(tg / Hkv);
        const int4 a = __ldg(qtiles + 2 * qt);
        const int pos1 = __ldg(&qtiles[2 * qt + 1].x);
        const int tok = c >> log2G, head = g * G + (c & (G - 1));
        float nl2 = -INFINITY, nds = 0.f;
        if (tok < a.y) {
            const int pos = tok < a.z ? a.w + tok : pos1 + (tok - a.z);
            const float l = lse[(long long)head * lse_T + pos];
            nl2 = (l == -INFINITY) ? -INFINITY : -l * 1.4426950408889634f;
            nds = -D[(long long)head * lse_T + pos] * scale;
        }
        out[(tg * 2 + 0) * 128 + c] = nl2;
        out[(tg * 2 + 1) * 128 + c] = nds;
    }
}

cudaError_t launch_tile_lse_d(const void *qtiles, int n_qtiles, int Hkv, int G, const float *lse, const float *D,
                              int64_t lse_T, float scale, float *out, cudaStream_t st) {
    if (n_qtiles <= 0) return cudaSuccess;
    int lg = 0;
    while ((1 << lg) < G) ++lg;
    const long long total = (long long)n_qtiles * Hkv * 128;
    const int blocks = (int)std::min<long long>((total + 255) / 256, (long long)num_sms() * 8);
    tile_lse_d_kernel<<<blocks, 256, 0, st>>>(static_cast<const int4 *>(qtiles), n_qtiles, Hkv, G, lg, lse, D, lse_T,
                                              scale, out);
    return cudaGetLastError();
}

// ------------------------------------------------------------------ cast
__global__ void __launch_bounds__(256) copy_from_host_kernel(const uint4 *__restrict__ src, uint4 *__restrict__ dst,
                                                            int64_t n16, const uint8_t *__restrict__ src_tail,
                                                            uint8_t *__restrict__ dst_tail, int tail) {
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n16; i += stride) dst[i] = src[i];
    if (blockIdx.x == 0 && (int)threadIdx.x < tail) dst_tail[threadIdx.x] = src_tail[threadIdx.x];
}

cudaError_t launch_copy_from_host(const void *src, void *dst, size_t n, cudaStream_t st) {
    if (n == 0) return cudaSuccess;
    if ((reinterpret_cast<uintptr_t>(src) | reinterpret_cast<uintptr_t>(dst)) & 15u) return cudaErrorInvalidValue;
    void *dsrc = nullptr;  // the device's address of the mapped host buffer
    cudaError_t e = cudaHostGetDevicePointer(&dsrc, const_cast<void *>(src), 0);
    if (e != cudaSuccess) return e;
    const int64_t n16 = (int64_t)(n / 16);
    const int tail = (int)(n % 16);
    const int64_t blocks = std::min<int64_t>(std::max<int64_t>((n16 + 255) / 256, 1), 1024);
    copy_from_host_kernel<<<(unsigned)blocks, 256, 0, st>>>(static_cast<const uint4 *>(dsrc), static_cast<uint4 *>(dst),
                                                           n16, static_cast<const uint8_t *>(dsrc) + n16 * 16,
                                                           static_cast<uint8_t *>(dst) + n16 * 16, tail);
    return cudaGetLastError();
}

__global__ void cast_bf16_kernel(const float *__restrict__ src, __nv_bfloat16 *__restrict__ dst, int64_t n) {
    const int64_t n4 = n / 4;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n4; i += (int64_t)gridDim.x * blockDim.x) {
        const float4 x = reinterpret_cast<const float4 *>(src)[i];
        uint2 pk;
        pk.x = dev::pack_bf16x2(x.x, x.y);
        pk.y = dev::pack_bf16x2(x.z, x.w);
        reinterpret_cast<uint2 *>(dst)[i] = pk;
    }
    for (int64_t i = n4 * 4 + (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x)
        dst[i] = __float2bfloat16_rn(src[i]);
}

cudaError_t launch_cast_f32(const float *src, void *dst, int dtype, int64_t n, cudaStream_t st) {
    if (n <= 0) return cudaSuccess;
    if (dtype == RA_FP32) {
        if (src != dst) return cudaMemcpyAsync(dst, src, (size_t)n * 4, cudaMemcpyDeviceToDevice, st);
        return cudaSuccess;
    }
    const int blocks = (int)std::min<int64_t>((n / 4 + 255) / 256 + 1, (int64_t)num_sms() * 8);
    cast_bf16_kernel<<<blocks, 256, 0, st>>>(src, static_cast<__nv_bfloat16 *>(dst), n);
    return cudaGetLastError();
}

// ------------------------------------------------------------------ self-test
// Waits on a barrier nothing arrives at; the guard must give up after the
// budget, record RA_ERR_TIMEOUT and let the kernel return.
__global__ void wait_selftest_kernel(uint64_t budget_ns, int *status) {
    __shared__ uint64_t bar;
    __shared__ int abort_flag;
    if (threadIdx.x == 0) {
        abort_flag = 0;
        dev::mbar_init(&bar, 1);
        dev::fence_mbar_init();
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        dev::WaitCtl w{&abort_flag, status, budget_ns};
        (void)dev::mbar_wait(&bar, 0, w);
    }
    __syncthreads();
}

cudaError_t launch_wait_selftest(uint64_t budget_ns, cudaStream_t st) {
    wait_selftest_kernel<<<1, 32, 0, st>>>(budget_ns, device_status_ptr());
    return cudaGetLastError();
}

}  // namespace ra
