// ra_simt.cu -- SIMT fp32 attention for the simulated ring: the exact path
// for fp32 inputs (a TF32 tensor-core path cannot reach 1e-5) and the
// fallback for shapes the tensor-core kernels do not take.
//
// Forward: one warp per (query row, head); the warp walks the ring steps
// t in [t0, t1) (rank r sees the KV shard of rank s = (r - t) mod cp, the
// ring schedule of "Question about varlen ring attention", MiniMax-01 #6)
// and the keys of its own document segment, with an fp32 online softmax.
// Backward: the textbook gradient from the saved LSE, dQ query-major and
// dK/dV key-major, accumulated (+=) in fp32.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cmath>

#include "ra_dev.cuh"
#include "ra_kernels.h"

namespace ra {

namespace {

template <typename T>
__device__ __forceinline__ float ld_f(const T *p) {
    return (float)(*p);
}
template <>
__device__ __forceinline__ float ld_f<__nv_bfloat16>(const __nv_bfloat16 *p) {
    return __bfloat162float(*p);
}

// largest index i in [0, n) with a[i] <= x (a non-decreasing, a[0] <= x)
__device__ __forceinline__ int upper_idx(const int32_t *a, int n, int64_t x) {
    int lo = 0, hi = n - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if ((int64_t)a[mid] <= x)
            lo = mid;
        else
            hi = mid - 1;
    }
    return lo;
}

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
    for (int s = 16; s; s >>= 1) x += __shfl_xor_sync(0xffffffffu, x, s);
    return x;
}

template <typename T, int NV>
__global__ void __launch_bounds__(256) simt_fwd_kernel(SimtArgs a) {
    const int lane = threadIdx.x & 31;
    const int64_t rows = a.Tq * a.Hq;
    const int64_t nw = (int64_t)gridDim.x * (blockDim.x >> 5);
    const int G = a.Hq / a.Hkv;
    const T *Q = static_cast<const T *>(a.q);
    const T *K = static_cast<const T *>(a.k);
    const T *V = static_cast<const T *>(a.v);
    for (int64_t w = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); w < rows; w += nw) {
        const int64_t i = w / a.Hq;
        const int h = (int)(w % a.Hq);
        const int g = h / G;
        const int r = upper_idx(a.qoff, a.cp + 1, i);
        const int64_t li = i - a.qoff[r];
        const int b = upper_idx(a.qcul + (int64_t)r * (a.B + 1), a.B + 1, li);
        const int32_t qp = a.qpos[i];
        float qv[NV], o[NV];
#pragma unroll
        for (int e = 0; e < NV; ++e) {
            qv[e] = ld_f(Q + (i * a.Hq + h) * a.d + lane + 32 * e);
            o[e] = 0.f;
        }
        float m = -INFINITY, l = 0.f;
        for (int t = a.t0; t < a.t1; ++t) {
            const int s = ((r - t) % a.cp + a.cp) % a.cp;
            const int32_t *kc = a.kcul + (int64_t)s * (a.B + 1);
            const int64_t j0 = a.koff[s] + kc[b], j1 = a.koff[s] + kc[b + 1];
            for (int64_t j = j0; j < j1; ++j) {
                if (a.causal && a.kpos[j] > qp) continue;
                if (a.window >= 0 && (int64_t)a.kpos[j] < (int64_t)qp - a.window) continue;
                float part = 0.f;
#pragma unroll
                for (int e = 0; e < NV; ++e) part += qv[e] * ld_f(K + (j * a.Hkv + g) * a.d + lane + 32 * e);
                const float sc = warp_sum(part) * a.scale;
                const float mn = fmaxf(m, sc);
                const float alpha = expf(m - mn);
                const float p = expf(sc - mn);
                l = l * alpha + p;
#pragma unroll
                for (int e = 0; e < NV; ++e)
                    o[e] = o[e] * alpha + p * ld_f(V + (j * a.Hkv + g) * a.d + lane + 32 * e);
                m = mn;
            }
        }
        const float inv = l > 0.f ? 1.f / l : 0.f;
        const float lse = l > 0.f ? m + logf(l) : -INFINITY;
        const int64_t orow = a.out_mode == kOutFinal ? (int64_t)qp : i;
        if (a.out_mode == kOutFinal && a.dtype == RA_BF16) {
            __nv_bfloat16 *O = static_cast<__nv_bfloat16 *>(a.out);
#pragma unroll
            for (int e = 0; e < NV; ++e) O[(orow * a.Hq + h) * a.d + lane + 32 * e] = __float2bfloat16_rn(o[e] * inv);
        } else {
            float *O = static_cast<float *>(a.out);
#pragma unroll
            for (int e = 0; e < NV; ++e) O[(orow * a.Hq + h) * a.d + lane + 32 * e] = o[e] * inv;
        }
        if (lane == 0) a.lse[(int64_t)h * a.lse_T + orow] = lse;
    }
}

// dQ: one warp per (query row, head).
template <typename T, int NV>
__global__ void __launch_bounds__(256) simt_bwd_dq_kernel(SimtBwdArgs a) {
    const int lane = threadIdx.x & 31;
    const int64_t rows = a.T * a.Hq;
    const int64_t nw = (int64_t)gridDim.x * (blockDim.x >> 5);
    const int G = a.Hq / a.Hkv;
    const T *Q = static_cast<const T *>(a.q);
    const T *K = static_cast<const T *>(a.k);
    const T *V = static_cast<const T *>(a.v);
    const T *dO = static_cast<const T *>(a.dout);
    for (int64_t w = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); w < rows; w += nw) {
        const int64_t i = w / a.Hq;
        const int h = (int)(w % a.Hq);
        const int g = h / G;
        const int r = upper_idx(a.off, a.cp + 1, i);
        const int64_t li = i - a.off[r];
        const int b = upper_idx(a.cul + (int64_t)r * (a.B + 1), a.B + 1, li);
        const int32_t qp = a.pos[i];
        const float lse = a.lse[(int64_t)h * a.lse_T + qp];
        const float Di = a.D[(int64_t)h * a.lse_T + qp];
        float qv[NV], dov[NV], dq[NV];
#pragma unroll
        for (int e = 0; e < NV; ++e) {
            qv[e] = ld_f(Q + (i * a.Hq + h) * a.d + lane + 32 * e);
            dov[e] = ld_f(dO + (i * a.Hq + h) * a.d + lane + 32 * e);
            dq[e] = 0.f;
        }
        if (lse != -INFINITY) {
            for (int t = a.t0; t < a.t1; ++t) {
                const int s = ((r - t) % a.cp + a.cp) % a.cp;
                const int32_t *kc = a.cul + (int64_t)s * (a.B + 1);
                const int64_t j0 = a.off[s] + kc[b], j1 = a.off[s] + kc[b + 1];
                for (int64_t j = j0; j < j1; ++j) {
                    if (a.causal && a.pos[j] > qp) continue;
                    if (a.window >= 0 && (int64_t)a.pos[j] < (int64_t)qp - a.window) continue;
                    float ps = 0.f, pd = 0.f;
#pragma unroll
                    for (int e = 0; e < NV; ++e) {
                        ps += qv[e] * ld_f(K + (j * a.Hkv + g) * a.d + lane + 32 * e);
                        pd += dov[e] * ld_f(V + (j * a.Hkv + g) * a.d + lane + 32 * e);
                    }
                    const float p = expf(warp_sum(ps) * a.scale - lse);
                    const float ds = p * (warp_sum(pd) - Di);
#pragma unroll
                    for (int e = 0; e < NV; ++e) dq[e] += a.scale * ds * ld_f(K + (j * a.Hkv + g) * a.d + lane + 32 * e);
                }
            }
        }
#pragma unroll
        for (int e = 0; e < NV; ++e) a.dq[((int64_t)qp * a.Hq + h) * a.d + lane + 32 * e] += dq[e];
    }
}

// dK, dV: one warp per (key row, KV head); the key's rank s meets the
// queries of rank (s + t) mod cp at ring step t.
template <typename T, int NV>
__global__ void __launch_bounds__(256) simt_bwd_dkv_kernel(SimtBwdArgs a) {
    const int lane = threadIdx.x & 31;
    const int64_t rows = a.T * a.Hkv;
    const int64_t nw = (int64_t)gridDim.x * (blockDim.x >> 5);
    const int G = a.Hq / a.Hkv;
    const T *Q = static_cast<const T *>(a.q);
    const T *K = static_cast<const T *>(a.k);
    const T *V = static_cast<const T *>(a.v);
    const T *dO = static_cast<const T *>(a.dout);
    for (int64_t w = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); w < rows; w += nw) {
        const int64_t j = w / a.Hkv;
        const int g = (int)(w % a.Hkv);
        const int s = upper_idx(a.off, a.cp + 1, j);
        const int64_t lj = j - a.off[s];
        const int b = upper_idx(a.cul + (int64_t)s * (a.B + 1), a.B + 1, lj);
        const int32_t kp = a.pos[j];
        float kv[NV], vv[NV], dk[NV], dv[NV];
#pragma unroll
        for (int e = 0; e < NV; ++e) {
            kv[e] = ld_f(K + (j * a.Hkv + g) * a.d + lane + 32 * e);
            vv[e] = ld_f(V + (j * a.Hkv + g) * a.d + lane + 32 * e);
            dk[e] = 0.f;
            dv[e] = 0.f;
        }
        for (int t = a.t0; t < a.t1; ++t) {
            const int r = (s + t) % a.cp;
            const int32_t *qc = a.cul + (int64_t)r * (a.B + 1);
            const int64_t i0 = a.off[r] + qc[b], i1 = a.off[r] + qc[b + 1];
            for (int64_t i = i0; i < i1; ++i) {
                const int32_t qp = a.pos[i];
                if (a.causal && kp > qp) continue;
                if (a.window >= 0 && (int64_t)kp < (int64_t)qp - a.window) continue;
                for (int h = g * G; h < (g + 1) * G; ++h) {
                    const float lse = a.lse[(int64_t)h * a.lse_T + qp];
                    if (lse == -INFINITY) continue;
                    const float Di = a.D[(int64_t)h * a.lse_T + qp];
                    float ps = 0.f, pd = 0.f;
                    float qv[NV], dov[NV];
#pragma unroll
                    for (int e = 0; e < NV; ++e) {
                        qv[e] = ld_f(Q + (i * a.Hq + h) * a.d + lane + 32 * e);
                        dov[e] = ld_f(dO + (i * a.Hq + h) * a.d + lane + 32 * e);
                        ps += qv[e] * kv[e];
                        pd += dov[e] * vv[e];
                    }
                    const float p = expf(warp_sum(ps) * a.scale - lse);
                    const float ds = p * (warp_sum(pd) - Di);
#pragma unroll
                    for (int e = 0; e < NV; ++e) {
                        dv[e] += p * dov[e];
                        dk[e] += a.scale * ds * qv[e];
                    }
                }
            }
        }
#pragma unroll
        for (int e = 0; e < NV; ++e) {
            a.dk[((int64_t)kp * a.Hkv + g) * a.d + lane + 32 * e] += dk[e];
            a.dv[((int64_t)kp * a.Hkv + g) * a.d + lane + 32 * e] += dv[e];
        }
    }
}

int sm_count() {
    int dev = 0, v = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev);
    return v > 0 ? v : 148;
}

}  // namespace

#define RA_SIMT_DISPATCH(KERNEL, T, NV_, ARGS, BLOCKS, ST)                         \
    switch (NV_) {                                                                 \
        case 1: KERNEL<T, 1><<<BLOCKS, 256, 0, ST>>>(ARGS); break;                 \
        case 2: KERNEL<T, 2><<<BLOCKS, 256, 0, ST>>>(ARGS); break;                 \
        case 3: KERNEL<T, 3><<<BLOCKS, 256, 0, ST>>>(ARGS); break;                 \
        case 4: KERNEL<T, 4><<<BLOCKS, 256, 0, ST>>>(ARGS); break;                 \
        case 5: KERNEL<T, 5><<<BLOCKS, 256, 0, ST>>>(ARGS); break;                 \
        case 6: KERNEL<T, 6><<<BLOCKS, 256, 0, ST>>>(ARGS); break;                 \
        case 7: KERNEL<T, 7><<<BLOCKS, 256, 0, ST>>>(ARGS); break;                 \
        default: KERNEL<T, 8><<<BLOCKS, 256, 0, ST>>>(ARGS); break;                \
    }

cudaError_t launch_simt_fwd(const SimtArgs &a, cudaStream_t st) {
    if (a.Tq <= 0) return cudaSuccess;
    const int nv = a.d / 32;
    const int64_t rows = a.Tq * a.Hq;
    const int blocks = (int)std::min<int64_t>((rows + 7) / 8, (int64_t)sm_count() * 16);
    if (a.dtype == RA_FP32) {
        RA_SIMT_DISPATCH(simt_fwd_kernel, float, nv, a, blocks, st)
    } else {
        RA_SIMT_DISPATCH(simt_fwd_kernel, __nv_bfloat16, nv, a, blocks, st)
    }
    return cudaGetLastError();
}

cudaError_t launch_simt_bwd(const SimtBwdArgs &a, cudaStream_t st) {
    if (a.T <= 0) return cudaSuccess;
    const int nv = a.d / 32;
    const int b1 = (int)std::min<int64_t>((a.T * a.Hq + 7) / 8, (int64_t)sm_count() * 16);
    const int b2 = (int)std::min<int64_t>((a.T * a.Hkv + 7) / 8, (int64_t)sm_count() * 16);
    if (a.dtype == RA_FP32) {
        RA_SIMT_DISPATCH(simt_bwd_dq_kernel, float, nv, a, b1, st)
        RA_SIMT_DISPATCH(simt_bwd_dkv_kernel, float, nv, a, b2, st)
    } else {
        RA_SIMT_DISPATCH(simt_bwd_dq_kernel, __nv_bfloat16, nv, a, b1, st)
        RA_SIMT_DISPATCH(simt_bwd_dkv_kernel, __nv_bfloat16, nv, a, b2, st)
    }
    return cudaGetLastError();
}

}  // namespace ra
