// exp_rate.cu -- throughput of the exponential the softmax needs, per SM
// sub-partition (SMSP), at 1, 2 and 4 warps per SMSP:
//   mufu: ex2.approx.ftz.f32 (the special-function unit)
//   poly: 2^x on the FMA pipe: x = j + f with j = round(x) (the 1.5 * 2^23
//         magic-number rounding), f in [-1/2, 1/2]; 2^f by a degree-3
//         polynomial whose coefficients were fitted here to minimise the
//         largest relative error on [-1/2, 1/2] (7.5e-5); 2^j added to the
//         exponent field
//   mix:  half of the elements each way
// Each thread runs 8 independent chains.
//
//   nvcc -gencode arch=compute_103a,code=sm_103a -O3 \
//        -o /tmp/exp_rate context_varlen_ring_gb300/microbench/exp_rate.cu && /tmp/exp_rate
#include <cstdio>
#include <cuda_runtime.h>
__device__ __forceinline__ float ex2a(float x) { float y; asm volatile("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x)); return y; }
__device__ __forceinline__ float ex2p(float x) {
    x = fmaxf(x, -127.f);
    const float t = x + 12582912.f;
    const float j = t - 12582912.f;
    const float f = x - j;
    float p = fmaf(0.05517134442925453f, f, 0.24261033535003662f);
    p = fmaf(p, f, 0.6932609677314758f);
    p = fmaf(p, f, 0.9999281167984009f);
    return __int_as_float(__float_as_int(p) + (__float_as_int(t) << 23));
}
template <int MODE>
__global__ void bench(float *out, long long *cyc, int iters) {
    float a[8];
    for (int i = 0; i < 8; ++i) a[i] = -0.001f * (threadIdx.x + i);
    __syncthreads();
    long long t0 = clock64();
    for (int it = 0; it < iters; ++it) {
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            if (MODE == 0) a[i] = ex2a(a[i]) - 1.5f;
            else if (MODE == 1) a[i] = ex2p(a[i]) - 1.5f;
            else a[i] = ((i & 1) ? ex2p(a[i]) : ex2a(a[i])) - 1.5f;
        }
    }
    __syncthreads();
    long long t1 = clock64();
    float s = 0; for (int i = 0; i < 8; ++i) s += a[i];
    out[blockIdx.x * blockDim.x + threadIdx.x] = s;
    if (threadIdx.x == 0) cyc[blockIdx.x] = t1 - t0;
}
int main() {
    int nsm = 0; cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, 0);
    float *out; long long *cyc; cudaMalloc(&out, nsm * 1024 * 4); cudaMalloc(&cyc, nsm * 8);
    long long h[1024];
    const int iters = 4096;
    for (int mode = 0; mode < 3; ++mode)
        for (int wps = 1; wps <= 4; wps *= 2) {
            int threads = 128 * wps;
            for (int rep = 0; rep < 2; ++rep) {
                if (mode == 0) bench<0><<<nsm, threads>>>(out, cyc, iters);
                if (mode == 1) bench<1><<<nsm, threads>>>(out, cyc, iters);
                if (mode == 2) bench<2><<<nsm, threads>>>(out, cyc, iters);
            }
            cudaDeviceSynchronize();
            cudaMemcpy(h, cyc, nsm * 8, cudaMemcpyDeviceToHost);
            double c = 0; for (int i = 0; i < nsm; ++i) c += h[i]; c /= nsm;
            double exps_per_smsp = (double)wps * 32 * 8 * iters;
            printf("mode=%s warps/SMSP=%d cycles=%.0f exps/clk/SMSP=%.2f\n", mode == 0 ? "mufu" : mode == 1 ? "poly" : "mix ",
                   wps, c, exps_per_smsp / c);
        }
    printf("err=%s\n", cudaGetErrorString(cudaGetLastError()));
    return 0;
}
