// softmax_mix.cu -- throughput of the forward softmax's inner loop per SM
// sub-partition (SMSP), at 1 and 2 warps per SMSP.  Per pair of scores the
// loop forms x = s * scale - m (fma.rn.f32x2), two ex2.approx, the running
// sum (add.rn.f32x2) and the bf16x2 pack of P; each thread runs 8
// independent chains (each pair feeds the next through e - 1.5).  Modes:
//   ex2 only        two ex2.approx per pair (the special-function unit alone)
//   ex2x2+cvt       plus the cvt.rn.bf16x2.f32 pack
//   mix cvt pack    the whole loop
//   mix int pack    the whole loop with the pack done on integer bits
//   cvt alone       the pack alone
// Prints cycles per warp-instruction of pairs (32 pairs).
//
//   nvcc -gencode arch=compute_103a,code=sm_103a -O3 \
//        -o /tmp/softmax_mix context_varlen_ring_gb300/microbench/softmax_mix.cu && /tmp/softmax_mix
#include <cstdio>
#include <cstdint>
#include <cuda_runtime.h>
#include <cuda_bf16.h>
__device__ __forceinline__ float ex2a(float x) { float y; asm volatile("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x)); return y; }
__device__ __forceinline__ uint32_t pack_rn(float lo, float hi) {
    __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&h);
}
__device__ __forceinline__ uint32_t pack_int(float lo, float hi) {
    // round half up on the bits, then take the high halves
    const uint32_t a = __float_as_uint(lo) + 0x8000u, b = __float_as_uint(hi) + 0x8000u;
    return __byte_perm(a, b, 0x7632);
}
__device__ __forceinline__ float2 fma2(float2 a, float2 b, float2 c) {
    float2 d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(*reinterpret_cast<unsigned long long *>(&d))
        : "l"(*reinterpret_cast<unsigned long long *>(&a)), "l"(*reinterpret_cast<unsigned long long *>(&b)),
          "l"(*reinterpret_cast<unsigned long long *>(&c)));
    return d;
}
__device__ __forceinline__ float2 add2(float2 a, float2 b) {
    float2 d;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(*reinterpret_cast<unsigned long long *>(&d))
        : "l"(*reinterpret_cast<unsigned long long *>(&a)), "l"(*reinterpret_cast<unsigned long long *>(&b)));
    return d;
}
template <int MODE>
__global__ void bench(float *out, long long *cyc, int iters) {
    float2 a[8];
    for (int i = 0; i < 8; ++i) a[i] = make_float2(-0.001f * (threadIdx.x + i), -0.002f * (threadIdx.x + i));
    float2 acc[4] = {};
    uint32_t x = 0;
    const float2 sl = make_float2(0.9f, 0.9f), nm = make_float2(-0.1f, -0.1f);
    __syncthreads();
    long long t0 = clock64();
    for (int it = 0; it < iters; ++it) {
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            if (MODE == 0) {  // ex2 only
                a[i] = make_float2(ex2a(a[i].x) - 1.5f, ex2a(a[i].y) - 1.5f);
            } else if (MODE == 1) {  // ex2 x2 + cvt pack
                const float2 e = make_float2(ex2a(a[i].x), ex2a(a[i].y));
                x ^= pack_rn(e.x, e.y);
                a[i] = make_float2(e.x - 1.5f, e.y - 1.5f);
            } else if (MODE == 2) {  // the softmax mix: fma2, ex2 x2, add2, cvt pack
                const float2 t = fma2(a[i], sl, nm);
                const float2 e = make_float2(ex2a(t.x), ex2a(t.y));
                acc[i & 3] = add2(acc[i & 3], e);
                x ^= pack_rn(e.x, e.y);
                a[i] = make_float2(e.x - 1.5f, e.y - 1.5f);
            } else if (MODE == 3) {  // the same mix with an integer pack
                const float2 t = fma2(a[i], sl, nm);
                const float2 e = make_float2(ex2a(t.x), ex2a(t.y));
                acc[i & 3] = add2(acc[i & 3], e);
                x ^= pack_int(e.x, e.y);
                a[i] = make_float2(e.x - 1.5f, e.y - 1.5f);
            } else {  // cvt pack alone
                x ^= pack_rn(a[i].x, a[i].y);
                a[i] = make_float2(a[i].y + 1.0f, a[i].x);
            }
        }
    }
    __syncthreads();
    long long t1 = clock64();
    float s = 0;
    for (int i = 0; i < 8; ++i) s += a[i].x + a[i].y;
    for (int i = 0; i < 4; ++i) s += acc[i].x + acc[i].y;
    out[blockIdx.x * blockDim.x + threadIdx.x] = s + (float)(x & 7);
    if (threadIdx.x == 0) cyc[blockIdx.x] = t1 - t0;
}
int main() {
    int nsm = 0; cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, 0);
    float *out; long long *cyc; cudaMalloc(&out, nsm * 1024 * 4); cudaMalloc(&cyc, nsm * 8);
    long long h[1024];
    const int iters = 2048;
    const char *names[5] = {"ex2 only       ", "ex2x2+cvt      ", "mix cvt pack   ", "mix int pack   ", "cvt alone      "};
    for (int mode = 0; mode < 5; ++mode)
        for (int wps = 1; wps <= 2; wps *= 2) {
            int threads = 128 * wps;
            for (int rep = 0; rep < 2; ++rep) {
                if (mode == 0) bench<0><<<nsm, threads>>>(out, cyc, iters);
                if (mode == 1) bench<1><<<nsm, threads>>>(out, cyc, iters);
                if (mode == 2) bench<2><<<nsm, threads>>>(out, cyc, iters);
                if (mode == 3) bench<3><<<nsm, threads>>>(out, cyc, iters);
                if (mode == 4) bench<4><<<nsm, threads>>>(out, cyc, iters);
            }
            cudaDeviceSynchronize();
            cudaMemcpy(h, cyc, nsm * 8, cudaMemcpyDeviceToHost);
            double c = 0; for (int i = 0; i < nsm; ++i) c += h[i]; c /= nsm;
            double pairs_per_smsp = (double)wps * 32 * 8 * iters;  // 8 pairs per iteration per thread
            printf("%s warps/SMSP=%d cycles=%.0f pairs/clk/SMSP=%.2f (cycles per warp-pair-instr %.2f)\n", names[mode],
                   wps, c, pairs_per_smsp / c, c / (wps * 8.0 * iters));
        }
    printf("err=%s\n", cudaGetErrorString(cudaGetLastError()));
    return 0;
}
