// red_rate.cu -- bandwidth of fp32 reductions into global memory, the cost
// a single-pass backward would pay to add every (query tile, KV tile) dQ
// contribution into an fp32 dQ buffer:
//   mode 0: atomicAdd on float4 per thread (512 coalesced bytes per warp)
//   mode 1: cp.reduce.async.bulk .add.f32 of 4 KB chunks from shared memory
// over a 1 GiB buffer (far above L2), reported as reduced bytes per second.
//
//   nvcc -gencode arch=compute_103a,code=sm_103a -O3 -std=c++17 \
//        -Icontext_varlen_ring_gb300/csrc -o /tmp/red_rate \
//        context_varlen_ring_gb300/microbench/red_rate.cu && /tmp/red_rate
#include <cuda_runtime.h>
#include <cstdint>
#include <cstdio>
#include "ra_dev.cuh"
using namespace ra::dev;

__global__ void __launch_bounds__(256) red_atomic(float* buf, long long n4, int iters) {
  long long tid = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  long long stride = (long long)gridDim.x * blockDim.x;
  float4 one = make_float4(1.f, 1.f, 1.f, 1.f);
  for (int it = 0; it < iters; ++it)
    for (long long i = tid; i < n4; i += stride)
      atomicAdd(reinterpret_cast<float4*>(buf) + i, one);
}

__global__ void __launch_bounds__(128) red_bulk(float* buf, long long nchunks, int iters) {
  __shared__ __align__(128) float src[8][1024];  // 8 x 4 KB
  for (int i = threadIdx.x; i < 8 * 1024; i += blockDim.x) (&src[0][0])[i] = 1.f;
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  __syncthreads();
  if (threadIdx.x < 8) {
    for (int it = 0; it < iters; ++it) {
      for (long long c = (long long)blockIdx.x * 8 + threadIdx.x; c < nchunks; c += (long long)gridDim.x * 8) {
        float* dst = buf + c * 1024;
        asm volatile("cp.reduce.async.bulk.global.shared::cta.bulk_group.add.f32 [%0], [%1], 4096;"
                     :: "l"(dst), "r"(smem_u32(&src[threadIdx.x][0])) : "memory");
        asm volatile("cp.async.bulk.commit_group;" ::: "memory");
        asm volatile("cp.async.bulk.wait_group.read 4;" ::: "memory");
      }
    }
    asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
  }
}

int main() {
  int nsm = 0;
  cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, 0);
  const long long nfloats = 1ll << 28;  // 1 GiB of fp32
  float *buf = nullptr;
  if (cudaMalloc(&buf, nfloats * 4) != cudaSuccess) return 1;
  cudaMemset(buf, 0, nfloats * 4);
  cudaEvent_t a, b;
  cudaEventCreate(&a);
  cudaEventCreate(&b);
  const int iters = 4;
  for (int mode = 0; mode < 2; ++mode) {
    for (int rep = 0; rep < 2; ++rep) {  // the first run warms up
      cudaEventRecord(a);
      if (mode == 0) red_atomic<<<nsm * 8, 256>>>(buf, nfloats / 4, iters);
      else red_bulk<<<nsm * 4, 128>>>(buf, nfloats / 1024, iters);
      cudaEventRecord(b);
      cudaEventSynchronize(b);
      float ms = 0.f;
      cudaEventElapsedTime(&ms, a, b);
      if (rep == 1)
        printf("%s: %.1f GB/s of fp32 reduced (%d passes over 1 GiB, %.2f ms)\n",
               mode == 0 ? "atomicAdd float4" : "bulk reduce 4 KB", nfloats * 4.0 * iters / (ms * 1e6), iters, ms);
    }
  }
  printf("err=%s\n", cudaGetErrorString(cudaDeviceSynchronize()));
  return 0;
}
