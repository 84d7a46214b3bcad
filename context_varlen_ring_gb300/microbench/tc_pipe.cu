// tc_pipe.cu -- the tensor pipe's ceiling for the forward kernel's MMA mix.
//
// One CTA per SM issues, from one converged warp, the tcgen05.mma products
// of one 128-key KV tile for two 128-row query tiles (S = Q K^T into TMEM,
// O += P V with P read from TMEM) in a loop, on data already in shared
// memory, and reports SM cycles per KV tile (ideal: 32 products of
// M=128 N=128 K=16 at 64 cycles = 2048).  Variants: S with both operands
// in shared memory (SS) or A from TMEM (TS), S as two N=64 halves, the
// forward kernel's six commits per KV tile, and its dependency pattern
// (each PV waits for the completion of its tile's S, as if the softmax
// took no time).  No loads, no softmax: what is left is the pipe.
//
//   nvcc -gencode arch=compute_103a,code=sm_103a -O3 -std=c++17 \
//        -Icontext_varlen_ring_gb300/csrc -Iinclude \
//        -o /tmp/tc_pipe context_varlen_ring_gb300/microbench/tc_pipe.cu && /tmp/tc_pipe
#include <cstdio>
#include <cuda_runtime.h>
#include "ra_dev.cuh"
using namespace ra::dev;
constexpr uint32_t kHalf = 16384, kTile = 32768;

__device__ __forceinline__ void s_ss(uint32_t d, uint32_t q_s, uint32_t k_s, uint32_t id, int n64, int nh) {
    // nh: key rows half (0/1) for N=64
#pragma unroll
    for (int ks = 0; ks < 8; ++ks) {
        const uint32_t off = (uint32_t)(ks >> 2) * kHalf + (uint32_t)(ks & 3) * 32u;
        tc_mma_ss_w(d, sdesc_sw128(q_s + off, 16, 1024), sdesc_sw128(k_s + off + (n64 ? nh * 8192u : 0u), 16, 1024), id, ks > 0);
    }
}
__device__ __forceinline__ void s_ts(uint32_t d, uint32_t a_t, uint32_t k_s, uint32_t id, int n64, int nh) {
#pragma unroll
    for (int ks = 0; ks < 8; ++ks) {
        const uint32_t off = (uint32_t)(ks >> 2) * kHalf + (uint32_t)(ks & 3) * 32u;
        tc_mma_ts_w(d, a_t + 8u * ks, sdesc_sw128(k_s + off + (n64 ? nh * 8192u : 0u), 16, 1024), id, ks > 0);
    }
}
__device__ __forceinline__ void pv(uint32_t d, uint32_t p_t, uint32_t v_s, uint32_t id, int k0, int k1) {
#pragma unroll
    for (int ks = k0; ks < k1; ++ks) tc_mma_ts_w(d, p_t + 8u * ks, sdesc_sw128(v_s + (uint32_t)ks * 2048u, kHalf, 1024), id, 1);
}

template <int MODE>
__global__ void __launch_bounds__(128, 1) bench(long long *out, int iters, int *status) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_s = smem_u32(smem_raw);
    const uint32_t base_s = (raw_s + 1023u) & ~1023u;
    uint8_t *base = smem_raw + (base_s - raw_s);
    uint64_t *bar = reinterpret_cast<uint64_t *>(base + 3 * kTile);
    uint64_t *cb = reinterpret_cast<uint64_t *>(base + 3 * kTile + 256);  // [8]
    uint32_t *slot = reinterpret_cast<uint32_t *>(base + 3 * kTile + 64);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(base + 3 * kTile + 128);
    const int warp = threadIdx.x >> 5;
    for (int i = threadIdx.x; i < 3 * kTile / 4; i += blockDim.x) reinterpret_cast<uint32_t *>(base)[i] = 0x3c003c00u;
    if (threadIdx.x == 0) {
        *abort_flag = 0;
        mbar_init(bar, 1);
        for (int i = 0; i < 8; ++i) mbar_init(cb + i, 1);
        fence_mbar_init();
    }
    fence_proxy_async_smem();
    if (warp == 0) {
        tmem_alloc(slot, 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *slot;
    if (warp == 1) {
        const WaitCtl wc{abort_flag, status, 2000000000ull};
        const uint32_t q_s = base_s, k_s = base_s + kTile, v_s = base_s + 2 * kTile;
        const uint32_t id128 = idesc_bf16_f32(128, 128, 0, 0), id64 = idesc_bf16_f32(128, 64, 0, 0);
        const uint32_t ido = idesc_bf16_f32(128, 128, 0, 1);
        const uint32_t S0 = tmem, S1 = tmem + 128, O0 = tmem + 256, O1 = tmem + 384;
        __syncwarp();
        const long long t0 = clock64();
        for (int it = 0; it < iters; ++it) {
            if (MODE == 0) {  // SS S, TS PV (the kernel's mix)
                s_ss(S0, q_s, k_s, id128, 0, 0); s_ss(S1, q_s, k_s, id128, 0, 0);
                pv(O0, S0, v_s, ido, 0, 8); pv(O1, S1, v_s, ido, 0, 8);
            } else if (MODE == 1) {  // S only, SS
                s_ss(S0, q_s, k_s, id128, 0, 0); s_ss(S1, q_s, k_s, id128, 0, 0);
                s_ss(S0, q_s, k_s, id128, 0, 0); s_ss(S1, q_s, k_s, id128, 0, 0);
            } else if (MODE == 2) {  // PV only
                pv(O0, S0, v_s, ido, 0, 8); pv(O1, S1, v_s, ido, 0, 8);
                pv(O0, S0, v_s, ido, 0, 8); pv(O1, S1, v_s, ido, 0, 8);
            } else if (MODE == 3) {  // S as TS (A from TMEM), PV TS
                s_ts(S0, O1, k_s, id128, 0, 0); s_ts(S1, O0, k_s, id128, 0, 0);
                pv(O0, S0, v_s, ido, 0, 8); pv(O1, S1, v_s, ido, 0, 8);
            } else if (MODE == 4) {  // S in N=64 halves SS, PV
                s_ss(S0, q_s, k_s, id64, 1, 0); s_ss(S0 + 64, q_s, k_s, id64, 1, 1);
                s_ss(S1, q_s, k_s, id64, 1, 0); s_ss(S1 + 64, q_s, k_s, id64, 1, 1);
                pv(O0, S0, v_s, ido, 0, 8); pv(O1, S1, v_s, ido, 0, 8);
            } else if (MODE == 6) {  // kernel mix + the kernel's 6 commits per KV tile
                pv(O0, S0, v_s, ido, 0, 8); tc_commit_w(cb + 0);
                s_ss(S0, q_s, k_s, id128, 0, 0); tc_commit_w(cb + 1);
                pv(O1, S1, v_s, ido, 0, 8); tc_commit_w(cb + 2);
                s_ss(S1, q_s, k_s, id128, 0, 0); tc_commit_w(cb + 3);
                tc_commit_w(cb + 4); tc_commit_w(cb + 5);
            } else if (MODE == 7 || MODE == 8) {  // the kernel's dependency: PV_k(j) after S_k(j) completes
                // (softmax instant): wait S0(j) -> PV0(j), S0(j+1); wait S1(j) -> PV1(j), S1(j+1)
                if (it == 0) {
                    s_ss(S0, q_s, k_s, id128, 0, 0); tc_commit_w(cb + 0);
                    s_ss(S1, q_s, k_s, id128, 0, 0); tc_commit_w(cb + 1);
                }
                (void)mbar_wait_warp(cb + 0, it & 1, wc);
                tc_fence_after();
                pv(O0, S0, v_s, ido, 0, 8);
                if (MODE == 8) tc_commit_w(cb + 2);
                s_ss(S0, q_s, k_s, id128, 0, 0); tc_commit_w(cb + 0);
                (void)mbar_wait_warp(cb + 1, it & 1, wc);
                tc_fence_after();
                pv(O1, S1, v_s, ido, 0, 8);
                if (MODE == 8) tc_commit_w(cb + 3);
                s_ss(S1, q_s, k_s, id128, 0, 0); tc_commit_w(cb + 1);
            } else if (MODE == 5) {  // S in N=64 halves TS, PV
                s_ts(S0, O1, k_s, id64, 1, 0); s_ts(S0 + 64, O1, k_s, id64, 1, 1);
                s_ts(S1, O0, k_s, id64, 1, 0); s_ts(S1 + 64, O0, k_s, id64, 1, 1);
                pv(O0, S0, v_s, ido, 0, 8); pv(O1, S1, v_s, ido, 0, 8);
            }
        }
        tc_commit_w(bar);
        (void)mbar_wait_warp(bar, 0, wc);
        const long long t1 = clock64();
        if ((threadIdx.x & 31) == 0) out[blockIdx.x] = t1 - t0;
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

int main() {
    int nsm = 0;
    cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, 0);
    long long *out;
    int *status;
    cudaMalloc(&out, nsm * 8);
    cudaMalloc(&status, 4);
    cudaMemset(status, 0, 4);
    const int smem = 3 * 32768 + 1024 + 1024;
    const int iters = 2000;
    void (*fns[9])(long long *, int, int *) = {bench<0>, bench<1>, bench<2>, bench<3>, bench<4>, bench<5>, bench<6>, bench<7>, bench<8>};
    const char *names[9] = {"S SS + PV TS (kernel mix)", "S SS only", "PV TS only", "S TS + PV TS", "S SS N=64 halves + PV",
                            "S TS N=64 halves + PV", "kernel mix + 6 commits", "wait S -> PV, S (instant softmax)", "same + PV commits"};
    long long h[1024];
    for (int m = 0; m < 9; ++m) {
        cudaFuncSetAttribute(fns[m], cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        for (int rep = 0; rep < 2; ++rep) fns[m]<<<nsm, 128, smem>>>(out, iters, status);
        cudaError_t e = cudaDeviceSynchronize();
        cudaMemcpy(h, out, nsm * 8, cudaMemcpyDeviceToHost);
        double c = 0;
        for (int i = 0; i < nsm; ++i) c += h[i];
        c /= nsm;
        // 32 MMAs of M128 N128 K16 (or equivalent work) per iteration = one KV tile of two query tiles
        printf("%-28s cycles per KV tile (2 query tiles) = %7.1f  (ideal 2048)  err=%s\n", names[m], c / iters,
               cudaGetErrorString(e));
    }
    int st = 0;
    cudaMemcpy(&st, status, 4, cudaMemcpyDeviceToHost);
    printf("status=%d\n", st);
    return 0;
}
