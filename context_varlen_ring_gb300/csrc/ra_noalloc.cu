// ra_noalloc.cu -- ra_varlen_attn_partial_noalloc: the single-step partial
// attention for callers that cannot allocate device memory.
//
// Some callers are handed only their input and output buffers and may not
// call cudaMalloc: a runtime whose memory pool already owns the device, a
// plugin inside another framework's allocator, or code that must not risk
// the implicit device-wide synchronisation cudaMalloc/cudaFree can cause.
// This entry point therefore keeps its scratch (the tile tables the kernel
// reads) in a file-scope __device__ array of RA_NOALLOC_SCRATCH_BYTES that
// exists on every GPU that loads the library, for the life of the process.
//
// Host code must not pass the array's name to a kernel: on the host it is
// only a stand-in symbol, not a device address.  The device address is
// fetched once per device with cudaGetSymbolAddress (on the first call made
// while that device is current) and cached for the life of the device's
// context (a cudaDeviceReset after that first call is not supported).
#include <cuda_runtime.h>

#include <mutex>
#include <string>

#include "ra_internal.h"
#include "ra_kernels.h"

namespace ra {
namespace {

static __device__ __align__(256) uint8_t g_partial_scratch[RA_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 128;
std::mutex g_scratch_mu;
void *g_scratch_addr[kMaxDevices] = {};

// Device address of this device's scratch array (set up on first use).
// The kernels run on the current device, so the caller's stream must
// belong to it: the address handed to them is the current device's copy.
ra_status scratch_address(void *stream, void **out) {
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return fail(RA_ERR_CUDA, std::string("cudaGetDevice: ") + cudaGetErrorString(e));
    if (dev < 0 || dev >= kMaxDevices) return fail(RA_ERR_UNSUPPORTED, "device index out of range");
    if (stream) {
        int sdev = -1;
        e = cudaStreamGetDevice(static_cast<cudaStream_t>(stream), &sdev);
        if (e != cudaSuccess) return fail(RA_ERR_CUDA, std::string("cudaStreamGetDevice: ") + cudaGetErrorString(e));
        if (sdev != dev)
            return fail(RA_ERR_INVALID_ARG, "stream belongs to device " + std::to_string(sdev) + ", but device " +
                                                std::to_string(dev) + " is current");
    }
    std::lock_guard<std::mutex> lk(g_scratch_mu);
    if (!g_scratch_addr[dev]) {
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_partial_scratch);
        if (e != cudaSuccess || !p)
            return fail(RA_ERR_CUDA, std::string("cudaGetSymbolAddress(scratch): ") + cudaGetErrorString(e));
        g_scratch_addr[dev] = p;
    }
    *out = g_scratch_addr[dev];
    return RA_OK;
}

}  // namespace
}  // namespace ra

extern "C" ra_status ra_varlen_attn_partial_noalloc(const void *q, const void *k, const void *v, int dtype,
                                                    int64_t Tq, int64_t Tk, int Hq, int Hkv, int d,
                                                    const int32_t *cu_seqlens_q, const int32_t *cu_seqlens_k,
                                                    int nseg, const int32_t *q_pos, const int32_t *k_pos,
                                                    int causal, int window, float scale, float *out, float *lse,
                                                    void *stream) {
    using namespace ra;
    const size_t need = ra_partial_workspace_bytes(Tq, Tk, nseg, Hq, Hkv, d, dtype);
    if (need > RA_NOALLOC_SCRATCH_BYTES)
        return fail(RA_ERR_WORKSPACE, "problem needs " + std::to_string(need) +
                                          " bytes of scratch, more than the static " +
                                          std::to_string((size_t)RA_NOALLOC_SCRATCH_BYTES) +
                                          " bytes; use ra_varlen_attn_partial with a caller workspace");
    void *scratch = nullptr;
    ra_status st = scratch_address(stream, &scratch);
    if (st) return st;
    // Every table the kernel reads is rewritten by this call (uploaded on
    // `stream` before the launch), so nothing in the shared array has to
    // start at zero.  Calls that overlap on the GPU share the array and race.
    return ra_varlen_attn_partial(q, k, v, dtype, Tq, Tk, Hq, Hkv, d, cu_seqlens_q, cu_seqlens_k, nseg, q_pos,
                                  k_pos, causal, window, scale, out, lse, scratch, RA_NOALLOC_SCRATCH_BYTES, stream);
}
