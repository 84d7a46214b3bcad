// ra_kernels.h -- launch interfaces of the library's kernels (host side).
// Included by the C-ABI drivers and by the .cu files that implement them.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <cstdint>

#include "../../include/ra.h"

namespace ra {

// ------------------------------------------------------------ status word
int *device_status_ptr();          // device address of this device's status word
uint64_t wait_budget_ns();         // budget of every device-side wait

// ------------------------------------------------------------ timing
// Brackets one launch with CUDA events on `st` when profiling is enabled.
class ProfScope {
  public:
    ProfScope(const char *name, cudaStream_t st);
    ~ProfScope();

  private:
    int id_ = -1;
    cudaStream_t st_;
};

// ------------------------------------------------------------ permute
struct PermJob {
    const void *src;
    void *dst;
    int64_t row_bytes;
    const uint8_t *only = nullptr;  // T bytes: move just the rows i with only[i] != 0
};
// inverse = 0: dst[i] = src[perm[i]];  inverse = 1: dst[perm[i]] = src[i].
// Up to 4 jobs share one launch (same perm, same T).
cudaError_t launch_permute(const PermJob *jobs, int njobs, const int32_t *perm, int64_t T, int inverse,
                           cudaStream_t st);
// [H, T] fp32: x[h, perm[i]] = y[h, i].
cudaError_t launch_unpermute_cols(const float *y, float *x, const int32_t *perm, int64_t T, int H,
                                  cudaStream_t st);

// ------------------------------------------------------------ merge & misc
constexpr int kMaxMergeParts = 64;
cudaError_t launch_merge(int n, const float *const *outs, const float *const *lses, int64_t Tq, int Hq, int d,
                         void *out, int out_dtype, float *lse_out, cudaStream_t st);
// D[h, t] = sum_c a[t, h, c] * b[t, h, c]   (a, b of dtype; fp32 result)
// Backward preprocess of bf16 tensors with head dim 128, one pass: permute
// the jobs (Q, K, V) and dO (dout -> dout_p, Hq heads) by perm, and
// D[h, p] = sum_c dO[p, h, c] * O[p, h, c] in fp32 at original rows p.
// All pointers and row sizes must be 16-byte aligned (else cudaErrorInvalidValue).
// With dout_only (T bytes) given, dout_p receives just the rows i with
// dout_only[i] != 0 (D is written for every row).
// Copies n bytes from page-locked host memory (mapped into the device's
// address space) to device memory with a kernel, so the copy never queues
// behind other streams' transfers on a copy engine.  src and dst must be
// 16-byte aligned (else cudaErrorInvalidValue).
cudaError_t launch_copy_from_host(const void *src, void *dst, size_t n, cudaStream_t st);
cudaError_t launch_permute_rowdot(const PermJob *jobs, int njobs, const void *dout, void *dout_p, const void *out,
                                  float *D, const int32_t *perm, int64_t T, int Hq, cudaStream_t st,
                                  const uint8_t *dout_only = nullptr);
cudaError_t launch_rowdot(const void *a, const void *b, int dtype, int64_t T, int H, int d, float *D,
                          cudaStream_t st);
// Per (query tile, KV head): 128 columns of -lse*log2(e) (-inf for empty
// rows) then 128 of -D*scale, contiguous (1 KB per tile and head), for the
// key-side backward's bulk copies.
cudaError_t launch_tile_lse_d(const void *qtiles, int n_qtiles, int Hkv, int G, const float *lse, const float *D,
                              int64_t lse_T, float scale, float *out, cudaStream_t st);
// dst (dtype) = src (fp32), n elements.
cudaError_t launch_cast_f32(const float *src, void *dst, int dtype, int64_t n, cudaStream_t st);

// ------------------------------------------------------------ attention
// Where an attention kernel writes its rows.
enum OutMode {
    kOutFinal = 0,    // dtype output at row = position (original order), lse[h*lse_T + position]
    kOutPartial = 1,  // fp32 output at the local row, lse[h*lse_T + local row]
};

// A ring over `cp` simulated ranks.  Query rows of rank r, segment b are
// [qoff[r] + qcul[r*(B+1)+b], qoff[r] + qcul[r*(B+1)+b+1]); key rows of rank s
// likewise with koff/kcul.  Positions (for the causal test and for kOutFinal
// rows) come from qpos / kpos.
struct SimtArgs {
    const void *q, *k, *v;
    int dtype, Hq, Hkv, d;
    int64_t Tq, Tk;
    const int32_t *qoff, *qcul, *qpos;
    const int32_t *koff, *kcul, *kpos;
    int cp, B, t0, t1;
    int causal;
    int window;                        // sliding window (keys at most this far behind), < 0: none
    float scale;
    int out_mode;
    void *out;
    float *lse;
    int64_t lse_T;
};
cudaError_t launch_simt_fwd(const SimtArgs &a, cudaStream_t st);

struct SimtBwdArgs {
    const void *q, *k, *v, *dout;
    int dtype, Hq, Hkv, d;
    int64_t T;                         // rows of the permuted buffers
    const int32_t *off, *cul, *pos;    // ring over cp ranks, q side = k side
    int cp, B, t0, t1;
    int causal;
    int window;                        // sliding window (keys at most this far behind), < 0: none
    float scale;
    const float *lse, *D;              // [Hq, lse_T] indexed by position
    int64_t lse_T;
    float *dq;                         // fp32 [T_orig, Hq, d] at position rows (+=)
    float *dk, *dv;                    // fp32 [T_orig, Hkv, d] at position rows (+=)
};
cudaError_t launch_simt_bwd(const SimtBwdArgs &a, cudaStream_t st);

// Tensor-core forward (bf16, d = 128).
struct TcFwdArgs {
    const void *q, *k, *v;             // permuted buffers
    const void *q_orig, *k_orig, *v_orig;  // nullable: Q / K and V in original order
                                       // (rows = positions); single-run tiles are read from them
    int64_t Tq, Tk;
    int Hq, Hkv, G;
    const void *qtiles, *kvtiles;      // Tile records (two int4 each)
    const int32_t *kv_off;             // [cp*(B+1)+1]
    const void *items;                 // WorkItem records
    int *sched;                        // [2] work counter, zero before the first launch
    int n_items;                       // item count (an upper bound when n_items_dev is given)
    const int *n_items_dev;            // nullable: the item count in device memory
    int cp, B;
    int t0, t1;                        // >= 0: override every item's step range
    int causal;
    int window;                        // sliding window (keys at most this far behind), < 0: none
    const void *qbounds;               // interval masks (else NULL): QBounds per query tile,
    const int32_t *key_lo, *key_hi;    // and each token's key bounds [Tq] at its original position
    float scale;
    int out_mode;
    void *out;
    float *lse;
    int64_t lse_T;
};
cudaError_t launch_tc_fwd(const TcFwdArgs &a, cudaStream_t st);
bool tc_fwd_supported(int dtype, int d, int Hq, int Hkv);

// Tensor-core key-side backward (bf16, d = 128): dK and dV, one CTA per KV
// tile and KV head.  out_mode: 0 bf16 store, 1 fp32 store, 2 fp32 +=.
struct TcBwdArgs {
    const void *q, *k, *v, *dout;      // permuted buffers
    const void *q_orig, *dout_orig;    // nullable pair: Q and dO in original order, read for
                                       // single-run query tiles
    const void *k_orig, *v_orig;       // nullable pair: K and V likewise for KV tiles
    int64_t T;
    int Hq, Hkv, G;
    const void *qtiles, *kvtiles;      // Tile records
    const int32_t *q_off;              // [cp*(B+1)+1]
    const void *items;                 // key-side WorkItem records (qt0 = KV tile)
    int n_items;
    int cp, B;
    int t0, t1;                        // >= 0: override every item's step range
    int causal;
    int window;                        // sliding window (keys at most this far behind), < 0: none
    const void *qbounds;               // interval masks (else NULL), as in TcFwdArgs
    const int32_t *key_lo, *key_hi;
    float scale;
    const float *tile_ld;              // launch_tile_lse_d output for these tiles
    void *dk, *dv;                     // [T, Hkv, d] at original positions
    int out_mode;
};
cudaError_t launch_tc_bwd(const TcBwdArgs &a, cudaStream_t st);

// Tensor-core dQ pass (bf16, d = 128): one CTA per query tile and KV head;
// no atomics.  out_mode: 0 bf16 store, 1 fp32 store, 2 fp32 +=.
struct TcDqArgs {
    const void *q, *k, *v, *dout;      // permuted buffers
    const void *q_orig, *dout_orig;    // nullable pairs, as in TcBwdArgs
    const void *k_orig, *v_orig;
    int64_t T;
    int Hq, Hkv, G;
    const void *qtiles, *kvtiles;
    const int32_t *kv_off;
    const void *items;                 // dQ WorkItem records (qt0 = query tile)
    int n_items;
    int cp, B;
    int t0, t1;
    int causal;
    int window;                        // sliding window (keys at most this far behind), < 0: none
    const void *qbounds;               // interval masks (else NULL), as in TcFwdArgs
    const int32_t *key_lo, *key_hi;
    float scale;
    const float *lse, *D;              // [Hq, lse_T] at original positions
    int64_t lse_T;
    void *dq;                          // [T, Hq, d] at original positions
    int out_mode;
};
cudaError_t launch_tc_dq(const TcDqArgs &a, cudaStream_t st);

// ------------------------------------------------------------ device tile tables
// The tile tables of one partial call built on the device (ra_tile_build.cu):
// query tiles of q_rows rows and KV tiles of 128 rows, at most two position
// runs each, per segment; forward items (pairs of query tiles x KV heads,
// head major), their count in *n_items and the work counter zeroed.  Tables
// sized by the host bound (a tile holds at least one row).  Malformed
// segment boundaries (or, with check_pos, positions outside [0, 2^30)) are
// recorded as RA_ERR_DEVICE_BOUNDS and leave *n_items = 0.
struct DevTileArgs {
    const int32_t *cu_q, *cu_k;        // DEVICE [nseg + 1]
    const int32_t *q_pos, *k_pos;      // DEVICE [Tq], [Tk]; NULL = row index
    int64_t Tq, Tk;
    int nseg, Hkv, q_rows, check_pos;
    void *qtiles, *kvtiles, *items;    // Tile [Tq + nseg], Tile [Tk + nseg], WorkItem [pairs x Hkv]
    int32_t *q_off, *kv_off;           // [nseg + 2]
    int32_t *q_cnt, *k_cnt, *pair_off; // scratch [nseg], [nseg], [nseg + 1]
    int *n_items, *sched;              // 1 int, 2 ints
};
cudaError_t launch_tile_build(const DevTileArgs &a, cudaStream_t st);

// Device-wait self-test (see ra_selftest_wait_timeout).
cudaError_t launch_wait_selftest(uint64_t budget_ns, cudaStream_t st);

}  // namespace ra
