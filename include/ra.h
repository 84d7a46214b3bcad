/*
 * ra.h -- C ABI of libra: packed causal varlen ring attention with zigzag
 * context-parallel (CP) load balancing, for NVIDIA GB300 (sm_103a).
 *
 * All CP ranks are simulated on one GPU: rank r's shard is the slice
 * [off[r], off[r+1]) of one zigzag-permuted buffer, and a ring step that
 * "receives" rank s's K/V reads that slice in place.
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 *  - Layout "THD": a token-major tensor [T, H, d], row-major, d contiguous
 *    (the packed layout of flash_attn_varlen_* named in "Attention Mask for
 *    Packed Sequences (via Attention Bias)", EasyDeL #129).
 *  - cu_seqlens: int32 cumulative document lengths, B+1 entries, cu[0] = 0,
 *    non-decreasing, cu[B] = T.  Documents never attend to each other
 *    (same page, opening request).
 *  - GQA: Hq = G * Hkv; query head h reads KV head floor(h / G).
 *  - LSE: natural-log log-sum-exp of the scaled scores, fp32, layout [Hq, T]
 *    (row h holds all tokens of head h).  A row with no allowed key has
 *    lse = -inf and output 0.
 *  - Device pointers must be 16-byte aligned.  "HOST" marks host arrays.
 *  - Every call is asynchronous on `stream` (a cudaStream_t; NULL = legacy
 *    default stream) unless it says otherwise.  The caller owns and
 *    allocates every device buffer, including the workspace; the library
 *    allocates no device memory.
 *  - Errors: argument checks happen on the host before any launch and
 *    return RA_ERR_INVALID_ARG / RA_ERR_UNSUPPORTED / RA_ERR_WORKSPACE with
 *    nothing launched; a failed launch returns RA_ERR_CUDA.  Device-side
 *    faults the kernels detect themselves (a wait that gave up, an index
 *    out of range) are recorded in a status word read by
 *    ra_get_device_status().  ra_last_error() gives a one-line detail of the
 *    last failure on the calling host thread.
 */
#ifndef RA_H_
#define RA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef int ra_status;
enum {
    RA_OK = 0,
    RA_ERR_INVALID_ARG = 1,   /* bad shape, cu_seqlens, pointer, cp, mode   */
    RA_ERR_UNSUPPORTED = 2,   /* valid but not implemented (dtype, d, align) */
    RA_ERR_CUDA = 3,          /* a CUDA runtime call or launch failed       */
    RA_ERR_WORKSPACE = 4,     /* workspace NULL or smaller than required    */
    RA_ERR_TIMEOUT = 5,       /* a device-side wait gave up (status word)   */
    RA_ERR_DEVICE_BOUNDS = 6  /* a kernel caught an out-of-range index      */
};

enum { RA_ZZ_GLOBAL = 0, RA_ZZ_PER_DOC = 1 };        /* zigzag modes       */
enum { RA_BF16 = 0, RA_FP32 = 1 };                   /* element types      */
enum { RA_SCHED_FUSED = 0, RA_SCHED_STEPWISE = 1, RA_SCHED_ALLGATHER = 2 };  /* CP schedules */

/* ------------------------------------------------------------------------
 * ra_zigzag_plan  (HOST, synchronous, no GPU needed)
 *
 * The zigzag split of ring-attention-pytorch #20 ("Zigzag attention
 * support?", the `extract_local` snippet) and maxtext PR #1133 (review
 * comment on load-balanced reordering): a stream of L tokens is cut into
 * n = 2*cp chunks, chunk c = [floor(c*L/n), floor((c+1)*L/n)), and rank r
 * holds chunks r and n-1-r.  When n does not divide L this balanced split
 * is used (chunks differ by at most one token; some may be empty).
 *   mode RA_ZZ_GLOBAL : the stream is the whole packed batch (T tokens).
 *   mode RA_ZZ_PER_DOC: every document is split on its own ("Question about
 *                       varlen ring attention", MiniMax-01 #6, notes that
 *                       zigzag under packing is the hard case).
 * Local token order is increasing packed index in both modes.
 *
 *   cu_seqlens HOST [B+1]             in
 *   perm       HOST [T]     int32     out: perm[i] = packed index of the
 *                                     token in permuted slot i
 *   off        HOST [cp+1]  int32     out: rank r owns slots [off[r], off[r+1])
 *   cu_local   HOST [cp*(B+1)] int32  out: rank r's local cu_seqlens (entry
 *                                     r*(B+1)+b); zero-length docs allowed
 * ------------------------------------------------------------------------ */
ra_status ra_zigzag_plan(const int32_t *cu_seqlens, int B, int cp, int mode,
                         int32_t *perm, int32_t *off, int32_t *cu_local);

/* ------------------------------------------------------------------------
 * ra_zigzag_permute / ra_zigzag_unpermute  (DEVICE)
 *
 * Applies the reordering the maxtext PR #1133 review says the framework
 * must perform before load-balanced CP attention (and undo afterwards):
 *   permute:    y[i, :] = x[perm[i], :]      for i in [0, T)
 *   unpermute:  x[perm[i], :] = y[i, :]
 * Rows are `row_bytes` bytes (H*d*element size for THD tensors); the copy
 * is bit-exact.  perm is a DEVICE int32 array [T] that must be a
 * permutation of [0, T) (an entry outside [0, T) is skipped and recorded
 * as RA_ERR_DEVICE_BOUNDS).  x and y must not overlap.
 * ------------------------------------------------------------------------ */
ra_status ra_zigzag_permute(const void *x, void *y, const int32_t *perm,
                            int64_t T, int64_t row_bytes, void *stream);
ra_status ra_zigzag_unpermute(const void *y, void *x, const int32_t *perm,
                              int64_t T, int64_t row_bytes, void *stream);

/* ------------------------------------------------------------------------
 * ra_varlen_attn_partial  (DEVICE tensors, HOST segment/position arrays)
 *
 * One ring step's attention: local queries against one KV shard, returning
 * the normalised output and its LSE so that partials can be merged
 * ("[Train] Support custom attention with context parallel", FlagScale
 * PR #910: RingAttention with a swappable forward_impl; this is that
 * step).  Allowed pairs:
 *   (i, j) with seg(i) == seg(j) and (causal == 0 or k_pos[j] <= q_pos[i])
 *          and (window < 0 or k_pos[j] >= q_pos[i] - window),
 * where seg is given by cu_seqlens_q / cu_seqlens_k (segment b of Q pairs
 * with segment b of K, nseg segments each).  window: the sliding window,
 * the number of positions a key may lie behind its query (the window_size
 * argument of the cuDNN flash-attention call in "Add Context Parallelism
 * support to cudnn Flash Attention #1133", maxtext); -1 = no window.
 *   q   DEVICE [Tq, Hq, d]      dtype RA_BF16 or RA_FP32
 *   k,v DEVICE [Tk, Hkv, d]     same dtype
 *   cu_seqlens_q, cu_seqlens_k  HOST [nseg+1]
 *   q_pos HOST [Tq], k_pos HOST [Tk]  int32 positions used by the causal
 *                               test (NULL = the local row index)
 *   out DEVICE [Tq, Hq, d] fp32, lse DEVICE [Hq, Tq] fp32 (written in full)
 *   workspace DEVICE, >= ra_partial_workspace_bytes(...) bytes
 * bf16 with d = 128 and G a power of two <= 16 runs on the tensor cores
 * (tcgen05, fp32 accumulation); other shapes and fp32 run a SIMT fp32 path.
 * Host arrays: every call tiles its segments on the host (O(Tq + Tk) work
 * plus O(query tiles x KV tiles) to classify tile pairs) and copies the
 * tables into the workspace on `stream` from host memory, so a call on a
 * capturing stream is refused with RA_ERR_UNSUPPORTED before any work
 * (the ring calls, which cache their plans, can be captured).
 * ra_partial_workspace_bytes is a bound over every position pattern;
 * ra_partial_table_bytes gives the exact bytes the tables of one call take
 * (HOST, no GPU needed; 0 for invalid arguments) and never exceeds it.
 * ------------------------------------------------------------------------ */
size_t ra_partial_workspace_bytes(int64_t Tq, int64_t Tk, int nseg, int Hq, int Hkv, int d, int dtype);
size_t ra_partial_table_bytes(int64_t Tq, int64_t Tk, int Hq, int Hkv, int d, int dtype,
                              const int32_t *cu_seqlens_q, const int32_t *cu_seqlens_k, int nseg,
                              const int32_t *q_pos, const int32_t *k_pos, int causal, int window);
ra_status ra_varlen_attn_partial(const void *q, const void *k, const void *v, int dtype,
                                 int64_t Tq, int64_t Tk, int Hq, int Hkv, int d,
                                 const int32_t *cu_seqlens_q, const int32_t *cu_seqlens_k, int nseg,
                                 const int32_t *q_pos, const int32_t *k_pos,
                                 int causal, int window, float scale,
                                 float *out, float *lse,
                                 void *workspace, size_t ws_bytes, void *stream);

/* ------------------------------------------------------------------------
 * ra_varlen_attn_partial_dev  (DEVICE tensors and DEVICE segment/position
 * arrays)
 *
 * ra_varlen_attn_partial with cu_seqlens_q, cu_seqlens_k [nseg+1], q_pos
 * [Tq] and k_pos [Tk] (NULL = the local row index) in DEVICE memory, as a
 * ring step holds them: the tile tables are built on the GPU (one small
 * kernel, the host planner's tiling row for row) ahead of the tensor-core
 * kernel, so the call makes no host round trip and can be captured in a
 * CUDA graph.  Same allowed pairs, results and workspace bound
 * (ra_partial_workspace_bytes) as ra_varlen_attn_partial; with the same
 * inputs the results are bit-identical to it.  Tensor-core path only
 * (bf16, d = 128, Hq / Hkv a power of two <= 16; else RA_ERR_UNSUPPORTED).
 * The device arrays are checked on the device: segment boundaries that do
 * not start at 0, decrease, or do not end at Tq / Tk (and, with a window,
 * positions outside [0, 2^30)) are recorded as RA_ERR_DEVICE_BOUNDS in the
 * status word (ra_get_device_status) and leave out / lse unwritten.
 * ------------------------------------------------------------------------ */
ra_status ra_varlen_attn_partial_dev(const void *q, const void *k, const void *v, int dtype,
                                     int64_t Tq, int64_t Tk, int Hq, int Hkv, int d,
                                     const int32_t *cu_seqlens_q, const int32_t *cu_seqlens_k, int nseg,
                                     const int32_t *q_pos, const int32_t *k_pos,
                                     int causal, int window, float scale,
                                     float *out, float *lse,
                                     void *workspace, size_t ws_bytes, void *stream);

/* ------------------------------------------------------------------------
 * ra_varlen_attn_partial_noalloc  (DEVICE tensors, HOST segment/position
 * arrays) -- the pages have no counterpart; this is a library convenience.
 *
 * The same computation, arguments and results as ra_varlen_attn_partial,
 * for callers that cannot allocate device memory: a runtime whose memory
 * pool already owns the GPU, a plugin that is handed only its input and
 * output buffers, or code that must not risk the implicit device
 * synchronisation cudaMalloc / cudaFree can cause.  Instead of a caller
 * workspace it uses a static device array of RA_NOALLOC_SCRATCH_BYTES
 * (8 MiB) that every GPU which loads the library holds until the process
 * exits; this call allocates nothing.
 *  - Size limit: a problem whose ra_partial_workspace_bytes(...) exceeds
 *    RA_NOALLOC_SCRATCH_BYTES is rejected with RA_ERR_WORKSPACE (the detail
 *    in ra_last_error() names both sizes); nothing is launched.
 *  - Set-up: the first call on a device (with that device current) looks up
 *    the array's device address and caches it.  Make that first call before
 *    any stream capture.  `stream` must belong to the current device (a
 *    stream of another device is rejected with RA_ERR_INVALID_ARG).  The
 *    cached address lives as long as the device's context: a
 *    cudaDeviceReset after the first call is not supported.
 *  - Sharing: all calls on a device share the one array, which keeps the
 *    last call's contents.  Each call rewrites every table it reads, so no
 *    state carries over, but calls that overlap on the GPU (different
 *    streams, or host threads) race on the array: serialise them.
 * ------------------------------------------------------------------------ */
#define RA_NOALLOC_SCRATCH_BYTES (8u << 20)
ra_status ra_varlen_attn_partial_noalloc(const void *q, const void *k, const void *v, int dtype,
                                         int64_t Tq, int64_t Tk, int Hq, int Hkv, int d,
                                         const int32_t *cu_seqlens_q, const int32_t *cu_seqlens_k, int nseg,
                                         const int32_t *q_pos, const int32_t *k_pos,
                                         int causal, int window, float scale,
                                         float *out, float *lse, void *stream);

/* ------------------------------------------------------------------------
 * ra_lse_merge  (DEVICE)
 *
 * Merges n_parts partial results of the same queries over disjoint key
 * sets (the step that combines ring partials; the pages name the ring
 * schedule, the merge is its textbook completion):
 *   M = max_p lse_p;  lse = M + log(sum_p exp(lse_p - M));
 *   out = sum_p exp(lse_p - lse) * out_p;   all -inf -> out 0, lse -inf.
 *   outs  HOST array [n_parts] of DEVICE fp32 [Tq, Hq, d] pointers
 *   lses  HOST array [n_parts] of DEVICE fp32 [Hq, Tq] pointers
 *   out   DEVICE [Tq, Hq, d] of out_dtype (RA_BF16 or RA_FP32)
 *   lse_out DEVICE [Hq, Tq] fp32 (may be NULL)
 * 1 <= n_parts <= 64, d a multiple of 4 and <= 256.  out may alias
 * outs[0] when out_dtype is RA_FP32 (each element is read before written).
 * ------------------------------------------------------------------------ */
ra_status ra_lse_merge(int n_parts, const float *const *outs, const float *const *lses,
                       int64_t Tq, int Hq, int d, void *out, int out_dtype, float *lse_out,
                       void *stream);

/* ------------------------------------------------------------------------
 * ra_ring_attn_fwd / ra_ring_attn_bwd  (DEVICE tensors, HOST cu_seqlens)
 *
 * The whole simulated ring: zigzag-permute Q/K/V, run the ring over cp
 * simulated ranks (rank r at step t attends to the K/V of rank
 * s = (r - t) mod cp), merge, and return results in the ORIGINAL token
 * order.
 *   sched RA_SCHED_FUSED    : one launch per direction; the ring steps are
 *                             the order in which each query tile visits KV
 *                             tiles and the merge is the on-chip online
 *                             softmax.  Fully masked tiles are skipped
 *                             (pruning, FlagScale PR #910).
 *   sched RA_SCHED_STEPWISE : one partial launch per ring step into fp32
 *                             buffers, then ra_lse_merge and unpermute
 *                             (backward: fp32 dK/dV accumulated per step).
 *   sched RA_SCHED_ALLGATHER: the all-gather form of context parallelism
 *                             (K/V of every rank gathered, then one pass of
 *                             each rank's zigzag queries over them: the
 *                             Llama 3 scheme discussed in "Zigzag attention
 *                             support?", ring-attention-pytorch issue #20,
 *                             and the Transformer-Engine path of maxtext PR
 *                             #1133).  The gathered K/V are the documents in
 *                             original order, tiled per document, so they
 *                             are read in place and never permuted.  Same
 *                             attention as the ring; only the tiling of
 *                             the key side and the rounding order differ.
 *                             Without tensor-core kernels (fp32, other
 *                             shapes) it runs as RA_SCHED_FUSED.
 * Forward:
 *   q DEVICE [T, Hq, d], k, v DEVICE [T, Hkv, d] (dtype), out DEVICE
 *   [T, Hq, d] (dtype), lse DEVICE [Hq, T] fp32.
 * Backward (from the saved lse, textbook gradient):
 *   out, dout DEVICE [T, Hq, d] (dtype), lse DEVICE [Hq, T];
 *   dq DEVICE [T, Hq, d], dk, dv DEVICE [T, Hkv, d] of grad_dtype
 *   (RA_BF16 or RA_FP32; dK/dV are always accumulated in fp32).
 * scale: softmax scale; pass 1/sqrt(d) for the usual attention (maxtext
 * PR #1133, cudnn_flash_attention diff).  cp >= 1.  window: sliding window
 * as in ra_varlen_attn_partial (-1 = none); positions are the original
 * (unpermuted) token indices, so the zigzag reorder leaves the mask intact.
 * workspace: DEVICE, >= ra_ring_workspace_bytes(...) for the same arguments
 * (the size holds for every causal and window setting: the planner's KV
 * tiling, which the mask selects, only changes the size of its tables and
 * the size covers every tiling).  ra_ring_workspace_bytes counts tiles on
 * the host (well under a millisecond for 32768 tokens) and keeps no state;
 * it returns 0 for invalid arguments.
 * On the tensor-core path (bf16, d = 128) the kernels read every tile whose
 * rows form one position run straight from q, k, v (and dout), and the
 * workspace receives rank-ordered copies of the rows of the other tiles
 * only (those that straddle two zigzag chunks); ra_zigzag_permute gives the
 * whole rank-ordered tensor where a caller needs it.
 * Asynchronous on `stream`.  The backward's fused tensor-core path runs its
 * key-side kernel on a second, library-owned stream forked from and joined
 * back to `stream` through events.  Both calls may be captured into a CUDA
 * graph once an uncaptured call with the same cu_seqlens, cp, zz_mode and
 * heads has run (it makes the page-locked table copy and the second
 * stream); otherwise a captured call returns RA_ERR_UNSUPPORTED.
 * ------------------------------------------------------------------------ */
size_t ra_ring_workspace_bytes(int64_t T, int Hq, int Hkv, int d, int dtype,
                               const int32_t *cu_seqlens, int B, int cp, int zz_mode,
                               int sched, int bwd);
ra_status ra_ring_attn_fwd(const void *q, const void *k, const void *v, int dtype,
                           int64_t T, int Hq, int Hkv, int d,
                           const int32_t *cu_seqlens, int B, int cp, int zz_mode,
                           int causal, int window, float scale, int sched,
                           void *out, float *lse,
                           void *workspace, size_t ws_bytes, void *stream);
/* flags of ra_ring_attn_bwd.
 * RA_BWD_FWD_RESERVE: the workspace is a reserve space left by the
 * preceding ra_ring_attn_fwd on the same stream with the same q, k, v
 * (unmodified), dtype, shapes, cu_seqlens, cp, zz_mode, causal and sched,
 * and nothing has written into it since: the rank-ordered Q, K, V rows and
 * the tile tables it holds are reused instead of rebuilt (they are the
 * forward's saved activations).  The library checks on the host that the
 * last forward on this workspace had the same pointers and plan and
 * ignores the flag otherwise; it cannot see changes to the contents. */
#define RA_BWD_FWD_RESERVE 1
ra_status ra_ring_attn_bwd(const void *q, const void *k, const void *v, int dtype,
                           int64_t T, int Hq, int Hkv, int d,
                           const int32_t *cu_seqlens, int B, int cp, int zz_mode,
                           int causal, int window, float scale, int sched,
                           const void *out, const float *lse, const void *dout,
                           void *dq, void *dk, void *dv, int grad_dtype, int flags,
                           void *workspace, size_t ws_bytes, void *stream);

/* ------------------------------------------------------------------------
 * ra_ring_attn_fwd_masked / ra_ring_attn_bwd_masked  (DEVICE tensors, HOST
 * cu_seqlens and bounds)
 *
 * The ring of ra_ring_attn_fwd / bwd under an interval mask instead of the
 * causal flag and the window: the dynamic, per-token attention masks that
 * "[Train] Support custom attention with context parallel" (FlagScale PR
 * #910, description) adds to context parallelism through flex attention,
 * in the form of one key interval per query token:
 *   query i sees key j  iff  same document  and  key_lo[i] <= j <= key_hi[i]
 * (original token indices).  This holds causal (lo = document start,
 * hi = i), sliding-window, chunked-local, prefix-LM (hi = max(i, end of
 * the prefix)) and bidirectional document masks.
 *   key_lo, key_hi HOST int32 [T]: both non-decreasing inside every
 *                  document (else RA_ERR_INVALID_ARG), values in
 *                  (-2^30, 2^30); a row with no key inside its interval
 *                  gets output 0 and lse -inf.
 * Fully masked tile pairs are skipped and fully visible ones run unmasked:
 * the block map comes from each query tile's bound extremes (the pruning
 * of the same PR).  Everything else is as in ra_ring_attn_fwd / bwd, with
 * these limits: the tensor-core path only (bf16, d = 128, Hq / Hkv a power
 * of two <= 16) and the RA_SCHED_FUSED or RA_SCHED_ALLGATHER schedule
 * (otherwise RA_ERR_UNSUPPORTED).  The plan (and so the workspace size)
 * depends on the bounds: size the workspace with
 * ra_ring_workspace_bytes_masked for the same bounds.
 * ------------------------------------------------------------------------ */
size_t ra_ring_workspace_bytes_masked(int64_t T, int Hq, int Hkv, int d, int dtype,
                                      const int32_t *cu_seqlens, int B, int cp, int zz_mode,
                                      const int32_t *key_lo, const int32_t *key_hi, int sched, int bwd);
ra_status ra_ring_attn_fwd_masked(const void *q, const void *k, const void *v, int dtype,
                                  int64_t T, int Hq, int Hkv, int d,
                                  const int32_t *cu_seqlens, int B, int cp, int zz_mode,
                                  const int32_t *key_lo, const int32_t *key_hi, float scale, int sched,
                                  void *out, float *lse, void *workspace, size_t ws_bytes, void *stream);
ra_status ra_ring_attn_bwd_masked(const void *q, const void *k, const void *v, int dtype,
                                  int64_t T, int Hq, int Hkv, int d,
                                  const int32_t *cu_seqlens, int B, int cp, int zz_mode,
                                  const int32_t *key_lo, const int32_t *key_hi, float scale, int sched,
                                  const void *out, const float *lse, const void *dout,
                                  void *dq, void *dk, void *dv, int grad_dtype, int flags,
                                  void *workspace, size_t ws_bytes, void *stream);

/* ------------------------------------------------------------------------
 * ra_ring_rank_pairs  (HOST, synchronous)
 *
 * Allowed (query, key) pairs each simulated rank computes over the whole
 * ring: the causal load that zigzag balances ("Question about varlen ring
 * attention", MiniMax-01 #6: causal imbalance; ring-attention-pytorch #20:
 * zigzag spreads it).  window as in ra_varlen_attn_partial (-1 = none).
 * counts HOST [cp] int64.
 * ------------------------------------------------------------------------ */
ra_status ra_ring_rank_pairs(const int32_t *cu_seqlens, int B, int cp, int zz_mode, int causal, int window,
                             int64_t *counts);

/* ------------------------------------------------------------------------
 * ra_ring_plan_stats  (HOST only; no GPU needed)
 *
 * What the tensor-core passes of ra_ring_attn_fwd / bwd visit for a packing
 * (bf16, d = 128; G = Hq / Hkv a power of two dividing 128), found by
 * walking every work item over its range of ring steps with the kernels'
 * own step-to-rank rule and tile classifier (tile-level skipping of fully
 * masked blocks, FlagScale PR #910).  stats HOST int64[RA_PLAN_STATS_N]:
 *   [0] query tiles (128/G tokens x G heads)   [1] key tiles (128 keys)
 *   [2] forward items  [3] dK/dV items  [4] dQ items (all KV heads)
 *   [5] forward visited (query tile, key tile) pairs, one KV head
 *   [6]   of which full (no mask inside)
 *   [7] rows of two-run query tiles  [8] rows of two-run key tiles
 *       (the rows the permutes copy into rank order)
 *   [9] token-pair capacity of the forward's visited pairs
 *       ([5] x 128/G x 128: the tensor work per head group / (2 d G))
 *   exact != 0 (brute force over the visited pairs; else -1):
 *   [10] allowed (query token, key) pairs inside the forward's visited pairs
 *   [11] disallowed pairs among valid rows and keys of "full" pairs
 *   [12] allowed pairs inside the dK/dV pass's visited pairs
 *   [13] allowed pairs inside the dQ pass's visited pairs
 *   [14] dK/dV visited pairs  [15] dQ visited pairs
 *   scheduling model over n_sm SMs, in tile-pair visits per SM (all KV
 *   heads; the ideal is the pass's total visits / n_sm):
 *   [16] forward (persistent CTAs claiming items in order)
 *   [17] dK/dV (one CTA per item, dispatched in order as SMs free up)
 *   [18] dQ (persistent CTAs, static stride over the items)
 *   [19] forward KV steps: KV tiles the forward items of one KV head walk
 *        with a product of either query tile ([5] counts one per query tile)
 * A correct plan covers each allowed pair once in every pass: [10], [12]
 * and [13] equal the sum of ra_ring_rank_pairs, and [11] is 0.
 * ------------------------------------------------------------------------ */
#define RA_PLAN_STATS_N 20
ra_status ra_ring_plan_stats(const int32_t *cu_seqlens, int B, int cp, int zz_mode, int G, int Hkv, int causal,
                             int window, int sched, int exact, int n_sm, int64_t *stats);
/* The same statistics under an interval mask (key_lo / key_hi as in
 * ra_ring_attn_fwd_masked; RA_SCHED_FUSED or RA_SCHED_ALLGATHER). */
ra_status ra_ring_plan_stats_masked(const int32_t *cu_seqlens, int B, int cp, int zz_mode, int G, int Hkv,
                                    const int32_t *key_lo, const int32_t *key_hi, int sched, int exact, int n_sm,
                                    int64_t *stats);

/* Reads and clears the device status word of the current device (waits for
 * `stream` first).  Returns RA_OK, RA_ERR_TIMEOUT or RA_ERR_DEVICE_BOUNDS. */
ra_status ra_get_device_status(void *stream);

/* Self-test of the device-wait guard: launches one CTA that waits on an
 * mbarrier nothing ever arrives at, with a budget of `budget_us`
 * microseconds (1..1000000).  The wait runs out, the kernel records
 * RA_ERR_TIMEOUT in the status word and returns; no copy or MMA is in
 * flight.  Read the result with ra_get_device_status().  Every real kernel
 * uses the same guard (2 s budget) on each of its waits. */
ra_status ra_selftest_wait_timeout(int64_t budget_us, void *stream);

/* ------------------------------------------------------------------------
 * Per-kernel timing (HOST).  While enabled, every kernel launch the library
 * makes is bracketed by two CUDA events recorded on its launching stream.
 * ra_profile_enable(1) clears earlier records; ra_profile_read waits for
 * the recorded events and reports, per kernel name (at most max_kernels,
 * names written as NUL-terminated strings of up to 64 bytes each into
 * `names`), the summed device time in ms and the launch count.  Returns
 * the number of kernels reported, or -1 on error.  Timing adds two event
 * records per launch; keep it off for throughput runs.  Independently of
 * this switch, each timed unit (a kernel launch, or the concurrent backward
 * pair "ra_tc_bwd") is also an NVTX range of the same name pushed on the
 * calling host thread, so a timeline tool shows the phases of a step and,
 * in STEPWISE mode, one range per ring step; with no tool attached the
 * range calls do nothing.
 * ------------------------------------------------------------------------ */
ra_status ra_profile_enable(int on);
int ra_profile_read(int max_kernels, char *names, double *total_ms, int64_t *launches);

const char *ra_status_string(ra_status s);
const char *ra_last_error(void);
const char *ra_version(void);

#ifdef __cplusplus
}
#endif
#endif /* RA_H_ */
