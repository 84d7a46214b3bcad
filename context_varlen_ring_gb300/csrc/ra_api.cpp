// ra_api.cpp -- the C ABI (include/ra.h): argument checks, plans, workspace
// carving and the drivers of the simulated ring.  Host code only; every
// step of the data path runs in the library's kernels.
#include <cuda_runtime.h>
#include <nvtx3/nvToolsExt.h>

#include <cmath>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <string>
#include <vector>

#include "ra_internal.h"
#include "ra_kernels.h"

namespace ra {

static thread_local std::string g_last_error;

ra_status fail(ra_status s, const std::string &msg) {
    g_last_error = msg;
    return s;
}

static ra_status cuda_fail(cudaError_t e, const char *what) {
    return fail(RA_ERR_CUDA, std::string(what) + ": " + cudaGetErrorString(e));
}

#define RA_CUDA(call, what)                             \
    do {                                                \
        cudaError_t e_ = (call);                        \
        if (e_ != cudaSuccess) return cuda_fail(e_, what); \
    } while (0)

// ---------------------------------------------------------------- timing
namespace {
struct ProfRec {
    std::string name;
    cudaEvent_t a, b;
};
std::mutex g_prof_mu;
bool g_prof_on = false;
std::vector<ProfRec> g_prof;
std::vector<cudaEvent_t> g_event_pool;

cudaEvent_t take_event() {
    if (!g_event_pool.empty()) {
        cudaEvent_t e = g_event_pool.back();
        g_event_pool.pop_back();
        return e;
    }
    cudaEvent_t e = nullptr;
    if (cudaEventCreate(&e) != cudaSuccess) return nullptr;
    return e;
}
}  // namespace

// Every scope is also an NVTX range (host side), so a timeline tool shows
// each phase and, in STEPWISE mode, each ring step by name; without a tool
// attached the range calls return at once.
ProfScope::ProfScope(const char *name, cudaStream_t st) : st_(st) {
    nvtxRangePushA(name);
    std::lock_guard<std::mutex> lk(g_prof_mu);
    if (!g_prof_on) return;
    cudaEvent_t a = take_event(), b = take_event();
    if (!a || !b) return;
    if (cudaEventRecord(a, st) != cudaSuccess) return;
    g_prof.push_back(ProfRec{name, a, b});
    id_ = (int)g_prof.size() - 1;
}

ProfScope::~ProfScope() {
    {
        std::lock_guard<std::mutex> lk(g_prof_mu);
        if (id_ >= 0 && id_ < (int)g_prof.size()) cudaEventRecord(g_prof[id_].b, st_);
    }
    nvtxRangePop();
}

static bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

static size_t esize(int dtype) { return dtype == RA_FP32 ? 4 : 2; }

static ra_status check_common(int dtype, int Hq, int Hkv, int d) {
    if (dtype != RA_BF16 && dtype != RA_FP32) return fail(RA_ERR_INVALID_ARG, "dtype must be RA_BF16 or RA_FP32");
    if (Hq <= 0 || Hkv <= 0 || Hq % Hkv != 0) return fail(RA_ERR_INVALID_ARG, "Hq must be a positive multiple of Hkv");
    if (d <= 0) return fail(RA_ERR_INVALID_ARG, "d must be positive");
    if (d % 32 != 0 || d > 256) return fail(RA_ERR_UNSUPPORTED, "d must be a multiple of 32 and <= 256");
    return RA_OK;
}

// Carves consecutive 256-byte aligned regions out of a workspace.
struct Carver {
    uint8_t *base;
    size_t used = 0;
    explicit Carver(void *b) : base(static_cast<uint8_t *>(b)) {}
    void *take(size_t bytes) {
        void *p = base ? base + used : nullptr;
        used = align_up(used + bytes, 256);
        return p;
    }
};

}  // namespace ra

using namespace ra;

namespace ra {

// Page-locked buffers of plans that left the cache, with the event of their
// last upload; a new plan reuses one once that upload has finished reading
// it.  Freeing page-locked memory would synchronise the device.
struct PinnedBuf {
    void *p;
    size_t n;
    void *ev;
    bool multi;
};
std::mutex g_pool_mu;
std::vector<PinnedBuf> g_pool;

static void pinned_buf_settle(const PinnedBuf &b) {
    if (b.multi) {
        (void)cudaDeviceSynchronize();  // uploads on several streams: rare
    } else if (b.ev) {
        (void)cudaEventSynchronize(static_cast<cudaEvent_t>(b.ev));
    }
    if (b.ev) (void)cudaEventDestroy(static_cast<cudaEvent_t>(b.ev));
}

static void *take_pinned(size_t n, size_t *got) {
    {
        std::lock_guard<std::mutex> lk(g_pool_mu);
        int best = -1;
        for (int i = 0; i < (int)g_pool.size(); ++i)
            if (g_pool[i].n >= n && (best < 0 || g_pool[i].n < g_pool[best].n)) best = i;
        if (best >= 0) {
            PinnedBuf b = g_pool[best];
            g_pool.erase(g_pool.begin() + best);
            pinned_buf_settle(b);
            *got = b.n;
            return b.p;
        }
    }
    const size_t sz = align_up(n, (size_t)1 << 16);
    void *h = nullptr;
    if (cudaMallocHost(&h, sz) != cudaSuccess) {
        (void)cudaGetLastError();
        return nullptr;
    }
    *got = sz;
    return h;
}

RingPlan::~RingPlan() {
    if (!pinned) return;
    if (in_graph) return;  // a captured graph may still copy from it
    std::lock_guard<std::mutex> lk(g_pool_mu);
    g_pool.push_back(PinnedBuf{pinned, pinned_bytes, uploaded, multi_stream});
    if (g_pool.size() > 32) {  // bound the pool: release the oldest
        PinnedBuf b = g_pool.front();
        g_pool.erase(g_pool.begin());
        pinned_buf_settle(b);
        (void)cudaFreeHost(b.p);
    }
}

ra_status upload_plan_tables(RingPlan &plan, void *dst, void *stream) {
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const size_t n = plan.dev.blob.size();
    if (n == 0) return RA_OK;
    std::lock_guard<std::mutex> lk(plan.pin_mu);
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(s, &cs) != cudaSuccess) {
        (void)cudaGetLastError();
        cs = cudaStreamCaptureStatusNone;
    }
    if (cs != cudaStreamCaptureStatusNone) {
        if (!plan.pinned)
            return fail(RA_ERR_UNSUPPORTED,
                        "stream capture: call once outside capture with these sequence lengths first "
                        "(the page-locked copy of the tables is made there)");
        plan.in_graph = true;
        RA_CUDA(launch_copy_from_host(plan.pinned, dst, n, s), "table upload");
        return RA_OK;
    }
    if (!plan.pinned) {
        plan.pinned = take_pinned(n, &plan.pinned_bytes);
        if (plan.pinned) std::memcpy(plan.pinned, plan.dev.blob.data(), n);
    }
    if (!plan.pinned) {  // no page-locked memory: pageable copy
        RA_CUDA(cudaMemcpyAsync(dst, plan.dev.blob.data(), n, cudaMemcpyHostToDevice, s), "table upload");
        return RA_OK;
    }
    // a kernel reads the mapped page-locked copy: a copy engine could queue
    // this small upload behind large transfers on other streams
    RA_CUDA(launch_copy_from_host(plan.pinned, dst, n, s), "table upload");
    if (!plan.uploaded) {
        cudaEvent_t e = nullptr;
        if (cudaEventCreateWithFlags(&e, cudaEventDisableTiming) == cudaSuccess) plan.uploaded = e;
        else (void)cudaGetLastError();
    }
    if (plan.upload_stream && plan.upload_stream != stream) plan.multi_stream = true;
    plan.upload_stream = stream;
    if (plan.uploaded) RA_CUDA(cudaEventRecord(static_cast<cudaEvent_t>(plan.uploaded), s), "upload event");
    else plan.multi_stream = true;  // nothing to wait on: settle by a device sync
    return RA_OK;
}

// A second stream per device, with a fork and a join event, for the query-side
// backward pass to run beside the key-side pass: both read the same inputs and
// write disjoint outputs.  The persistent dQ grid is issued first and holds one
// CTA per SM; each key-side CTA takes an SM as soon as the dQ CTA there
// retires, so the uneven ends of the dQ CTAs leave no SM idle.  The mutex is
// held across a whole fork/join so that another thread cannot re-record the
// events between a record and its wait.
struct SideStream {
    cudaStream_t st = nullptr;
    cudaEvent_t fork = nullptr, join = nullptr;
};
std::mutex g_side_mu;

SideStream *side_stream_locked(bool may_create) {
    static SideStream ss[128];
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 128) return nullptr;
    SideStream &s = ss[dev];
    if (!s.st) {
        if (!may_create) return nullptr;
        cudaStream_t st = nullptr;
        cudaEvent_t a = nullptr, b = nullptr;
        if (cudaStreamCreateWithFlags(&st, cudaStreamNonBlocking) != cudaSuccess ||
            cudaEventCreateWithFlags(&a, cudaEventDisableTiming) != cudaSuccess ||
            cudaEventCreateWithFlags(&b, cudaEventDisableTiming) != cudaSuccess) {
            (void)cudaGetLastError();
            if (st) (void)cudaStreamDestroy(st);
            if (a) (void)cudaEventDestroy(a);
            return nullptr;
        }
        s.st = st;
        s.fork = a;
        s.join = b;
    }
    return &s;
}

// Host record of what the last ring forward left in each workspace (the
// reserve space a backward may reuse with RA_BWD_FWD_RESERVE).
struct ReserveRec {
    const void *plan, *q, *k, *v;
    int dtype, Hq, Hkv, d, causal, sched;
    int64_t T;
};
static std::mutex g_reserve_mu;
static std::vector<std::pair<const void *, ReserveRec>> g_reserve;  // few workspaces, linear scan

void reserve_record(const void *ws, const void *plan, const void *q, const void *k, const void *v, int dtype,
                    int64_t T, int Hq, int Hkv, int d, int causal, int sched) {
    std::lock_guard<std::mutex> lk(g_reserve_mu);
    const ReserveRec r{plan, q, k, v, dtype, Hq, Hkv, d, causal, sched, T};
    for (auto &e : g_reserve)
        if (e.first == ws) {
            e.second = r;
            return;
        }
    if (g_reserve.size() >= 64) g_reserve.erase(g_reserve.begin());
    g_reserve.emplace_back(ws, r);
}

bool reserve_matches(const void *ws, const void *plan, const void *q, const void *k, const void *v, int dtype,
                     int64_t T, int Hq, int Hkv, int d, int causal, int sched) {
    std::lock_guard<std::mutex> lk(g_reserve_mu);
    for (const auto &e : g_reserve)
        if (e.first == ws) {
            const ReserveRec &r = e.second;
            return r.plan == plan && r.q == q && r.k == k && r.v == v && r.dtype == dtype && r.T == T &&
                   r.Hq == Hq && r.Hkv == Hkv && r.d == d && r.causal == causal && r.sched == sched;
        }
    return false;
}

}  // namespace ra

extern "C" {

const char *ra_version(void) { return "libra 0.1 (sm_103a)"; }

ra_status ra_profile_enable(int on) {
    std::lock_guard<std::mutex> lk(g_prof_mu);
    if (on) {
        for (auto &r : g_prof) {
            g_event_pool.push_back(r.a);
            g_event_pool.push_back(r.b);
        }
        g_prof.clear();
    }
    g_prof_on = on != 0;
    return RA_OK;
}

int ra_profile_read(int max_kernels, char *names, double *total_ms, int64_t *launches) {
    std::lock_guard<std::mutex> lk(g_prof_mu);
    std::vector<std::string> keys;
    std::vector<double> ms;
    std::vector<int64_t> cnt;
    for (auto &r : g_prof) {
        if (cudaEventSynchronize(r.b) != cudaSuccess) return -1;
        float t = 0.f;
        if (cudaEventElapsedTime(&t, r.a, r.b) != cudaSuccess) return -1;
        size_t i = 0;
        while (i < keys.size() && keys[i] != r.name) ++i;
        if (i == keys.size()) {
            keys.push_back(r.name);
            ms.push_back(0.0);
            cnt.push_back(0);
        }
        ms[i] += t;
        cnt[i] += 1;
    }
    const int n = (int)std::min<size_t>(keys.size(), (size_t)std::max(max_kernels, 0));
    for (int i = 0; i < n; ++i) {
        if (names) {
            std::strncpy(names + (size_t)i * 64, keys[i].c_str(), 63);
            names[(size_t)i * 64 + 63] = 0;
        }
        if (total_ms) total_ms[i] = ms[i];
        if (launches) launches[i] = cnt[i];
    }
    return n;
}

const char *ra_last_error(void) { return g_last_error.c_str(); }

const char *ra_status_string(ra_status s) {
    switch (s) {
        case RA_OK: return "ok";
        case RA_ERR_INVALID_ARG: return "invalid argument";
        case RA_ERR_UNSUPPORTED: return "unsupported";
        case RA_ERR_CUDA: return "CUDA error";
        case RA_ERR_WORKSPACE: return "workspace too small";
        case RA_ERR_TIMEOUT: return "device wait timed out";
        case RA_ERR_DEVICE_BOUNDS: return "device index out of range";
        default: return "unknown status";
    }
}

ra_status ra_zigzag_plan(const int32_t *cu, int B, int cp, int mode, int32_t *perm, int32_t *off,
                         int32_t *cu_local) {
    if (!perm || !off || !cu_local) return fail(RA_ERR_INVALID_ARG, "output pointer is NULL");
    ZigzagPlan zp;
    ra_status st = build_zigzag(cu, B, cp, mode, zp);
    if (st) return st;
    std::memcpy(perm, zp.perm.data(), zp.perm.size() * 4);
    std::memcpy(off, zp.off.data(), zp.off.size() * 4);
    std::memcpy(cu_local, zp.cu_local.data(), zp.cu_local.size() * 4);
    return RA_OK;
}

static ra_status permute_common(const void *src, void *dst, const int32_t *perm, int64_t T, int64_t row_bytes,
                                void *stream, int inverse) {
    if (T < 0 || row_bytes <= 0) return fail(RA_ERR_INVALID_ARG, "T must be >= 0 and row_bytes > 0");
    if (T == 0) return RA_OK;
    if (!src || !dst || !perm) return fail(RA_ERR_INVALID_ARG, "NULL pointer");
    if (T > INT32_MAX) return fail(RA_ERR_UNSUPPORTED, "T must fit in int32");
    PermJob job{src, dst, row_bytes};
    {
        ProfScope ps(inverse ? "ra_unpermute" : "ra_permute", static_cast<cudaStream_t>(stream));
        RA_CUDA(launch_permute(&job, 1, perm, T, inverse, static_cast<cudaStream_t>(stream)), "permute launch");
    }
    return RA_OK;
}

ra_status ra_zigzag_permute(const void *x, void *y, const int32_t *perm, int64_t T, int64_t row_bytes,
                            void *stream) {
    return permute_common(x, y, perm, T, row_bytes, stream, 0);
}

ra_status ra_zigzag_unpermute(const void *y, void *x, const int32_t *perm, int64_t T, int64_t row_bytes,
                              void *stream) {
    return permute_common(y, x, perm, T, row_bytes, stream, 1);
}

ra_status ra_ring_rank_pairs(const int32_t *cu, int B, int cp, int mode, int causal, int window, int64_t *counts) {
    if (!counts) return fail(RA_ERR_INVALID_ARG, "counts is NULL");
    ZigzagPlan zp;
    ra_status st = build_zigzag(cu, B, cp, mode, zp);
    if (st) return st;
    for (int r = 0; r < cp; ++r) {
        int64_t c = 0;
        for (int b = 0; b < B; ++b) {
            const int64_t lo = zp.off[r] + zp.cu_local[(size_t)r * (B + 1) + b];
            const int64_t hi = zp.off[r] + zp.cu_local[(size_t)r * (B + 1) + b + 1];
            const int64_t L = (int64_t)cu[b + 1] - cu[b];
            for (int64_t i = lo; i < hi; ++i) {
                // keys of the document in [first, last]
                const int64_t pos = zp.perm[i];
                int64_t first = cu[b];
                const int64_t last = causal ? pos : (int64_t)cu[b] + L - 1;
                if (window >= 0 && pos - window > first) first = pos - window;
                if (last >= first) c += last - first + 1;
            }
        }
        counts[r] = c;
    }
    return RA_OK;
}

ra_status ra_get_device_status(void *stream) {
    RA_CUDA(cudaStreamSynchronize(static_cast<cudaStream_t>(stream)), "stream synchronize");
    int *p = device_status_ptr();
    if (!p) return fail(RA_ERR_CUDA, "status word unavailable");
    int v = 0;
    RA_CUDA(cudaMemcpy(&v, p, sizeof(int), cudaMemcpyDeviceToHost), "status read");
    if (v != 0) {
        const int zero = 0;
        RA_CUDA(cudaMemcpy(p, &zero, sizeof(int), cudaMemcpyHostToDevice), "status clear");
        return fail(v, std::string("device status: ") + ra_status_string(v));
    }
    return RA_OK;
}

ra_status ra_selftest_wait_timeout(int64_t budget_us, void *stream) {
    if (budget_us < 1 || budget_us > 1000000) return fail(RA_ERR_INVALID_ARG, "budget_us must be in [1, 1e6]");
    RA_CUDA(launch_wait_selftest((uint64_t)budget_us * 1000ull, static_cast<cudaStream_t>(stream)), "selftest launch");
    return RA_OK;
}

// ---------------------------------------------------------------- merge
ra_status ra_lse_merge(int n_parts, const float *const *outs, const float *const *lses, int64_t Tq, int Hq, int d,
                       void *out, int out_dtype, float *lse_out, void *stream) {
    if (n_parts < 1 || n_parts > kMaxMergeParts) return fail(RA_ERR_INVALID_ARG, "n_parts must be in [1, 64]");
    if (!outs || !lses) return fail(RA_ERR_INVALID_ARG, "outs/lses is NULL");
    if (Tq < 0 || Hq <= 0 || d <= 0) return fail(RA_ERR_INVALID_ARG, "bad shape");
    if (d % 4 != 0 || d > 256) return fail(RA_ERR_UNSUPPORTED, "d must be a multiple of 4 and <= 256");
    if (out_dtype != RA_BF16 && out_dtype != RA_FP32) return fail(RA_ERR_INVALID_ARG, "bad out_dtype");
    if (Tq == 0) return RA_OK;
    if (!out) return fail(RA_ERR_INVALID_ARG, "out is NULL");
    for (int p = 0; p < n_parts; ++p) {
        if (!outs[p] || !lses[p]) return fail(RA_ERR_INVALID_ARG, "NULL partial");
        if (!aligned16(outs[p])) return fail(RA_ERR_UNSUPPORTED, "partial outputs must be 16-byte aligned");
    }
    if (!aligned16(out)) return fail(RA_ERR_UNSUPPORTED, "out must be 16-byte aligned");
    ProfScope ps("ra_lse_merge", static_cast<cudaStream_t>(stream));
    RA_CUDA(launch_merge(n_parts, outs, lses, Tq, Hq, d, out, out_dtype, lse_out, static_cast<cudaStream_t>(stream)),
            "merge launch");
    return RA_OK;
}

// ---------------------------------------------------------------- partial
size_t ra_partial_workspace_bytes(int64_t Tq, int64_t Tk, int nseg, int Hq, int Hkv, int d, int dtype) {
    (void)d;
    (void)dtype;
    if (Tq < 0 || Tk < 0 || nseg < 1 || Hkv <= 0 || Hq <= 0) return 0;
    // Upper bound over any positions (a tile holds at least one row, so there
    // are at most Tq query tiles and Tk KV tiles) of the tables a call
    // uploads: query and KV tile records, their per-segment offsets, the
    // forward items (two query tiles of one segment per item and KV head)
    // and the work counter; the SIMT path's position and offset arrays are
    // added on top.
    const size_t qt = (size_t)Tq + nseg, kt = (size_t)Tk + nseg;
    size_t s = 0;
    s += align_up(qt * sizeof(Tile), 256) + align_up(kt * sizeof(Tile), 256);
    s += 2 * align_up(((size_t)nseg + 2) * 4, 256);
    s += align_up(((qt + 1) / 2 + nseg) * (size_t)Hkv * sizeof(WorkItem), 256);
    // SIMT path: positions and offsets
    s += align_up((size_t)Tq * 4, 256) + align_up((size_t)Tk * 4, 256) + 4 * align_up(((size_t)nseg + 2) * 4, 256);
    return s + 4096;
}

size_t ra_partial_table_bytes(int64_t Tq, int64_t Tk, int Hq, int Hkv, int d, int dtype, const int32_t *cu_q,
                              const int32_t *cu_k, int nseg, const int32_t *q_pos, const int32_t *k_pos, int causal,
                              int window) {
    if (check_common(dtype, Hq, Hkv, d) || Tq < 0 || Tk < 0 || Tq > INT32_MAX || Tk > INT32_MAX || nseg < 1)
        return 0;
    if (validate_cu(cu_q, nseg, Tq) || validate_cu(cu_k, nseg, Tk)) return 0;
    if (tc_fwd_supported(dtype, d, Hq, Hkv)) {
        TilePlan tp;
        if (build_partial_tiles(cu_q, cu_k, nseg, q_pos, k_pos, Tq, Tk, Hq / Hkv, Hkv, causal, window, tp)) return 0;
        tp.bitems.clear();
        tp.qitems.clear();
        DeviceTables dt;
        pack_tables(nullptr, &tp, dt);
        return dt.blob.size();
    }
    auto a64 = [](size_t n) { return align_up(n, 64); };
    return 4 * (a64((size_t)Tq) + a64((size_t)Tk) + 2 * a64(2) + 2 * a64((size_t)nseg + 1));
}

ra_status ra_varlen_attn_partial(const void *q, const void *k, const void *v, int dtype, int64_t Tq, int64_t Tk,
                                 int Hq, int Hkv, int d, const int32_t *cu_q, const int32_t *cu_k, int nseg,
                                 const int32_t *q_pos, const int32_t *k_pos, int causal, int window, float scale,
                                 float *out, float *lse, void *workspace, size_t ws_bytes, void *stream) {
    ra_status st = check_common(dtype, Hq, Hkv, d);
    if (st) return st;
    if (window >= 0) {
        // the kernels take position + window in 32-bit arithmetic
        const int32_t lim = 1 << 30;
        if (window >= lim) {
            window = -1;  // reaches back further than any position
        } else {
            for (int64_t i = 0; i < Tq; ++i)
                if ((q_pos ? q_pos[i] : i) >= lim || (q_pos && q_pos[i] < 0))
                    return fail(RA_ERR_UNSUPPORTED, "with a window, positions must be in [0, 2^30)");
            for (int64_t i = 0; i < Tk; ++i)
                if ((k_pos ? k_pos[i] : i) >= lim || (k_pos && k_pos[i] < 0))
                    return fail(RA_ERR_UNSUPPORTED, "with a window, positions must be in [0, 2^30)");
        }
    }
    if (Tq < 0 || Tk < 0 || Tq > INT32_MAX || Tk > INT32_MAX) return fail(RA_ERR_INVALID_ARG, "bad Tq/Tk");
    if (nseg < 1) return fail(RA_ERR_INVALID_ARG, "nseg must be >= 1");
    if ((st = validate_cu(cu_q, nseg, Tq))) return st;
    if ((st = validate_cu(cu_k, nseg, Tk))) return st;
    if (!std::isfinite(scale)) return fail(RA_ERR_INVALID_ARG, "scale must be finite");
    if (Tq == 0) return RA_OK;
    if (!q || !out || !lse || (Tk > 0 && (!k || !v))) return fail(RA_ERR_INVALID_ARG, "NULL tensor");
    if (!aligned16(q) || !aligned16(out) || (Tk > 0 && (!aligned16(k) || !aligned16(v))))
        return fail(RA_ERR_UNSUPPORTED, "tensors must be 16-byte aligned");
    const size_t need = ra_partial_workspace_bytes(Tq, Tk, nseg, Hq, Hkv, d, dtype);
    if (!workspace || ws_bytes < need) return fail(RA_ERR_WORKSPACE, "workspace must be >= " + std::to_string(need));
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    {
        // The segment and position arrays are host arrays: each call plans
        // on the host and uploads its tables from host memory on `stream`,
        // which a captured graph could not replay (the host copy is gone
        // after the call), so a capturing stream is refused before any work.
        cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
        if (cudaStreamIsCapturing(s, &cs) != cudaSuccess) {
            (void)cudaGetLastError();
            cs = cudaStreamCaptureStatusNone;
        }
        if (cs != cudaStreamCaptureStatusNone)
            return fail(RA_ERR_UNSUPPORTED,
                        "the partial calls upload per-call tables from host memory and cannot be captured");
    }
    const int G = Hq / Hkv;
    const bool tc = tc_fwd_supported(dtype, d, Hq, Hkv);
    Carver cv(workspace);
    if (tc) {
        TilePlan tp;
        if ((st = build_partial_tiles(cu_q, cu_k, nseg, q_pos, k_pos, Tq, Tk, G, Hkv, causal, window, tp))) return st;
        // one forward pass: the backward passes' items are not uploaded (the
        // same tables ra_partial_table_bytes sizes)
        tp.bitems.clear();
        tp.qitems.clear();
        DeviceTables dt;
        pack_tables(nullptr, &tp, dt);
        if (dt.blob.size() > ws_bytes)
            return fail(RA_ERR_WORKSPACE, "tile tables need " + std::to_string(dt.blob.size()) +
                                              " bytes, more than the workspace's " + std::to_string(ws_bytes));
        void *tab = cv.take(dt.blob.size());
        RA_CUDA(cudaMemcpyAsync(tab, dt.blob.data(), dt.blob.size(), cudaMemcpyHostToDevice, s), "table upload");
        const uint8_t *tb = static_cast<const uint8_t *>(tab);
        TcFwdArgs a{};
        a.q = q;
        a.k = k ? k : q;
        a.v = v ? v : q;
        a.Tq = Tq;
        a.Tk = Tk;
        a.Hq = Hq;
        a.Hkv = Hkv;
        a.G = G;
        a.qtiles = tb + dt.o_qt;
        a.kvtiles = tb + dt.o_kt;
        a.kv_off = reinterpret_cast<const int32_t *>(tb + dt.o_kvoff);
        a.items = tb + dt.o_items;
        a.sched = reinterpret_cast<int *>(const_cast<uint8_t *>(tb) + dt.o_sched);
        a.n_items = dt.n_items;
        a.cp = 1;
        a.B = nseg;
        a.t0 = 0;
        a.t1 = 1;
        a.causal = causal;
        a.window = window;
        a.scale = scale;
        a.out_mode = kOutPartial;
        a.out = out;
        a.lse = lse;
        a.lse_T = Tq;
        ProfScope ps("ra_tc_fwd", s);
        RA_CUDA(launch_tc_fwd(a, s), "tensor-core partial launch");
        return RA_OK;
    }
    // SIMT path: a one-rank ring with explicit position arrays.
    std::vector<int32_t> qp((size_t)Tq), kp((size_t)Tk);
    for (int64_t i = 0; i < Tq; ++i) qp[i] = q_pos ? q_pos[i] : (int32_t)i;
    for (int64_t i = 0; i < Tk; ++i) kp[i] = k_pos ? k_pos[i] : (int32_t)i;
    std::vector<int32_t> host;
    const int32_t offq[2] = {0, (int32_t)Tq}, offk[2] = {0, (int32_t)Tk};
    size_t o_qp = 0, o_kp, o_offq, o_offk, o_cuq, o_cuk;
    auto put = [&](const int32_t *src, size_t n) {
        size_t at = host.size();
        host.insert(host.end(), src, src + n);
        host.resize(align_up(host.size(), 64), 0);
        return at;
    };
    o_qp = put(qp.data(), qp.size());
    o_kp = put(kp.data(), kp.size());
    o_offq = put(offq, 2);
    o_offk = put(offk, 2);
    o_cuq = put(cu_q, (size_t)nseg + 1);
    o_cuk = put(cu_k, (size_t)nseg + 1);
    if (host.size() * 4 > ws_bytes)
        return fail(RA_ERR_WORKSPACE, "position tables need " + std::to_string(host.size() * 4) +
                                          " bytes, more than the workspace's " + std::to_string(ws_bytes));
    int32_t *dh = static_cast<int32_t *>(cv.take(host.size() * 4));
    RA_CUDA(cudaMemcpyAsync(dh, host.data(), host.size() * 4, cudaMemcpyHostToDevice, s), "table upload");
    SimtArgs a{};
    a.q = q;
    a.k = k;
    a.v = v;
    a.dtype = dtype;
    a.Hq = Hq;
    a.Hkv = Hkv;
    a.d = d;
    a.Tq = Tq;
    a.Tk = Tk;
    a.qoff = dh + o_offq;
    a.qcul = dh + o_cuq;
    a.qpos = dh + o_qp;
    a.koff = dh + o_offk;
    a.kcul = dh + o_cuk;
    a.kpos = dh + o_kp;
    a.cp = 1;
    a.B = nseg;
    a.t0 = 0;
    a.t1 = 1;
    a.causal = causal;
    a.window = window;
    a.scale = scale;
    a.out_mode = kOutPartial;
    a.out = out;
    a.lse = lse;
    a.lse_T = Tq;
    ProfScope ps("ra_simt_fwd", s);
    RA_CUDA(launch_simt_fwd(a, s), "SIMT partial launch");
    return RA_OK;
}

ra_status ra_varlen_attn_partial_dev(const void *q, const void *k, const void *v, int dtype, int64_t Tq, int64_t Tk,
                                     int Hq, int Hkv, int d, const int32_t *cu_q, const int32_t *cu_k, int nseg,
                                     const int32_t *q_pos, const int32_t *k_pos, int causal, int window, float scale,
                                     float *out, float *lse, void *workspace, size_t ws_bytes, void *stream) {
    ra_status st = check_common(dtype, Hq, Hkv, d);
    if (st) return st;
    if (!tc_fwd_supported(dtype, d, Hq, Hkv))
        return fail(RA_ERR_UNSUPPORTED, "device-array partials run on the tensor-core path (bf16, d = 128, Hq / Hkv "
                                        "a power of two <= 16); use ra_varlen_attn_partial");
    if (Tq < 0 || Tk < 0 || Tq > INT32_MAX || Tk > INT32_MAX) return fail(RA_ERR_INVALID_ARG, "bad Tq/Tk");
    if (nseg < 1) return fail(RA_ERR_INVALID_ARG, "nseg must be >= 1");
    if (!std::isfinite(scale)) return fail(RA_ERR_INVALID_ARG, "scale must be finite");
    if (window >= (1 << 30)) window = -1;  // reaches back further than any position
    if (window >= 0 && (Tq >= (1 << 30) || Tk >= (1 << 30)))
        return fail(RA_ERR_UNSUPPORTED, "with a window, Tq and Tk must be < 2^30");
    if (Tq == 0) return RA_OK;
    if (!q || !out || !lse || !cu_q || !cu_k || (Tk > 0 && (!k || !v))) return fail(RA_ERR_INVALID_ARG, "NULL pointer");
    if (!aligned16(q) || !aligned16(out) || (Tk > 0 && (!aligned16(k) || !aligned16(v))))
        return fail(RA_ERR_UNSUPPORTED, "tensors must be 16-byte aligned");
    const size_t need = ra_partial_workspace_bytes(Tq, Tk, nseg, Hq, Hkv, d, dtype);
    if (!workspace || ws_bytes < need) return fail(RA_ERR_WORKSPACE, "workspace must be >= " + std::to_string(need));
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const int G = Hq / Hkv;
    const size_t qt = (size_t)Tq + nseg, kt = (size_t)Tk + nseg;
    Carver cv(workspace);
    DevTileArgs b{};
    b.cu_q = cu_q;
    b.cu_k = cu_k;
    b.q_pos = q_pos;
    b.k_pos = k_pos;
    b.Tq = Tq;
    b.Tk = Tk;
    b.nseg = nseg;
    b.Hkv = Hkv;
    b.q_rows = kBM / G;
    b.check_pos = window >= 0;
    b.qtiles = cv.take(qt * sizeof(Tile));
    b.kvtiles = cv.take(kt * sizeof(Tile));
    b.q_off = static_cast<int32_t *>(cv.take(((size_t)nseg + 2) * 4));
    b.kv_off = static_cast<int32_t *>(cv.take(((size_t)nseg + 2) * 4));
    b.items = cv.take(((qt + 1) / 2 + nseg) * (size_t)Hkv * sizeof(WorkItem));
    b.sched = static_cast<int *>(cv.take(64));
    b.n_items = static_cast<int *>(cv.take(16));
    b.q_cnt = static_cast<int32_t *>(cv.take((size_t)nseg * 4));
    b.k_cnt = static_cast<int32_t *>(cv.take((size_t)nseg * 4));
    b.pair_off = static_cast<int32_t *>(cv.take(((size_t)nseg + 1) * 4));
    if (cv.used > ws_bytes) return fail(RA_ERR_WORKSPACE, "internal: device tables exceed the workspace bound");
    {
        ProfScope ps("ra_tile_build", s);
        RA_CUDA(launch_tile_build(b, s), "tile build launch");
    }
    TcFwdArgs a{};
    a.q = q;
    a.k = k ? k : q;
    a.v = v ? v : q;
    a.Tq = Tq;
    a.Tk = Tk;
    a.Hq = Hq;
    a.Hkv = Hkv;
    a.G = G;
    a.qtiles = b.qtiles;
    a.kvtiles = b.kvtiles;
    a.kv_off = b.kv_off;
    a.items = b.items;
    a.sched = b.sched;
    a.n_items = INT32_MAX;  // the count is on the device: one CTA per SM
    a.n_items_dev = b.n_items;
    a.cp = 1;
    a.B = nseg;
    a.t0 = 0;
    a.t1 = 1;
    a.causal = causal;
    a.window = window;
    a.scale = scale;
    a.out_mode = kOutPartial;
    a.out = out;
    a.lse = lse;
    a.lse_T = Tq;
    ProfScope ps("ra_tc_fwd", s);
    RA_CUDA(launch_tc_fwd(a, s), "tensor-core partial launch");
    return RA_OK;
}

// ---------------------------------------------------------------- ring
namespace {

struct RingLayout {
    size_t total = 0;
    size_t tables = 0, qp = 0, kp = 0, vp = 0;
    // stepwise forward
    size_t parts_o = 0, parts_l = 0, op = 0, lp = 0;
    // backward
    size_t dop = 0, Dv = 0, dq = 0, dk = 0, dv = 0, tile_ld = 0;
};

// The workspace regions of a ring call whose tables take blob_bytes and
// whose plan has n_qtiles query tiles.
static RingLayout ring_layout_sized(size_t blob_bytes, size_t n_qtiles, int64_t T, int Hq, int Hkv, int d, int dtype,
                                    int cp, int sched, int bwd) {
    RingLayout L;
    Carver c(nullptr);
    auto at = [&](size_t bytes) {
        size_t o = c.used;
        c.take(bytes);
        return o;
    };
    const size_t es = esize(dtype);
    L.tables = at(blob_bytes);
    L.qp = at((size_t)T * Hq * d * es);
    L.kp = at((size_t)T * Hkv * d * es);
    L.vp = at((size_t)T * Hkv * d * es);
    if (!bwd && sched == RA_SCHED_STEPWISE) {
        L.parts_o = at((size_t)cp * T * Hq * d * 4);
        L.parts_l = at((size_t)cp * Hq * T * 4);
        L.op = at((size_t)T * Hq * d * es);
        L.lp = at((size_t)Hq * T * 4);
    }
    if (bwd) {
        L.dop = at((size_t)T * Hq * d * es);
        L.Dv = at((size_t)Hq * T * 4);
        L.dq = at((size_t)T * Hq * d * 4);
        L.dk = at((size_t)T * Hkv * d * 4);
        L.dv = at((size_t)T * Hkv * d * 4);
        L.tile_ld = at(n_qtiles * (size_t)Hkv * 1024);
    }
    L.total = c.used + 256;
    return L;
}

RingLayout ring_layout(const RingPlan &plan, int64_t T, int Hq, int Hkv, int d, int dtype, int cp, int sched, int bwd) {
    return ring_layout_sized(plan.dev.blob.size(), plan.tiles.qtiles.size(), T, Hq, Hkv, d, dtype, cp, sched, bwd);
}

// Interval masks: both bounds or neither; they run on the tensor-core
// path in the fused and all-gather schedules; each bound must keep the
// kernels' 32-bit position arithmetic exact.  With bounds the causal flag
// and the window are not used (the intervals hold them).
static ra_status bounds_checks(const int32_t *key_lo, const int32_t *key_hi, int64_t T, bool tc, int sched,
                               int *causal, int *window) {
    if (!key_lo && !key_hi) return RA_OK;
    if (!key_lo || !key_hi) return fail(RA_ERR_INVALID_ARG, "key_lo and key_hi go together");
    if (!tc)
        return fail(RA_ERR_UNSUPPORTED, "interval masks run on the tensor-core path (bf16, d = 128, Hq / Hkv a "
                                        "power of two <= 16)");
    if (sched == RA_SCHED_STEPWISE)
        return fail(RA_ERR_UNSUPPORTED, "interval masks run in the fused and all-gather schedules");
    const int32_t lim = 1 << 30;
    for (int64_t i = 0; i < T; ++i)
        if (key_lo[i] <= -lim || key_lo[i] >= lim || key_hi[i] <= -lim || key_hi[i] >= lim)
            return fail(RA_ERR_UNSUPPORTED, "interval bounds must lie in (-2^30, 2^30)");
    *causal = 0;
    *window = -1;
    return RA_OK;
}

// A window >= T reaches every earlier key of every document: no window.
// Positions (< T) plus the window must fit the kernels' 32-bit arithmetic.
static ra_status ring_window(int64_t T, int *window) {
    if (*window < 0 || *window >= T) {
        *window = -1;
        return RA_OK;
    }
    if (T >= ((int64_t)1 << 30)) return fail(RA_ERR_UNSUPPORTED, "with a window, T must be < 2^30");
    return RA_OK;
}

ra_status ring_checks(const void *q, const void *k, const void *v, int dtype, int64_t T, int Hq, int Hkv, int d,
                      const int32_t *cu, int B, int cp, int mode, int sched, float scale) {
    ra_status st = check_common(dtype, Hq, Hkv, d);
    if (st) return st;
    if (T < 0 || T > INT32_MAX) return fail(RA_ERR_INVALID_ARG, "T must be in [0, 2^31)");
    if ((st = validate_cu(cu, B, T))) return st;
    if (cp < 1 || cp > kMaxMergeParts) return fail(RA_ERR_INVALID_ARG, "cp must be in [1, 64]");
    if (mode != RA_ZZ_GLOBAL && mode != RA_ZZ_PER_DOC) return fail(RA_ERR_INVALID_ARG, "unknown zigzag mode");
    if (sched != RA_SCHED_FUSED && sched != RA_SCHED_STEPWISE && sched != RA_SCHED_ALLGATHER)
        return fail(RA_ERR_INVALID_ARG, "unknown schedule");
    if (!std::isfinite(scale)) return fail(RA_ERR_INVALID_ARG, "scale must be finite");
    if (T > 0 && (!q || !k || !v)) return fail(RA_ERR_INVALID_ARG, "NULL tensor");
    if (T > 0 && (!aligned16(q) || !aligned16(k) || !aligned16(v)))
        return fail(RA_ERR_UNSUPPORTED, "tensors must be 16-byte aligned");
    return RA_OK;
}

}  // namespace

size_t ra_ring_workspace_bytes(int64_t T, int Hq, int Hkv, int d, int dtype, const int32_t *cu, int B, int cp,
                               int mode, int sched, int bwd) {
    if (check_common(dtype, Hq, Hkv, d) != RA_OK || T < 0) return 0;
    ra_status st;
    const bool tc = tc_fwd_supported(dtype, d, Hq, Hkv);
    if (sched != RA_SCHED_FUSED && sched != RA_SCHED_STEPWISE && sched != RA_SCHED_ALLGATHER) return 0;
    // Only the plan's tables depend on the mask: each rank's KV tiles of a
    // document have at most two position runs or one, whichever the mask
    // visits less (a sliding window usually takes tiles of one run), so the
    // size is that of the tables with every KV tile of one run, the most
    // tiles; counted from the tiles alone (no plan is built or cached).
    size_t blob = 0, nq = 0;
    st = ring_tables_bound(cu, B, cp, mode, Hq / Hkv, Hkv, tc, tc && sched == RA_SCHED_ALLGATHER, &blob, &nq);
    if (st) return 0;
    return ring_layout_sized(blob, nq, T, Hq, Hkv, d, dtype, cp, sched, bwd).total;
}

size_t ra_ring_workspace_bytes_masked(int64_t T, int Hq, int Hkv, int d, int dtype, const int32_t *cu, int B, int cp,
                                      int mode, const int32_t *key_lo, const int32_t *key_hi, int sched, int bwd) {
    if (check_common(dtype, Hq, Hkv, d) != RA_OK || T < 0 || T > INT32_MAX) return 0;
    if (sched != RA_SCHED_FUSED && sched != RA_SCHED_ALLGATHER) return 0;
    if (!tc_fwd_supported(dtype, d, Hq, Hkv) || !key_lo || !key_hi) return 0;
    if (validate_cu(cu, B, T) != RA_OK) return 0;
    ra_status st;
    int causal = 0, window = -1;
    if (bounds_checks(key_lo, key_hi, T, true, sched, &causal, &window) != RA_OK) return 0;
    auto plan = get_ring_plan(cu, B, cp, mode, Hq / Hkv, Hkv, 0, -1, true, sched == RA_SCHED_ALLGATHER, &st, key_lo,
                              key_hi);
    if (!plan) return 0;
    return ring_layout(*plan, T, Hq, Hkv, d, dtype, cp, sched, bwd).total;
}

static ra_status ring_fwd_impl(const void *q, const void *k, const void *v, int dtype, int64_t T, int Hq, int Hkv,
                               int d, const int32_t *cu, int B, int cp, int mode, int causal, int window, float scale,
                               int sched, void *out, float *lse, void *workspace, size_t ws_bytes, void *stream,
                               const int32_t *key_lo, const int32_t *key_hi) {
    ra_status st = ring_checks(q, k, v, dtype, T, Hq, Hkv, d, cu, B, cp, mode, sched, scale);
    if (st) return st;
    const int G = Hq / Hkv;
    const bool tc = tc_fwd_supported(dtype, d, Hq, Hkv);
    if ((st = bounds_checks(key_lo, key_hi, T, tc, sched, &causal, &window))) return st;
    if (T == 0) return RA_OK;
    if (!out || !lse) return fail(RA_ERR_INVALID_ARG, "out/lse is NULL");
    if (!aligned16(out)) return fail(RA_ERR_UNSUPPORTED, "out must be 16-byte aligned");
    // all-gather: one pass of each rank's queries over every document's K/V
    // in original order (tensor cores); elsewhere the fused ring computes the
    // same attention
    const bool allgather = sched == RA_SCHED_ALLGATHER && tc;
    if (sched == RA_SCHED_ALLGATHER && !tc) sched = RA_SCHED_FUSED;
    if ((st = ring_window(T, &window))) return st;
    auto plan = get_ring_plan(cu, B, cp, mode, G, Hkv, causal ? 1 : 0, window, tc, allgather, &st, key_lo, key_hi);
    if (!plan) return st;
    const RingLayout L = ring_layout(*plan, T, Hq, Hkv, d, dtype, cp, sched, 0);
    if (!workspace || ws_bytes < L.total)
        return fail(RA_ERR_WORKSPACE, "workspace must be >= " + std::to_string(L.total) + " bytes");
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    uint8_t *ws = static_cast<uint8_t *>(workspace);
    const DeviceTables &dt = plan->dev;
    uint8_t *tab = ws + L.tables;
    {
        ProfScope ps("ra_table_upload", s);
        if ((st = upload_plan_tables(*plan, tab, s))) return st;
    }
    const int32_t *perm = reinterpret_cast<const int32_t *>(tab + dt.o_perm);
    const int32_t *off = reinterpret_cast<const int32_t *>(tab + dt.o_off);
    const int32_t *cul = reinterpret_cast<const int32_t *>(tab + dt.o_cul);
    const size_t es = esize(dtype);
    void *Qp = ws + L.qp, *Kp = ws + L.kp, *Vp = ws + L.vp;
    // a3: zigzag-permute Q, K, V into the ranks' shards (one launch).  The
    // tensor-core kernels read a tile of one position run straight from q, k
    // and v, so the copies are made only for the rows of two-run tiles.
    const uint8_t *qmask = tc ? tab + dt.o_qmask : nullptr;
    const uint8_t *kvmask = tc ? tab + dt.o_kvmask : nullptr;
    PermJob jobs[3] = {{q, Qp, (int64_t)Hq * d * (int64_t)es, qmask},
                       {k, Kp, (int64_t)Hkv * d * (int64_t)es, kvmask},
                       {v, Vp, (int64_t)Hkv * d * (int64_t)es, kvmask}};
    {
        // all-gather: K and V are read in original order, never copied
        ProfScope ps("ra_permute_fwd", s);
        RA_CUDA(launch_permute(jobs, allgather ? 1 : 3, perm, T, 0, s), "permute launch");
    }
    reserve_record(workspace, plan.get(), q, k, v, dtype, T, Hq, Hkv, d, causal, sched);

    auto run_partial = [&](int t0, int t1, int out_mode, void *o, float *l, int64_t lse_T) -> ra_status {
        if (tc) {
            TcFwdArgs a{};
            a.q = Qp;
            a.q_orig = q;
            a.k = allgather ? k : Kp;
            a.v = allgather ? v : Vp;
            a.k_orig = k;
            a.v_orig = v;
            a.Tq = T;
            a.Tk = T;
            a.Hq = Hq;
            a.Hkv = Hkv;
            a.G = G;
            a.qtiles = tab + dt.o_qt;
            a.kvtiles = tab + dt.o_kt;
            a.kv_off = reinterpret_cast<const int32_t *>(tab + dt.o_kvoff);
            a.items = tab + dt.o_items;
            a.sched = reinterpret_cast<int *>(tab + dt.o_sched);
            a.n_items = dt.n_items;
            a.cp = cp;
            a.B = B;
            a.t0 = t0;
            a.t1 = t1;
            a.causal = causal;
            a.window = window;
            if (dt.bounds) {
                a.qbounds = tab + dt.o_qb;
                a.key_lo = reinterpret_cast<const int32_t *>(tab + dt.o_klo);
                a.key_hi = reinterpret_cast<const int32_t *>(tab + dt.o_khi);
            }
            a.scale = scale;
            a.out_mode = out_mode;
            a.out = o;
            a.lse = l;
            a.lse_T = lse_T;
            ProfScope ps("ra_tc_fwd", s);
            RA_CUDA(launch_tc_fwd(a, s), "tensor-core forward launch");
        } else {
            SimtArgs a{};
            a.q = Qp;
            a.k = Kp;
            a.v = Vp;
            a.dtype = dtype;
            a.Hq = Hq;
            a.Hkv = Hkv;
            a.d = d;
            a.Tq = T;
            a.Tk = T;
            a.qoff = off;
            a.qcul = cul;
            a.qpos = perm;
            a.koff = off;
            a.kcul = cul;
            a.kpos = perm;
            a.cp = cp;
            a.B = B;
            a.t0 = t0 < 0 ? 0 : t0;  // the SIMT kernel walks [t0, t1) for every row
            a.t1 = t1;
            a.causal = causal;
            a.window = window;
            a.scale = scale;
            a.out_mode = out_mode;
            a.out = o;
            a.lse = l;
            a.lse_T = lse_T;
            ProfScope ps("ra_simt_fwd", s);
            RA_CUDA(launch_simt_fwd(a, s), "SIMT forward launch");
        }
        return RA_OK;
    };

    if (sched == RA_SCHED_FUSED || sched == RA_SCHED_ALLGATHER) {
        // a4+a5+a6 in one launch: ring order inside each tile, on-chip merge,
        // rows written straight back to their original positions.  t0 = -1:
        // each item walks only the ring steps that hold its visited KV tiles.
        return run_partial(-1, cp, kOutFinal, out, lse, T);
    }
    // STEPWISE: one launch per ring step into fp32 partials (local order),
    // then the n-way LSE merge, then un-permute O and LSE.
    std::vector<const float *> po((size_t)cp), pl((size_t)cp);
    for (int t = 0; t < cp; ++t) {
        float *o_t = reinterpret_cast<float *>(ws + L.parts_o) + (size_t)t * T * Hq * d;
        float *l_t = reinterpret_cast<float *>(ws + L.parts_l) + (size_t)t * Hq * T;
        if ((st = run_partial(t, t + 1, kOutPartial, o_t, l_t, T))) return st;
        po[t] = o_t;
        pl[t] = l_t;
    }
    void *Op = ws + L.op;
    float *Lp = reinterpret_cast<float *>(ws + L.lp);
    {
        ProfScope ps("ra_lse_merge", s);
        RA_CUDA(launch_merge(cp, po.data(), pl.data(), T, Hq, d, Op, dtype, Lp, s), "merge launch");
    }
    PermJob uj{Op, out, (int64_t)Hq * d * (int64_t)es};
    {
        ProfScope ps("ra_unpermute", s);
        RA_CUDA(launch_permute(&uj, 1, perm, T, 1, s), "unpermute launch");
    }
    {
        ProfScope ps("ra_unpermute_lse", s);
        RA_CUDA(launch_unpermute_cols(Lp, lse, perm, T, Hq, s), "lse unpermute launch");
    }
    return RA_OK;
}

static ra_status ring_bwd_impl(const void *q, const void *k, const void *v, int dtype, int64_t T, int Hq, int Hkv,
                               int d, const int32_t *cu, int B, int cp, int mode, int causal, int window, float scale,
                               int sched, const void *out, const float *lse, const void *dout, void *dq, void *dk,
                               void *dv, int grad_dtype, int flags, void *workspace, size_t ws_bytes, void *stream,
                               const int32_t *key_lo, const int32_t *key_hi) {
    ra_status st = ring_checks(q, k, v, dtype, T, Hq, Hkv, d, cu, B, cp, mode, sched, scale);
    if (st) return st;
    if (grad_dtype != RA_BF16 && grad_dtype != RA_FP32) return fail(RA_ERR_INVALID_ARG, "bad grad_dtype");
    const int G = Hq / Hkv;
    const bool tc = tc_fwd_supported(dtype, d, Hq, Hkv);
    if ((st = bounds_checks(key_lo, key_hi, T, tc, sched, &causal, &window))) return st;
    if (T == 0) return RA_OK;
    if (!out || !lse || !dout || !dq || !dk || !dv) return fail(RA_ERR_INVALID_ARG, "NULL tensor");
    if (!aligned16(out) || !aligned16(dout) || !aligned16(dq) || !aligned16(dk) || !aligned16(dv))
        return fail(RA_ERR_UNSUPPORTED, "tensors must be 16-byte aligned");
    const bool allgather = sched == RA_SCHED_ALLGATHER && tc;
    if (sched == RA_SCHED_ALLGATHER && !tc) sched = RA_SCHED_FUSED;
    if ((st = ring_window(T, &window))) return st;
    auto plan = get_ring_plan(cu, B, cp, mode, G, Hkv, causal ? 1 : 0, window, tc, allgather, &st, key_lo, key_hi);
    if (!plan) return st;
    const RingLayout L = ring_layout(*plan, T, Hq, Hkv, d, dtype, cp, sched, 1);
    if (!workspace || ws_bytes < L.total)
        return fail(RA_ERR_WORKSPACE, "workspace must be >= " + std::to_string(L.total) + " bytes");
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    uint8_t *ws = static_cast<uint8_t *>(workspace);
    const DeviceTables &dt = plan->dev;
    uint8_t *tab = ws + L.tables;
    // the forward's reserve space: tables and rank-ordered Q, K, V (same
    // offsets in both layouts) when the caller asks and the host record agrees
    const bool reserve = (flags & RA_BWD_FWD_RESERVE) &&
                         reserve_matches(workspace, plan.get(), q, k, v, dtype, T, Hq, Hkv, d, causal, sched);
    if (!reserve) {
        ProfScope ps("ra_table_upload", s);
        if ((st = upload_plan_tables(*plan, tab, s))) return st;
    }
    const int32_t *perm = reinterpret_cast<const int32_t *>(tab + dt.o_perm);
    const int32_t *off = reinterpret_cast<const int32_t *>(tab + dt.o_off);
    const int32_t *cul = reinterpret_cast<const int32_t *>(tab + dt.o_cul);
    const size_t es = esize(dtype);
    void *Qp = ws + L.qp, *Kp = ws + L.kp, *Vp = ws + L.vp, *dOp = ws + L.dop;
    float *D = reinterpret_cast<float *>(ws + L.Dv);
    float *dqa = reinterpret_cast<float *>(ws + L.dq);
    float *dka = reinterpret_cast<float *>(ws + L.dk);
    float *dva = reinterpret_cast<float *>(ws + L.dv);
    // a7: permute Q, K, V, dO; D = rowsum(dO * O) in original order.  With
    // the tensor cores the copies are made only for the rows of two-run
    // tiles (the kernels read the others straight from q, k, v and dout).
    const uint8_t *qmask = tc ? tab + dt.o_qmask : nullptr;
    const uint8_t *kvmask = tc ? tab + dt.o_kvmask : nullptr;
    PermJob jobs[4] = {{q, Qp, (int64_t)Hq * d * (int64_t)es, qmask},
                       {k, Kp, (int64_t)Hkv * d * (int64_t)es, kvmask},
                       {v, Vp, (int64_t)Hkv * d * (int64_t)es, kvmask},
                       {dout, dOp, (int64_t)Hq * d * (int64_t)es, qmask}};
    if (dtype == RA_BF16 && d == 128 && aligned16(out) && aligned16(dout)) {
        // one pass: the permutes and D from the same dO reads
        ProfScope ps("ra_permute_rowdot", s);
        // (all-gather: K and V are read in original order, never copied)
        RA_CUDA(launch_permute_rowdot(jobs, reserve ? 0 : (allgather ? 1 : 3), dout, dOp, out, D, perm, T, Hq, s,
                                      qmask),
                "permute+rowdot launch");
    } else {
        {
            ProfScope ps("ra_permute_bwd", s);
            if (reserve)
                RA_CUDA(launch_permute(jobs + 3, 1, perm, T, 0, s), "permute launch");
            else
                RA_CUDA(launch_permute(jobs, 4, perm, T, 0, s), "permute launch");
        }
        ProfScope ps("ra_rowdot", s);
        RA_CUDA(launch_rowdot(dout, out, dtype, T, Hq, d, D, s), "rowdot launch");
    }
    const bool fused_tc = tc && (sched == RA_SCHED_FUSED || sched == RA_SCHED_ALLGATHER);
    if (!fused_tc) {
        RA_CUDA(cudaMemsetAsync(dqa, 0, (size_t)T * Hq * d * 4, s), "memset dq");
        RA_CUDA(cudaMemsetAsync(dka, 0, (size_t)T * Hkv * d * 4, s), "memset dk");
        RA_CUDA(cudaMemsetAsync(dva, 0, (size_t)T * Hkv * d * 4, s), "memset dv");
    }
    // a8: the ring backward.  Tensor cores: a key-side pass (dK, dV in TMEM
    // across ring steps) and a query-side pass (dQ in TMEM, no atomics).
    // STEPWISE: one launch of each per ring step, accumulating in fp32.
    if (tc) {
        float *tld = reinterpret_cast<float *>(ws + L.tile_ld);
        {
            ProfScope ps("ra_tile_lse_d", s);
            RA_CUDA(launch_tile_lse_d(tab + dt.o_qt, (int)plan->tiles.qtiles.size(), Hkv, G, lse, D, T, scale, tld, s),
                    "tile lse/D launch");
        }
        TcBwdArgs a{};
        a.q = Qp;
        a.k = allgather ? k : Kp;
        a.v = allgather ? v : Vp;
        a.dout = dOp;
        a.q_orig = q;
        a.dout_orig = dout;
        a.k_orig = k;
        a.v_orig = v;
        a.T = T;
        a.Hq = Hq;
        a.Hkv = Hkv;
        a.G = G;
        a.qtiles = tab + dt.o_qt;
        a.kvtiles = tab + dt.o_kt;
        a.q_off = reinterpret_cast<const int32_t *>(tab + dt.o_qoff);
        a.items = tab + dt.o_bitems;
        a.n_items = dt.n_bitems;
        a.cp = cp;
        a.B = B;
        a.causal = causal;
        a.window = window;
        a.scale = scale;
        a.tile_ld = tld;
        if (dt.bounds) {
            a.qbounds = tab + dt.o_qb;
            a.key_lo = reinterpret_cast<const int32_t *>(tab + dt.o_klo);
            a.key_hi = reinterpret_cast<const int32_t *>(tab + dt.o_khi);
        }
        TcDqArgs qa{};
        qa.q = Qp;
        qa.k = allgather ? k : Kp;
        qa.v = allgather ? v : Vp;
        qa.dout = dOp;
        qa.q_orig = q;
        qa.dout_orig = dout;
        qa.k_orig = k;
        qa.v_orig = v;
        qa.T = T;
        qa.Hq = Hq;
        qa.Hkv = Hkv;
        qa.G = G;
        qa.qtiles = tab + dt.o_qt;
        qa.kvtiles = tab + dt.o_kt;
        qa.kv_off = reinterpret_cast<const int32_t *>(tab + dt.o_kvoff);
        qa.items = tab + dt.o_qitems;
        qa.n_items = dt.n_qitems;
        qa.cp = cp;
        qa.B = B;
        qa.causal = causal;
        qa.window = window;
        qa.qbounds = a.qbounds;
        qa.key_lo = a.key_lo;
        qa.key_hi = a.key_hi;
        qa.scale = scale;
        qa.lse = lse;
        qa.D = D;
        qa.lse_T = T;
        if (fused_tc) {
            a.t0 = -1;  // each item's own range of ring steps with visited tiles
            a.t1 = cp;
            // complete per KV tile: written once in the gradient dtype
            a.dk = dk;
            a.dv = dv;
            a.out_mode = grad_dtype == RA_BF16 ? 0 : 1;
            qa.t0 = -1;
            qa.t1 = cp;
            qa.dq = dq;  // complete per query tile: written once in the gradient dtype
            qa.out_mode = grad_dtype == RA_BF16 ? 0 : 1;
            std::lock_guard<std::mutex> lk(g_side_mu);
            // under stream capture the side stream is joined into the graph
            // (fork/join through events); it is created outside capture only
            cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
            if (cudaStreamIsCapturing(s, &cs) != cudaSuccess) {
                (void)cudaGetLastError();
                cs = cudaStreamCaptureStatusActive;
            }
            SideStream *side = side_stream_locked(cs == cudaStreamCaptureStatusNone);
            if (side) {
                // one timing scope over both kernels: they share the SMs
                ProfScope ps("ra_tc_bwd", s);
                RA_CUDA(cudaEventRecord(side->fork, s), "fork record");
                RA_CUDA(launch_tc_dq(qa, s), "tensor-core dQ launch");
                RA_CUDA(cudaStreamWaitEvent(side->st, side->fork, 0), "fork wait");
                RA_CUDA(launch_tc_bwd(a, side->st), "tensor-core dK/dV launch");
                RA_CUDA(cudaEventRecord(side->join, side->st), "join record");
                RA_CUDA(cudaStreamWaitEvent(s, side->join, 0), "join wait");
            } else {
                {
                    ProfScope ps("ra_tc_bwd_dq", s);
                    RA_CUDA(launch_tc_dq(qa, s), "tensor-core dQ launch");
                }
                ProfScope ps("ra_tc_bwd_dkdv", s);
                RA_CUDA(launch_tc_bwd(a, s), "tensor-core dK/dV launch");
            }
        } else {
            a.dk = dka;
            a.dv = dva;
            a.out_mode = 2;
            qa.dq = dqa;
            qa.out_mode = 2;
            for (int t = 0; t < cp; ++t) {
                a.t0 = qa.t0 = t;
                a.t1 = qa.t1 = t + 1;
                {
                    ProfScope ps("ra_tc_bwd_dkdv", s);
                    RA_CUDA(launch_tc_bwd(a, s), "tensor-core dK/dV launch");
                }
                {
                    ProfScope ps("ra_tc_bwd_dq", s);
                    RA_CUDA(launch_tc_dq(qa, s), "tensor-core dQ launch");
                }
            }
        }
    } else {
        SimtBwdArgs a{};
        a.q = Qp;
        a.k = Kp;
        a.v = Vp;
        a.dout = dOp;
        a.dtype = dtype;
        a.Hq = Hq;
        a.Hkv = Hkv;
        a.d = d;
        a.T = T;
        a.off = off;
        a.cul = cul;
        a.pos = perm;
        a.cp = cp;
        a.B = B;
        a.causal = causal;
        a.window = window;
        a.scale = scale;
        a.lse = lse;
        a.D = D;
        a.lse_T = T;
        a.dq = dqa;
        a.dk = dka;
        a.dv = dva;
        if (sched == RA_SCHED_FUSED) {
            a.t0 = 0;
            a.t1 = cp;
            ProfScope ps("ra_simt_bwd", s);
            RA_CUDA(launch_simt_bwd(a, s), "SIMT backward launch");
        } else {
            for (int t = 0; t < cp; ++t) {
                a.t0 = t;
                a.t1 = t + 1;
                ProfScope ps("ra_simt_bwd", s);
                RA_CUDA(launch_simt_bwd(a, s), "SIMT backward launch");
            }
        }
    }
    // a9: cast to the gradient dtype (rows are already in original order); the
    // fused tensor-core passes write the gradient dtype directly
    if (!fused_tc) {
        ProfScope ps("ra_cast", s);
        RA_CUDA(launch_cast_f32(dqa, dq, grad_dtype, T * Hq * d, s), "cast dq");
        RA_CUDA(launch_cast_f32(dka, dk, grad_dtype, T * Hkv * d, s), "cast dk");
        RA_CUDA(launch_cast_f32(dva, dv, grad_dtype, T * Hkv * d, s), "cast dv");
    }
    return RA_OK;
}

ra_status ra_ring_attn_fwd(const void *q, const void *k, const void *v, int dtype, int64_t T, int Hq, int Hkv, int d,
                           const int32_t *cu, int B, int cp, int mode, int causal, int window, float scale, int sched,
                           void *out, float *lse, void *workspace, size_t ws_bytes, void *stream) {
    return ring_fwd_impl(q, k, v, dtype, T, Hq, Hkv, d, cu, B, cp, mode, causal, window, scale, sched, out, lse,
                         workspace, ws_bytes, stream, nullptr, nullptr);
}

ra_status ra_ring_attn_bwd(const void *q, const void *k, const void *v, int dtype, int64_t T, int Hq, int Hkv, int d,
                           const int32_t *cu, int B, int cp, int mode, int causal, int window, float scale, int sched,
                           const void *out, const float *lse, const void *dout, void *dq, void *dk, void *dv,
                           int grad_dtype, int flags, void *workspace, size_t ws_bytes, void *stream) {
    return ring_bwd_impl(q, k, v, dtype, T, Hq, Hkv, d, cu, B, cp, mode, causal, window, scale, sched, out, lse, dout,
                         dq, dk, dv, grad_dtype, flags, workspace, ws_bytes, stream, nullptr, nullptr);
}

ra_status ra_ring_attn_fwd_masked(const void *q, const void *k, const void *v, int dtype, int64_t T, int Hq,
                                  int Hkv, int d, const int32_t *cu, int B, int cp, int mode, const int32_t *key_lo,
                                  const int32_t *key_hi, float scale, int sched, void *out, float *lse,
                                  void *workspace, size_t ws_bytes, void *stream) {
    if (!key_lo || !key_hi) return fail(RA_ERR_INVALID_ARG, "key_lo / key_hi is NULL");
    return ring_fwd_impl(q, k, v, dtype, T, Hq, Hkv, d, cu, B, cp, mode, 0, -1, scale, sched, out, lse, workspace,
                         ws_bytes, stream, key_lo, key_hi);
}

ra_status ra_ring_attn_bwd_masked(const void *q, const void *k, const void *v, int dtype, int64_t T, int Hq,
                                  int Hkv, int d, const int32_t *cu, int B, int cp, int mode, const int32_t *key_lo,
                                  const int32_t *key_hi, float scale, int sched, const void *out, const float *lse,
                                  const void *dout, void *dq, void *dk, void *dv, int grad_dtype, int flags,
                                  void *workspace, size_t ws_bytes, void *stream) {
    if (!key_lo || !key_hi) return fail(RA_ERR_INVALID_ARG, "key_lo / key_hi is NULL");
    return ring_bwd_impl(q, k, v, dtype, T, Hq, Hkv, d, cu, B, cp, mode, 0, -1, scale, sched, out, lse, dout, dq, dk,
                         dv, grad_dtype, flags, workspace, ws_bytes, stream, key_lo, key_hi);
}

}  // extern "C"
