// C ABI of the dropless MoE layer forward (declared in include/moe.h).
//
// Host-side argument checks run before anything touches CUDA, so a bad call
// returns an error and launches nothing.  The library allocates nothing: every
// buffer, scratch included, is the caller's.
#include "../../include/moe.h"
#include "kernels.h"

#include <nvtx3/nvToolsExt.h>

#include <atomic>
#include <mutex>
#include <vector>

namespace {

constexpr int kMaxE = 256;
constexpr int kMaxK = 16;
constexpr uint64_t kWaitLimitNs = 1000000000ull;  // bounded device waits: 1 s

std::atomic<uint64_t> g_launches{0};

__device__ int g_device_status = 0;

// Copies the device status word into the caller's word and clears it, in
// stream order: it sees what every kernel queued before it on the stream
// recorded.  One thread; the exchange clears the word atomically, so a
// kernel on another stream that records a timeout meanwhile is not lost
// (it shows in the next read).
__global__ void read_status_kernel(int32_t *out) { *out = atomicExch(&g_device_status, 0); }

struct DeviceState {
    bool ready = false;
    int num_sms = 0;
    int *status = nullptr;
    moe::GemmLaunch gemm;
};
constexpr int kMaxDevices = 64;
DeviceState g_dev[kMaxDevices];
std::mutex g_mu;

// Per-device one-time set-up: SM count, kernel attributes, status word address.
moe_status_t device_state(DeviceState **out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return MOE_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_mu);
    DeviceState &s = g_dev[dev];
    if (!s.ready) {
        if (cudaDeviceGetAttribute(&s.num_sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return MOE_ERR_CUDA;
        int major = 0, minor = 0;
        cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
        if (major != 10) return MOE_ERR_UNSUPPORTED;  // built for sm_103a only
        if (moe::grouped_gemm_setup(s.num_sms, &s.gemm) != cudaSuccess) return MOE_ERR_CUDA;
        if (moe::router_setup() != cudaSuccess) return MOE_ERR_CUDA;
        if (moe::grouped_gemm_mx_setup(&s.gemm) != cudaSuccess) return MOE_ERR_CUDA;
        if (moe::wgrad_setup(&s.gemm) != cudaSuccess) return MOE_ERR_CUDA;
        if (cudaGetSymbolAddress(reinterpret_cast<void **>(&s.status), g_device_status) != cudaSuccess)
            return MOE_ERR_CUDA;
        s.ready = true;
    }
    *out = &s;
    return MOE_OK;
}

inline bool aligned(const void *p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// One NVTX range per C-ABI call, named after the entry point, so that a
// profiler's timeline shows which call queued which kernels.  Without a
// profiler attached the push and pop return at once.
struct Range {
    explicit Range(const char *name) { nvtxRangePushA(name); }
    ~Range() { nvtxRangePop(); }
    Range(const Range &) = delete;
    Range &operator=(const Range &) = delete;
};
#define MOE_RANGE() Range moe_nvtx_range_(__func__)

// Copy streams and events of the pipelined host runner, created once and
// reused: a call takes a set from its device's pool (or creates one) and
// gives it back once everything is queued.  Reusing them is safe: every wait
// a call queues refers to an event recorded earlier in the same call, and a
// later record of the same event does not change a wait already queued.
struct Runner {
    int dev = -1;
    cudaStream_t cin = nullptr, cout = nullptr;
    cudaEvent_t ev[7] = {};
};
std::vector<Runner> g_runners;
std::mutex g_runner_mu;

bool acquire_runner(Runner *r) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return false;
    {
        std::lock_guard<std::mutex> lock(g_runner_mu);
        for (size_t i = 0; i < g_runners.size(); ++i) {
            if (g_runners[i].dev == dev) {
                *r = g_runners[i];
                g_runners.erase(g_runners.begin() + static_cast<std::ptrdiff_t>(i));
                return true;
            }
        }
    }
    Runner n;
    n.dev = dev;
    bool ok = cudaStreamCreateWithFlags(&n.cin, cudaStreamNonBlocking) == cudaSuccess &&
              cudaStreamCreateWithFlags(&n.cout, cudaStreamNonBlocking) == cudaSuccess;
    for (int i = 0; ok && i < 7; ++i) ok = cudaEventCreateWithFlags(&n.ev[i], cudaEventDisableTiming) == cudaSuccess;
    if (!ok) {
        for (int i = 0; i < 7; ++i)
            if (n.ev[i]) cudaEventDestroy(n.ev[i]);
        if (n.cin) cudaStreamDestroy(n.cin);
        if (n.cout) cudaStreamDestroy(n.cout);
        return false;
    }
    *r = n;
    return true;
}

void release_runner(const Runner &r) {
    std::lock_guard<std::mutex> lock(g_runner_mu);
    g_runners.push_back(r);
}

moe_status_t check_shape(int T, int d, int E, int K, int f, bool need_d, bool need_f) {
    if (T < 1 || E < 1 || K < 1 || K > E) return MOE_ERR_INVALID_ARG;
    if (E > kMaxE || K > kMaxK) return MOE_ERR_UNSUPPORTED;
    if (static_cast<int64_t>(T) * K >= (int64_t(1) << 31)) return MOE_ERR_UNSUPPORTED;
    if (need_d && (d < 64 || d % 64 != 0)) return d < 1 ? MOE_ERR_INVALID_ARG : MOE_ERR_UNSUPPORTED;
    if (need_f && (f < 64 || f % 64 != 0)) return f < 1 ? MOE_ERR_INVALID_ARG : MOE_ERR_UNSUPPORTED;
    if (need_d && need_f && static_cast<int64_t>(E) * 2 * f >= (int64_t(1) << 31)) return MOE_ERR_UNSUPPORTED;
    if (need_d && need_f && static_cast<int64_t>(E) * d >= (int64_t(1) << 31)) return MOE_ERR_UNSUPPORTED;
    return MOE_OK;
}

inline moe_status_t cuda_status(cudaError_t e) { return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA; }

size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

bool forward_layout(int T, int d, int E, int K, int f, moe_forward_layout_t *L) {
    const size_t TK = static_cast<size_t>(T) * K;
    size_t o = 0;
    auto take = [&](size_t bytes) {
        const size_t at = o;
        o = align_up(o + bytes, 256);
        return at;
    };
    L->logits = take(static_cast<size_t>(T) * E * 4);
    L->topk_idx = take(TK * 4);
    L->topk_w = take(TK * 4);
    L->counts = take(static_cast<size_t>(E) * 4);
    L->offsets = take(static_cast<size_t>(E + 1) * 4);
    L->row_of = take(TK * 4);
    L->src_tok = take(TK * 4);
    L->route_ws = take(moe::route_workspace_bytes(T, E));
    L->router_ws = take(moe::router_workspace_bytes(d, E));
    L->x_perm = take(TK * d * 2);
    L->h = take(TK * f * 2);
    L->y_perm = take(TK * d * 2);
    L->x_dev = take(static_cast<size_t>(T) * d * 2);
    L->y_dev = take(static_cast<size_t>(T) * d * 2);
    L->total = o;
    return true;
}

bool forward_mxfp8_layout(int T, int d, int E, int K, int f, moe_forward_mxfp8_layout_t *L) {
    const size_t TK = static_cast<size_t>(T) * K;
    size_t o = 0;
    auto take = [&](size_t bytes) {
        const size_t at = o;
        o = align_up(o + bytes, 256);
        return at;
    };
    L->logits = take(static_cast<size_t>(T) * E * 4);
    L->topk_idx = take(TK * 4);
    L->topk_w = take(TK * 4);
    L->counts = take(static_cast<size_t>(E) * 4);
    L->offsets = take(static_cast<size_t>(E + 1) * 4);
    L->row_of = take(TK * 4);
    L->src_tok = take(TK * 4);
    L->route_ws = take(moe::route_workspace_bytes(T, E));
    L->router_ws = take(moe::router_workspace_bytes(d, E));
    L->xq_perm = take(TK * d);
    L->sfa = take(moe::mxfp8_perm_scales_bytes(static_cast<int>(TK), E, d));
    L->hq = take(TK * f);
    L->sfh = take(moe::mxfp8_perm_scales_bytes(static_cast<int>(TK), E, f));
    L->y_perm = take(TK * d * 2);
    L->total = o;
    return true;
}

bool backward_layout(int T, int d, int E, int K, int f, moe_backward_layout_t *L) {
    const size_t TK = static_cast<size_t>(T) * K;
    size_t o = 0;
    auto take = [&](size_t bytes) {
        const size_t at = o;
        o = align_up(o + bytes, 256);
        return at;
    };
    L->dw = take(TK * 4);
    L->dl = take(TK * 4);
    L->dl_row = take(TK * 4);
    L->dy_perm = take(TK * d * 2);
    L->dh = take(TK * f * 2);
    L->a = take(TK * 2 * f * 2);
    L->da = take(TK * 2 * f * 2);
    L->dx_perm = take(TK * d * 2);
    L->WrT = take(static_cast<size_t>(E) * d * 4);
    L->rw_part = take(moe::router_wgrad_slices(static_cast<int>(TK), E) * (static_cast<size_t>(d) + 1) * 4);
    L->tmaps = take(moe::WGRAD_MAP_BYTES * static_cast<size_t>(E));
    L->total = o;
    return true;
}

moe_status_t check_mx_shape(int T, int d, int E, int K, int f) {
    moe_status_t st = check_shape(T, d, E, K, f, true, true);
    if (st != MOE_OK) return st;
    if (d % 128 != 0 || f % 128 != 0) return MOE_ERR_UNSUPPORTED;
    return MOE_OK;
}

moe_status_t run_gemm(bool swiglu, const void *A, const int32_t *offsets, int E, int TK, int d, int f,
                      const void *W, void *out, cudaStream_t stream, void *preact = nullptr) {
    DeviceState *ds = nullptr;
    moe_status_t st = device_state(&ds);
    if (st != MOE_OK) return st;
    const int Kdim = swiglu ? d : f;
    const int n_out = swiglu ? f : d;
    g_launches.fetch_add(1, std::memory_order_relaxed);
    return cuda_status(moe::launch_grouped_gemm(swiglu, A, TK, Kdim, W, E, n_out, offsets, out, ds->gemm,
                                                ds->status, kWaitLimitNs, stream, nullptr, false, preact));
}

// Runs n batches through `compute(x_dev, y_dev)` on `stream` with
// double-buffered device copies: batch i's host->device copy (copy stream
// `cin`) and batch i-1's device->host copy (copy stream `cout`) overlap
// batch i-1's and batch i's compute.  Buffer b = i % 2 is refilled only after
// the compute of batch i-2 that read it, and recomputed only after the copy
// out of batch i-2 that read it.  `stream` ends waiting for the last copy out,
// so its completion means every y_hosts[i] is written.  The copy streams and
// events come from the device's runner pool (created on first use, reused).
template <typename F>
moe_status_t run_pipelined(const uint16_t *const *x_hosts, uint16_t *const *y_hosts, int n, size_t bytes,
                           uint16_t *const xbuf[2], uint16_t *const ybuf[2], cudaStream_t stream, F compute) {
    Runner run;
    if (!acquire_runner(&run)) return MOE_ERR_CUDA;
    cudaStream_t cin = run.cin, cout = run.cout;
    cudaEvent_t *ev = run.ev;
    moe_status_t st = MOE_OK;
    cudaEvent_t entry = ev[0], *xready = ev + 1, *done = ev + 3, *yfree = ev + 5;
    auto chk = [&](cudaError_t e) {
        if (st == MOE_OK && e != cudaSuccess) st = MOE_ERR_CUDA;
        return st == MOE_OK;
    };
    // the copies start after the work the caller queued before this call
    if (chk(cudaEventRecord(entry, stream)) && chk(cudaStreamWaitEvent(cin, entry, 0)))
        chk(cudaStreamWaitEvent(cout, entry, 0));
    for (int i = 0; st == MOE_OK && i < n; ++i) {
        const int b = i & 1;
        if (i >= 2 && !chk(cudaStreamWaitEvent(cin, done[b], 0))) break;
        if (!chk(cudaMemcpyAsync(xbuf[b], x_hosts[i], bytes, cudaMemcpyHostToDevice, cin))) break;
        if (!chk(cudaEventRecord(xready[b], cin))) break;
        if (!chk(cudaStreamWaitEvent(stream, xready[b], 0))) break;
        if (i >= 2 && !chk(cudaStreamWaitEvent(stream, yfree[b], 0))) break;
        if ((st = compute(xbuf[b], ybuf[b])) != MOE_OK) break;
        if (!chk(cudaEventRecord(done[b], stream))) break;
        if (!chk(cudaStreamWaitEvent(cout, done[b], 0))) break;
        if (!chk(cudaMemcpyAsync(y_hosts[i], ybuf[b], bytes, cudaMemcpyDeviceToHost, cout))) break;
        if (!chk(cudaEventRecord(yfree[b], cout))) break;
    }
    if (st == MOE_OK && n > 0) chk(cudaStreamWaitEvent(stream, yfree[(n - 1) & 1], 0));
    release_runner(run);
    return st;
}

}  // namespace

extern "C" {

const char *moe_status_string(int status) {
    switch (status) {
        case MOE_OK: return "MOE_OK";
        case MOE_ERR_INVALID_ARG: return "MOE_ERR_INVALID_ARG: null or misaligned pointer, or size out of range";
        case MOE_ERR_UNSUPPORTED: return "MOE_ERR_UNSUPPORTED: sizes outside what the kernels cover";
        case MOE_ERR_WORKSPACE: return "MOE_ERR_WORKSPACE: workspace smaller than required";
        case MOE_ERR_CUDA: return "MOE_ERR_CUDA: a CUDA call or kernel launch failed";
        case MOE_ERR_DEVICE_TIMEOUT: return "MOE_ERR_DEVICE_TIMEOUT: a bounded device-side wait expired";
        default: return "unknown moe_status_t";
    }
}

int moe_abi_version(void) { return 403; }

uint64_t moe_launch_count(void) { return g_launches.load(std::memory_order_relaxed); }

size_t moe_router_workspace_size(int d, int E) {
    if (d < 64 || d % 64 != 0 || E < 1 || E > kMaxE) return 0;
    return moe::router_workspace_bytes(d, E);
}

moe_status_t moe_router_logits(const uint16_t *x, const float *Wr, const float *bias, int T, int d, int E,
                               float *logits, void *workspace, size_t workspace_bytes, cudaStream_t stream) {
    MOE_RANGE();
    if (!x || !Wr || !logits || !workspace) return MOE_ERR_INVALID_ARG;
    if (!aligned(x, 16) || !aligned(Wr, 4) || !aligned(logits, 4) || (bias && !aligned(bias, 4)) ||
        !aligned(workspace, 16))
        return MOE_ERR_INVALID_ARG;
    moe_status_t st = check_shape(T, d, E, 1, 64, true, false);
    if (st != MOE_OK) return st;
    if (static_cast<int64_t>(E) * d >= (int64_t(1) << 31)) return MOE_ERR_UNSUPPORTED;
    if (workspace_bytes < moe::router_workspace_bytes(d, E)) return MOE_ERR_WORKSPACE;
    DeviceState *ds = nullptr;
    if ((st = device_state(&ds)) != MOE_OK) return st;
    g_launches.fetch_add(2, std::memory_order_relaxed);
    return cuda_status(
        moe::launch_router_logits(x, Wr, bias, T, d, E, logits, workspace, ds->status, kWaitLimitNs, stream));
}

size_t moe_route_workspace_size(int T, int E, int K) {
    if (T < 1 || E < 1 || K < 1) return 0;
    return moe::route_workspace_bytes(T, E);
}

moe_status_t moe_route(const float *logits, int T, int E, int K, int32_t *topk_idx, float *topk_w,
                       int32_t *counts, int32_t *offsets, int32_t *row_of, int32_t *src_tok, void *workspace,
                       size_t workspace_bytes, cudaStream_t stream) {
    MOE_RANGE();
    if (!logits || !topk_idx || !topk_w || !counts || !offsets || !row_of || !src_tok || !workspace)
        return MOE_ERR_INVALID_ARG;
    if (!aligned(logits, 4) || !aligned(topk_idx, 4) || !aligned(topk_w, 4) || !aligned(counts, 4) ||
        !aligned(offsets, 4) || !aligned(row_of, 4) || !aligned(src_tok, 4) || !aligned(workspace, 4))
        return MOE_ERR_INVALID_ARG;
    moe_status_t st = check_shape(T, 64, E, K, 64, false, false);
    if (st != MOE_OK) return st;
    if (workspace_bytes < moe::route_workspace_bytes(T, E)) return MOE_ERR_WORKSPACE;
    g_launches.fetch_add(3, std::memory_order_relaxed);
    return cuda_status(moe::launch_route(logits, T, E, K, topk_idx, topk_w, counts, offsets, row_of, src_tok,
                                         static_cast<int32_t *>(workspace), stream));
}

moe_status_t moe_permute(const uint16_t *x, const int32_t *row_of, int T, int K, int d, uint16_t *x_perm,
                         cudaStream_t stream) {
    MOE_RANGE();
    if (!x || !row_of || !x_perm) return MOE_ERR_INVALID_ARG;
    if (!aligned(x, 16) || !aligned(x_perm, 16) || !aligned(row_of, 4)) return MOE_ERR_INVALID_ARG;
    moe_status_t st = check_shape(T, d, K, K, 64, true, false);
    if (st != MOE_OK) return st;
    g_launches.fetch_add(1, std::memory_order_relaxed);
    return cuda_status(moe::launch_permute(x, row_of, T, K, d, x_perm, stream));
}

moe_status_t moe_grouped_gemm1_swiglu(const uint16_t *x_perm, const int32_t *offsets, int E, int TK, int d, int f,
                                      const uint16_t *W1, uint16_t *h, cudaStream_t stream) {
    MOE_RANGE();
    if (!x_perm || !offsets || !W1 || !h) return MOE_ERR_INVALID_ARG;
    if (!aligned(x_perm, 16) || !aligned(W1, 16) || !aligned(h, 16) || !aligned(offsets, 4))
        return MOE_ERR_INVALID_ARG;
    moe_status_t st = check_shape(TK, d, E, 1, f, true, true);
    if (st != MOE_OK) return st;
    return run_gemm(true, x_perm, offsets, E, TK, d, f, W1, h, stream);
}

moe_status_t moe_grouped_gemm1_swiglu_preact(const uint16_t *x_perm, const int32_t *offsets, int E, int TK, int d,
                                             int f, const uint16_t *W1, uint16_t *h, uint16_t *preact,
                                             cudaStream_t stream) {
    MOE_RANGE();
    if (!x_perm || !offsets || !W1 || !h || !preact) return MOE_ERR_INVALID_ARG;
    if (!aligned(x_perm, 16) || !aligned(W1, 16) || !aligned(h, 16) || !aligned(preact, 16) ||
        !aligned(offsets, 4))
        return MOE_ERR_INVALID_ARG;
    moe_status_t st = check_shape(TK, d, E, 1, f, true, true);
    if (st != MOE_OK) return st;
    return run_gemm(true, x_perm, offsets, E, TK, d, f, W1, h, stream, preact);
}

moe_status_t moe_grouped_gemm2(const uint16_t *h, const int32_t *offsets, int E, int TK, int d, int f,
                               const uint16_t *W2, uint16_t *y_perm, cudaStream_t stream) {
    MOE_RANGE();
    if (!h || !offsets || !W2 || !y_perm) return MOE_ERR_INVALID_ARG;
    if (!aligned(h, 16) || !aligned(W2, 16) || !aligned(y_perm, 16) || !aligned(offsets, 4))
        return MOE_ERR_INVALID_ARG;
    moe_status_t st = check_shape(TK, d, E, 1, f, true, true);
    if (st != MOE_OK) return st;
    return run_gemm(false, h, offsets, E, TK, d, f, W2, y_perm, stream);
}

moe_status_t moe_grouped_gemm1_swiglu_gather(const uint16_t *x, const int32_t *src_tok, const int32_t *offsets,
                                             int T, int E, int TK, int d, int f, const uint16_t *W1, uint16_t *h,
                                             cudaStream_t stream) {
    MOE_RANGE();
    if (!x || !src_tok || !offsets || !W1 || !h) return MOE_ERR_INVALID_ARG;
    if (!aligned(x, 16) || !aligned(W1, 16) || !aligned(h, 16) || !aligned(src_tok, 4) || !aligned(offsets, 4))
        return MOE_ERR_INVALID_ARG;
    moe_status_t st = check_shape(TK, d, E, 1, f, true, true);
    if (st != MOE_OK) return st;
    if (T < 1) return MOE_ERR_INVALID_ARG;
    DeviceState *ds = nullptr;
    if ((st = device_state(&ds)) != MOE_OK) return st;
    const moe::GatherArgs g{src_tok, T};
    g_launches.fetch_add(1, std::memory_order_relaxed);
    return cuda_status(moe::launch_grouped_gemm(true, x, TK, d, W1, E, f, offsets, h, ds->gemm, ds->status,
                                                kWaitLimitNs, stream, nullptr, false, nullptr, &g));
}

size_t moe_combine_counters_size(int T, int d) {
    if (T < 1 || d < 64 || d % 64 != 0) return 0;
    return static_cast<size_t>(T) * ((d + 255) / 256) * sizeof(int32_t);
}

moe_status_t moe_grouped_gemm2_combine(const uint16_t *h, const int32_t *offsets, int E, int TK, int d, int f,
                                       const uint16_t *W2, const int32_t *src_tok, const int32_t *row_of,
                                       const float *topk_w, int T, int K, uint16_t *y_perm, int32_t *counters,
                                       size_t counters_bytes, uint16_t *y, cudaStream_t stream) {
    MOE_RANGE();
    if (!h || !offsets || !W2 || !src_tok || !row_of || !topk_w || !y_perm || !counters || !y)
        return MOE_ERR_INVALID_ARG;
    if (!aligned(h, 16) || !aligned(W2, 16) || !aligned(y_perm, 16) || !aligned(y, 16) || !aligned(offsets, 4) ||
        !aligned(src_tok, 4) || !aligned(row_of, 4) || !aligned(topk_w, 4) || !aligned(counters, 4))
        return MOE_ERR_INVALID_ARG;
    moe_status_t st = check_shape(T, d, E, K, f, true, true);
    if (st != MOE_OK) return st;
    if (static_cast<int64_t>(T) * K != TK) return MOE_ERR_INVALID_ARG;
    const size_t need = moe_combine_counters_size(T, d);
    if (counters_bytes < need) return MOE_ERR_WORKSPACE;
    DeviceState *ds = nullptr;
    if ((st = device_state(&ds)) != MOE_OK) return st;
    if (cudaMemsetAsync(counters, 0, need, stream) != cudaSuccess) return MOE_ERR_CUDA;
    moe::CombineArgs cb{src_tok, row_of, topk_w, T, K, counters, y};
    g_launches.fetch_add(1, std::memory_order_relaxed);
    return cuda_status(moe::launch_grouped_gemm(false, h, TK, f, W2, E, d, offsets, y_perm, ds->gemm, ds->status,
                                                kWaitLimitNs, stream, &cb));
}

moe_status_t moe_grouped_mlp(const uint16_t *x_perm, const int32_t *offsets, int E, int TK, int d, int f,
                             const uint16_t *W1, const uint16_t *W2, uint16_t *h, uint16_t *y_perm,
                             cudaStream_t stream) {
    MOE_RANGE();
    if (!W2 || !y_perm || !aligned(W2, 16) || !aligned(y_perm, 16)) return MOE_ERR_INVALID_ARG;
    moe_status_t st = moe_grouped_gemm1_swiglu(x_perm, offsets, E, TK, d, f, W1, h, stream);
    if (st != MOE_OK) return st;
    return moe_grouped_gemm2(h, offsets, E, TK, d, f, W2, y_perm, stream);
}

moe_status_t moe_unpermute(const uint16_t *y_perm, const int32_t *row_of, const float *topk_w, int T, int K, int d,
                           uint16_t *y, cudaStream_t stream) {
    MOE_RANGE();
    if (!y_perm || !row_of || !topk_w || !y) return MOE_ERR_INVALID_ARG;
    if (!aligned(y_perm, 16) || !aligned(y, 16) || !aligned(row_of, 4) || !aligned(topk_w, 4))
        return MOE_ERR_INVALID_ARG;
    moe_status_t st = check_shape(T, d, K, K, 64, true, false);
    if (st != MOE_OK) return st;
    g_launches.fetch_add(1, std::memory_order_relaxed);
    return cuda_status(moe::launch_unpermute(y_perm, row_of, topk_w, T, K, d, y, stream));
}

size_t moe_forward_workspace_size(int T, int d, int E, int K, int f) {
    if (check_shape(T, d, E, K, f, true, true) != MOE_OK) return 0;
    moe_forward_layout_t L;
    forward_layout(T, d, E, K, f, &L);
    return L.total;
}

moe_status_t moe_forward_views(int T, int d, int E, int K, int f, moe_forward_layout_t *layout) {
    MOE_RANGE();
    if (!layout) return MOE_ERR_INVALID_ARG;
    moe_status_t st = check_shape(T, d, E, K, f, true, true);
    if (st != MOE_OK) return st;
    forward_layout(T, d, E, K, f, layout);
    return MOE_OK;
}

}  // extern "C"

namespace {

// The forward of moe_forward and moe_forward_train.  `fuse_permute`: GEMM1
// reads its rows straight from x (the permute fused into its operand load)
// and x_perm is not written.
moe_status_t forward_impl(const uint16_t *x, const float *Wr, const float *bias, const uint16_t *W1,
                          const uint16_t *W2, int T, int d, int E, int K, int f, uint16_t *y, void *workspace,
                          size_t workspace_bytes, uint16_t *preact, bool fuse_permute, cudaStream_t stream) {
    if (!x || !Wr || !W1 || !W2 || !y || !workspace) return MOE_ERR_INVALID_ARG;
    if (preact && !aligned(preact, 16)) return MOE_ERR_INVALID_ARG;
    if (!aligned(x, 16) || !aligned(W1, 16) || !aligned(W2, 16) || !aligned(y, 16) || !aligned(workspace, 16) ||
        !aligned(Wr, 4) || (bias && !aligned(bias, 4)))
        return MOE_ERR_INVALID_ARG;
    moe_status_t st = check_shape(T, d, E, K, f, true, true);
    if (st != MOE_OK) return st;
    moe_forward_layout_t L;
    forward_layout(T, d, E, K, f, &L);
    if (workspace_bytes < L.total) return MOE_ERR_WORKSPACE;
    uint8_t *ws = static_cast<uint8_t *>(workspace);
    auto at = [&](size_t off) { return static_cast<void *>(ws + off); };
    const int TK = T * K;
    float *logits = static_cast<float *>(at(L.logits));
    int32_t *idx = static_cast<int32_t *>(at(L.topk_idx));
    float *w = static_cast<float *>(at(L.topk_w));
    int32_t *counts = static_cast<int32_t *>(at(L.counts));
    int32_t *offsets = static_cast<int32_t *>(at(L.offsets));
    int32_t *row_of = static_cast<int32_t *>(at(L.row_of));
    int32_t *src_tok = static_cast<int32_t *>(at(L.src_tok));
    uint16_t *x_perm = static_cast<uint16_t *>(at(L.x_perm));
    uint16_t *h = static_cast<uint16_t *>(at(L.h));
    uint16_t *y_perm = static_cast<uint16_t *>(at(L.y_perm));
    if ((st = moe_router_logits(x, Wr, bias, T, d, E, logits, at(L.router_ws), L.x_perm - L.router_ws,
                                stream)) != MOE_OK)
        return st;
    if ((st = moe_route(logits, T, E, K, idx, w, counts, offsets, row_of, src_tok, at(L.route_ws),
                        L.router_ws - L.route_ws, stream)) != MOE_OK)
        return st;
    if (fuse_permute) {
        st = moe_grouped_gemm1_swiglu_gather(x, src_tok, offsets, T, E, TK, d, f, W1, h, stream);
    } else {
        if ((st = moe_permute(x, row_of, T, K, d, x_perm, stream)) != MOE_OK) return st;
        if (preact)
            st = moe_grouped_gemm1_swiglu_preact(x_perm, offsets, E, TK, d, f, W1, h, preact, stream);
        else
            st = moe_grouped_gemm1_swiglu(x_perm, offsets, E, TK, d, f, W1, h, stream);
    }
    if (st != MOE_OK) return st;
    if ((st = moe_grouped_gemm2(h, offsets, E, TK, d, f, W2, y_perm, stream)) != MOE_OK) return st;
    return moe_unpermute(y_perm, row_of, w, T, K, d, y, stream);
}

}  // namespace

extern "C" {

int moe_forward_fuses_permute(int T, int d, int E, int K, int f) {
    if (check_shape(T, d, E, K, f, true, true) != MOE_OK) return 0;
    return moe::grouped_gemm1_prefers_gather(T * K, E, f) ? 1 : 0;
}

moe_status_t moe_forward_train(const uint16_t *x, const float *Wr, const float *bias, const uint16_t *W1,
                               const uint16_t *W2, int T, int d, int E, int K, int f, uint16_t *y, void *workspace,
                               size_t workspace_bytes, uint16_t *preact, cudaStream_t stream) {
    MOE_RANGE();
    // the backward reads x_perm: the training forward always writes it
    return forward_impl(x, Wr, bias, W1, W2, T, d, E, K, f, y, workspace, workspace_bytes, preact, false, stream);
}

moe_status_t moe_forward(const uint16_t *x, const float *Wr, const float *bias, const uint16_t *W1,
                         const uint16_t *W2, int T, int d, int E, int K, int f, uint16_t *y, void *workspace,
                         size_t workspace_bytes, cudaStream_t stream) {
    MOE_RANGE();
    return forward_impl(x, Wr, bias, W1, W2, T, d, E, K, f, y, workspace, workspace_bytes, nullptr,
                        moe_forward_fuses_permute(T, d, E, K, f) != 0, stream);
}

moe_status_t moe_forward_host(const uint16_t *x_host, const float *Wr, const float *bias, const uint16_t *W1,
                              const uint16_t *W2, int T, int d, int E, int K, int f, uint16_t *y_host,
                              void *workspace, size_t workspace_bytes, cudaStream_t stream) {
    MOE_RANGE();
    if (!x_host || !y_host || !workspace) return MOE_ERR_INVALID_ARG;
    moe_status_t st = check_shape(T, d, E, K, f, true, true);
    if (st != MOE_OK) return st;
    moe_forward_layout_t L;
    forward_layout(T, d, E, K, f, &L);
    if (workspace_bytes < L.total) return MOE_ERR_WORKSPACE;
    uint8_t *ws = static_cast<uint8_t *>(workspace);
    uint16_t *x_dev = reinterpret_cast<uint16_t *>(ws + L.x_dev);
    uint16_t *y_dev = reinterpret_cast<uint16_t *>(ws + L.y_dev);
    const size_t bytes = static_cast<size_t>(T) * d * 2;
    if (cudaMemcpyAsync(x_dev, x_host, bytes, cudaMemcpyHostToDevice, stream) != cudaSuccess) return MOE_ERR_CUDA;
    if ((st = moe_forward(x_dev, Wr, bias, W1, W2, T, d, E, K, f, y_dev, workspace, workspace_bytes, stream)) !=
        MOE_OK)
        return st;
    return cuda_status(cudaMemcpyAsync(y_host, y_dev, bytes, cudaMemcpyDeviceToHost, stream));
}

size_t moe_forward_host_pipelined_workspace_size(int T, int d, int E, int K, int f) {
    if (check_shape(T, d, E, K, f, true, true) != MOE_OK) return 0;
    moe_forward_layout_t L;
    forward_layout(T, d, E, K, f, &L);
    // a second x and y buffer after the layer's workspace
    return L.total + 2 * align_up(static_cast<size_t>(T) * d * 2, 256);
}

moe_status_t moe_forward_host_pipelined(const uint16_t *const *x_hosts, uint16_t *const *y_hosts, int n_batches,
                                        const float *Wr, const float *bias, const uint16_t *W1, const uint16_t *W2,
                                        int T, int d, int E, int K, int f, void *workspace, size_t workspace_bytes,
                                        cudaStream_t stream) {
    MOE_RANGE();
    if (!x_hosts || !y_hosts || n_batches < 1 || !workspace) return MOE_ERR_INVALID_ARG;
    for (int i = 0; i < n_batches; ++i)
        if (!x_hosts[i] || !y_hosts[i]) return MOE_ERR_INVALID_ARG;
    if (!aligned(workspace, 256)) return MOE_ERR_INVALID_ARG;
    moe_status_t st = check_shape(T, d, E, K, f, true, true);
    if (st != MOE_OK) return st;
    if (workspace_bytes < moe_forward_host_pipelined_workspace_size(T, d, E, K, f)) return MOE_ERR_WORKSPACE;
    moe_forward_layout_t L;
    forward_layout(T, d, E, K, f, &L);
    uint8_t *ws = static_cast<uint8_t *>(workspace);
    const size_t bytes = static_cast<size_t>(T) * d * 2;
    const size_t extra = align_up(bytes, 256);
    uint16_t *const xbuf[2] = {reinterpret_cast<uint16_t *>(ws + L.x_dev), reinterpret_cast<uint16_t *>(ws + L.total)};
    uint16_t *const ybuf[2] = {reinterpret_cast<uint16_t *>(ws + L.y_dev),
                               reinterpret_cast<uint16_t *>(ws + L.total + extra)};
    return run_pipelined(x_hosts, y_hosts, n_batches, bytes, xbuf, ybuf, stream, [&](uint16_t *xd, uint16_t *yd) {
        return moe_forward(xd, Wr, bias, W1, W2, T, d, E, K, f, yd, workspace, workspace_bytes, stream);
    });
}

size_t moe_mxfp8_scales_size(int rows, int K) {
    if (rows < 1 || K < 128 || K % 128 != 0) return 0;
    return moe::mxfp8_scales_bytes(rows, K);
}

moe_status_t moe_mxfp8_quantize(const uint16_t *src, int rows, int K, uint8_t *codes, uint8_t *scales,
                                cudaStream_t stream) {
    MOE_RANGE();
    if (!src || !codes || !scales) return MOE_ERR_INVALID_ARG;
    if (!aligned(src, 16) || !aligned(codes, 16) || !aligned(scales, 16)) return MOE_ERR_INVALID_ARG;
    if (rows < 1 || K < 1) return MOE_ERR_INVALID_ARG;
    if (K % 128 != 0) return MOE_ERR_UNSUPPORTED;
    g_launches.fetch_add(1, std::memory_order_relaxed);
    return cuda_status(moe::launch_mxfp8_quantize(src, rows, K, codes, scales, stream));
}

size_t moe_mxfp8_act_scales_size(int TK, int E, int K) {
    if (TK < 1 || E < 1 || E > kMaxE || K < 128 || K % 128 != 0) return 0;
    return moe::mxfp8_perm_scales_bytes(TK, E, K);
}

moe_status_t moe_permute_mxfp8(const uint16_t *x, const int32_t *topk_idx, const int32_t *row_of,
                               const int32_t *offsets, int T, int K, int d, int E, uint8_t *xq_perm, uint8_t *sfa,
                               size_t sfa_bytes, cudaStream_t stream) {
    MOE_RANGE();
    if (!x || !topk_idx || !row_of || !offsets || !xq_perm || !sfa) return MOE_ERR_INVALID_ARG;
    if (!aligned(x, 16) || !aligned(xq_perm, 16) || !aligned(sfa, 16) || !aligned(topk_idx, 4) ||
        !aligned(row_of, 4) || !aligned(offsets, 4))
        return MOE_ERR_INVALID_ARG;
    moe_status_t st = check_shape(T, d, E, K, 64, true, false);
    if (st != MOE_OK) return st;
    if (d % 128 != 0) return MOE_ERR_UNSUPPORTED;
    if (sfa_bytes < moe::mxfp8_perm_scales_bytes(T * K, E, d)) return MOE_ERR_WORKSPACE;
    g_launches.fetch_add(1, std::memory_order_relaxed);
    return cuda_status(moe::launch_permute_mxfp8(x, topk_idx, row_of, offsets, T, K, d, E, xq_perm, sfa, stream));
}

moe_status_t moe_grouped_gemm1_swiglu_mxfp8(const uint8_t *xq_perm, const uint8_t *sfa, size_t sfa_bytes,
                                            const int32_t *offsets, int E, int TK, int d, int f, const uint8_t *W1q,
                                            const uint8_t *W1s, uint8_t *hq, uint8_t *sfh, size_t sfh_bytes,
                                            cudaStream_t stream) {
    MOE_RANGE();
    if (!xq_perm || !sfa || !offsets || !W1q || !W1s || !hq || !sfh) return MOE_ERR_INVALID_ARG;
    if (!aligned(xq_perm, 16) || !aligned(sfa, 16) || !aligned(W1q, 16) || !aligned(W1s, 16) || !aligned(hq, 16) ||
        !aligned(sfh, 16) || !aligned(offsets, 4))
        return MOE_ERR_INVALID_ARG;
    moe_status_t st = check_mx_shape(TK, d, E, 1, f);
    if (st != MOE_OK) return st;
    if (sfa_bytes < moe::mxfp8_perm_scales_bytes(TK, E, d) || sfh_bytes < moe::mxfp8_perm_scales_bytes(TK, E, f))
        return MOE_ERR_WORKSPACE;
    DeviceState *ds = nullptr;
    if ((st = device_state(&ds)) != MOE_OK) return st;
    g_launches.fetch_add(1, std::memory_order_relaxed);
    return cuda_status(moe::launch_grouped_gemm_mx(true, xq_perm, sfa, sfa_bytes, TK, d, W1q, W1s,
                                                   moe::mxfp8_scales_bytes(E * 2 * f, d), E, f, offsets, hq, sfh,
                                                   sfh_bytes, ds->gemm, ds->status, kWaitLimitNs, stream));
}

moe_status_t moe_grouped_gemm2_mxfp8(const uint8_t *hq, const uint8_t *sfh, size_t sfh_bytes, const int32_t *offsets,
                                     int E, int TK, int d, int f, const uint8_t *W2q, const uint8_t *W2s,
                                     uint16_t *y_perm, cudaStream_t stream) {
    MOE_RANGE();
    if (!hq || !sfh || !offsets || !W2q || !W2s || !y_perm) return MOE_ERR_INVALID_ARG;
    if (!aligned(hq, 16) || !aligned(sfh, 16) || !aligned(W2q, 16) || !aligned(W2s, 16) || !aligned(y_perm, 16) ||
        !aligned(offsets, 4))
        return MOE_ERR_INVALID_ARG;
    moe_status_t st = check_mx_shape(TK, d, E, 1, f);
    if (st != MOE_OK) return st;
    if (sfh_bytes < moe::mxfp8_perm_scales_bytes(TK, E, f)) return MOE_ERR_WORKSPACE;
    DeviceState *ds = nullptr;
    if ((st = device_state(&ds)) != MOE_OK) return st;
    g_launches.fetch_add(1, std::memory_order_relaxed);
    return cuda_status(moe::launch_grouped_gemm_mx(false, hq, sfh, sfh_bytes, TK, f, W2q, W2s,
                                                   moe::mxfp8_scales_bytes(E * d, f), E, d, offsets, y_perm, nullptr,
                                                   0, ds->gemm, ds->status, kWaitLimitNs, stream));
}

size_t moe_forward_mxfp8_workspace_size(int T, int d, int E, int K, int f) {
    if (check_mx_shape(T, d, E, K, f) != MOE_OK) return 0;
    moe_forward_mxfp8_layout_t L;
    forward_mxfp8_layout(T, d, E, K, f, &L);
    return L.total;
}

moe_status_t moe_forward_mxfp8_views(int T, int d, int E, int K, int f, moe_forward_mxfp8_layout_t *layout) {
    MOE_RANGE();
    if (!layout) return MOE_ERR_INVALID_ARG;
    moe_status_t st = check_mx_shape(T, d, E, K, f);
    if (st != MOE_OK) return st;
    forward_mxfp8_layout(T, d, E, K, f, layout);
    return MOE_OK;
}

moe_status_t moe_forward_mxfp8(const uint16_t *x, const float *Wr, const float *bias, const uint8_t *W1q,
                               const uint8_t *W1s, const uint8_t *W2q, const uint8_t *W2s, int T, int d, int E, int K,
                               int f, uint16_t *y, void *workspace, size_t workspace_bytes, cudaStream_t stream) {
    MOE_RANGE();
    if (!x || !Wr || !W1q || !W1s || !W2q || !W2s || !y || !workspace) return MOE_ERR_INVALID_ARG;
    if (!aligned(x, 16) || !aligned(y, 16) || !aligned(workspace, 16) || !aligned(Wr, 4) ||
        (bias && !aligned(bias, 4)))
        return MOE_ERR_INVALID_ARG;
    moe_status_t st = check_mx_shape(T, d, E, K, f);
    if (st != MOE_OK) return st;
    moe_forward_mxfp8_layout_t L;
    forward_mxfp8_layout(T, d, E, K, f, &L);
    if (workspace_bytes < L.total) return MOE_ERR_WORKSPACE;
    uint8_t *ws = static_cast<uint8_t *>(workspace);
    auto at = [&](size_t off) { return static_cast<void *>(ws + off); };
    const int TK = T * K;
    float *logits = static_cast<float *>(at(L.logits));
    int32_t *idx = static_cast<int32_t *>(at(L.topk_idx));
    float *w = static_cast<float *>(at(L.topk_w));
    int32_t *counts = static_cast<int32_t *>(at(L.counts));
    int32_t *offsets = static_cast<int32_t *>(at(L.offsets));
    int32_t *row_of = static_cast<int32_t *>(at(L.row_of));
    int32_t *src_tok = static_cast<int32_t *>(at(L.src_tok));
    uint8_t *xq = static_cast<uint8_t *>(at(L.xq_perm));
    uint8_t *sfa = static_cast<uint8_t *>(at(L.sfa));
    uint8_t *hq = static_cast<uint8_t *>(at(L.hq));
    uint8_t *sfh = static_cast<uint8_t *>(at(L.sfh));
    uint16_t *y_perm = static_cast<uint16_t *>(at(L.y_perm));
    if ((st = moe_router_logits(x, Wr, bias, T, d, E, logits, at(L.router_ws), L.xq_perm - L.router_ws, stream)) !=
        MOE_OK)
        return st;
    if ((st = moe_route(logits, T, E, K, idx, w, counts, offsets, row_of, src_tok, at(L.route_ws),
                        L.router_ws - L.route_ws, stream)) != MOE_OK)
        return st;
    if ((st = moe_permute_mxfp8(x, idx, row_of, offsets, T, K, d, E, xq, sfa, L.hq - L.sfa, stream)) != MOE_OK)
        return st;
    if ((st = moe_grouped_gemm1_swiglu_mxfp8(xq, sfa, L.hq - L.sfa, offsets, E, TK, d, f, W1q, W1s, hq, sfh,
                                             L.y_perm - L.sfh, stream)) != MOE_OK)
        return st;
    if ((st = moe_grouped_gemm2_mxfp8(hq, sfh, L.y_perm - L.sfh, offsets, E, TK, d, f, W2q, W2s, y_perm, stream)) !=
        MOE_OK)
        return st;
    return moe_unpermute(y_perm, row_of, w, T, K, d, y, stream);
}

size_t moe_forward_mxfp8_host_pipelined_workspace_size(int T, int d, int E, int K, int f) {
    if (check_mx_shape(T, d, E, K, f) != MOE_OK) return 0;
    moe_forward_mxfp8_layout_t L;
    forward_mxfp8_layout(T, d, E, K, f, &L);
    // two x and two y buffers after the layer's workspace
    return L.total + 4 * align_up(static_cast<size_t>(T) * d * 2, 256);
}

moe_status_t moe_forward_mxfp8_host_pipelined(const uint16_t *const *x_hosts, uint16_t *const *y_hosts,
                                              int n_batches, const float *Wr, const float *bias,
                                              const uint8_t *W1q, const uint8_t *W1s, const uint8_t *W2q,
                                              const uint8_t *W2s, int T, int d, int E, int K, int f,
                                              void *workspace, size_t workspace_bytes, cudaStream_t stream) {
    MOE_RANGE();
    if (!x_hosts || !y_hosts || n_batches < 1 || !workspace) return MOE_ERR_INVALID_ARG;
    for (int i = 0; i < n_batches; ++i)
        if (!x_hosts[i] || !y_hosts[i]) return MOE_ERR_INVALID_ARG;
    if (!aligned(workspace, 256)) return MOE_ERR_INVALID_ARG;
    moe_status_t st = check_mx_shape(T, d, E, K, f);
    if (st != MOE_OK) return st;
    if (workspace_bytes < moe_forward_mxfp8_host_pipelined_workspace_size(T, d, E, K, f)) return MOE_ERR_WORKSPACE;
    moe_forward_mxfp8_layout_t L;
    forward_mxfp8_layout(T, d, E, K, f, &L);
    uint8_t *ws = static_cast<uint8_t *>(workspace);
    const size_t bytes = static_cast<size_t>(T) * d * 2;
    const size_t extra = align_up(bytes, 256);
    uint16_t *const xbuf[2] = {reinterpret_cast<uint16_t *>(ws + L.total),
                               reinterpret_cast<uint16_t *>(ws + L.total + extra)};
    uint16_t *const ybuf[2] = {reinterpret_cast<uint16_t *>(ws + L.total + 2 * extra),
                               reinterpret_cast<uint16_t *>(ws + L.total + 3 * extra)};
    return run_pipelined(x_hosts, y_hosts, n_batches, bytes, xbuf, ybuf, stream, [&](uint16_t *xd, uint16_t *yd) {
        return moe_forward_mxfp8(xd, Wr, bias, W1q, W1s, W2q, W2s, T, d, E, K, f, yd, workspace, L.total, stream);
    });
}

size_t moe_backward_workspace_size(int T, int d, int E, int K, int f) {
    if (check_shape(T, d, E, K, f, true, true) != MOE_OK) return 0;
    moe_backward_layout_t L;
    backward_layout(T, d, E, K, f, &L);
    return L.total;
}

moe_status_t moe_backward_views(int T, int d, int E, int K, int f, moe_backward_layout_t *layout) {
    MOE_RANGE();
    if (!layout) return MOE_ERR_INVALID_ARG;
    moe_status_t st = check_shape(T, d, E, K, f, true, true);
    if (st != MOE_OK) return st;
    backward_layout(T, d, E, K, f, layout);
    return MOE_OK;
}

moe_status_t moe_backward(const uint16_t *x, const float *Wr, const float *bias, const uint16_t *W1,
                          const uint16_t *W2, int T, int d, int E, int K, int f, const uint16_t *dy,
                          const void *fwd_workspace, size_t fwd_workspace_bytes, const uint16_t *preact,
                          uint16_t *dx, float *dWr, float *dbias, float *dW1, float *dW2, void *workspace,
                          size_t workspace_bytes, cudaStream_t stream) {
    MOE_RANGE();
    (void)bias;  // the bias enters the gradients only through the routing recorded by the forward
    if (!x || !Wr || !W1 || !W2 || !dy || !fwd_workspace || !dx || !dWr || !dbias || !dW1 || !dW2 || !workspace)
        return MOE_ERR_INVALID_ARG;
    if (!aligned(x, 16) || !aligned(W1, 16) || !aligned(W2, 16) || !aligned(dy, 16) || !aligned(dx, 16) ||
        !aligned(fwd_workspace, 16) || !aligned(workspace, 128) || !aligned(Wr, 4) || !aligned(dWr, 4) ||
        !aligned(dbias, 4) || !aligned(dW1, 16) || !aligned(dW2, 16) || (preact && !aligned(preact, 16)))
        return MOE_ERR_INVALID_ARG;
    moe_status_t st = check_shape(T, d, E, K, f, true, true);
    if (st != MOE_OK) return st;
    moe_forward_layout_t F;
    forward_layout(T, d, E, K, f, &F);
    moe_backward_layout_t B;
    backward_layout(T, d, E, K, f, &B);
    if (fwd_workspace_bytes < F.total || workspace_bytes < B.total) return MOE_ERR_WORKSPACE;
    DeviceState *ds = nullptr;
    if ((st = device_state(&ds)) != MOE_OK) return st;
    const uint8_t *fw = static_cast<const uint8_t *>(fwd_workspace);
    uint8_t *bw = static_cast<uint8_t *>(workspace);
    auto fv = [&](size_t off) { return fw + off; };
    auto bv = [&](size_t off) { return bw + off; };
    const int32_t *topk_idx = reinterpret_cast<const int32_t *>(fv(F.topk_idx));
    const float *topk_w = reinterpret_cast<const float *>(fv(F.topk_w));
    const int32_t *offsets = reinterpret_cast<const int32_t *>(fv(F.offsets));
    const int32_t *row_of = reinterpret_cast<const int32_t *>(fv(F.row_of));
    const uint16_t *x_perm = reinterpret_cast<const uint16_t *>(fv(F.x_perm));
    const uint16_t *h = reinterpret_cast<const uint16_t *>(fv(F.h));
    const uint16_t *y_perm = reinterpret_cast<const uint16_t *>(fv(F.y_perm));
    float *dw = reinterpret_cast<float *>(bv(B.dw));
    float *dl = reinterpret_cast<float *>(bv(B.dl));
    float *dl_row = reinterpret_cast<float *>(bv(B.dl_row));
    uint16_t *dy_perm = reinterpret_cast<uint16_t *>(bv(B.dy_perm));
    uint16_t *dh = reinterpret_cast<uint16_t *>(bv(B.dh));
    uint16_t *a = reinterpret_cast<uint16_t *>(bv(B.a));
    uint16_t *da = reinterpret_cast<uint16_t *>(bv(B.da));
    uint16_t *dx_perm = reinterpret_cast<uint16_t *>(bv(B.dx_perm));
    float *WrT = reinterpret_cast<float *>(bv(B.WrT));
    float *rw_part = reinterpret_cast<float *>(bv(B.rw_part));
    void *tmaps = bv(B.tmaps);
    const int TK = T * K;
    const moe::GemmLaunch &g = ds->gemm;
    cudaError_t e = cudaSuccess;
    auto go = [&](cudaError_t r, int launches) {
        if (e == cudaSuccess) e = r;
        g_launches.fetch_add(launches, std::memory_order_relaxed);
    };
    // Wr transposed for dx (the dgrad GEMMs read W1 and W2 as stored, MN-major)
    go(moe::launch_transpose_f32(Wr, 1, d, E, WrT, stream), 1);
    // combine and router
    go(moe::launch_combine_bwd(dy, y_perm, row_of, topk_w, T, K, d, dw, dy_perm, stream), 1);
    go(moe::launch_router_bwd(topk_w, dw, row_of, T, K, dl, dl_row, stream), 1);
    // GEMM2 dgrad: dh = dy_perm . W2[e]
    go(moe::launch_grouped_gemm(false, dy_perm, TK, d, W2, E, f, offsets, dh, g, ds->status, kWaitLimitNs, stream,
                                nullptr, true),
       1);
    // GEMM1 pre-activations: as the forward saved them, else computed again; then SwiGLU backward
    if (!preact)
        go(moe::launch_grouped_gemm(false, x_perm, TK, d, W1, E, 2 * f, offsets, a, g, ds->status, kWaitLimitNs,
                                    stream),
           1);
    go(moe::launch_swiglu_bwd(preact ? preact : a, dh, TK, f, da, stream), 1);
    // GEMM1 dgrad: dx_perm = da . W1[e]
    go(moe::launch_grouped_gemm(false, da, TK, 2 * f, W1, E, d, offsets, dx_perm, g, ds->status, kWaitLimitNs,
                                stream, nullptr, true),
       1);
    // weight gradients over each expert's rows: dW2[e] = dy_perm[e]^T h[e], dW1[e] = da[e]^T x_perm[e]
    // (the two share the per-expert tensor-map scratch: stream order separates them)
    go(moe::launch_wgrad(dy_perm, h, d, f, offsets, E, TK, dW2, tmaps, g, ds->status, kWaitLimitNs, stream), 2);
    go(moe::launch_wgrad(da, x_perm, 2 * f, d, offsets, E, TK, dW1, tmaps, g, ds->status, kWaitLimitNs, stream), 2);
    // router weights and the input gradient
    go(moe::launch_router_wgrad(x_perm, dl_row, offsets, E, TK, d, rw_part, dWr, dbias, stream), 2);
    go(moe::launch_dx(dx_perm, WrT, row_of, topk_idx, dl, T, K, E, d, dx, stream), 1);
    return cuda_status(e);
}

moe_status_t moe_check_bounded_wait(uint64_t limit_ns, cudaStream_t stream) {
    MOE_RANGE();
    if (limit_ns < 1000ull || limit_ns > kWaitLimitNs) return MOE_ERR_INVALID_ARG;
    DeviceState *ds = nullptr;
    moe_status_t st = device_state(&ds);
    if (st != MOE_OK) return st;
    g_launches.fetch_add(1, std::memory_order_relaxed);
    return cuda_status(moe::launch_bounded_wait_probe(ds->status, limit_ns, stream));
}

moe_status_t moe_last_device_status(int32_t *dev_status_word, cudaStream_t stream) {
    MOE_RANGE();
    if (!dev_status_word || !aligned(dev_status_word, 4)) return MOE_ERR_INVALID_ARG;
    DeviceState *ds = nullptr;
    moe_status_t st = device_state(&ds);
    if (st != MOE_OK) return st;
    g_launches.fetch_add(1, std::memory_order_relaxed);
    read_status_kernel<<<1, 1, 0, stream>>>(dev_status_word);
    return cuda_status(cudaGetLastError());
}

moe_status_t moe_device_status(int *status_out) {
    MOE_RANGE();
    if (!status_out) return MOE_ERR_INVALID_ARG;
    DeviceState *ds = nullptr;
    moe_status_t st = device_state(&ds);
    if (st != MOE_OK) return st;
    int v = 0;
    if (cudaMemcpyFromSymbol(&v, g_device_status, sizeof(int)) != cudaSuccess) return MOE_ERR_CUDA;
    const int zero = 0;
    if (cudaMemcpyToSymbol(g_device_status, &zero, sizeof(int)) != cudaSuccess) return MOE_ERR_CUDA;
    *status_out = v;
    return MOE_OK;
}

}  // extern "C"
