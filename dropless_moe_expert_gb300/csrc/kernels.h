// Internal launchers of the sm_103a kernels (not part of the C ABI).
#pragma once

#include <cuda_runtime_api.h>
#include <stddef.h>
#include <stdint.h>

#include <algorithm>
#include <atomic>

namespace moe {

// Blocks of `kernel` (launched with `threads` threads and no dynamic shared
// memory) that are resident on the current device at once: one wave.
// Worked out on the first call per device and kept in `cache`, one slot per
// device (at most 64 devices).
template <class Kernel>
cudaError_t one_wave(Kernel kernel, int threads, std::atomic<int> (&cache)[64], int *blocks) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    int wave = cache[dev].load(std::memory_order_relaxed);
    if (wave == 0) {
        int sms = 0, per_sm = 0;
        cudaError_t err = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        if (err == cudaSuccess) err = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, threads, 0);
        if (err != cudaSuccess) return err;
        wave = std::max(1, sms * std::max(1, per_sm));
        cache[dev].store(wave, std::memory_order_relaxed);
    }
    *blocks = wave;
    return cudaSuccess;
}

// Tokens per routing chunk: the unit of the per-chunk histograms that make the
// dispatch order deterministic.
constexpr int kRouteChunk = 64;

inline int route_num_chunks(int T) { return (T + kRouteChunk - 1) / kRouteChunk; }
// chunk_counts [C, E] and chunk_base [C, E], int32
inline size_t route_workspace_bytes(int T, int E) {
    return static_cast<size_t>(route_num_chunks(T)) * static_cast<size_t>(E) * 2 * sizeof(int32_t);
}

// Router: the exact three-piece bf16 split of Wr [3][E][d] lives in caller
// scratch of router_workspace_bytes(d, E) bytes (16-byte aligned).
size_t router_workspace_bytes(int d, int E);
// Kernel attributes; once per device, before any capture.
cudaError_t router_setup();
// Width (experts) of one router tile for this shape: 32, 64 or 128.
int router_tile_n(int T, int E);
cudaError_t launch_router_logits(const uint16_t *x, const float *Wr, const float *bias, int T, int d, int E,
                                 float *logits, void *workspace, int *status, uint64_t timeout_ns,
                                 cudaStream_t stream);

cudaError_t launch_route(const float *logits, int T, int E, int K, int32_t *topk_idx, float *topk_w,
                         int32_t *counts, int32_t *offsets, int32_t *row_of, int32_t *src_tok, int32_t *workspace,
                         cudaStream_t stream);

cudaError_t launch_permute(const uint16_t *x, const int32_t *row_of, int T, int K, int d, uint16_t *x_perm,
                           cudaStream_t stream);

cudaError_t launch_unpermute(const uint16_t *y_perm, const int32_t *row_of, const float *topk_w, int T, int K,
                             int d, uint16_t *y, cudaStream_t stream);

// MXFP8 (E4M3 codes, one power-of-two scale byte per 32 elements along K,
// scales stored as 512-byte atoms of 128 rows x one 128-wide K slice).
size_t mxfp8_scales_bytes(int rows, int K);
size_t mxfp8_perm_scales_bytes(int TK, int E, int K);
cudaError_t launch_mxfp8_quantize(const uint16_t *src, int rows, int K, uint8_t *codes, uint8_t *scales,
                                  cudaStream_t stream);
cudaError_t launch_permute_mxfp8(const uint16_t *x, const int32_t *topk_idx, const int32_t *row_of,
                                 const int32_t *offsets, int T, int K, int d, int E, uint8_t *xq, uint8_t *sfa,
                                 cudaStream_t stream);

// MXFP8 grouped GEMMs (single-CTA tiles; GEMM2 on CTA pairs where its groups
// are large and Kdim < 4096).  swiglu: GEMM1 (A = x codes [TK, d],
// W = W1 codes [E, 2f, d], out = h codes [TK, f], sfo = h scale atoms);
// else GEMM2 (A = h codes [TK, f], W = W2 codes [E, d, f], out = y_perm bf16).
cudaError_t grouped_gemm_mx_setup(struct GemmLaunch *cfg);
cudaError_t launch_grouped_gemm_mx(bool swiglu, const uint8_t *A, const uint8_t *sfa, size_t sfa_bytes, int TK,
                                   int Kdim, const uint8_t *W, const uint8_t *sfw, size_t sfw_bytes, int E, int n_out,
                                   const int32_t *offsets, void *out, uint8_t *sfo, size_t sfo_bytes,
                                   const struct GemmLaunch &cfg, int *status, uint64_t timeout_ns, cudaStream_t stream);

// Backward (backward.cu, wgrad.cu).
// dst[b] = src[b]^T (fp32)
cudaError_t launch_transpose_f32(const float *src, int B, int R, int C, float *dst, cudaStream_t s);
cudaError_t launch_combine_bwd(const uint16_t *dy, const uint16_t *y_perm, const int32_t *row_of, const float *topk_w,
                               int T, int K, int d, float *dw, uint16_t *dy_perm, cudaStream_t s);
cudaError_t launch_router_bwd(const float *topk_w, const float *dw, const int32_t *row_of, int T, int K, float *dl,
                              float *dl_row, cudaStream_t s);
cudaError_t launch_swiglu_bwd(const uint16_t *a, const uint16_t *dh, int TK, int f, uint16_t *da, cudaStream_t s);
// scratch `part` holds router_wgrad_slices(TK, E) * (d + 1) floats; two launches
size_t router_wgrad_slices(int TK, int E);
cudaError_t launch_router_wgrad(const uint16_t *x_perm, const float *dl_row, const int32_t *offsets, int E, int TK,
                                int d, float *part, float *dWr, float *dbias, cudaStream_t s);
cudaError_t launch_dx(const uint16_t *dx_perm, const float *WrT, const int32_t *row_of, const int32_t *topk_idx,
                      const float *dl, int T, int K, int E, int d, uint16_t *dx, cudaStream_t s);
cudaError_t wgrad_setup(struct GemmLaunch *cfg);
// D[e] [M, N] fp32 = A[group e]^T . B[group e] for rows grouped by expert, A [TK, M], B [TK, N];
// `maps` (128-byte aligned) is scratch for WGRAD_MAP_BYTES * E bytes of per-expert tensor maps.  Two launches.
constexpr size_t WGRAD_MAP_BYTES = 2 * 128;
cudaError_t launch_wgrad(const uint16_t *A, const uint16_t *B, int M, int N, const int32_t *offsets, int E, int TK,
                         float *D, void *maps, const struct GemmLaunch &lc, int *status, uint64_t timeout_ns,
                         cudaStream_t stream);

// Per-device launch shape of the grouped GEMM: SM count, and how many CTA
// pairs of the pair kernel can be resident at once (0: single-CTA only).
struct GemmLaunch {
    int num_sms = 0;
    int pairs_swiglu = 0;
    int pairs_plain = 0;
    int wgrad_pairs = 0;  // resident CTA pairs of the weight-gradient pair kernel
    int mx_pairs = 0;  // ... of the MXFP8 GEMM2 pair kernel
    int device = -1;
    int *sched_base = nullptr;  // device address of the dynamic tile order's counter table
};
// Kernel attributes and occupancy queries; once per device, before any capture.
cudaError_t grouped_gemm_setup(int num_sms, GemmLaunch *cfg);
// True when the CTA-pair kernel is used for this shape (decided on host
// sizes only, so the choice is the same for every routing).
bool grouped_gemm_use_pair(int TK, int E);
// True when the whole-layer forward fuses the permute into GEMM1 for this
// shape (host sizes only).
bool grouped_gemm1_prefers_gather(int TK, int E, int f);
// GEMM2 with the combine fused into its epilogue: y [T, n_out] bf16 from the
// rows it stores in `out` (then scratch); counters [T, ceil(n_out / 256)]
// int32 must be zero at launch.
struct CombineArgs {
    const int32_t *src_tok;
    const int32_t *row_of;
    const float *topk_w;
    int T, K;
    int *counters;
    void *y;
};
// GEMM1 with the permute fused into its operand load: A is the token matrix
// x [T, Kdim] and row r of the grouped operand is x[src_tok[r]].
struct GatherArgs {
    const int32_t *src_tok;  // [TK]
    int T;
};
// swiglu: GEMM1 (out [TK, n_out=f], W [E, 2f, Kdim=d]); else GEMM2 (out [TK, n_out=d], W [E, d, Kdim=f]).
// b_trans (plain only): W is [E, Kdim, n_out] and out = A . W[e] (no transpose in memory).
// preact (GEMM1 only, nullable): also store the bf16 pre-activations [TK, 2 n_out] (gate | up).
// gather (GEMM1 only, nullable): the fused permute (single-CTA kernel for every shape).
cudaError_t launch_grouped_gemm(bool swiglu, const void *A, int TK, int Kdim, const void *W, int E, int n_out,
                                const int32_t *offsets, void *out, const GemmLaunch &cfg, int *status,
                                uint64_t timeout_ns, cudaStream_t stream, const CombineArgs *comb = nullptr,
                                bool b_trans = false, void *preact = nullptr, const GatherArgs *gather = nullptr);

// A kernel whose only wait never completes: it times out after limit_ns and
// records MOE_ERR_DEVICE_TIMEOUT in *status.
cudaError_t launch_bounded_wait_probe(int *status, uint64_t limit_ns, cudaStream_t stream);

}  // namespace moe
