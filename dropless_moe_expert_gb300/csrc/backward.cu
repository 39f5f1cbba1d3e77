// Backward of the dropless MoE layer: the small kernels around the grouped
// GEMMs (the dgrad GEMMs reuse the forward's grouped GEMM, the weight
// gradients are wgrad.cu).
//
// "Accelerating dropless MoE training in JAX with NVIDIA Transformer Engine"
// is about training; the gradients are those of the forward's definition for
// an output gradient dy (the top-K choice is piecewise constant, the gate
// weights a softmax over the K selected logits):
//   combine:   dw[t,k] = <dy[t], y_perm[r]>,  dy_perm[r] = w[t,k] dy[t]   (r = row_of[t,k])
//   router:    dl[t,k] = w[t,k] (dw[t,k] - sum_j w[t,j] dw[t,j]),
//              dbias[e] = sum of dl over e's rows, dWr[:, e] = sum of dl x over e's rows
//   SwiGLU:    dg = dh u (s + g s (1 - s)), du = dh g s,  s = sigmoid(g)
//   permute:   dx[t] = sum_k dx_perm[row_of[t,k]] + sum_k dl[t,k] Wr[:, idx[t,k]]
// Every sum runs in a fixed order (warp shuffles of a fixed shape, rows in
// group order, k ascending): the gradients are deterministic.
#include "kernels.h"

#include <cuda_bf16.h>

#include <algorithm>

namespace moe {
namespace bw {

__device__ __forceinline__ void unpack8(const uint4 &u, float *o) {
    const uint32_t p[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        o[2 * i] = __uint_as_float(p[i] << 16);
        o[2 * i + 1] = __uint_as_float(p[i] & 0xffff0000u);
    }
}

__device__ __forceinline__ uint4 pack8(const float *v) {
    uint32_t p[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const __nv_bfloat162 b = __floats2bfloat162_rn(v[2 * i], v[2 * i + 1]);
        p[i] = *reinterpret_cast<const uint32_t *>(&b);
    }
    return make_uint4(p[0], p[1], p[2], p[3]);
}

// dst[b][c][r] = src[b][r][c]: 32 x 32 tiles through shared memory.
template <typename T>
__global__ void __launch_bounds__(256)
transpose_kernel(const T *__restrict__ src, int B, int R, int C, T *__restrict__ dst) {
    __shared__ T tile[32][33];
    const int b = blockIdx.z;
    const int r0 = blockIdx.y * 32, c0 = blockIdx.x * 32;
    const int tx = threadIdx.x & 31, ty = threadIdx.x >> 5;
    const T *s = src + static_cast<size_t>(b) * R * C;
    T *d = dst + static_cast<size_t>(b) * R * C;
    for (int i = ty; i < 32; i += 8) {
        const int r = r0 + i, c = c0 + tx;
        if (r < R && c < C) tile[i][tx] = s[static_cast<size_t>(r) * C + c];
    }
    __syncthreads();
    for (int i = ty; i < 32; i += 8) {
        const int c = c0 + i, r = r0 + tx;
        if (r < R && c < C) d[static_cast<size_t>(c) * R + r] = tile[tx][i];
    }
}

// Combine backward: one warp per token.  Lanes hold 8 columns of a 256-wide
// chunk; the dot products reduce by a fixed shuffle tree.
__global__ void __launch_bounds__(256)
combine_bwd_kernel(const uint4 *__restrict__ dy, const uint4 *__restrict__ y_perm, const int32_t *__restrict__ row_of,
                   const float *__restrict__ topk_w, int T, int K, int nvec, float *__restrict__ dw,
                   uint4 *__restrict__ dy_perm) {
    const int lane = threadIdx.x & 31;
    const int gw = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int nw = (gridDim.x * blockDim.x) >> 5;
    for (int t = gw; t < T; t += nw) {
        for (int k = 0; k < K; ++k) {
            const int r = row_of[static_cast<size_t>(t) * K + k];
            const float w = topk_w[static_cast<size_t>(t) * K + k];
            float dot = 0.0f;
            const bool row_ok = r >= 0 && r < T * K;  // outside the contract: no access, dw = 0
            for (int v = lane; row_ok && v < nvec; v += 32) {
                float a[8], b[8];
                unpack8(__ldg(dy + static_cast<size_t>(t) * nvec + v), a);
                unpack8(__ldg(y_perm + static_cast<size_t>(r) * nvec + v), b);
                float o[8];
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    dot = __fmaf_rn(a[i], b[i], dot);
                    o[i] = w * a[i];
                }
                dy_perm[static_cast<size_t>(r) * nvec + v] = pack8(o);
            }
#pragma unroll
            for (int s = 16; s >= 1; s >>= 1) dot += __shfl_xor_sync(0xffffffffu, dot, s);
            if (lane == 0) dw[static_cast<size_t>(t) * K + k] = dot;
        }
    }
}

// Softmax backward over the K selected logits: dl per (t, k) and per row.
__global__ void router_bwd_kernel(const float *__restrict__ topk_w, const float *__restrict__ dw,
                                  const int32_t *__restrict__ row_of, int T, int K, float *__restrict__ dl,
                                  float *__restrict__ dl_row, int TK) {
    const int t = blockIdx.x * blockDim.x + threadIdx.x;
    if (t >= T) return;
    float s = 0.0f;
    for (int k = 0; k < K; ++k) s = __fmaf_rn(topk_w[static_cast<size_t>(t) * K + k], dw[static_cast<size_t>(t) * K + k], s);
    for (int k = 0; k < K; ++k) {
        const size_t i = static_cast<size_t>(t) * K + k;
        const float v = topk_w[i] * (dw[i] - s);
        dl[i] = v;
        const int r = row_of[i];
        if (r >= 0 && r < TK) dl_row[r] = v;
    }
}

// SwiGLU backward, 8 elements per thread: a = [g | u] [TK, 2f], dh [TK, f]
// -> da = [dg | du] [TK, 2f].
__global__ void __launch_bounds__(256)
swiglu_bwd_kernel(const uint4 *__restrict__ a, const uint4 *__restrict__ dh, int TK, int f, uint4 *__restrict__ da) {
    const int fv = f / 8;
    const size_t n = static_cast<size_t>(TK) * fv;
    for (size_t p = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x; p < n;
         p += static_cast<size_t>(gridDim.x) * blockDim.x) {
        const size_t r = p / fv, c = p % fv;
        float g[8], u[8], d[8], dg[8], du[8];
        unpack8(a[r * 2 * fv + c], g);
        unpack8(a[r * 2 * fv + fv + c], u);
        unpack8(dh[r * fv + c], d);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const float s = 1.0f / (1.0f + __expf(-g[i]));
            dg[i] = d[i] * u[i] * (s + g[i] * s * (1.0f - s));
            du[i] = d[i] * g[i] * s;
        }
        da[r * 2 * fv + c] = pack8(dg);
        da[r * 2 * fv + fv + c] = pack8(du);
    }
}

// dWr[:, e] and dbias[e]: sums over expert e's rows, in two passes so that
// a heavy expert's rows spread over many blocks.  Each expert's rows are cut
// into slices of RW_SLICE rows (slice w of all experts in order: the prefix
// s_pre over experts of ceil(count / RW_SLICE)); pass 1 sums one slice per
// block into part[w], pass 2 adds an expert's slices in slice order.  Every
// addition has a fixed order: deterministic.
constexpr int RW_SLICE = 256;
constexpr int RW_MAX_E = 256;

// Group starts, counts (clamped to [0, TK]) and the slice prefix; one warp.
__device__ __forceinline__ void slice_prefix(const int32_t *offsets, int E, int TK, int lane, int *s_off, int *s_cnt,
                                             int *s_pre) {
    int carry = 0;
    for (int base = 0; base < E; base += 32) {
        const int e = base + lane;
        int v = 0;
        if (e < E) {
            const int o0 = min(max(offsets[e], 0), TK);
            const int o1 = min(max(offsets[e + 1], o0), TK);
            s_off[e] = o0;
            s_cnt[e] = o1 - o0;
            v = (o1 - o0 + RW_SLICE - 1) / RW_SLICE;
        }
        int incl = v;
#pragma unroll
        for (int sh = 1; sh < 32; sh <<= 1) {
            const int n = __shfl_up_sync(0xffffffffu, incl, sh);
            if (lane >= sh) incl += n;
        }
        if (e < E) s_pre[e] = carry + incl - v;
        carry += __shfl_sync(0xffffffffu, incl, 31);
    }
    if (lane == 0) s_pre[E] = carry;
}

// Pass 1: block (column chunk of 256, slice w).  Lane l of warp q owns 8
// columns and the slice's rows q, q + 8, q + 16, ... (four loads in flight);
// the 8 warps' sums are added in warp order into part[w][cols]; the chunk-0
// block also writes the slice's sum of dl into bpart[w].
__global__ void __launch_bounds__(256)
router_wgrad_partial_kernel(const uint4 *__restrict__ x_perm, const float *__restrict__ dl_row,
                            const int32_t *__restrict__ offsets, int E, int TK, int d, float *__restrict__ part,
                            float *__restrict__ bpart) {
    __shared__ int s_off[RW_MAX_E], s_cnt[RW_MAX_E], s_pre[RW_MAX_E + 1];
    __shared__ float red[8][256 + 1];
    __shared__ float bred[8];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (warp == 0) slice_prefix(offsets, E, TK, lane, s_off, s_cnt, s_pre);
    __syncthreads();
    const int w = blockIdx.y;
    if (w >= s_pre[E]) return;  // block-uniform
    int lo = 0, hi = E - 1;     // the expert whose slices hold w
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (s_pre[mid] <= w) lo = mid; else hi = mid - 1;
    }
    const int e = lo;
    const int r0 = s_off[e] + (w - s_pre[e]) * RW_SLICE;
    const int r1 = min(r0 + RW_SLICE, s_off[e] + s_cnt[e]);
    const int nvec = d / 8;
    const int v = blockIdx.x * 32 + lane;  // 8-column vector index
    const bool col_ok = v < nvec;
    float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    float bsum = 0.0f;
    for (int r = r0 + warp; r < r1; r += 32) {
        uint4 xr[4];
        float g[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int rr = r + 8 * j;
            const bool ok = rr < r1;
            g[j] = ok ? dl_row[rr] : 0.0f;
            xr[j] = (ok && col_ok) ? __ldg(x_perm + static_cast<size_t>(rr) * nvec + v) : make_uint4(0u, 0u, 0u, 0u);
        }
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            if (r + 8 * j >= r1) break;
            bsum += g[j];
            float xv[8];
            unpack8(xr[j], xv);
#pragma unroll
            for (int i = 0; i < 8; ++i) acc[i] = __fmaf_rn(g[j], xv[i], acc[i]);
        }
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) red[warp][lane * 8 + i] = acc[i];
    if (lane == 0) bred[warp] = bsum;
    __syncthreads();
    if (warp == 0) {
        if (col_ok) {
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                float t = 0.0f;
                for (int q = 0; q < 8; ++q) t += red[q][lane * 8 + i];
                part[static_cast<size_t>(w) * d + v * 8 + i] = t;
            }
        }
        if (blockIdx.x == 0 && lane == 0) {
            float t = 0.0f;
            for (int q = 0; q < 8; ++q) t += bred[q];
            bpart[w] = t;
        }
    }
}

// Pass 2: block (column chunk of 256, expert e): dWr[col, e] = the expert's
// slices' partial sums added in slice order (0 for an expert without rows).
__global__ void __launch_bounds__(256)
router_wgrad_reduce_kernel(const float *__restrict__ part, const float *__restrict__ bpart,
                           const int32_t *__restrict__ offsets, int E, int TK, int d, int W, float *__restrict__ dWr,
                           float *__restrict__ dbias) {
    __shared__ int s_off[RW_MAX_E], s_cnt[RW_MAX_E], s_pre[RW_MAX_E + 1];
    if (threadIdx.x < 32) slice_prefix(offsets, E, TK, threadIdx.x, s_off, s_cnt, s_pre);
    __syncthreads();
    const int e = blockIdx.y;
    // (clamped to the W slices pass 1 had: offsets that are not monotone
    // cannot send a read past `part`)
    const int w0 = min(s_pre[e], W), w1 = min(s_pre[e + 1], W);
    const int col = blockIdx.x * 256 + threadIdx.x;
    if (col < d) {
        float t = 0.0f;
        for (int w = w0; w < w1; ++w) t += part[static_cast<size_t>(w) * d + col];
        dWr[static_cast<size_t>(col) * E + e] = t;
    }
    if (blockIdx.x == 0 && threadIdx.x == 0) {
        float t = 0.0f;
        for (int w = w0; w < w1; ++w) t += bpart[w];
        dbias[e] = t;
    }
}

// dx[t] = sum_k dx_perm[row_of[t,k]] + sum_k dl[t,k] Wr^T[idx[t,k]]; one warp
// per token, fp32 in ascending k, then bf16.  Lane k holds the token's k-th
// row, expert and dl (K <= 32), handed to every lane by shuffles.  KT > 0: K
// is KT and the K rows' vectors are all loaded before they are summed (KT
// loads in flight per lane); KT == 0: any K.
template <int KT>
__global__ void __launch_bounds__(256)
dx_kernel(const uint4 *__restrict__ dx_perm, const float *__restrict__ WrT, const int32_t *__restrict__ row_of,
          const int32_t *__restrict__ topk_idx, const float *__restrict__ dl, int T, int K, int E, int TK, int nvec,
          uint4 *__restrict__ dx) {
    const int lane = threadIdx.x & 31;
    const int gw = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int nw = (gridDim.x * blockDim.x) >> 5;
    const int k_n = KT > 0 ? KT : K;
    for (int t = gw; t < T; t += nw) {
        int my_r = -1, my_e = -1;
        float my_g = 0.0f;
        if (lane < k_n) {
            my_r = row_of[static_cast<size_t>(t) * k_n + lane];
            my_e = topk_idx[static_cast<size_t>(t) * k_n + lane];
            my_g = dl[static_cast<size_t>(t) * k_n + lane];
        }
        // the loop is warp-uniform (the shuffles need every lane); lanes past
        // the row's end load and store nothing
        for (int v0 = 0; v0 < nvec; v0 += 32) {
            const int v = v0 + lane;
            const bool col_ok = v < nvec;
            float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
            if (KT > 0) {
                uint4 buf[KT > 0 ? KT : 1];
#pragma unroll
                for (int k = 0; k < KT; ++k) {
                    const int r = __shfl_sync(0xffffffffu, my_r, k);
                    const bool ok = col_ok && r >= 0 && r < TK;
                    buf[k] = ok ? __ldg(dx_perm + static_cast<size_t>(r) * nvec + v) : make_uint4(0u, 0u, 0u, 0u);
                }
#pragma unroll
                for (int k = 0; k < KT; ++k) {
                    float xv[8];
                    unpack8(buf[k], xv);
#pragma unroll
                    for (int i = 0; i < 8; ++i) acc[i] += xv[i];
                }
            } else {
                for (int k = 0; k < k_n; ++k) {
                    const int r = __shfl_sync(0xffffffffu, my_r, k);
                    if (r < 0 || r >= TK || !col_ok) continue;
                    float xv[8];
                    unpack8(__ldg(dx_perm + static_cast<size_t>(r) * nvec + v), xv);
#pragma unroll
                    for (int i = 0; i < 8; ++i) acc[i] += xv[i];
                }
            }
            for (int k = 0; k < k_n; ++k) {
                const int e = __shfl_sync(0xffffffffu, my_e, k);
                const float g = __shfl_sync(0xffffffffu, my_g, k);
                if (e < 0 || e >= E || !col_ok) continue;
                const float4 *wr = reinterpret_cast<const float4 *>(WrT + static_cast<size_t>(e) * nvec * 8) + 2 * v;
                const float4 w0 = __ldg(wr), w1 = __ldg(wr + 1);
                const float wv[8] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w};
#pragma unroll
                for (int i = 0; i < 8; ++i) acc[i] = __fmaf_rn(g, wv[i], acc[i]);
            }
            if (col_ok) dx[static_cast<size_t>(t) * nvec + v] = pack8(acc);
        }
    }
}

int warps_grid(int n) { return std::max(1, std::min((n + 7) / 8, 152 * 8)); }

}  // namespace bw

cudaError_t launch_transpose_f32(const float *src, int B, int R, int C, float *dst, cudaStream_t s) {
    dim3 grid((C + 31) / 32, (R + 31) / 32, B);
    bw::transpose_kernel<float><<<grid, 256, 0, s>>>(src, B, R, C, dst);
    return cudaGetLastError();
}

cudaError_t launch_combine_bwd(const uint16_t *dy, const uint16_t *y_perm, const int32_t *row_of, const float *topk_w,
                               int T, int K, int d, float *dw, uint16_t *dy_perm, cudaStream_t s) {
    bw::combine_bwd_kernel<<<bw::warps_grid(T), 256, 0, s>>>(
        reinterpret_cast<const uint4 *>(dy), reinterpret_cast<const uint4 *>(y_perm), row_of, topk_w, T, K, d / 8, dw,
        reinterpret_cast<uint4 *>(dy_perm));
    return cudaGetLastError();
}

cudaError_t launch_router_bwd(const float *topk_w, const float *dw, const int32_t *row_of, int T, int K, float *dl,
                              float *dl_row, cudaStream_t s) {
    bw::router_bwd_kernel<<<(T + 255) / 256, 256, 0, s>>>(topk_w, dw, row_of, T, K, dl, dl_row, T * K);
    return cudaGetLastError();
}

cudaError_t launch_swiglu_bwd(const uint16_t *a, const uint16_t *dh, int TK, int f, uint16_t *da, cudaStream_t s) {
    const size_t n = static_cast<size_t>(TK) * (f / 8);
    const int blocks = static_cast<int>(std::min<size_t>((n + 255) / 256, 152 * 16));
    bw::swiglu_bwd_kernel<<<std::max(blocks, 1), 256, 0, s>>>(reinterpret_cast<const uint4 *>(a),
                                                              reinterpret_cast<const uint4 *>(dh), TK, f,
                                                              reinterpret_cast<uint4 *>(da));
    return cudaGetLastError();
}

size_t router_wgrad_slices(int TK, int E) {
    return (static_cast<size_t>(TK) + bw::RW_SLICE - 1) / bw::RW_SLICE + static_cast<size_t>(E);
}

cudaError_t launch_router_wgrad(const uint16_t *x_perm, const float *dl_row, const int32_t *offsets, int E, int TK,
                                int d, float *part, float *dWr, float *dbias, cudaStream_t s) {
    if (E > bw::RW_MAX_E) return cudaErrorInvalidValue;
    const int chunks = (d / 8 + 31) / 32;
    const size_t Ws = router_wgrad_slices(TK, E);  // at least the slices of all experts
    if (Ws > 65535) return cudaErrorInvalidValue;   // grid.y
    const int W = static_cast<int>(Ws);
    float *bpart = part + static_cast<size_t>(W) * d;
    bw::router_wgrad_partial_kernel<<<dim3(chunks, W), 256, 0, s>>>(reinterpret_cast<const uint4 *>(x_perm), dl_row,
                                                                   offsets, E, TK, d, part, bpart);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    bw::router_wgrad_reduce_kernel<<<dim3((d + 255) / 256, E), 256, 0, s>>>(part, bpart, offsets, E, TK, d, W, dWr,
                                                                           dbias);
    return cudaGetLastError();
}

cudaError_t launch_dx(const uint16_t *dx_perm, const float *WrT, const int32_t *row_of, const int32_t *topk_idx,
                      const float *dl, int T, int K, int E, int d, uint16_t *dx, cudaStream_t s) {
    const auto *src = reinterpret_cast<const uint4 *>(dx_perm);
    auto *dst = reinterpret_cast<uint4 *>(dx);
    const int g = bw::warps_grid(T), TK = T * K, nv = d / 8;
    switch (K) {
        case 1: bw::dx_kernel<1><<<g, 256, 0, s>>>(src, WrT, row_of, topk_idx, dl, T, K, E, TK, nv, dst); break;
        case 2: bw::dx_kernel<2><<<g, 256, 0, s>>>(src, WrT, row_of, topk_idx, dl, T, K, E, TK, nv, dst); break;
        case 4: bw::dx_kernel<4><<<g, 256, 0, s>>>(src, WrT, row_of, topk_idx, dl, T, K, E, TK, nv, dst); break;
        case 6: bw::dx_kernel<6><<<g, 256, 0, s>>>(src, WrT, row_of, topk_idx, dl, T, K, E, TK, nv, dst); break;
        case 8: bw::dx_kernel<8><<<g, 256, 0, s>>>(src, WrT, row_of, topk_idx, dl, T, K, E, TK, nv, dst); break;
        default: bw::dx_kernel<0><<<g, 256, 0, s>>>(src, WrT, row_of, topk_idx, dl, T, K, E, TK, nv, dst); break;
    }
    return cudaGetLastError();
}

}  // namespace moe
