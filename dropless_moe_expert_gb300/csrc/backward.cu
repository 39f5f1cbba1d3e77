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
            for (int v = lane; v < nvec; v += 32) {
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

// dWr[:, e] and dbias[e]: sums over expert e's rows.  One block per (expert,
// 256-column chunk): lane l of warp w owns 8 columns and the rows
// w, w + 8, w + 16, ... of the group; the 8 warps' partial sums are then
// added in warp order.  The order of every addition is fixed: deterministic.
__global__ void __launch_bounds__(256)
router_wgrad_kernel(const uint4 *__restrict__ x_perm, const float *__restrict__ dl_row,
                    const int32_t *__restrict__ offsets, int E, int TK, int d, float *__restrict__ dWr,
                    float *__restrict__ dbias) {
    __shared__ float part[8][256 + 1];
    __shared__ float bpart[8];
    const int e = blockIdx.y;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int nvec = d / 8;
    const int v = blockIdx.x * 32 + lane;  // 8-column vector index
    const int o0 = min(max(offsets[e], 0), TK);
    const int o1 = min(max(offsets[e + 1], o0), TK);
    float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    float bsum = 0.0f;
    for (int r = o0 + warp; r < o1; r += 8) {
        const float g = dl_row[r];
        bsum += g;
        if (v < nvec) {
            float xv[8];
            unpack8(__ldg(x_perm + static_cast<size_t>(r) * nvec + v), xv);
#pragma unroll
            for (int i = 0; i < 8; ++i) acc[i] = __fmaf_rn(g, xv[i], acc[i]);
        }
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) part[warp][lane * 8 + i] = acc[i];
    if (lane == 0) bpart[warp] = bsum;
    __syncthreads();
    // warp 0 adds the 8 partial sums in warp order and writes
    if (warp == 0) {
        if (v < nvec) {
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                float t = 0.0f;
                for (int w = 0; w < 8; ++w) t += part[w][lane * 8 + i];
                dWr[static_cast<size_t>(v * 8 + i) * E + e] = t;
            }
        }
        if (blockIdx.x == 0 && lane == 0) {
            float t = 0.0f;
            for (int w = 0; w < 8; ++w) t += bpart[w];
            dbias[e] = t;
        }
    }
}

// dx[t] = sum_k dx_perm[row_of[t,k]] + sum_k dl[t,k] Wr^T[idx[t,k]]; one warp
// per token, fp32 in ascending k, then bf16.
__global__ void __launch_bounds__(256)
dx_kernel(const uint4 *__restrict__ dx_perm, const float *__restrict__ WrT, const int32_t *__restrict__ row_of,
          const int32_t *__restrict__ topk_idx, const float *__restrict__ dl, int T, int K, int E, int TK, int nvec,
          uint4 *__restrict__ dx) {
    const int lane = threadIdx.x & 31;
    const int gw = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int nw = (gridDim.x * blockDim.x) >> 5;
    for (int t = gw; t < T; t += nw) {
        for (int v = lane; v < nvec; v += 32) {
            float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
            for (int k = 0; k < K; ++k) {
                const int r = row_of[static_cast<size_t>(t) * K + k];
                if (r < 0 || r >= TK) continue;
                float xv[8];
                unpack8(__ldg(dx_perm + static_cast<size_t>(r) * nvec + v), xv);
#pragma unroll
                for (int i = 0; i < 8; ++i) acc[i] += xv[i];
            }
            for (int k = 0; k < K; ++k) {
                const int e = topk_idx[static_cast<size_t>(t) * K + k];
                if (e < 0 || e >= E) continue;
                const float g = dl[static_cast<size_t>(t) * K + k];
                const float4 *wr = reinterpret_cast<const float4 *>(WrT + static_cast<size_t>(e) * nvec * 8) + 2 * v;
                const float4 w0 = __ldg(wr), w1 = __ldg(wr + 1);
                const float wv[8] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w};
#pragma unroll
                for (int i = 0; i < 8; ++i) acc[i] = __fmaf_rn(g, wv[i], acc[i]);
            }
            dx[static_cast<size_t>(t) * nvec + v] = pack8(acc);
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

cudaError_t launch_router_wgrad(const uint16_t *x_perm, const float *dl_row, const int32_t *offsets, int E, int TK,
                                int d, float *dWr, float *dbias, cudaStream_t s) {
    dim3 grid((d / 8 + 31) / 32, E);
    bw::router_wgrad_kernel<<<grid, 256, 0, s>>>(reinterpret_cast<const uint4 *>(x_perm), dl_row, offsets, E, TK, d,
                                                dWr, dbias);
    return cudaGetLastError();
}

cudaError_t launch_dx(const uint16_t *dx_perm, const float *WrT, const int32_t *row_of, const int32_t *topk_idx,
                      const float *dl, int T, int K, int E, int d, uint16_t *dx, cudaStream_t s) {
    bw::dx_kernel<<<bw::warps_grid(T), 256, 0, s>>>(reinterpret_cast<const uint4 *>(dx_perm), WrT, row_of, topk_idx,
                                                   dl, T, K, E, T * K, d / 8, reinterpret_cast<uint4 *>(dx));
    return cudaGetLastError();
}

}  // namespace moe
