// Steps a3 and a6: permute (local dispatch) and weighted unpermute (local
// combine).  Both are HBM-bound row moves with 16-byte vectors.
//
// Figure 3 caption of "Accelerating dropless MoE training in JAX with NVIDIA
// Transformer Engine": dispatch moves each token to its experts, combine
// reverses the exchange and restores the original token order; "Optimization
// 2" notes that a naive dispatch/combine reads and writes the data many times.
//
// permute : x_perm[row_of[t,k], :] = x[t, :] -- each token row is read once
//           and written K times (scatter form: T*d reads, T*K*d writes).
// combine : y[t, :] = bf16( sum_k w[t,k] * y_perm[row_of[t,k], :] ), fp32
//           fused multiply-add in ascending k.
// One warp per token, lanes own 16-byte column vectors.  permute keeps UV
// vectors in flight per lane; combine loads all K rows of a round before
// accumulating them (for the common K), so K*UVK loads are in flight; for
// K = 8 the combine's unit is a (token, 256-column round) pair instead.
#include "kernels.h"

#include <cuda_bf16.h>

#include <algorithm>
#include <atomic>

namespace moe {
namespace pm {

constexpr int THREADS = 256;
constexpr int UV = 4;

__global__ void __launch_bounds__(THREADS)
permute_kernel(const uint4 *__restrict__ x, const int32_t *__restrict__ row_of, int T, int K, int nvec,
               uint4 *__restrict__ x_perm) {
    const int lane = threadIdx.x & 31;
    const int gw = (blockIdx.x * THREADS + threadIdx.x) >> 5;
    const int nw = (gridDim.x * THREADS) >> 5;
    for (int t = gw; t < T; t += nw) {
        const int my_row = lane < K ? row_of[static_cast<size_t>(t) * K + lane] : 0;
        const uint4 *src = x + static_cast<size_t>(t) * nvec;
        for (int v0 = 0; v0 < nvec; v0 += 32 * UV) {
            uint4 buf[UV];
#pragma unroll
            for (int u = 0; u < UV; ++u) {
                const int v = v0 + u * 32 + lane;
                if (v < nvec) buf[u] = __ldg(src + v);
            }
            for (int k = 0; k < K; ++k) {
                const int r = __shfl_sync(0xffffffffu, my_row, k);
                if (r < 0 || r >= T * K) continue;  // outside the contract: no write (warp-uniform)
                uint4 *dst = x_perm + static_cast<size_t>(r) * nvec;
#pragma unroll
                for (int u = 0; u < UV; ++u) {
                    const int v = v0 + u * 32 + lane;
                    if (v < nvec) dst[v] = buf[u];
                }
            }
        }
    }
}

__device__ __forceinline__ void fma_bf16x8(float (&acc)[8], float w, const uint4 &v) {
    const uint32_t p[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        acc[2 * i] = __fmaf_rn(w, __uint_as_float(p[i] << 16), acc[2 * i]);
        acc[2 * i + 1] = __fmaf_rn(w, __uint_as_float(p[i] & 0xffff0000u), acc[2 * i + 1]);
    }
}

__device__ __forceinline__ uint4 to_bf16x8(const float (&acc)[8]) {
    uint32_t p[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const __nv_bfloat162 b = __floats2bfloat162_rn(acc[2 * i], acc[2 * i + 1]);
        p[i] = *reinterpret_cast<const uint32_t *>(&b);
    }
    return make_uint4(p[0], p[1], p[2], p[3]);
}

// KT > 0: K is KT, and all K rows' vectors of a round are loaded before any
// is accumulated, so a lane keeps KT*UVK loads in flight.  KT == 0: any K.
template <int KT, int UVK>
__global__ void __launch_bounds__(THREADS)
unpermute_kernel(const uint4 *__restrict__ y_perm, const int32_t *__restrict__ row_of,
                 const float *__restrict__ topk_w, int T, int K, int nvec, uint4 *__restrict__ y) {
    const int lane = threadIdx.x & 31;
    const int gw = (blockIdx.x * THREADS + threadIdx.x) >> 5;
    const int nw = (gridDim.x * THREADS) >> 5;
    for (int t = gw; t < T; t += nw) {
        const int my_row = lane < K ? row_of[static_cast<size_t>(t) * K + lane] : 0;
        const float my_w = lane < K ? topk_w[static_cast<size_t>(t) * K + lane] : 0.0f;
        for (int v0 = 0; v0 < nvec; v0 += 32 * UVK) {
            float acc[UVK][8];
#pragma unroll
            for (int u = 0; u < UVK; ++u)
#pragma unroll
                for (int i = 0; i < 8; ++i) acc[u][i] = 0.0f;
            if (KT > 0) {
                uint4 buf[KT > 0 ? KT : 1][UVK];
#pragma unroll
                for (int k = 0; k < KT; ++k) {
                    const int r = __shfl_sync(0xffffffffu, my_row, k);
                    const bool row_ok = r >= 0 && r < T * K;  // outside the contract: read as zeros
                    const uint4 *src = y_perm + static_cast<size_t>(row_ok ? r : 0) * nvec;
#pragma unroll
                    for (int u = 0; u < UVK; ++u) {
                        const int v = v0 + u * 32 + lane;
                        buf[k][u] = (row_ok && v < nvec) ? __ldg(src + v) : make_uint4(0, 0, 0, 0);
                    }
                }
#pragma unroll
                for (int k = 0; k < KT; ++k) {
                    const float w = __shfl_sync(0xffffffffu, my_w, k);
#pragma unroll
                    for (int u = 0; u < UVK; ++u) fma_bf16x8(acc[u], w, buf[k][u]);
                }
            } else {
                for (int k = 0; k < K; ++k) {
                    const int r = __shfl_sync(0xffffffffu, my_row, k);
                    const float w = __shfl_sync(0xffffffffu, my_w, k);
                    const bool row_ok = r >= 0 && r < T * K;  // outside the contract: read as zeros
                    const uint4 *src = y_perm + static_cast<size_t>(row_ok ? r : 0) * nvec;
                    uint4 buf[UVK];
#pragma unroll
                    for (int u = 0; u < UVK; ++u) {
                        const int v = v0 + u * 32 + lane;
                        buf[u] = (row_ok && v < nvec) ? __ldg(src + v) : make_uint4(0, 0, 0, 0);
                    }
#pragma unroll
                    for (int u = 0; u < UVK; ++u) fma_bf16x8(acc[u], w, buf[u]);
                }
            }
            uint4 *dst = y + static_cast<size_t>(t) * nvec;
#pragma unroll
            for (int u = 0; u < UVK; ++u) {
                const int v = v0 + u * 32 + lane;
                if (v < nvec) dst[v] = to_bf16x8(acc[u]);
            }
        }
    }
}

// K = 8: one warp per (token, 256-column round) unit, warps taking units in
// grid-stride order (token-major, so neighbouring warps read neighbouring
// columns of the same rows).  A lane holds one vector of each of the K rows
// (60 registers, four blocks per SM, against 116 registers and two blocks
// for the per-token form with two vectors per lane), and the next
// unit's routing is loaded while the current unit's rows are in flight.
// The arithmetic per element is the per-token form's: fp32 FMAs in
// ascending k, so y is bit-identical.
template <int KT>
__global__ void __launch_bounds__(THREADS, 4)
unpermute_unit_kernel(const uint4 *__restrict__ y_perm, const int32_t *__restrict__ row_of,
                      const float *__restrict__ topk_w, int T, int nvec, uint4 *__restrict__ y) {
    const int lane = threadIdx.x & 31;
    const int gw = (blockIdx.x * THREADS + threadIdx.x) >> 5;
    const int nw = (gridDim.x * THREADS) >> 5;
    const int R = (nvec + 31) / 32;  // rounds per token
    const long long U = static_cast<long long>(T) * R;
    long long u = gw;
    if (u >= U) return;
    int t = static_cast<int>(u / R);
    int my_row = lane < KT ? row_of[static_cast<size_t>(t) * KT + lane] : 0;
    float my_w = lane < KT ? topk_w[static_cast<size_t>(t) * KT + lane] : 0.0f;
    while (true) {
        const int v = static_cast<int>(u % R) * 32 + lane;
        const long long un = u + nw;
        uint4 buf[KT];
#pragma unroll
        for (int k = 0; k < KT; ++k) {
            const int r = __shfl_sync(0xffffffffu, my_row, k);
            const bool row_ok = r >= 0 && r < T * KT;  // outside the contract: read as zeros
            buf[k] = (row_ok && v < nvec) ? __ldg(y_perm + static_cast<size_t>(r) * nvec + v) : make_uint4(0, 0, 0, 0);
        }
        int n_row = 0;
        float n_w = 0.0f;
        if (un < U && lane < KT) {
            const int tn = static_cast<int>(un / R);
            n_row = row_of[static_cast<size_t>(tn) * KT + lane];
            n_w = topk_w[static_cast<size_t>(tn) * KT + lane];
        }
        float acc[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) acc[i] = 0.0f;
#pragma unroll
        for (int k = 0; k < KT; ++k) fma_bf16x8(acc, __shfl_sync(0xffffffffu, my_w, k), buf[k]);
        if (v < nvec) y[static_cast<size_t>(t) * nvec + v] = to_bf16x8(acc);
        if (un >= U) break;
        u = un;
        t = static_cast<int>(u / R);
        my_row = n_row;
        my_w = n_w;
    }
}

int grid_for(int T) {
    const int warps_per_block = THREADS / 32;
    const int blocks = (T + warps_per_block - 1) / warps_per_block;
    return blocks < 1 ? 1 : blocks;
}

}  // namespace pm

cudaError_t launch_permute(const uint16_t *x, const int32_t *row_of, int T, int K, int d, uint16_t *x_perm,
                           cudaStream_t stream) {
    pm::permute_kernel<<<pm::grid_for(T), pm::THREADS, 0, stream>>>(
        reinterpret_cast<const uint4 *>(x), row_of, T, K, d / 8, reinterpret_cast<uint4 *>(x_perm));
    return cudaGetLastError();
}

cudaError_t launch_unpermute(const uint16_t *y_perm, const int32_t *row_of, const float *topk_w, int T, int K,
                             int d, uint16_t *y, cudaStream_t stream) {
    const uint4 *src = reinterpret_cast<const uint4 *>(y_perm);
    uint4 *dst = reinterpret_cast<uint4 *>(y);
    const int g = pm::grid_for(T), nvec = d / 8;
#define MOE_UNPERMUTE(KT, UVK) \
    pm::unpermute_kernel<KT, UVK><<<g, pm::THREADS, 0, stream>>>(src, row_of, topk_w, T, K, nvec, dst)
    switch (K) {
        case 1: MOE_UNPERMUTE(1, 4); break;
        case 2: MOE_UNPERMUTE(2, 4); break;
        case 4: MOE_UNPERMUTE(4, 2); break;
        case 6: MOE_UNPERMUTE(6, 2); break;
        case 8: {
            // one wave of the unit form (measured in a CUDA graph: the
            // DSv3-shaped combine 88.7 -> 79.7 us, the Qwen-shaped 99.6 -> 91.3
            // us; for K = 2 and 6 the per-token form stays faster)
            static std::atomic<int> resident[64];
            int wave = 0;
            const cudaError_t err = one_wave(pm::unpermute_unit_kernel<8>, pm::THREADS, resident, &wave);
            if (err != cudaSuccess) return err;
            const long long units = static_cast<long long>(T) * ((nvec + 31) / 32);
            const int blocks = static_cast<int>(std::max(1LL, std::min((units + 7) / 8, static_cast<long long>(wave))));
            pm::unpermute_unit_kernel<8><<<blocks, pm::THREADS, 0, stream>>>(src, row_of, topk_w, T, nvec, dst);
            break;
        }
        default: MOE_UNPERMUTE(0, 4); break;
    }
#undef MOE_UNPERMUTE
    return cudaGetLastError();
}

}  // namespace moe
