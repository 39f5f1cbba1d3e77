// Steps a1 + a2: top-K softmax routing, expert histogram, offsets and the
// stable dispatch order, all on the device.
//
// "Accelerating dropless MoE training in JAX with NVIDIA Transformer Engine":
// the router activates the Top-K experts of each token (introduction); the
// per-expert counts are data dependent and must not be copied to the host,
// which would stall the critical path and break CUDA graphs ("What specialized
// optimizations are needed for dropless MoE?", "Optimization 1: Grouped GEMM").
//
// Three kernels, no atomics whose order could show in a result:
//  1. route_topk: a group of G lanes per token (G = 8, 16 or 32; 32/G tokens
//     per warp); each lane holds E/G logits as 64-bit keys (order-preserving
//     float bits << 32 | ~expert), K rounds of group max via shuffles pick the
//     experts (descending, lower index on ties, -0.0 == +0.0); softmax over
//     the K picks.  The CTA then marks, per
//     expert, which of its 256 tokens chose it in a shared bitmap (atomicOr:
//     the final bitmap does not depend on order), and from it writes the
//     chunk's per-expert count and every pair's rank inside the chunk.
//  2. route_scan: one CTA; counts = sum over chunks, offsets = exclusive
//     scan over experts, chunk_base[c][e] = offsets[e] + rows of expert e in
//     earlier chunks.
//  3. route_scatter: row_of[t,k] = chunk_base[chunk(t)][e] + rank;
//     src_tok[row] = t.  Rows of a group are thus in ascending token order.
#include "kernels.h"

#include <math.h>

#include <algorithm>

namespace moe {
namespace rt {

constexpr int CH = kRouteChunk;  // tokens per CTA
constexpr int THREADS = 1024;    // 32 warps: each ranks 8 of the chunk's tokens
constexpr int WARPS = THREADS / 32;
constexpr int MAX_E = 256;
constexpr int MAX_K = 16;

__device__ __forceinline__ uint32_t order_key(float v) {
    if (v == 0.0f) v = 0.0f;  // -0.0 and +0.0 compare equal: give them one key
    const uint32_t u = __float_as_uint(v);
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ float key_value(uint32_t k) {
    const uint32_t u = (k & 0x80000000u) ? (k & 0x7fffffffu) : ~k;
    return __uint_as_float(u);
}

// G lanes per token (a power of two, G >= E / EPL), EPL logits per lane, so
// that few experts do not leave most of a warp idle: 32/G tokens per warp.
template <int G, int EPL>
__global__ void __launch_bounds__(THREADS)
route_topk_kernel(const float *__restrict__ L, int T, int E, int K, int32_t *__restrict__ topk_idx,
                  float *__restrict__ topk_w, int32_t *__restrict__ row_rank, int32_t *__restrict__ chunk_counts) {
    constexpr int TPW = 32 / G;  // tokens per warp at a time
    __shared__ uint32_t bits[MAX_E][CH / 32];
    __shared__ int32_t s_idx[CH * MAX_K];
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int glane = lane % G;                 // lane inside the token's group
    const int group = lane / G;
    const unsigned gmask = (G == 32) ? 0xffffffffu : (((1u << G) - 1u) << (group * G));
    const int t0 = blockIdx.x * CH;
    const int nt = min(CH, T - t0);

    for (int i = threadIdx.x; i < E * (CH / 32); i += THREADS) (&bits[0][0])[i] = 0u;
    __syncthreads();

    // the logits of the group's next token are loaded while the current one is
    // ranked, so a warp does not pay one global-load latency per token
    float nxt[EPL];
    auto load_logits = [&](int tl) {
        const float *row = L + static_cast<size_t>(t0 + tl) * E;
#pragma unroll
        for (int j = 0; j < EPL; ++j) {
            const int e = glane + G * j;
            nxt[j] = (tl < nt && e < E) ? row[e] : 0.0f;
        }
    };
    load_logits(warp * TPW + group);
    for (int tl = warp * TPW + group; tl < nt; tl += WARPS * TPW) {
        const int t = t0 + tl;
        unsigned long long key[EPL];
#pragma unroll
        for (int j = 0; j < EPL; ++j) {
            const int e = glane + G * j;
            key[j] = (e < E) ? ((static_cast<unsigned long long>(order_key(nxt[j])) << 32) |
                                static_cast<unsigned long long>(0xffffffffu - static_cast<uint32_t>(e)))
                             : 0ull;  // below every real key
        }
        load_logits(tl + WARPS * TPW);
        int my_e = 0;
        float my_z = 0.0f;
        float v0 = 0.0f, sum = 0.0f;
        for (int k = 0; k < K; ++k) {
            unsigned long long best = key[0];
#pragma unroll
            for (int j = 1; j < EPL; ++j) best = key[j] > best ? key[j] : best;
#pragma unroll
            for (int s = G / 2; s >= 1; s >>= 1) {
                const unsigned long long o = __shfl_xor_sync(gmask, best, s, G);
                best = o > best ? o : best;
            }
            const int e = static_cast<int>(0xffffffffu - static_cast<uint32_t>(best & 0xffffffffull));
            const float v = key_value(static_cast<uint32_t>(best >> 32));
            const bool mine = (e % G) == glane;
#pragma unroll
            for (int j = 0; j < EPL; ++j) key[j] = (mine && j == e / G) ? 0ull : key[j];
            if (k == 0) v0 = v;
            const float z = expf(v - v0);
            sum += z;
            if (glane == k) { my_e = e; my_z = z; }
        }
        if (glane < K) {
            topk_idx[static_cast<size_t>(t) * K + glane] = my_e;
            topk_w[static_cast<size_t>(t) * K + glane] = my_z / sum;
            s_idx[tl * K + glane] = my_e;
            atomicOr(&bits[my_e][tl >> 5], 1u << (tl & 31));
        }
    }
    __syncthreads();

    // per-expert count of this chunk
    for (int e = threadIdx.x; e < E; e += THREADS) {
        int c = 0;
#pragma unroll
        for (int w = 0; w < CH / 32; ++w) c += __popc(bits[e][w]);
        chunk_counts[static_cast<size_t>(blockIdx.x) * E + e] = c;
    }
    // rank of each (t, k) among the chunk's tokens that chose the same expert
    for (int p = threadIdx.x; p < nt * K; p += THREADS) {
        const int tl = p / K;
        const int e = s_idx[p];
        int r = __popc(bits[e][tl >> 5] & ((1u << (tl & 31)) - 1u));
        for (int w = 0; w < (tl >> 5); ++w) r += __popc(bits[e][w]);
        row_rank[static_cast<size_t>(t0) * K + p] = r;
    }
}

__global__ void __launch_bounds__(MAX_E)
route_scan_kernel(const int32_t *__restrict__ chunk_counts, int C, int E, int32_t *__restrict__ counts,
                  int32_t *__restrict__ offsets, int32_t *__restrict__ chunk_base) {
    __shared__ int32_t warp_tot[MAX_E / 32];
    const int e = threadIdx.x;
    const int lane = e & 31, warp = e >> 5;
    int cnt = 0;
    if (e < E) {
#pragma unroll 8
        for (int c = 0; c < C; ++c) cnt += chunk_counts[static_cast<size_t>(c) * E + e];
    }
    // exclusive scan of cnt over experts
    int v = cnt;
#pragma unroll
    for (int s = 1; s < 32; s <<= 1) {
        const int n = __shfl_up_sync(0xffffffffu, v, s);
        if (lane >= s) v += n;
    }
    if (lane == 31) warp_tot[warp] = v;
    __syncthreads();
    int before = 0;
    for (int w = 0; w < warp; ++w) before += warp_tot[w];
    const int excl = before + v - cnt;
    if (e < E) {
        counts[e] = cnt;
        offsets[e] = excl;
        if (e == E - 1) offsets[E] = excl + cnt;
        int run = excl;
#pragma unroll 8
        for (int c = 0; c < C; ++c) {
            chunk_base[static_cast<size_t>(c) * E + e] = run;
            run += chunk_counts[static_cast<size_t>(c) * E + e];
        }
    }
}

__global__ void route_scatter_kernel(const int32_t *__restrict__ topk_idx, const int32_t *__restrict__ chunk_base,
                                     int T, int E, int K, int32_t *__restrict__ row_of,
                                     int32_t *__restrict__ src_tok) {
    const size_t TK = static_cast<size_t>(T) * K;
    for (size_t p = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x; p < TK;
         p += static_cast<size_t>(gridDim.x) * blockDim.x) {
        const int t = static_cast<int>(p / K);
        const int e = topk_idx[p];
        const int r = chunk_base[static_cast<size_t>(t / CH) * E + e] + row_of[p];
        row_of[p] = r;
        src_tok[r] = t;
    }
}

}  // namespace rt

cudaError_t launch_route(const float *logits, int T, int E, int K, int32_t *topk_idx, float *topk_w,
                         int32_t *counts, int32_t *offsets, int32_t *row_of, int32_t *src_tok, int32_t *workspace,
                         cudaStream_t stream) {
    const int C = route_num_chunks(T);
    int32_t *chunk_counts = workspace;
    int32_t *chunk_base = workspace + static_cast<size_t>(C) * E;
    if (E <= 8)
        rt::route_topk_kernel<8, 1><<<C, rt::THREADS, 0, stream>>>(logits, T, E, K, topk_idx, topk_w, row_of, chunk_counts);
    else if (E <= 16)
        rt::route_topk_kernel<16, 1><<<C, rt::THREADS, 0, stream>>>(logits, T, E, K, topk_idx, topk_w, row_of, chunk_counts);
    else if (E <= 32)
        rt::route_topk_kernel<32, 1><<<C, rt::THREADS, 0, stream>>>(logits, T, E, K, topk_idx, topk_w, row_of, chunk_counts);
    else if (E <= 64)
        rt::route_topk_kernel<32, 2><<<C, rt::THREADS, 0, stream>>>(logits, T, E, K, topk_idx, topk_w, row_of, chunk_counts);
    else if (E <= 128)
        rt::route_topk_kernel<32, 4><<<C, rt::THREADS, 0, stream>>>(logits, T, E, K, topk_idx, topk_w, row_of, chunk_counts);
    else
        rt::route_topk_kernel<32, 8><<<C, rt::THREADS, 0, stream>>>(logits, T, E, K, topk_idx, topk_w, row_of, chunk_counts);
    cudaError_t err = cudaGetLastError();
    if (err != cudaSuccess) return err;
    rt::route_scan_kernel<<<1, rt::MAX_E, 0, stream>>>(chunk_counts, C, E, counts, offsets, chunk_base);
    err = cudaGetLastError();
    if (err != cudaSuccess) return err;
    const size_t TK = static_cast<size_t>(T) * K;
    const int blocks = static_cast<int>(std::min<size_t>((TK + 255) / 256, 152 * 8));
    rt::route_scatter_kernel<<<blocks, 256, 0, stream>>>(topk_idx, chunk_base, T, E, K, row_of, src_tok);
    return cudaGetLastError();
}

}  // namespace moe
