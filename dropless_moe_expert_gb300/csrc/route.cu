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
//  1. route_topk: one CTA of 32 warps per chunk of 64 tokens.  A group of G
//     lanes per token (G = 8, 16 or 32; 32/G tokens per warp); each lane holds E/G
//     logits as order-preserving 32-bit keys (-0.0 == +0.0).  K rounds pick
//     the experts, descending, lower index on ties.  With G = 32 a round is
//     two warp reductions (redux.sync): the largest key, then the lowest
//     expert among the lanes whose best key equals it; with G < 32 a round is
//     a group max of 64-bit (key << 32 | ~expert) values via shuffles.
//     Softmax over the K picks.  The CTA then marks, per expert, which of its
//     tokens chose it in a shared bitmap (atomicOr: the final bitmap does not
//     depend on order), and from it writes the chunk's per-expert count and
//     every pair's rank inside the chunk.
//  2. route_scan: one CTA of 1024 threads per 32 experts, each thread owning
//     one expert and a slice of chunks; counts = sum over chunks,
//     chunk_base[c][e] = rows of expert e in earlier chunks.
//  3. route_scatter: every CTA scans counts over the experts (CTA 0 writes
//     them as offsets); row_of[t,k] = offsets[e] + chunk_base[chunk(t)][e] +
//     rank; src_tok[row] = t.  Rows of a group are thus in ascending token
//     order.
#include "kernels.h"

#include <math.h>

#include <algorithm>

namespace moe {
namespace rt {

constexpr int CH = kRouteChunk;  // tokens per CTA
constexpr int SCAN_THREADS = 1024;
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
template <int G, int EPL, int THREADS>
__global__ void __launch_bounds__(THREADS)
route_topk_kernel(const float *__restrict__ L, int T, int E, int K, int32_t *__restrict__ topk_idx,
                  float *__restrict__ topk_w, int32_t *__restrict__ row_rank, int32_t *__restrict__ chunk_counts) {
    constexpr int TPW = 32 / G;  // tokens per warp at a time
    constexpr int WARPS = THREADS / 32;
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
        int my_e = 0;
        float my_z = 0.0f;
        float v0 = 0.0f, sum = 0.0f;
        if constexpr (G == 32) {
            // keys of experts lane + 32 j; 0 is below every real key
            uint32_t vk[EPL];
#pragma unroll
            for (int j = 0; j < EPL; ++j) vk[j] = (glane + 32 * j < E) ? order_key(nxt[j]) : 0u;
            load_logits(tl + WARPS * TPW);
            // this lane's best key; the lowest j (lowest expert) on ties
            uint32_t bv = vk[0];
            int bj = 0;
#pragma unroll
            for (int j = 1; j < EPL; ++j)
                if (vk[j] > bv) { bv = vk[j]; bj = j; }
            for (int k = 0; k < K; ++k) {
                const uint32_t vmax = __reduce_max_sync(0xffffffffu, bv);
                const uint32_t cand = (bv == vmax) ? static_cast<uint32_t>(glane + 32 * bj) : 0xffffffffu;
                const int e = static_cast<int>(__reduce_min_sync(0xffffffffu, cand));
                if ((e & 31) == glane) {
                    // the winner is this lane's best key: drop it, find the next
#pragma unroll
                    for (int j = 0; j < EPL; ++j) vk[j] = (j == bj) ? 0u : vk[j];
                    bv = vk[0];
                    bj = 0;
#pragma unroll
                    for (int j = 1; j < EPL; ++j)
                        if (vk[j] > bv) { bv = vk[j]; bj = j; }
                }
                const float v = key_value(vmax);
                if (k == 0) v0 = v;
                const float z = expf(v - v0);
                sum += z;
                if (glane == k) { my_e = e; my_z = z; }
            }
        } else {
            unsigned long long key[EPL];
#pragma unroll
            for (int j = 0; j < EPL; ++j) {
                const int e = glane + G * j;
                key[j] = (e < E) ? ((static_cast<unsigned long long>(order_key(nxt[j])) << 32) |
                                    static_cast<unsigned long long>(0xffffffffu - static_cast<uint32_t>(e)))
                                 : 0ull;  // below every real key
            }
            load_logits(tl + WARPS * TPW);
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

// Per-expert prefix over the chunks, spread over CTAs of SCAN_E experts.
// Thread (e, s) of a CTA: expert e0 + e, slice s of S = SCAN_THREADS / SCAN_E
// consecutive chunk ranges, so a warp's loads of one chunk row are coalesced
// across its experts.  Writes counts[e] and chunk_base[c][e], the rows of
// expert e in chunks before c (the base within the expert's group; the
// scatter adds the group's offset).
constexpr int SCAN_E = 32;
__global__ void __launch_bounds__(SCAN_THREADS)
route_scan_kernel(const int32_t *__restrict__ chunk_counts, int C, int E, int32_t *__restrict__ counts,
                  int32_t *__restrict__ chunk_base) {
    __shared__ int32_t part[SCAN_THREADS];  // [s][e]: rows of expert e in slice s, then the slice's base
    constexpr int S = SCAN_THREADS / SCAN_E;
    const int el = threadIdx.x % SCAN_E;
    const int sl = threadIdx.x / SCAN_E;
    const int e = blockIdx.x * SCAN_E + el;
    const int CS = (C + S - 1) / S;
    const int c0 = min(C, sl * CS), c1 = min(C, c0 + CS);
    int sum = 0;
    if (e < E) {
#pragma unroll 8
        for (int c = c0; c < c1; ++c) sum += chunk_counts[static_cast<size_t>(c) * E + e];
    }
    part[sl * SCAN_E + el] = sum;
    __syncthreads();
    if (sl == 0) {
        int run = 0;
        for (int q = 0; q < S; ++q) {
            const int pq = part[q * SCAN_E + el];
            part[q * SCAN_E + el] = run;
            run += pq;
        }
        if (e < E) counts[e] = run;
    }
    __syncthreads();
    if (e < E) {
        int run = part[sl * SCAN_E + el];
#pragma unroll 8
        for (int c = c0; c < c1; ++c) {
            chunk_base[static_cast<size_t>(c) * E + e] = run;
            run += chunk_counts[static_cast<size_t>(c) * E + e];
        }
    }
}

// Every CTA forms the exclusive scan of counts over the experts (E <= 256)
// in shared memory, and CTA 0 writes it to offsets (E + 1 entries).  Then
// row_of[t, k] = offsets[e] + chunk_base[chunk of t][e] + (the rank within
// the chunk that row_of holds on entry), and src_tok of that row is t.
__global__ void route_scatter_kernel(const int32_t *__restrict__ topk_idx, const int32_t *__restrict__ chunk_base,
                                     const int32_t *__restrict__ counts, int T, int E, int K,
                                     int32_t *__restrict__ offsets, int32_t *__restrict__ row_of,
                                     int32_t *__restrict__ src_tok) {
    __shared__ int32_t s_off[MAX_E + 1];
    if (threadIdx.x < 32) {
        const int lane = threadIdx.x;
        int carry = 0;
        for (int base = 0; base < E; base += 32) {
            const int v = base + lane < E ? counts[base + lane] : 0;
            int incl = v;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int n = __shfl_up_sync(0xffffffffu, incl, o);
                if (lane >= o) incl += n;
            }
            if (base + lane < E) s_off[base + lane] = carry + incl - v;
            carry += __shfl_sync(0xffffffffu, incl, 31);
        }
        if (lane == 0) s_off[E] = carry;
    }
    __syncthreads();
    if (blockIdx.x == 0)
        for (int e = threadIdx.x; e <= E; e += blockDim.x) offsets[e] = s_off[e];
    const size_t TK = static_cast<size_t>(T) * K;
    for (size_t p = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x; p < TK;
         p += static_cast<size_t>(gridDim.x) * blockDim.x) {
        const int t = static_cast<int>(p / K);
        const int e = topk_idx[p];
        const int r = s_off[e] + chunk_base[static_cast<size_t>(t / CH) * E + e] + row_of[p];
        row_of[p] = r;
        src_tok[r] = t;
    }
}

}  // namespace rt

cudaError_t launch_route(const float *logits, int T, int E, int K, int32_t *topk_idx, float *topk_w,
                         int32_t *counts, int32_t *offsets, int32_t *row_of, int32_t *src_tok, int32_t *workspace,
                         cudaStream_t stream) {
    const int C = route_num_chunks(T);
    // 32 warps per 64-token chunk: in a graph of back-to-back routing calls,
    // 256 -> 1024 threads took the DSv3-shaped routing from 22.0 to 17.0 us
    // and the Qwen-shaped from 24.9 to 22.5 us (the others unchanged)
    constexpr int TOPK_THREADS = 1024;
    int32_t *chunk_counts = workspace;
    int32_t *chunk_base = workspace + static_cast<size_t>(C) * E;
    if (E <= 8)
        rt::route_topk_kernel<8, 1, TOPK_THREADS><<<C, TOPK_THREADS, 0, stream>>>(logits, T, E, K, topk_idx, topk_w, row_of, chunk_counts);
    else if (E <= 16)
        rt::route_topk_kernel<16, 1, TOPK_THREADS><<<C, TOPK_THREADS, 0, stream>>>(logits, T, E, K, topk_idx, topk_w, row_of, chunk_counts);
    else if (E <= 32)
        rt::route_topk_kernel<32, 1, TOPK_THREADS><<<C, TOPK_THREADS, 0, stream>>>(logits, T, E, K, topk_idx, topk_w, row_of, chunk_counts);
    else if (E <= 64)
        rt::route_topk_kernel<32, 2, TOPK_THREADS><<<C, TOPK_THREADS, 0, stream>>>(logits, T, E, K, topk_idx, topk_w, row_of, chunk_counts);
    else if (E <= 128)
        rt::route_topk_kernel<32, 4, TOPK_THREADS><<<C, TOPK_THREADS, 0, stream>>>(logits, T, E, K, topk_idx, topk_w, row_of, chunk_counts);
    else
        rt::route_topk_kernel<32, 8, TOPK_THREADS><<<C, TOPK_THREADS, 0, stream>>>(logits, T, E, K, topk_idx, topk_w, row_of, chunk_counts);
    cudaError_t err = cudaGetLastError();
    if (err != cudaSuccess) return err;
    rt::route_scan_kernel<<<(E + rt::SCAN_E - 1) / rt::SCAN_E, rt::SCAN_THREADS, 0, stream>>>(chunk_counts, C, E,
                                                                                              counts, chunk_base);
    err = cudaGetLastError();
    if (err != cudaSuccess) return err;
    const size_t TK = static_cast<size_t>(T) * K;
    const int blocks = static_cast<int>(std::min<size_t>((TK + 255) / 256, 152 * 8));
    rt::route_scatter_kernel<<<blocks, 256, 0, stream>>>(topk_idx, chunk_base, counts, T, E, K, offsets, row_of,
                                                         src_tok);
    return cudaGetLastError();
}

}  // namespace moe
