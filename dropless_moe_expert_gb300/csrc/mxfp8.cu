// MXFP8 quantisation for the block-scaled grouped GEMMs.
//
// "Optimization 1: Grouped GEMM" of "Accelerating dropless MoE training in JAX
// with NVIDIA Transformer Engine": on Blackwell the grouped GEMM path runs the
// expert matmuls with MXFP8 block scaling, fed by grouped quantisation
// kernels.  Format (MX, E4M3 elements): every 32 consecutive elements along
// the reduction dimension share one power-of-two scale 2^e stored as the
// byte e + 127; e is the smallest exponent with 448 * 2^e >= the block's
// largest magnitude (no element saturates), and each element is v * 2^-e
// rounded to the nearest E4M3 value (ties to even).
//
// Scale layout ("atoms").  The tensor cores read block scales from tensor
// memory, where tcgen05.cp 32x128b.warpx4 puts a 512-byte shared-memory
// atom: 128 rows x 4 blocks (one 128-wide K slice), byte
//     (row % 32) * 16 + (row / 32) * 4 + block
// lands in TMEM lane row % 32 (of every lane quarter), column row / 32, byte
// `block`, which is where a block-scaled MMA with scale-factor id `block`
// reads the scale of `row`.  Scales are stored in global memory as these
// atoms, one per (128-row block, K slice), so that a stage's scales are one
// 512-byte bulk copy:
//   * a plain matrix [R, K]: atom (r / 128) * (K / 128) + k / 128;
//   * the permuted activations (rows grouped by expert): the rows of each
//     expert group are cut into 128-row blocks from the group's first row,
//     and block b of expert e is atom row block rb = rb_prefix[e] + b, with
//     rb_prefix[e] = sum over e' < e of ceil(count[e'] / 128).  A GEMM tile
//     is one such row block, so its scales are whole atoms.
#include "kernels.h"
#include "mxfp8.cuh"

#include <cuda_bf16.h>

#include <algorithm>

namespace moe {
namespace mx {

constexpr int MAX_E = 256;

__device__ __forceinline__ void unpack_bf16x8(const uint4 &u, float *out) {
    const uint32_t p[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        out[2 * i] = __uint_as_float(p[i] << 16);
        out[2 * i + 1] = __uint_as_float(p[i] & 0xffff0000u);
    }
}

// One 128-wide K slice of one row: 256 bytes of bf16 in, 128 code bytes and
// one word of 4 scale bytes out.
__device__ __forceinline__ uint32_t quant_slice(const uint4 *__restrict__ src, uint4 (&codes)[8]) {
    uint32_t scales = 0;
#pragma unroll
    for (int b = 0; b < 4; ++b) {
        float v[32];
#pragma unroll
        for (int j = 0; j < 4; ++j) unpack_bf16x8(__ldg(src + 4 * b + j), v + 8 * j);
        uint32_t packed[8];
        scales |= quant_block(v, packed) << (8 * b);
        codes[2 * b] = make_uint4(packed[0], packed[1], packed[2], packed[3]);
        codes[2 * b + 1] = make_uint4(packed[4], packed[5], packed[6], packed[7]);
    }
    return scales;
}

// Plain matrix [R, K]: one thread per (row, K slice).
__global__ void __launch_bounds__(256)
quantize_kernel(const uint4 *__restrict__ src, int R, int K, uint4 *__restrict__ codes, uint32_t *__restrict__ sf) {
    const int ns = K / 128;
    const size_t n = static_cast<size_t>(R) * ns;
    for (size_t p = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x; p < n;
         p += static_cast<size_t>(gridDim.x) * blockDim.x) {
        const int r = static_cast<int>(p / ns), ks = static_cast<int>(p % ns);
        uint4 c[8];
        const uint32_t s = quant_slice(src + (static_cast<size_t>(r) * K + ks * 128) / 8, c);
        uint4 *dst = codes + (static_cast<size_t>(r) * K + ks * 128) / 16;
#pragma unroll
        for (int i = 0; i < 8; ++i) dst[i] = c[i];
        sf[atom_word(r / 128, ks, ns, r % 128)] = s;
    }
}

// Row-block prefix of the expert groups, from offsets[E+1] (clamped to
// [0, TK] like the GEMMs do), into shared memory; one warp.
__device__ __forceinline__ void row_block_prefix(const int32_t *__restrict__ offsets, int E, int TK, int lane,
                                                 int *s_off, int *s_rb) {
    int carry = 0;
    for (int base = 0; base < E; base += 32) {
        const int e = base + lane;
        int cnt = 0;
        if (e < E) {
            const int o0 = min(max(offsets[e], 0), TK);
            const int o1 = min(max(offsets[e + 1], o0), TK);
            s_off[e] = o0;
            cnt = (o1 - o0 + 127) / 128;
        }
        int v = cnt;
#pragma unroll
        for (int s = 1; s < 32; s <<= 1) {
            const int n = __shfl_up_sync(0xffffffffu, v, s);
            if (lane >= s) v += n;
        }
        if (e < E) s_rb[e] = carry + v - cnt;
        carry += __shfl_sync(0xffffffffu, v, 31);
    }
}

// Permute + quantise: one warp per token.  The warp walks the row in chunks
// of 256 elements, lane l holding elements 8l..8l+7 (one 16-byte load, so the
// warp reads 512 contiguous bytes); a block of 32 elements is 4 lanes, which
// combine their maxima with two shuffles.  Each lane writes its 8 codes (8
// bytes: 256 contiguous bytes per warp) to every row of x_perm the token
// occupies, and lane 16 s (s = 0, 1) gathers the 4 scale bytes of the chunk's
// s-th 128-element slice and writes them as one word of that row's atom.
__global__ void __launch_bounds__(256)
permute_kernel(const uint4 *__restrict__ x, const int32_t *__restrict__ topk_idx, const int32_t *__restrict__ row_of,
               const int32_t *__restrict__ offsets, int T, int K, int d, int E, uint2 *__restrict__ xq,
               uint32_t *__restrict__ sf) {
    __shared__ int s_off[MAX_E];
    __shared__ int s_rb[MAX_E];
    const int lane = threadIdx.x & 31;
    const int TK = T * K;
    if (threadIdx.x < 32) row_block_prefix(offsets, E, TK, lane, s_off, s_rb);
    __syncthreads();
    const int ns = d / 128;
    const int gw = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int nw = (gridDim.x * blockDim.x) >> 5;
    for (int t = gw; t < T; t += nw) {
        // lanes k < K hold the token's k-th row and expert
        int my_r = -1, my_e = -1;
        if (lane < K) {
            my_r = __ldg(row_of + static_cast<size_t>(t) * K + lane);
            my_e = __ldg(topk_idx + static_cast<size_t>(t) * K + lane);
        }
        // the next 256 columns' load is in flight while these are quantised and stored
        const uint4 *xrow = x + static_cast<size_t>(t) * d / 8;
        uint4 nxt = 8 * lane < d ? __ldg(xrow + lane) : make_uint4(0u, 0u, 0u, 0u);
        for (int c0 = 0; c0 < d; c0 += 256) {
            const bool valid = c0 + 8 * lane < d;  // d is a multiple of 128: whole blocks
            const uint4 cur = nxt;
            if (c0 + 256 + 8 * lane < d) nxt = __ldg(xrow + (c0 + 256) / 8 + lane);
            float v[8];
            if (valid) {
                unpack_bf16x8(cur, v);
            } else {
#pragma unroll
                for (int i = 0; i < 8; ++i) v[i] = 0.0f;
            }
            float amax = 0.0f;
#pragma unroll
            for (int i = 0; i < 8; ++i) amax = fmaxf(amax, fabsf(v[i]));
            amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
            amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
            const uint32_t sbyte = scale_byte(amax);
            const float inv = __uint_as_float((254u - sbyte) << 23);  // 2^-(s-127)
            uint2 code;
            code.x = pack4(v[0] * inv, v[1] * inv, v[2] * inv, v[3] * inv);
            code.y = pack4(v[4] * inv, v[5] * inv, v[6] * inv, v[7] * inv);
            // the chunk's two slices: bytes of blocks 0..3 from lanes 0, 4, 8, 12
            // (slice 0) and 16, 20, 24, 28 (slice 1)
            const uint32_t b1 = __shfl_down_sync(0xffffffffu, sbyte, 4);
            const uint32_t b2 = __shfl_down_sync(0xffffffffu, sbyte, 8);
            const uint32_t b3 = __shfl_down_sync(0xffffffffu, sbyte, 12);
            const uint32_t word = sbyte | (b1 << 8) | (b2 << 16) | (b3 << 24);
            const int ks = c0 / 128 + (lane >> 4);
            for (int k = 0; k < K; ++k) {
                const int r = __shfl_sync(0xffffffffu, my_r, k);
                const int e = __shfl_sync(0xffffffffu, my_e, k);
                if (r < 0 || r >= TK || e < 0 || e >= E) continue;  // outside the contract: skip (warp-uniform)
                const int local = r - s_off[e];
                if (local < 0) continue;
                if (valid) xq[(static_cast<size_t>(r) * d + c0 + 8 * lane) / 8] = code;
                if ((lane & 15) == 0 && valid) sf[atom_word(s_rb[e] + local / 128, ks, ns, local % 128)] = word;
            }
        }
    }
}

}  // namespace mx

size_t mxfp8_scales_bytes(int rows, int K) {
    return static_cast<size_t>((rows + 127) / 128) * (K / 128) * 512;
}

size_t mxfp8_perm_scales_bytes(int TK, int E, int K) {
    // row blocks of all groups: at most ceil(TK / 128) + E
    return (static_cast<size_t>((TK + 127) / 128) + E) * (K / 128) * 512;
}

cudaError_t launch_mxfp8_quantize(const uint16_t *src, int rows, int K, uint8_t *codes, uint8_t *scales,
                                  cudaStream_t stream) {
    const size_t n = static_cast<size_t>(rows) * (K / 128);
    const int blocks = static_cast<int>(std::min<size_t>((n + 255) / 256, 152 * 16));
    mx::quantize_kernel<<<blocks, 256, 0, stream>>>(reinterpret_cast<const uint4 *>(src), rows, K,
                                                   reinterpret_cast<uint4 *>(codes), reinterpret_cast<uint32_t *>(scales));
    return cudaGetLastError();
}

cudaError_t launch_permute_mxfp8(const uint16_t *x, const int32_t *topk_idx, const int32_t *row_of,
                                 const int32_t *offsets, int T, int K, int d, int E, uint8_t *xq, uint8_t *sfa,
                                 cudaStream_t stream) {
    const int warps = 8;
    const int blocks = std::max(1, std::min((T + warps - 1) / warps, 152 * 8));
    mx::permute_kernel<<<blocks, 32 * warps, 0, stream>>>(reinterpret_cast<const uint4 *>(x), topk_idx, row_of,
                                                         offsets, T, K, d, E, reinterpret_cast<uint2 *>(xq),
                                                         reinterpret_cast<uint32_t *>(sfa));
    return cudaGetLastError();
}

}  // namespace moe
