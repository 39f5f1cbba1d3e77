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
#include <atomic>

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
// [0, TK] like the GEMMs do), into shared memory; one warp.  Group e holds
// rows [s_off[e], s_end[e]) and its scale atoms start at row block s_rb[e].
__device__ __forceinline__ void row_block_prefix(const int32_t *__restrict__ offsets, int E, int TK, int lane,
                                                 int *s_off, int *s_end, int *s_rb) {
    int carry = 0;
    for (int base = 0; base < E; base += 32) {
        const int e = base + lane;
        int cnt = 0;
        if (e < E) {
            const int o0 = min(max(offsets[e], 0), TK);
            const int o1 = min(max(offsets[e + 1], o0), TK);
            s_off[e] = o0;
            s_end[e] = o1;
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

constexpr int PERMUTE_WARPS = 8;
constexpr int MAX_K = 16;

// Where one of a token's rows goes: its row r of x_perm (-1 for a row
// outside the contract, a row index outside [0, TK) or outside its expert's
// group, which is skipped) and its scale word in the atom of its group's row
// block at K slice 0 (slice ks adds 128 words).
struct RowDest {
    int row;
    int sf;
};

// 16 consecutive elements (32 bytes of bf16) of one lane, zeros past d.
__device__ __forceinline__ void load16(const uint4 *__restrict__ row, int c, int d, uint4 &a, uint4 &b) {
    if (c < d) {
        a = __ldg(row + c / 8);
        b = __ldg(row + c / 8 + 1);
    } else {
        a = b = make_uint4(0u, 0u, 0u, 0u);
    }
}

// Lane k < K: the destination of the token's k-th row (row r, expert e).
__device__ __forceinline__ RowDest row_dest(int r, int e, int E, int ns, const int *s_off, const int *s_end,
                                            const int *s_rb) {
    RowDest rd;
    rd.row = -1;
    rd.sf = 0;
    if (e >= 0 && e < E && r >= s_off[e] && r < s_end[e]) {
        const int local = r - s_off[e];
        rd.row = r;
        rd.sf = static_cast<int>(atom_word(s_rb[e] + local / 128, 0, ns, local % 128));
    }
    return rd;
}

// Permute + quantise.  A token row is cut into chunks of 512 elements.
// With W warps in the grid, warp w first takes whole tokens w, w + W, ...
// for R = floor(T / W) rounds, so that the warps sweep the tokens in order;
// the chunks of the last T - R W tokens are then cut into W equal
// contiguous runs, one per warp, so that the warps also end together.  In
// a chunk lane l holds elements 16l..16l+15 (two 16-byte loads; the warp
// reads 1 KB contiguous), so a 32-element block is a lane pair, whose maxima
// meet in one shuffle, and its 16 codes are one 16-byte store per
// destination row (512 contiguous bytes per warp).  Lane 8 s (s = 0..3)
// collects the 4 scale bytes of the chunk's s-th 128-element slice from
// lanes 8s, 8s+2, 8s+4, 8s+6 and writes them as one word of the row's atom.
// When a warp reaches a new token, lanes k < K work out its K destinations
// into shared memory, read back as one broadcast per row and chunk (the
// next row's read issued before this row's stores).  The next chunk and the
// next token's routing are loaded while the current chunk is quantised and
// stored.
__global__ void __launch_bounds__(32 * PERMUTE_WARPS, 5)
permute_kernel(const uint4 *__restrict__ x, const int32_t *__restrict__ topk_idx, const int32_t *__restrict__ row_of,
               const int32_t *__restrict__ offsets, int T, int K, int d, int E, uint8_t *__restrict__ xq,
               uint32_t *__restrict__ sf) {
    __shared__ int s_off[MAX_E];
    __shared__ int s_end[MAX_E];
    __shared__ int s_rb[MAX_E];
    __shared__ RowDest s_dst[PERMUTE_WARPS][MAX_K];
    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const int TK = T * K;
    if (threadIdx.x < 32) row_block_prefix(offsets, E, TK, lane, s_off, s_end, s_rb);
    __syncthreads();
    const int ns = d / 128;
    const int nch = (d + 511) / 512;
    const int W = gridDim.x * PERMUTE_WARPS;
    const int w = blockIdx.x * PERMUTE_WARPS + warp;
    const int R = T / W;
    const int tail0 = R * W;  // first token of the tail
    const long long tail_chunks = static_cast<long long>(T - tail0) * nch;
    const long long q0 = tail_chunks * w / W, q1 = tail_chunks * (w + 1) / W;
    const int tail_t = tail0 + static_cast<int>(q0 / nch);  // this warp's run of the tail
    const int tail_c = static_cast<int>(q0 % nch) * 512;
    const int tail_last = tail0 + static_cast<int>((q1 - 1) / nch);  // used only when q1 > q0
    int left = R * nch + static_cast<int>(q1 - q0);                  // chunks this warp quantises
    if (left == 0) return;
    // the token after tt in this warp's sequence (T when there is none)
    auto after = [&](int tt) -> int {
        if (tt < tail0) return tt + W < tail0 ? tt + W : (q1 > q0 ? tail_t : T);
        return tt < tail_last ? tt + 1 : T;
    };
    int t = R > 0 ? w : tail_t;
    int c0 = R > 0 ? 0 : tail_c;
    int t_next = after(t);
    RowDest *dst = s_dst[warp];
    int my_r = -1, my_e = -1;
    if (lane < K) {
        my_r = __ldg(row_of + static_cast<size_t>(t) * K + lane);
        my_e = __ldg(topk_idx + static_cast<size_t>(t) * K + lane);
        dst[lane] = row_dest(my_r, my_e, E, ns, s_off, s_end, s_rb);
        if (t_next < T) {
            my_r = __ldg(row_of + static_cast<size_t>(t_next) * K + lane);
            my_e = __ldg(topk_idx + static_cast<size_t>(t_next) * K + lane);
        }
    }
    uint4 na, nb;
    load16(x + static_cast<size_t>(t) * d / 8, c0 + 16 * lane, d, na, nb);
    __syncwarp();
    const bool scale_lane = (lane & 7) == 0;
    for (; left > 0; --left) {
        const bool more = left > 1;
        const int c = c0 + 16 * lane;
        const bool valid = c < d;  // d is a multiple of 128: whole slices
        const uint4 a = na, b = nb;
        int tn = t, cn = c0 + 512;
        if (cn >= d) {
            tn = t_next;
            cn = (t < tail0 && tn == tail_t) ? tail_c : 0;
        }
        if (more) load16(x + static_cast<size_t>(tn) * d / 8, cn + 16 * lane, d, na, nb);
        float v[16];
        unpack_bf16x8(a, v);
        unpack_bf16x8(b, v + 8);
        float amax = 0.0f;
#pragma unroll
        for (int i = 0; i < 16; ++i) amax = fmaxf(amax, fabsf(v[i]));
        amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
        const uint32_t sbyte = scale_byte(amax);
        const float inv = __uint_as_float((254u - sbyte) << 23);  // 2^-(s-127)
        uint4 code;
        code.x = pack4(v[0] * inv, v[1] * inv, v[2] * inv, v[3] * inv);
        code.y = pack4(v[4] * inv, v[5] * inv, v[6] * inv, v[7] * inv);
        code.z = pack4(v[8] * inv, v[9] * inv, v[10] * inv, v[11] * inv);
        code.w = pack4(v[12] * inv, v[13] * inv, v[14] * inv, v[15] * inv);
        const uint32_t b1 = __shfl_down_sync(0xffffffffu, sbyte, 2);
        const uint32_t b2 = __shfl_down_sync(0xffffffffu, sbyte, 4);
        const uint32_t b3 = __shfl_down_sync(0xffffffffu, sbyte, 6);
        const uint32_t word = sbyte | (b1 << 8) | (b2 << 16) | (b3 << 24);
        const int sf_col = (c0 / 128 + (lane >> 3)) * 128;
        uint8_t *xq_c = xq + c;
        RowDest nxt = dst[0];
        for (int k = 0; k < K; ++k) {
            const RowDest rd = nxt;
            if (k + 1 < K) nxt = dst[k + 1];
            if (rd.row >= 0 && valid) {  // rd is warp-uniform
                *reinterpret_cast<uint4 *>(xq_c + static_cast<size_t>(rd.row) * d) = code;
                if (scale_lane) sf[rd.sf + sf_col] = word;
            }
        }
        if (tn != t && more) {
            // next token: its destinations from the routing loaded a token ago
            __syncwarp();
            t_next = after(tn);
            if (lane < K) {
                dst[lane] = row_dest(my_r, my_e, E, ns, s_off, s_end, s_rb);
                if (t_next < T) {
                    my_r = __ldg(row_of + static_cast<size_t>(t_next) * K + lane);
                    my_e = __ldg(topk_idx + static_cast<size_t>(t_next) * K + lane);
                }
            }
            __syncwarp();
        }
        t = tn;
        c0 = cn;
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
    static std::atomic<int> resident[64];
    int wave = 0;
    const cudaError_t err = one_wave(mx::permute_kernel, 32 * mx::PERMUTE_WARPS, resident, &wave);
    if (err != cudaSuccess) return err;
    const long long chunks = static_cast<long long>(T) * ((d + 511) / 512);
    const int blocks = static_cast<int>(std::max(1LL, std::min((chunks + mx::PERMUTE_WARPS - 1) / mx::PERMUTE_WARPS,
                                                                static_cast<long long>(wave))));
    mx::permute_kernel<<<blocks, 32 * mx::PERMUTE_WARPS, 0, stream>>>(reinterpret_cast<const uint4 *>(x), topk_idx,
                                                                      row_of, offsets, T, K, d, E, xq,
                                                                      reinterpret_cast<uint32_t *>(sfa));
    return cudaGetLastError();
}

}  // namespace moe
