// Step a0: router logits, strict fp32 on the CUDA cores.
//
// Introduction of "Accelerating dropless MoE training in JAX with NVIDIA
// Transformer Engine": a learned router scores the experts of every token and
// activates the Top-K.  The score is the fp32 dot product of the token (bf16,
// converted exactly) with the expert's router column, accumulated in index
// order with one fused multiply-add per term, plus the expert's bias added
// once at the end.  Every output is one sequential FMA chain, so the logits
// are bit-reproducible, and the routing decisions taken on them are too.
//
// Two kernels: one for few experts (one chain per thread) and a register-tiled
// SIMT GEMM for many experts; both walk the reduction in index order.
#include "kernels.h"

#include <cuda_bf16.h>

namespace moe {
namespace rl {

// Many experts: register-tiled SIMT GEMM.  A CTA of NTH = (BE/TN)*(BT/TM)
// threads owns BT tokens x BE experts, each thread TM tokens x TN experts
// (TM x TN independent FMA chains).  The reduction walks 64-wide chunks
// staged in shared memory: x transposed to [k][token] as fp32 (consecutive
// lanes write consecutive tokens: no bank conflicts), Wr as [k][expert].  The
// next chunk is loaded into registers while the current one is consumed.
// Per k a warp reads TM/4 + 1 float4 per lane from shared memory for TM*TN
// FMAs, which keeps the FMA pipe, not the shared-memory pipe, the limit.
template <int BE, int BT, int TM, int TN>
__global__ void __launch_bounds__((BE / TN) * (BT / TM))
router_logits_kernel(const uint16_t *__restrict__ x, const float *__restrict__ Wr, const float *__restrict__ bias,
                     int T, int d, int E, float *__restrict__ L) {
    constexpr int BK = 64;
    constexpr int GX = BE / TN;
    constexpr int GY = BT / TM;
    constexpr int NTH = GX * GY;
    constexpr int XPAD = BT + 4;
    constexpr int XV = (BT * BK / 8 + NTH - 1) / NTH;   // 16-byte x vectors per thread per chunk
    constexpr int WV4 = (BK * BE / 4 + NTH - 1) / NTH;  // float4 of Wr per thread per chunk
    static_assert(TM % 4 == 0 && TN == 4, "float4 fragments");
    __shared__ __align__(16) float xs[BK][XPAD];
    __shared__ __align__(16) float ws[BK][BE];

    const int tid = threadIdx.x;
    const int tx = tid % GX;
    const int ty = tid / GX;
    const int t0 = blockIdx.x * BT;
    const int e0 = blockIdx.y * BE;
    const bool w_vec = (E % 4) == 0;  // Wr rows are 16-byte aligned: float4 loads

    uint4 xr[XV];
    float4 wr[WV4];
    auto load_chunk = [&](int k0) {
#pragma unroll
        for (int i = 0; i < XV; ++i) {
            const int v = tid + i * NTH;
            const int tl = v % BT, kv = (v / BT) * 8;
            const int t = t0 + tl;
            xr[i] = (v < BT * (BK / 8) && t < T)
                        ? *reinterpret_cast<const uint4 *>(x + static_cast<size_t>(t) * d + k0 + kv)
                        : make_uint4(0, 0, 0, 0);
        }
#pragma unroll
        for (int i = 0; i < WV4; ++i) {
            const int v = tid + i * NTH;
            const int kk = v / (BE / 4), e = e0 + (v % (BE / 4)) * 4;
            float4 w = make_float4(0.f, 0.f, 0.f, 0.f);
            if (v < BK * BE / 4) {
                const float *row = Wr + static_cast<size_t>(k0 + kk) * E;
                if (w_vec && e + 3 < E) {
                    w = *reinterpret_cast<const float4 *>(row + e);
                } else {
                    if (e < E) w.x = row[e];
                    if (e + 1 < E) w.y = row[e + 1];
                    if (e + 2 < E) w.z = row[e + 2];
                    if (e + 3 < E) w.w = row[e + 3];
                }
            }
            wr[i] = w;
        }
    };

    float acc[TM][TN];
#pragma unroll
    for (int i = 0; i < TM; ++i)
#pragma unroll
        for (int j = 0; j < TN; ++j) acc[i][j] = 0.0f;

    load_chunk(0);
    for (int k0 = 0; k0 < d; k0 += BK) {
#pragma unroll
        for (int i = 0; i < XV; ++i) {
            const int v = tid + i * NTH;
            if (v < BT * (BK / 8)) {
                const int tl = v % BT, kv = (v / BT) * 8;
                const uint32_t w4[4] = {xr[i].x, xr[i].y, xr[i].z, xr[i].w};
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    xs[kv + 2 * q][tl] = __uint_as_float(w4[q] << 16);
                    xs[kv + 2 * q + 1][tl] = __uint_as_float(w4[q] & 0xffff0000u);
                }
            }
        }
#pragma unroll
        for (int i = 0; i < WV4; ++i) {
            const int v = tid + i * NTH;
            if (v < BK * BE / 4) *reinterpret_cast<float4 *>(&ws[v / (BE / 4)][(v % (BE / 4)) * 4]) = wr[i];
        }
        __syncthreads();
        if (k0 + BK < d) load_chunk(k0 + BK);  // in flight during this chunk's FMAs
#pragma unroll 8
        for (int kk = 0; kk < BK; ++kk) {
            float a[TM];
#pragma unroll
            for (int i = 0; i < TM; i += 4) {
                const float4 a4 = *reinterpret_cast<const float4 *>(&xs[kk][ty * TM + i]);
                a[i] = a4.x; a[i + 1] = a4.y; a[i + 2] = a4.z; a[i + 3] = a4.w;
            }
            const float4 b4 = *reinterpret_cast<const float4 *>(&ws[kk][tx * TN]);
            const float b[4] = {b4.x, b4.y, b4.z, b4.w};
#pragma unroll
            for (int i = 0; i < TM; ++i)
#pragma unroll
                for (int j = 0; j < TN; ++j) acc[i][j] = __fmaf_rn(a[i], b[j], acc[i][j]);
        }
        __syncthreads();
    }

#pragma unroll
    for (int i = 0; i < TM; ++i) {
        const int t = t0 + ty * TM + i;
        if (t >= T) continue;
#pragma unroll
        for (int j = 0; j < TN; ++j) {
            const int e = e0 + tx * TN + j;
            if (e >= E) continue;
            const float v = bias ? __fadd_rn(acc[i][j], bias[e]) : acc[i][j];
            L[static_cast<size_t>(t) * E + e] = v;
        }
    }
}

// Few experts (E <= 16): one thread per (token, expert) pair, so there are
// T*E chains in flight instead of T*E/16; EP lanes of a warp share one token.
// Each 128-wide reduction chunk is staged in shared memory as fp32 (x once per
// token, Wr transposed to [expert][k]) while the next chunk is already being
// loaded into registers.
template <int EP>
__global__ void __launch_bounds__(256)
router_logits_small_e_kernel(const uint16_t *__restrict__ x, const float *__restrict__ Wr,
                             const float *__restrict__ bias, int T, int d, int E, float *__restrict__ L) {
    constexpr int SK = 128;               // reduction chunk
    constexpr int TPW = 32 / EP;          // tokens per warp
    constexpr int TPC = 8 * TPW;          // tokens per CTA
    constexpr int XV = TPC * SK / 8 / 256; // 16-byte x vectors per thread per chunk
    constexpr int WV = SK * EP / 256;      // Wr values per thread per chunk
    static_assert(XV >= 1 && WV >= 1, "tile does not cover the CTA");
    __shared__ __align__(16) float xs[TPC][SK + 4];
    __shared__ __align__(16) float ws[EP][SK + 4];

    const int tid = threadIdx.x;
    const int lane = tid & 31;
    const int tl = (tid >> 5) * TPW + lane / EP;
    const int e = lane % EP;
    const int t0 = blockIdx.x * TPC;

    uint4 xr[XV];
    float wr[WV];
    auto load_chunk = [&](int k0) {
#pragma unroll
        for (int i = 0; i < XV; ++i) {
            const int v = tid + i * 256;
            const int r = v / (SK / 8), c = (v % (SK / 8)) * 8;
            const int t = t0 + r;
            xr[i] = (t < T) ? *reinterpret_cast<const uint4 *>(x + static_cast<size_t>(t) * d + k0 + c)
                            : make_uint4(0, 0, 0, 0);
        }
#pragma unroll
        for (int i = 0; i < WV; ++i) {
            const int v = tid + i * 256;
            const int kk = v / EP, ee = v % EP;
            wr[i] = (ee < E) ? Wr[static_cast<size_t>(k0 + kk) * E + ee] : 0.0f;
        }
    };

    float acc = 0.0f;
    load_chunk(0);
    for (int k0 = 0; k0 < d; k0 += SK) {
#pragma unroll
        for (int i = 0; i < XV; ++i) {
            const int v = tid + i * 256;
            const int r = v / (SK / 8), c = (v % (SK / 8)) * 8;
            const uint32_t w4[4] = {xr[i].x, xr[i].y, xr[i].z, xr[i].w};
            float4 lo, hi;
            lo.x = __uint_as_float(w4[0] << 16); lo.y = __uint_as_float(w4[0] & 0xffff0000u);
            lo.z = __uint_as_float(w4[1] << 16); lo.w = __uint_as_float(w4[1] & 0xffff0000u);
            hi.x = __uint_as_float(w4[2] << 16); hi.y = __uint_as_float(w4[2] & 0xffff0000u);
            hi.z = __uint_as_float(w4[3] << 16); hi.w = __uint_as_float(w4[3] & 0xffff0000u);
            *reinterpret_cast<float4 *>(&xs[r][c]) = lo;
            *reinterpret_cast<float4 *>(&xs[r][c + 4]) = hi;
        }
#pragma unroll
        for (int i = 0; i < WV; ++i) {
            const int v = tid + i * 256;
            ws[v % EP][v / EP] = wr[i];
        }
        __syncthreads();
        if (k0 + SK < d) load_chunk(k0 + SK);  // in flight during this chunk's FMAs
#pragma unroll
        for (int kk = 0; kk < SK; kk += 4) {
            const float4 a = *reinterpret_cast<const float4 *>(&xs[tl][kk]);
            const float4 b = *reinterpret_cast<const float4 *>(&ws[e][kk]);
            acc = __fmaf_rn(a.x, b.x, acc);
            acc = __fmaf_rn(a.y, b.y, acc);
            acc = __fmaf_rn(a.z, b.z, acc);
            acc = __fmaf_rn(a.w, b.w, acc);
        }
        __syncthreads();
    }
    const int t = t0 + tl;
    if (t < T && e < E) L[static_cast<size_t>(t) * E + e] = bias ? __fadd_rn(acc, bias[e]) : acc;
}

template <int EP>
cudaError_t launch_small_e(const uint16_t *x, const float *Wr, const float *bias, int T, int d, int E, float *L,
                           cudaStream_t s) {
    constexpr int TPC = 8 * (32 / EP);
    router_logits_small_e_kernel<EP><<<(T + TPC - 1) / TPC, 256, 0, s>>>(x, Wr, bias, T, d, E, L);
    return cudaGetLastError();
}

template <int BE, int BT, int TM, int TN>
cudaError_t launch(const uint16_t *x, const float *Wr, const float *bias, int T, int d, int E, float *L,
                   cudaStream_t s) {
    dim3 grid((T + BT - 1) / BT, (E + BE - 1) / BE);
    router_logits_kernel<BE, BT, TM, TN><<<grid, (BE / TN) * (BT / TM), 0, s>>>(x, Wr, bias, T, d, E, L);
    return cudaGetLastError();
}

}  // namespace rl

cudaError_t launch_router_logits(const uint16_t *x, const float *Wr, const float *bias, int T, int d, int E,
                                 float *logits, cudaStream_t stream) {
    // d is a multiple of 64 (checked by the caller); the small-E kernel walks
    // the reduction in 128-wide chunks
    if (d % 128 == 0) {
        if (E <= 8) return rl::launch_small_e<8>(x, Wr, bias, T, d, E, logits, stream);
        if (E <= 16) return rl::launch_small_e<16>(x, Wr, bias, T, d, E, logits, stream);
    }
    if (E <= 16) return rl::launch<16, 64, 4, 4>(x, Wr, bias, T, d, E, logits, stream);
    if (E <= 32) return rl::launch<32, 64, 8, 4>(x, Wr, bias, T, d, E, logits, stream);
    return rl::launch<64, 64, 8, 4>(x, Wr, bias, T, d, E, logits, stream);
}

}  // namespace moe
