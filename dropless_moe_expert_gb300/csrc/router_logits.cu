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
// Register-tiled SIMT GEMM: a CTA owns BT tokens x BE experts; each thread
// owns TM tokens x TN experts and walks the reduction in order through
// 32-wide chunks staged in shared memory (x transposed to [k][token]).
#include "kernels.h"

#include <cuda_bf16.h>

namespace moe {
namespace rl {

constexpr int BK = 32;

template <int BE, int BT, int TM, int TN>
__global__ void __launch_bounds__((BE / TN) * (BT / TM))
router_logits_kernel(const uint16_t *__restrict__ x, const float *__restrict__ Wr, const float *__restrict__ bias,
                     int T, int d, int E, float *__restrict__ L) {
    constexpr int GX = BE / TN;
    constexpr int GY = BT / TM;
    constexpr int NTH = GX * GY;
    constexpr int XPAD = BT + 4;
    __shared__ __align__(16) float xs[BK][XPAD];
    __shared__ __align__(16) float ws[BK][BE];

    const int tid = threadIdx.x;
    const int tx = tid % GX;
    const int ty = tid / GX;
    const int t0 = blockIdx.x * BT;
    const int e0 = blockIdx.y * BE;

    float acc[TM][TN];
#pragma unroll
    for (int i = 0; i < TM; ++i)
#pragma unroll
        for (int j = 0; j < TN; ++j) acc[i][j] = 0.0f;

    for (int k0 = 0; k0 < d; k0 += BK) {
        // x chunk: BT tokens x 32 bf16 = BT * 4 vectors of 8 bf16
        for (int v = tid; v < BT * (BK / 8); v += NTH) {
            const int tl = v / (BK / 8);
            const int kv = (v % (BK / 8)) * 8;
            const int t = t0 + tl;
            uint4 raw = make_uint4(0, 0, 0, 0);
            if (t < T) raw = *reinterpret_cast<const uint4 *>(x + static_cast<size_t>(t) * d + k0 + kv);
            const uint32_t w4[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                xs[kv + 2 * q][tl] = __uint_as_float(w4[q] << 16);
                xs[kv + 2 * q + 1][tl] = __uint_as_float(w4[q] & 0xffff0000u);
            }
        }
        // Wr chunk: 32 rows x BE experts
        for (int v = tid; v < BK * BE; v += NTH) {
            const int kk = v / BE;
            const int el = v % BE;
            const int e = e0 + el;
            ws[kk][el] = (e < E) ? Wr[static_cast<size_t>(k0 + kk) * E + e] : 0.0f;
        }
        __syncthreads();
#pragma unroll 8
        for (int kk = 0; kk < BK; ++kk) {
            float a[TM], b[TN];
#pragma unroll
            for (int i = 0; i < TM; ++i) a[i] = xs[kk][ty * TM + i];
#pragma unroll
            for (int j = 0; j < TN; ++j) b[j] = ws[kk][tx * TN + j];
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
    if (E <= 8) return rl::launch<8, 32, 1, 2>(x, Wr, bias, T, d, E, logits, stream);
    if (E <= 16) return rl::launch<16, 64, 2, 4>(x, Wr, bias, T, d, E, logits, stream);
    if (E <= 32) return rl::launch<32, 64, 4, 4>(x, Wr, bias, T, d, E, logits, stream);
    return rl::launch<64, 64, 4, 4>(x, Wr, bias, T, d, E, logits, stream);
}

}  // namespace moe
