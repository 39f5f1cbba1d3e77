// Weight gradients of the grouped GEMMs: for every expert e,
//     D[e] = A^T[:, group e] . B^T[:, group e]^T    (M x N, fp32)
// i.e. dW2[e] = dy_perm[e]^T h[e] (M = d, N = f) and dW1[e] = da[e]^T x_perm[e]
// (M = 2f, N = d): a sum over the expert's own rows, a ragged reduction
// length per expert.
//
// The pages are about training with the grouped GEMM ("Optimization 1:
// Grouped GEMM" of "Accelerating dropless MoE training in JAX with NVIDIA
// Transformer Engine"); its weight gradients reduce over each expert's actual
// token rows, again without padding to a capacity.
//
// Operands are the transposed activations, K-major: A^T [M, Rp] and B^T
// [N, Rp] bf16, in which group e occupies columns pstart[e] ..
// pstart[e] + count[e] - 1 with pstart[e] = sum over e' < e of
// round_up(count[e'], 64) and zeros in the padding columns.  Every TMA K
// coordinate is then a multiple of 64 (16-byte aligned) and the padding adds
// nothing to the sums.
//
// Persistent kernel, one CTA per SM: tiles (e, 128-row block, 256-column
// block) of every expert; a 4-stage ring of 64-wide K slices (A 128 x 64,
// B 2 x 128 x 64, 128-byte swizzle); tcgen05.mma M=128 N=256 K=16 into two
// 256-column TMEM accumulators, so a tile's epilogue (fp32 stores, masked at
// M and N) overlaps the next tile's mainloop.  Experts without rows get their
// tiles written as zeros.  Bounded waits as in the forward GEMMs.
#include "kernels.h"
#include "ptx.cuh"
#include "tmap.h"

namespace moe {
namespace wg {

constexpr int BM = 128;
constexpr int BN = 256;
constexpr int BK = 64;
constexpr int UMMA_K = 16;
constexpr int THREADS = 192;
constexpr int STAGES = 4;
constexpr int MAX_E = 256;
constexpr int A_BYTES = BM * BK * 2;
constexpr int B_BYTES = BN * BK * 2;
constexpr int STAGE = A_BYTES + B_BYTES;
constexpr int TMEM_COLS = 2 * BN;
constexpr int OFF_BARS = STAGES * STAGE;
constexpr int NUM_BARS = 2 * STAGES + 5;  // full, empty, tfull[2], tempty[2], drain
constexpr int OFF_TMEM = OFF_BARS + NUM_BARS * 8;
constexpr int OFF_ABORT = OFF_TMEM + 4;
constexpr int OFF_PST = OFF_ABORT + 4;
constexpr int OFF_PCNT = OFF_PST + MAX_E * 4;
constexpr int SMEM_BYTES = OFF_PCNT + MAX_E * 4 + 1024;
static_assert(SMEM_BYTES <= 227 * 1024, "shared memory budget");

struct Params {
    const int32_t *offsets;  // [E+1]
    int E, TK, M, N, MT, NT;
    float *D;                // [E, M, N]
    int *status;
    uint64_t timeout_ns;
};

// Padded group starts and K lengths from offsets (clamped to [0, TK]); one warp.
__device__ __forceinline__ void padded_groups(const Params &p, int lane, int *s_pst, int *s_pcnt) {
    int carry = 0;
    for (int base = 0; base < p.E; base += 32) {
        const int e = base + lane;
        int v = 0;
        if (e < p.E) {
            const int o0 = min(max(p.offsets[e], 0), p.TK);
            const int o1 = min(max(p.offsets[e + 1], o0), p.TK);
            v = (o1 - o0 + BK - 1) / BK * BK;
            s_pcnt[e] = v;
        }
        int incl = v;
#pragma unroll
        for (int s = 1; s < 32; s <<= 1) {
            const int n = __shfl_up_sync(0xffffffffu, incl, s);
            if (lane >= s) incl += n;
        }
        if (e < p.E) s_pst[e] = carry + incl - v;
        carry += __shfl_sync(0xffffffffu, incl, 31);
    }
}

struct Tile {
    int e, m0, n0;
};

__device__ __forceinline__ Tile decode(const Params &p, int tile) {
    Tile t;
    const int per = p.MT * p.NT;
    t.e = tile / per;
    const int rem = tile - t.e * per;
    // column blocks vary fastest: neighbouring CTAs share the A rows in L2
    t.m0 = (rem / p.NT) * BM;
    t.n0 = (rem % p.NT) * BN;
    return t;
}

// One warp's 32 rows of a tile: fp32 out, masked at M and N.  `zero`: the
// expert has no rows, the accumulator is not read.
__device__ __forceinline__ void epilogue(const Params &p, const Tile &t, uint32_t tbase, int q, int lane, bool zero) {
    const int m = t.m0 + q * 32 + lane;
    const bool row_ok = m < p.M;
    float *row = p.D + (static_cast<size_t>(t.e) * p.M + m) * p.N;
#pragma unroll 1
    for (int c = 0; c < BN; c += 32) {
        const int n = t.n0 + c;
        if (n >= p.N) break;  // uniform
        uint32_t v[32];
        if (!zero) {
            tmem_ld_32x32b_x32(tbase + c, v);
            tmem_ld_wait();
        } else {
#pragma unroll
            for (int i = 0; i < 32; ++i) v[i] = 0u;
        }
        if (row_ok) {
            if (n + 32 <= p.N && (p.N % 4) == 0) {
#pragma unroll
                for (int i = 0; i < 32; i += 4)
                    *reinterpret_cast<float4 *>(row + n + i) = make_float4(
                        __uint_as_float(v[i]), __uint_as_float(v[i + 1]), __uint_as_float(v[i + 2]),
                        __uint_as_float(v[i + 3]));
            } else {
#pragma unroll
                for (int i = 0; i < 32; ++i)
                    if (n + i < p.N) row[n + i] = __uint_as_float(v[i]);
            }
        }
        __syncwarp();  // converged before the next tcgen05.ld
    }
}

__global__ void __launch_bounds__(THREADS, 1)
wgrad_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB, const Params p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + OFF_BARS);
    uint64_t *full = bars;
    uint64_t *empty = bars + STAGES;
    uint64_t *tfull = bars + 2 * STAGES;
    uint64_t *tempty = tfull + 2;
    uint64_t *drain = tfull + 4;
    uint32_t *s_tmem = reinterpret_cast<uint32_t *>(smem + OFF_TMEM);
    volatile int *s_abort = reinterpret_cast<volatile int *>(smem + OFF_ABORT);
    int *s_pst = reinterpret_cast<int *>(smem + OFF_PST);
    int *s_pcnt = reinterpret_cast<int *>(smem + OFF_PCNT);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int i = 0; i < STAGES; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&tfull[i], 1);
            mbar_init(&tempty[i], 4);
        }
        mbar_init(drain, 1);
        *s_abort = 0;
        fence_mbar_init();
        tma_prefetch_desc(&tmA);
        tma_prefetch_desc(&tmB);
    }
    if (warp == 1) {
        tmem_alloc(s_tmem, TMEM_COLS);
        tmem_relinquish();
    }
    if (warp == 2) padded_groups(p, lane, s_pst, s_pcnt);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *s_tmem;
    const int total = p.E * p.MT * p.NT;

    if (warp == 0) {
        if (lane == 0) {
            int armed_phase[STAGES];
#pragma unroll
            for (int i = 0; i < STAGES; ++i) armed_phase[i] = -1;
            uint32_t stage = 0, phase = 0;
            bool ok = true;
            for (int tile = blockIdx.x; ok && tile < total; tile += gridDim.x) {
                const Tile t = decode(p, tile);
                const int KB = s_pcnt[t.e] / BK;
                const int k0 = s_pst[t.e];
                for (int kb = 0; kb < KB; ++kb) {
                    if (!mbar_wait(&empty[stage], phase ^ 1u, s_abort, p.status, p.timeout_ns)) { ok = false; break; }
                    uint8_t *sa = smem + stage * STAGE;
                    uint8_t *sb = sa + A_BYTES;
                    mbar_arrive_expect_tx(&full[stage], STAGE);
                    tma_load_2d(sa, &tmA, &full[stage], k0 + kb * BK, t.m0);
                    tma_load_2d(sb, &tmB, &full[stage], k0 + kb * BK, t.n0);
                    tma_load_2d(sb + B_BYTES / 2, &tmB, &full[stage], k0 + kb * BK, t.n0 + BN / 2);
                    armed_phase[stage] = static_cast<int>(phase);
                    if (++stage == STAGES) { stage = 0; phase ^= 1u; }
                }
            }
            if (!ok) {
                volatile int no_abort = 0;
                for (int i = 0; i < STAGES; ++i)
                    if (armed_phase[i] >= 0)
                        mbar_wait(&full[i], static_cast<uint32_t>(armed_phase[i]), &no_abort, p.status, p.timeout_ns);
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {
            constexpr uint32_t idesc = idesc_bf16_f32(BM, BN);
            uint32_t stage = 0, phase = 0, acc = 0, acc_phase = 0;
            bool ok = true, issued = false;
            for (int tile = blockIdx.x; ok && tile < total; tile += gridDim.x) {
                const Tile t = decode(p, tile);
                const int KB = s_pcnt[t.e] / BK;
                if (!mbar_wait(&tempty[acc], acc_phase ^ 1u, s_abort, p.status, p.timeout_ns)) { ok = false; break; }
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + acc * BN;
                for (int kb = 0; kb < KB; ++kb) {
                    if (!mbar_wait(&full[stage], phase, s_abort, p.status, p.timeout_ns)) { ok = false; break; }
                    tc_fence_after();
                    const uint32_t sa = smem_u32(smem + stage * STAGE);
                    const uint64_t adesc = smem_desc_kmajor_sw128(sa);
                    const uint64_t bdesc = smem_desc_kmajor_sw128(sa + A_BYTES);
#pragma unroll
                    for (int j = 0; j < BK / UMMA_K; ++j)
                        umma_bf16(d_tmem, adesc + 2 * j, bdesc + 2 * j, idesc, (kb | j) != 0);
                    issued = true;
                    umma_commit(&empty[stage]);
                    if (++stage == STAGES) { stage = 0; phase ^= 1u; }
                }
                if (!ok) break;
                umma_commit(&tfull[acc]);  // with no MMAs (empty expert) it arrives at once
                acc ^= 1u;
                if (acc == 0) acc_phase ^= 1u;
            }
            if (!ok && issued) {
                volatile int no_abort = 0;
                umma_commit(drain);
                mbar_wait(drain, 0, &no_abort, p.status, p.timeout_ns);
            }
        }
    } else {
        const int q = warp & 3;
        uint32_t acc = 0, acc_phase = 0;
        for (int tile = blockIdx.x; tile < total; tile += gridDim.x) {
            const Tile t = decode(p, tile);
            if (!mbar_wait(&tfull[acc], acc_phase, s_abort, p.status, p.timeout_ns)) break;
            tc_fence_after();
            const uint32_t tbase = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + acc * BN;
            epilogue(p, t, tbase, q, lane, s_pcnt[t.e] == 0);
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&tempty[acc]);
            acc ^= 1u;
            if (acc == 0) acc_phase ^= 1u;
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem_base, TMEM_COLS);
    }
}

}  // namespace wg

size_t wgrad_padded_rows(int TK, int E) {
    // every group padded to a multiple of 64 rows, and the total a multiple
    // of 64 (16-byte row strides for TMA)
    return (static_cast<size_t>(TK) + 63) / 64 * 64 + static_cast<size_t>(E) * wg::BK;
}

cudaError_t wgrad_setup() {
    return cudaFuncSetAttribute(wg::wgrad_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, wg::SMEM_BYTES);
}

cudaError_t launch_wgrad(const uint16_t *At, const uint16_t *Bt, int M, int N, int Rp, const int32_t *offsets, int E,
                         int TK, float *D, int num_sms, int *status, uint64_t timeout_ns, cudaStream_t stream) {
    CUtensorMap tmA, tmB;
    if (!make_tmap(&tmA, At, static_cast<uint64_t>(M), static_cast<uint64_t>(Rp), wg::BM, wg::BK))
        return cudaErrorInvalidValue;
    if (!make_tmap(&tmB, Bt, static_cast<uint64_t>(N), static_cast<uint64_t>(Rp), wg::BN / 2, wg::BK))
        return cudaErrorInvalidValue;
    wg::Params p;
    p.offsets = offsets;
    p.E = E;
    p.TK = TK;
    p.M = M;
    p.N = N;
    p.MT = (M + wg::BM - 1) / wg::BM;
    p.NT = (N + wg::BN - 1) / wg::BN;
    p.D = D;
    p.status = status;
    p.timeout_ns = timeout_ns;
    wg::wgrad_kernel<<<num_sms, wg::THREADS, wg::SMEM_BYTES, stream>>>(tmA, tmB, p);
    return cudaGetLastError();
}

}  // namespace moe
