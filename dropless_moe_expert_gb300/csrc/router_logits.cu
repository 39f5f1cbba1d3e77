// Step a0: router logits on the tensor cores, with fp32-exact products.
//
// Introduction of "Accelerating dropless MoE training in JAX with NVIDIA
// Transformer Engine": a learned router scores the experts of every token and
// activates the Top-K.  The score is the fp32 dot product of the token with
// the expert's router column, plus the expert's bias:
//     L[t, e] = sum_i x[t, i] * Wr[i, e] + bias[e]
// with x bf16 and Wr, bias and L fp32.
//
// Exact split of the fp32 weights.  Every fp32 value w is the exact sum of
// three bf16 values, w = hi + mid + lo, with hi = bf16(w), mid = bf16(w - hi),
// lo = bf16(w - hi - mid): each difference is exact in fp32 (the operands are
// within a factor of two), the first residual has at most 16 significant bits
// and the second at most 8, so lo takes it without rounding.  A bf16 x bf16
// product has at most 16 significant bits, so it is exact in fp32.  Hence
//     L[t, e] = sum_p sum_i x[t, i] * Wp[e, i],   p in {hi, mid, lo},
// is one bf16 contraction of depth 3d with exact products and fp32
// accumulation: the same operands and precision as the fp32 dot product,
// summed in the tensor core's order instead of index order (each piece's
// sum in its own fp32 accumulator, the three added at the end).  The result
// is deterministic (fixed tile shapes, no atomics, no split reduction).  A
// one-hot token gives every weight exactly: hi + mid is representable in
// fp32, and adding lo restores w.
//
// Two kernels:
//   router_split_kernel : Wr [d, E] fp32 -> Ws [3][E][d] bf16 (hi, mid, lo,
//                         each K-major, i.e. transposed) in caller scratch;
//   router_gemm_kernel  : one tile of MB x 128 tokens x BN experts per CTA;
//                         per 64-wide K slice TMA brings the MB x tiles and
//                         the three weight pieces' tiles (128-byte swizzle),
//                         which lie one after the other in shared memory and
//                         so form one K-major B operand of 3 BN rows.  One
//                         thread issues, per 128-token block, 4 tcgen05.mma
//                         (M=128, N=3 BN, K=16; for BN = 128 two per K step,
//                         N = 256 and 128) into the block's accumulator:
//                         TMEM columns [0, BN) accumulate x.hi, [BN, 2BN)
//                         x.mid and [2BN, 3BN) x.lo, each in fp32.  Tiles of
//                         two blocks (MB = 2) share the weight tiles, halving
//                         their bytes per token; they are used where one-block
//                         tiles would take more than one wave of the GPU.  Four warps form
//                         L = (x.hi + x.mid) + x.lo + bias and store fp32
//                         rows.  (Three MMAs of N = BN per K step measured
//                         2-3x slower: small-N MMAs are bound by their issue
//                         cost, not by the tensor pipe.)  Expert rows past E
//                         and token rows past T come from TMA zero fill and
//                         are not stored.
#include <atomic>

#include "kernels.h"
#include "ptx.cuh"
#include "tmap.h"

#include <cuda_bf16.h>

namespace moe {
namespace rt {

constexpr int BM = 128;
constexpr int BK = 64;
constexpr int UMMA_K = 16;
constexpr int THREADS = 128;
constexpr int A_BYTES = BM * BK * 2;

template <int BN, int MB>
struct Cfg {
    static constexpr int B_PIECE = BN * BK * 2;
    static constexpr int STAGE = MB * A_BYTES + 3 * B_PIECE;
    static constexpr int STAGES = (200 * 1024) / STAGE < 8 ? (200 * 1024) / STAGE : 8;
    static constexpr int OFF_BARS = STAGES * STAGE;  // whole KBs: tiles stay 1024-aligned
    static constexpr int NUM_BARS = 2 * STAGES + 2;  // full, empty, accumulator full, drain
    static constexpr int OFF_TMEM = OFF_BARS + NUM_BARS * 8;
    static constexpr int OFF_ABORT = OFF_TMEM + 4;
    static constexpr int BYTES = OFF_ABORT + 4 + 1024;  // slack for 1024-byte alignment
    static constexpr int ACC = BN == 32 ? 128 : (BN == 64 ? 256 : 512);  // 3 BN, rounded up to a power of two
    static constexpr int TMEM_COLS = MB * ACC;
    // one MMA of N = 3 BN where that fits (N <= 256); for BN = 128 two, of
    // N = 256 (hi and mid) and N = 128 (lo)
    static constexpr bool SPLIT_MMA = 3 * BN > 256;
    static_assert(BN == 32 || BN == 64 || BN == 128, "accumulator width");
    static_assert(MB == 1 || (MB == 2 && BN <= 64), "accumulators of a tile fit in TMEM");
    static_assert(STAGES >= 2 && BYTES <= 227 * 1024, "shared memory budget");
    static_assert(B_PIECE % 1024 == 0, "swizzled tiles must stay 1024-byte aligned");
};

struct Params {
    int T, d, E, NT;         // NT: expert tiles per token tile
    const float *bias;       // [E] or null
    float *L;                // [T, E]
    int vec4;                // rows of L are 16-byte aligned (E % 4 == 0 and L aligned)
    int *status;
    uint64_t timeout_ns;
};

// Wr [d, E] fp32 -> Ws[p][e][k] bf16, p = 0 (hi), 1 (mid), 2 (lo); 32 x 32
// tiles transposed through shared memory.
__global__ void __launch_bounds__(256)
router_split_kernel(const float *__restrict__ Wr, int d, int E, __nv_bfloat16 *__restrict__ Ws) {
    __shared__ float tile[32][33];
    const int k0 = blockIdx.x * 32, e0 = blockIdx.y * 32;
    const int tx = threadIdx.x & 31, ty = threadIdx.x >> 5;
#pragma unroll
    for (int r = ty; r < 32; r += 8) {
        const int k = k0 + r, e = e0 + tx;
        tile[r][tx] = (k < d && e < E) ? Wr[static_cast<size_t>(k) * E + e] : 0.0f;
    }
    __syncthreads();
    const size_t piece = static_cast<size_t>(E) * d;
#pragma unroll
    for (int r = ty; r < 32; r += 8) {
        const int e = e0 + r, k = k0 + tx;
        if (e >= E || k >= d) continue;
        const float w = tile[tx][r];
        const __nv_bfloat16 hi = __float2bfloat16_rn(w);
        const float r1 = w - __bfloat162float(hi);
        const __nv_bfloat16 mid = __float2bfloat16_rn(r1);
        const float r2 = r1 - __bfloat162float(mid);
        const __nv_bfloat16 lo = __float2bfloat16_rn(r2);
        const size_t o = static_cast<size_t>(e) * d + k;
        Ws[o] = hi;
        Ws[piece + o] = mid;
        Ws[2 * piece + o] = lo;
    }
}

template <int BN, int MB>
__global__ void __launch_bounds__(THREADS, 1)
router_gemm_kernel(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmW0,
                   const __grid_constant__ CUtensorMap tmW1, const __grid_constant__ CUtensorMap tmW2,
                   const Params p) {
    using C = Cfg<BN, MB>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + C::OFF_BARS);
    uint64_t *full = bars;
    uint64_t *empty = bars + C::STAGES;
    uint64_t *accfull = bars + 2 * C::STAGES;
    uint64_t *drain = accfull + 1;
    uint32_t *s_tmem = reinterpret_cast<uint32_t *>(smem + C::OFF_TMEM);
    volatile int *s_abort = reinterpret_cast<volatile int *>(smem + C::OFF_ABORT);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int n_blk = blockIdx.x % p.NT;
    const int m_blk = blockIdx.x / p.NT;  // expert tiles of one token tile are neighbours: x tile shared in L2
    const int n0 = n_blk * BN;
    const int m0 = m_blk * MB * BM;

    if (threadIdx.x == 0) {
        for (int i = 0; i < C::STAGES; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], 1);
        }
        mbar_init(accfull, 1);
        mbar_init(drain, 1);
        *s_abort = 0;
        fence_mbar_init();
        tma_prefetch_desc(&tmX);
        tma_prefetch_desc(&tmW0);
        tma_prefetch_desc(&tmW1);
        tma_prefetch_desc(&tmW2);
    }
    if (warp == 1) {
        tmem_alloc(s_tmem, C::TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *s_tmem;
    const int KB = p.d / BK;
    bool committed = false;  // MMA thread: the accumulator commit was issued

    if (warp == 0 && lane == 0) {
        // TMA producer
        int armed_phase[C::STAGES];
#pragma unroll
        for (int i = 0; i < C::STAGES; ++i) armed_phase[i] = -1;
        uint32_t stage = 0, phase = 0;
        bool ok = true;
        for (int kb = 0; kb < KB; ++kb) {
            if (!mbar_wait(&empty[stage], phase ^ 1u, s_abort, p.status, p.timeout_ns)) { ok = false; break; }
            uint8_t *sa = smem + stage * C::STAGE;
            uint8_t *sb = sa + MB * A_BYTES;
            mbar_arrive_expect_tx(&full[stage], C::STAGE);
#pragma unroll
            for (int b = 0; b < MB; ++b) tma_load_2d(sa + b * A_BYTES, &tmX, &full[stage], kb * BK, m0 + b * BM);
            tma_load_2d(sb, &tmW0, &full[stage], kb * BK, n0);
            tma_load_2d(sb + C::B_PIECE, &tmW1, &full[stage], kb * BK, n0);
            tma_load_2d(sb + 2 * C::B_PIECE, &tmW2, &full[stage], kb * BK, n0);
            armed_phase[stage] = static_cast<int>(phase);
            if (++stage == C::STAGES) { stage = 0; phase ^= 1u; }
        }
        if (!ok) {
            // every armed stage completes once its bytes have landed
            volatile int no_abort = 0;
            for (int i = 0; i < C::STAGES; ++i)
                if (armed_phase[i] >= 0)
                    mbar_wait(&full[i], static_cast<uint32_t>(armed_phase[i]), &no_abort, p.status, p.timeout_ns);
        }
    } else if (warp == 1 && lane == 0) {
        // MMA issuer: per K slice, the hi, mid and lo pieces in turn
        constexpr uint32_t idesc = idesc_bf16_f32(BM, C::SPLIT_MMA ? 2 * BN : 3 * BN);
        constexpr uint32_t idesc_lo = idesc_bf16_f32(BM, BN);
        uint32_t stage = 0, phase = 0;
        bool ok = true, issued = false;
        for (int kb = 0; kb < KB; ++kb) {
            if (!mbar_wait(&full[stage], phase, s_abort, p.status, p.timeout_ns)) { ok = false; break; }
            tc_fence_after();
            const uint32_t sa = smem_u32(smem + stage * C::STAGE);
            const uint64_t bdesc = smem_desc_kmajor_sw128(sa + MB * A_BYTES);  // hi, mid, lo rows: 3 BN
            const uint64_t bdesc_lo = smem_desc_kmajor_sw128(sa + MB * A_BYTES + 2 * C::B_PIECE);
#pragma unroll
            for (int b = 0; b < MB; ++b) {
                const uint64_t adesc = smem_desc_kmajor_sw128(sa + b * A_BYTES);
                const uint32_t acc = tmem_base + b * C::ACC;
#pragma unroll
                for (int j = 0; j < BK / UMMA_K; ++j) {
                    umma_bf16(acc, adesc + 2 * j, bdesc + 2 * j, idesc, (kb | j) != 0);
                    if (C::SPLIT_MMA)
                        umma_bf16(acc + 2 * BN, adesc + 2 * j, bdesc_lo + 2 * j, idesc_lo, (kb | j) != 0);
                }
            }
            issued = true;
            umma_commit(&empty[stage]);
            if (++stage == C::STAGES) { stage = 0; phase ^= 1u; }
        }
        committed = ok;
        if (ok) {
            umma_commit(accfull);
        } else if (issued) {
            volatile int no_abort = 0;
            umma_commit(drain);
            mbar_wait(drain, 0, &no_abort, p.status, p.timeout_ns);
        }
    }
    __syncwarp();

    // epilogue: warp w owns TMEM lanes 32w..32w+31 = token rows m0+32w.. of
    // each 128-token block
    const bool acc_ready = __all_sync(0xffffffffu, mbar_wait(accfull, 0, s_abort, p.status, p.timeout_ns));
    tc_fence_after();
#pragma unroll 1
    for (int b = 0; acc_ready && b < MB; ++b) {
        const int row = m0 + b * BM + warp * 32 + lane;
        const uint32_t tbase = tmem_base + (static_cast<uint32_t>(warp * 32) << 16) + b * C::ACC;
        float *Lrow = p.L + static_cast<size_t>(row) * p.E;
#pragma unroll 1
        for (int c = 0; c < BN; c += 32) {
            uint32_t vh[32], vm[32], vl[32];
            tmem_ld_32x32b_x32(tbase + c, vh);
            tmem_ld_32x32b_x32(tbase + BN + c, vm);
            tmem_ld_32x32b_x32(tbase + 2 * BN + c, vl);
            tmem_ld_wait();
            const int e0 = n0 + c;
            if (row < p.T && e0 < p.E) {
            float o[32];
#pragma unroll
            for (int i = 0; i < 32; ++i) {
                const int e = e0 + i;
                const float a = __fadd_rn(__fadd_rn(__uint_as_float(vh[i]), __uint_as_float(vm[i])),
                                          __uint_as_float(vl[i]));
                o[i] = (p.bias && e < p.E) ? __fadd_rn(a, p.bias[e]) : a;
            }
            if (p.vec4) {
#pragma unroll
                for (int i = 0; i < 32; i += 4)
                    if (e0 + i < p.E) *reinterpret_cast<float4 *>(Lrow + e0 + i) = make_float4(o[i], o[i + 1], o[i + 2], o[i + 3]);
            } else {
#pragma unroll
                for (int i = 0; i < 32; ++i)
                    if (e0 + i < p.E) Lrow[e0 + i] = o[i];
            }
            }
            __syncwarp();  // converged before the next tcgen05.ld
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        if (lane == 0 && committed && !acc_ready) {
            // the epilogue gave up: the MMAs still finish before TMEM is freed
            volatile int no_abort = 0;
            mbar_wait(accfull, 0, &no_abort, p.status, p.timeout_ns);
        }
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem_base, C::TMEM_COLS);
    }
}

template <int BN, int MB>
cudaError_t launch_gemm(const CUtensorMap &tmX, const CUtensorMap (&tmW)[3], const Params &p, int tiles,
                        cudaStream_t s) {
    router_gemm_kernel<BN, MB><<<tiles, THREADS, Cfg<BN, MB>::BYTES, s>>>(tmX, tmW[0], tmW[1], tmW[2], p);
    return cudaGetLastError();
}

}  // namespace rt

size_t router_workspace_bytes(int d, int E) { return static_cast<size_t>(3) * E * d * 2; }

int router_tile_n(int T, int E) {
    // widest accumulator that still gives about one wave of tiles
    const int mt = (T + rt::BM - 1) / rt::BM;
    int bn = E <= 32 ? 32 : (E <= 64 ? 64 : 128);
    while (bn > 32 && static_cast<int64_t>(mt) * ((E + bn - 1) / bn) < 120) bn /= 2;
    return bn;
}

cudaError_t router_setup() {
    cudaError_t e;
#define MOE_ROUTER_SMEM(BN, MB)                                                                               \
    if ((e = cudaFuncSetAttribute(rt::router_gemm_kernel<BN, MB>, cudaFuncAttributeMaxDynamicSharedMemorySize, \
                                  rt::Cfg<BN, MB>::BYTES)) != cudaSuccess)                                      \
        return e;
    MOE_ROUTER_SMEM(32, 1)
    MOE_ROUTER_SMEM(64, 1)
    MOE_ROUTER_SMEM(128, 1)
    MOE_ROUTER_SMEM(32, 2)
    MOE_ROUTER_SMEM(64, 2)
#undef MOE_ROUTER_SMEM
    return cudaSuccess;
}

cudaError_t launch_router_logits(const uint16_t *x, const float *Wr, const float *bias, int T, int d, int E,
                                 float *logits, void *workspace, int *status, uint64_t timeout_ns,
                                 cudaStream_t stream) {
    __nv_bfloat16 *Ws = static_cast<__nv_bfloat16 *>(workspace);
    rt::router_split_kernel<<<dim3((d + 31) / 32, (E + 31) / 32), 256, 0, stream>>>(Wr, d, E, Ws);
    cudaError_t err = cudaGetLastError();
    if (err != cudaSuccess) return err;

    const int bn = router_tile_n(T, E);
    CUtensorMap tmX, tmW[3];
    if (!make_tmap(&tmX, x, static_cast<uint64_t>(T), static_cast<uint64_t>(d), rt::BM, rt::BK))
        return cudaErrorInvalidValue;
    const size_t piece = static_cast<size_t>(E) * d;
    for (int pc = 0; pc < 3; ++pc)
        if (!make_tmap(&tmW[pc], Ws + pc * piece, static_cast<uint64_t>(E), static_cast<uint64_t>(d),
                       static_cast<uint32_t>(bn), rt::BK))
            return cudaErrorInvalidValue;
    rt::Params p;
    p.T = T;
    p.d = d;
    p.E = E;
    p.NT = (E + bn - 1) / bn;
    p.bias = bias;
    p.L = logits;
    p.vec4 = (E % 4 == 0) && (reinterpret_cast<uintptr_t>(logits) % 16 == 0);
    p.status = status;
    p.timeout_ns = timeout_ns;
    // Tiles of two 128-token blocks where one-block tiles would take more
    // than one wave: the busiest SMs then take in x for 256 tokens and the
    // weight tiles once, instead of both twice.
    const int mt = (T + rt::BM - 1) / rt::BM;
    static std::atomic<int> sm_count[64];  // per device, read once
    int dev = 0;
    if ((err = cudaGetDevice(&dev)) != cudaSuccess) return err;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    int sms = sm_count[dev].load(std::memory_order_relaxed);
    if (sms == 0) {
        if ((err = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return err;
        sm_count[dev].store(sms, std::memory_order_relaxed);
    }
    const bool two = bn <= 64 && mt * p.NT > sms;
    const int tiles = (two ? (mt + 1) / 2 : mt) * p.NT;
    switch (bn) {
        case 32: return two ? rt::launch_gemm<32, 2>(tmX, tmW, p, tiles, stream)
                            : rt::launch_gemm<32, 1>(tmX, tmW, p, tiles, stream);
        case 64: return two ? rt::launch_gemm<64, 2>(tmX, tmW, p, tiles, stream)
                            : rt::launch_gemm<64, 1>(tmX, tmW, p, tiles, stream);
        default: return rt::launch_gemm<128, 1>(tmX, tmW, p, tiles, stream);
    }
}

}  // namespace moe
