// Persistent grouped GEMM over ragged per-expert row groups, sm_103a.
//
// "Optimization 1: Grouped GEMM" of "Accelerating dropless MoE training in JAX
// with NVIDIA Transformer Engine": every expert's matmul runs inside one kernel
// call with its actual token count, only valid-token rows are computed, and
// the counts never travel to the host.  Figure 3 caption: the grouped MLP is
// two such GEMMs over the variable-length groups.
//
//   GEMM1 (SWIGLU = true):  h[r, n]      = bf16( silu(x_perm[r].W1[e,n]) * (x_perm[r].W1[e,f+n]) )
//   GEMM2 (SWIGLU = false): y_perm[r, n] = bf16( h[r].W2[e,n] )
// for every row r of expert e's group offsets[e]..offsets[e+1]-1.
//
// Design:
//  * One CTA per SM, persistent over a device-side tile list.  Every CTA reads
//    offsets[] (E+1 ints) and builds the tile prefix itself, so the host never
//    sees a count and the launch is the same for every routing.
//  * Tile = 128 rows x 256 accumulator columns.  GEMM1 stacks the gate rows
//    n0..n0+127 and the up rows f+n0..f+n0+127 of W1[e] into one 256-row B tile,
//    so one MMA produces both halves of SwiGLU for 128 output columns; GEMM2
//    uses 256 consecutive rows of W2[e].  A tile that runs past its group
//    reads neighbouring rows (or TMA zero fill); the epilogue masks them.
//  * Warp roles: warp 0 = TMA producer, warp 1 = tcgen05.mma issuer (and TMEM
//    owner), warps 2..5 = epilogue (TMEM -> registers -> global).
//  * 4-stage smem ring (48 KB per stage: A 128x64, B 256x64 bf16, 128-byte
//    swizzle) with full/empty mbarriers; two 256-column fp32 accumulators in
//    TMEM (512 columns) so the epilogue of tile i overlaps the mainloop of
//    tile i+1.
//  * Tiles are ordered expert by expert; inside an expert, bands of 16 row
//    blocks sweep all column blocks, so concurrent CTAs share the weight tile
//    through L2 and the band's activation rows stay L2-resident.
//  * Every wait is bounded: on expiry the kernel records a timeout, drains its
//    copies and MMAs, frees TMEM and returns.
#include <cudaTypedefs.h>

#include "kernels.h"
#include "ptx.cuh"

namespace moe {
namespace gg {

constexpr int BM = 128;
constexpr int BK = 64;
constexpr int BN_ACC = 256;
constexpr int STAGES = 4;
constexpr int A_BYTES = BM * BK * 2;
constexpr int B_BYTES = BN_ACC * BK * 2;
constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
constexpr int UMMA_K = 16;
constexpr int TMEM_COLS = 2 * BN_ACC;
constexpr int BAND = 16;
constexpr int THREADS = 192;
constexpr int MAX_E = 256;

constexpr int OFF_BARS = STAGES * STAGE_BYTES;
constexpr int NUM_BARS = 2 * STAGES + 5;  // full, empty, tfull[2], tempty[2], drain
constexpr int OFF_TMEM = OFF_BARS + NUM_BARS * 8;
constexpr int OFF_ABORT = OFF_TMEM + 4;
constexpr int OFF_OFFS = OFF_ABORT + 4;
constexpr int OFF_ENDS = OFF_OFFS + MAX_E * 4;
constexpr int OFF_PRE = OFF_ENDS + MAX_E * 4;
constexpr int SMEM_USED = OFF_PRE + (MAX_E + 1) * 4;
constexpr int SMEM_BYTES = SMEM_USED + 1024;  // slack for 1024-byte alignment

struct Params {
    const int32_t *offsets;  // [E+1] device
    int E;
    int TK;         // rows of the activation matrix
    int Kdim;       // reduction length (d for GEMM1, f for GEMM2)
    int n_out;      // output columns (f for GEMM1, d for GEMM2)
    int w_rows;     // weight rows per expert (2f or d)
    int NT;         // column blocks per row block
    __nv_bfloat16 *out;  // [TK, n_out]
    int *status;
    uint64_t timeout_ns;
};

struct Tile {
    int e, m_blk, n_blk, row0, rows, grp_end;
};

__device__ __forceinline__ Tile decode_tile(int tile, const int *s_pre, const int *s_off, const int *s_end, int E,
                                            int NT) {
    int lo = 0, hi = E - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (s_pre[mid] <= tile) lo = mid; else hi = mid - 1;
    }
    Tile t;
    t.e = lo;
    const int local = tile - s_pre[lo];
    const int g0 = s_off[lo], g1 = s_end[lo];
    const int cnt = g1 - g0;
    const int MT = (cnt + BM - 1) / BM;
    const int band = local / (BAND * NT);
    const int within = local - band * BAND * NT;
    const int mb0 = band * BAND;
    const int bm = min(BAND, MT - mb0);
    t.n_blk = within / bm;
    t.m_blk = mb0 + (within - t.n_blk * bm);
    t.row0 = g0 + t.m_blk * BM;
    t.rows = min(BM, cnt - t.m_blk * BM);
    t.grp_end = g1;
    return t;
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<const uint32_t *>(&v);
}

template <bool SWIGLU>
__global__ void __launch_bounds__(THREADS, 1)
grouped_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                    const Params p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + OFF_BARS);
    uint64_t *full = bars;
    uint64_t *empty = bars + STAGES;
    uint64_t *tfull = bars + 2 * STAGES;
    uint64_t *tempty = bars + 2 * STAGES + 2;
    uint64_t *drain = bars + 2 * STAGES + 4;
    uint32_t *s_tmem = reinterpret_cast<uint32_t *>(smem + OFF_TMEM);
    volatile int *s_abort = reinterpret_cast<volatile int *>(smem + OFF_ABORT);
    int *s_off = reinterpret_cast<int *>(smem + OFF_OFFS);
    int *s_end = reinterpret_cast<int *>(smem + OFF_ENDS);
    int *s_pre = reinterpret_cast<int *>(smem + OFF_PRE);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int E = p.E;
    const int NT = p.NT;

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
    if (warp == 2) {
        // Group bounds [s_off[e], s_end[e]), clamped to [0, TK] so that no
        // content of offsets[] can send a store out of bounds, and the
        // per-expert tile prefix s_pre (tiles of experts < e).
        int carry = 0;
        for (int base = 0; base < E; base += 32) {
            const int e = base + lane;
            int v = 0;
            if (e < E) {
                const int o0 = min(max(p.offsets[e], 0), p.TK);
                const int o1 = min(max(p.offsets[e + 1], o0), p.TK);
                s_off[e] = o0;
                s_end[e] = o1;
                v = ((o1 - o0 + BM - 1) / BM) * NT;
            }
#pragma unroll
            for (int s = 1; s < 32; s <<= 1) {
                const int n = __shfl_up_sync(0xffffffffu, v, s);
                if (lane >= s) v += n;
            }
            if (e < E) s_pre[e + 1] = carry + v;
            carry += __shfl_sync(0xffffffffu, v, 31);
        }
        if (lane == 0) s_pre[0] = 0;
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();

    const uint32_t tmem_base = *s_tmem;
    const int total_tiles = s_pre[E];
    const int KB = p.Kdim / BK;

    if (warp == 0) {
        if (lane == 0) {
            int armed_phase[STAGES];
#pragma unroll
            for (int i = 0; i < STAGES; ++i) armed_phase[i] = -1;
            uint32_t stage = 0, phase = 0;
            bool ok = true;
            for (int tile = blockIdx.x; ok && tile < total_tiles; tile += gridDim.x) {
                const Tile t = decode_tile(tile, s_pre, s_off, s_end, E, NT);
                int brow0, brow1;
                if (SWIGLU) {
                    brow0 = t.e * p.w_rows + t.n_blk * (BN_ACC / 2);
                    brow1 = brow0 + p.n_out;  // the up half starts f rows later
                } else {
                    brow0 = t.e * p.w_rows + t.n_blk * BN_ACC;
                    brow1 = brow0 + BN_ACC / 2;
                }
                for (int kb = 0; kb < KB; ++kb) {
                    if (!mbar_wait(&empty[stage], phase ^ 1u, s_abort, p.status, p.timeout_ns)) { ok = false; break; }
                    uint8_t *sa = smem + stage * STAGE_BYTES;
                    uint8_t *sb = sa + A_BYTES;
                    mbar_arrive_expect_tx(&full[stage], STAGE_BYTES);
                    tma_load_2d(sa, &tmA, &full[stage], kb * BK, t.row0);
                    tma_load_2d(sb, &tmB, &full[stage], kb * BK, brow0);
                    tma_load_2d(sb + B_BYTES / 2, &tmB, &full[stage], kb * BK, brow1);
                    armed_phase[stage] = static_cast<int>(phase);
                    if (++stage == STAGES) { stage = 0; phase ^= 1u; }
                }
            }
            if (!ok) {
                // Drain: every armed stage completes once its bytes have landed.
                volatile int no_abort = 0;
                for (int i = 0; i < STAGES; ++i)
                    if (armed_phase[i] >= 0)
                        mbar_wait(&full[i], static_cast<uint32_t>(armed_phase[i]), &no_abort, p.status, p.timeout_ns);
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {
            constexpr uint32_t idesc = idesc_bf16_f32(BM, BN_ACC);
            uint32_t stage = 0, phase = 0, acc = 0, acc_phase = 0;
            bool ok = true;
            bool issued = false;
            for (int tile = blockIdx.x; ok && tile < total_tiles; tile += gridDim.x) {
                if (!mbar_wait(&tempty[acc], acc_phase ^ 1u, s_abort, p.status, p.timeout_ns)) { ok = false; break; }
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + acc * BN_ACC;
                for (int kb = 0; kb < KB; ++kb) {
                    if (!mbar_wait(&full[stage], phase, s_abort, p.status, p.timeout_ns)) { ok = false; break; }
                    tc_fence_after();
                    const uint32_t sa = smem_u32(smem + stage * STAGE_BYTES);
                    const uint64_t adesc = smem_desc_kmajor_sw128(sa);
                    const uint64_t bdesc = smem_desc_kmajor_sw128(sa + A_BYTES);
#pragma unroll
                    for (int j = 0; j < BK / UMMA_K; ++j) {
                        // advance 16 elements (32 bytes) along K inside the swizzled row
                        umma_bf16(d_tmem, adesc + 2 * j, bdesc + 2 * j, idesc, (kb | j) != 0);
                    }
                    issued = true;
                    umma_commit(&empty[stage]);
                    if (++stage == STAGES) { stage = 0; phase ^= 1u; }
                }
                if (!ok) break;
                umma_commit(&tfull[acc]);
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
        const int q = warp & 3;  // TMEM lane quarter this warp may access
        const int row_local = q * 32 + lane;
        uint32_t acc = 0, acc_phase = 0;
        for (int tile = blockIdx.x; tile < total_tiles; tile += gridDim.x) {
            const Tile t = decode_tile(tile, s_pre, s_off, s_end, E, NT);
            if (!mbar_wait(&tfull[acc], acc_phase, s_abort, p.status, p.timeout_ns)) break;
            tc_fence_after();
            const uint32_t tbase = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + acc * BN_ACC;
            const int grow = t.row0 + row_local;
            const bool row_ok = row_local < t.rows && grow < t.grp_end;
            if (SWIGLU) {
#pragma unroll 1
                for (int c = 0; c < BN_ACC / 2; c += 32) {
                    uint32_t g[32], u[32];
                    tmem_ld_32x32b_x32(tbase + c, g);
                    tmem_ld_32x32b_x32(tbase + BN_ACC / 2 + c, u);
                    tmem_ld_wait();
                    const int col = t.n_blk * (BN_ACC / 2) + c;
                    if (row_ok && col < p.n_out) {
                        uint32_t packed[16];
#pragma unroll
                        for (int i = 0; i < 16; ++i) {
                            float h2[2];
#pragma unroll
                            for (int k = 0; k < 2; ++k) {
                                const float gv = __uint_as_float(g[2 * i + k]);
                                const float uv = __uint_as_float(u[2 * i + k]);
                                h2[k] = gv * __frcp_rn(1.0f + __expf(-gv)) * uv;
                            }
                            packed[i] = pack_bf16x2(h2[0], h2[1]);
                        }
                        uint4 *dst = reinterpret_cast<uint4 *>(p.out + static_cast<size_t>(grow) * p.n_out + col);
#pragma unroll
                        for (int i = 0; i < 4; ++i)
                            dst[i] = make_uint4(packed[4 * i], packed[4 * i + 1], packed[4 * i + 2], packed[4 * i + 3]);
                    }
                }
            } else {
#pragma unroll 1
                for (int c = 0; c < BN_ACC; c += 32) {
                    uint32_t v[32];
                    tmem_ld_32x32b_x32(tbase + c, v);
                    tmem_ld_wait();
                    const int col = t.n_blk * BN_ACC + c;
                    if (row_ok && col < p.n_out) {
                        uint32_t packed[16];
#pragma unroll
                        for (int i = 0; i < 16; ++i)
                            packed[i] = pack_bf16x2(__uint_as_float(v[2 * i]), __uint_as_float(v[2 * i + 1]));
                        uint4 *dst = reinterpret_cast<uint4 *>(p.out + static_cast<size_t>(grow) * p.n_out + col);
#pragma unroll
                        for (int i = 0; i < 4; ++i)
                            dst[i] = make_uint4(packed[4 * i], packed[4 * i + 1], packed[4 * i + 2], packed[4 * i + 3]);
                    }
                }
            }
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

}  // namespace gg

// ------------------------------------------------------------------ host side
namespace {

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static bool tried = false;
    if (!tried) {
        tried = true;
        void *ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
    }
    return fn;
}

// 2D bf16 row-major [rows, cols] with a (box_rows x 64) box and 128-byte swizzle.
bool make_tmap(CUtensorMap *m, const void *base, uint64_t rows, uint64_t cols, uint32_t box_rows) {
    auto fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[2] = {cols, rows};
    cuuint64_t strides[1] = {cols * 2};
    cuuint32_t box[2] = {static_cast<cuuint32_t>(gg::BK), box_rows};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

}  // namespace

int grouped_gemm_smem_bytes() { return gg::SMEM_BYTES; }

cudaError_t launch_grouped_gemm(bool swiglu, const void *A, int TK, int Kdim, const void *W, int E, int n_out,
                                const int32_t *offsets, void *out, int num_sms, int *status, uint64_t timeout_ns,
                                cudaStream_t stream) {
    CUtensorMap tmA, tmB;
    const int w_rows = swiglu ? 2 * n_out : n_out;
    if (!make_tmap(&tmA, A, static_cast<uint64_t>(TK), static_cast<uint64_t>(Kdim), gg::BM)) return cudaErrorInvalidValue;
    if (!make_tmap(&tmB, W, static_cast<uint64_t>(E) * w_rows, static_cast<uint64_t>(Kdim), gg::BN_ACC / 2))
        return cudaErrorInvalidValue;
    gg::Params p;
    p.offsets = offsets;
    p.E = E;
    p.TK = TK;
    p.Kdim = Kdim;
    p.n_out = n_out;
    p.w_rows = w_rows;
    p.NT = swiglu ? (n_out + gg::BN_ACC / 2 - 1) / (gg::BN_ACC / 2) : (n_out + gg::BN_ACC - 1) / gg::BN_ACC;
    p.out = static_cast<__nv_bfloat16 *>(out);
    p.status = status;
    p.timeout_ns = timeout_ns;
    if (swiglu)
        gg::grouped_gemm_kernel<true><<<num_sms, gg::THREADS, gg::SMEM_BYTES, stream>>>(tmA, tmB, p);
    else
        gg::grouped_gemm_kernel<false><<<num_sms, gg::THREADS, gg::SMEM_BYTES, stream>>>(tmA, tmB, p);
    return cudaGetLastError();
}

cudaError_t grouped_gemm_set_attributes() {
    cudaError_t e = cudaFuncSetAttribute(gg::grouped_gemm_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         gg::SMEM_BYTES);
    if (e != cudaSuccess) return e;
    return cudaFuncSetAttribute(gg::grouped_gemm_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                gg::SMEM_BYTES);
}

}  // namespace moe
