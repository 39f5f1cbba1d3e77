// MXFP8 block-scaled persistent grouped GEMM over ragged expert groups, sm_103a.
//
// "Optimization 1: Grouped GEMM" of "Accelerating dropless MoE training in JAX
// with NVIDIA Transformer Engine": all expert matmuls in one kernel call with
// their actual token counts, and on Blackwell with MXFP8 block scaling.
//
//   GEMM1 (SWIGLU = true):  h = silu(xq . W1q_gate^T) * (xq . W1q_up^T), then
//                           h is quantised to MXFP8 (blocks of 32 along f):
//                           codes hq [TK, f] and scale atoms for GEMM2's A
//   GEMM2 (SWIGLU = false): y_perm = bf16(hq . W2q^T)
// Operands are E4M3 codes with one UE8M0 scale per 32 elements of K; the
// products of the dequantised values are accumulated in fp32 in TMEM.
//
// Design (single CTA per tile, 128 rows x 256 accumulator columns; the tile
// scheduler, raster order and bf16 epilogue are the bf16 kernel's; GEMM2 of
// large groups with short reductions runs on the CTA-pair variant further
// down):
//  * Stage = one 128-element K slice: the A tile (128 rows x 128 B), the B
//    tile (two 128-row boxes: GEMM1 gate and up rows, GEMM2 256 rows), both
//    by TMA with 128-byte swizzle, and three 512-byte scale atoms (A, two B
//    row blocks) by bulk copies.  4 stages of 50 KB.
//  * The MMA thread copies a stage's atoms into that stage's slot of a TMEM
//    scale ring (tcgen05.cp 32x128b.warpx4: A at columns +0..3, B at
//    +4..11), then issues four tcgen05.mma kind::mxf8f6f4 block_scale
//    (M=128, N=256, K=32), the k-th reading scale byte k.  The copies and the
//    MMAs of one thread execute in issue order, and a slot is rewritten only
//    after its stage's MMAs completed (the shared-memory stage was freed by
//    their commit), so the ring needs no further synchronisation.
//  * One accumulator (256 columns); the other 256 TMEM columns hold the
//    scale ring.  GEMM1's epilogue, which forms and quantises h, is spread
//    over eight warps; each thread loads its 128 accumulator values first
//    and hands the accumulator back before the arithmetic and the stores, so
//    those overlap the next tile's mainloop.  GEMM2's epilogue (256 columns
//    per row) holds the accumulator until its last TMEM load.
//  * Scale atoms are addressed by 128-row blocks: A and h by the tile's row
//    block (rb = row blocks of earlier experts + the tile's block inside its
//    expert), the weights by their global row / 128.  Every atom index is
//    clamped to its buffer, so no content of offsets[] can send a bulk copy
//    out of bounds.
//  * Bounded waits as in the bf16 kernel.
#include <algorithm>

#include "gemm_common.cuh"
#include "kernels.h"
#include "mxfp8.cuh"
#include "ptx.cuh"
#include "tmap.h"

namespace moe {
namespace gmx {

using gg::BN_ACC;
using gg::EPI_BUF;
using gg::EPI_BYTES;
using gg::MAX_E;

constexpr int BM = 128;
constexpr int BK = 128;          // elements (= bytes) of K per stage
constexpr int UMMA_K = 32;
constexpr int BAND = 16;
// warps 0 and 1: TMA producer and MMA issuer; then eight epilogue warps, two
// per TMEM lane quarter, each owning half of the tile's columns (GEMM1: 64 of
// its 128 h columns, GEMM2: 128 of its 256 output columns).  With a single
// accumulator the epilogue would hold the next tile's MMAs for its whole
// length, so each thread first loads all of its accumulator values and hands
// the accumulator back, then forms and stores its outputs beside the next
// tile's mainloop.
template <bool SWIGLU>
struct Roles {
    static constexpr int EPI_WARPS = 8;
    static constexpr int THREADS = 64 + 32 * EPI_WARPS;
};
constexpr int STAGES = 4;
constexpr int A_BYTES = BM * BK;
constexpr int B_BYTES = BN_ACC * BK;
constexpr int SF_OFF = A_BYTES + B_BYTES;
constexpr int SF_BYTES = 3 * 512;
constexpr int STAGE = 51200;     // 1024-aligned
constexpr int TX_BYTES = A_BYTES + B_BYTES + SF_BYTES;
constexpr int TMEM_COLS = 512;
constexpr int SF_COL0 = BN_ACC;  // scale ring after the accumulator
constexpr int SF_SLOT = 16;
static_assert(SF_OFF + SF_BYTES <= STAGE && STAGE % 1024 == 0, "stage layout");
static_assert(SF_COL0 + STAGES * SF_SLOT <= TMEM_COLS, "TMEM budget");

constexpr int OFF_EPI = STAGES * STAGE;
constexpr int OFF_BARS = OFF_EPI + EPI_BYTES;
constexpr int NUM_BARS = 2 * STAGES + 3;  // full, empty, tfull, tempty, drain
constexpr int OFF_TMEM = OFF_BARS + NUM_BARS * 8;
constexpr int OFF_ABORT = OFF_TMEM + 4;
constexpr int OFF_OFFS = OFF_ABORT + 4;
constexpr int OFF_ENDS = OFF_OFFS + MAX_E * 4;
constexpr int OFF_PRE = OFF_ENDS + MAX_E * 4;
constexpr int OFF_MIX = OFF_PRE + (MAX_E + 1) * 4;
constexpr int SMEM_BYTES = OFF_MIX + 4 + 1024;
static_assert(SMEM_BYTES <= 227 * 1024, "shared memory budget");

struct MxParams {
    gg::Params g;
    const uint8_t *sfa;   // A scale atoms (row blocks of the expert groups)
    size_t sfa_atoms;
    const uint8_t *sfb;   // weight scale atoms (row blocks of the weight matrix)
    size_t sfb_atoms;
    uint8_t *hq;          // GEMM1: h codes [TK, n_out]
    uint32_t *sfh;        // GEMM1: h scale atoms, as words
    size_t sfh_atoms;
};

__device__ __forceinline__ size_t clamp_atom(size_t a, size_t n) { return a < n ? a : n - 1; }

// GEMM1 epilogue of one warp: 32 rows and half (64) of the tile's 128 output
// columns of h (gate columns 0..127 and up columns 128..255 of the
// accumulator).  Each thread owns one row.  It first loads all 128 of its
// accumulator values (the gate and up halves of its 64 columns) and then
// releases the accumulator (`release`: fence, warp sync, arrive on tempty),
// so the next tile's MMAs start while it forms h, quantises it per 32-column
// block and stores the codes; its two blocks' scale bytes are one half-word
// of the row's word in the h atom for this row block and slice.
template <typename Release>
__device__ __forceinline__ void epilogue_swiglu_mx(const MxParams &mp, uint32_t tbase, const gg::Tile &t, int q,
                                                   int half, int lane, int rb, Release release) {
    const gg::Params &p = mp.g;
    const int wrow0 = t.row0 + q * 32;
    if (wrow0 >= t.grp_end) {  // warp-uniform: nothing of this warp's rows to store
        release();
        return;
    }
    const int grow = wrow0 + lane;
    const bool row_ok = grow < t.grp_end;
    uint32_t g[2][32], u[2][32];
    tmem_ld_32x32b_x32(tbase + half * 64, g[0]);
    tmem_ld_32x32b_x32(tbase + BN_ACC / 2 + half * 64, u[0]);
    tmem_ld_32x32b_x32(tbase + half * 64 + 32, g[1]);
    tmem_ld_32x32b_x32(tbase + BN_ACC / 2 + half * 64 + 32, u[1]);
    tmem_ld_wait();
    release();
    uint32_t scales = 0;
#pragma unroll
    for (int b = 0; b < 2; ++b) {
        const int c = half * 64 + 32 * b;
        float h[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) {
            const float gv = __uint_as_float(g[b][i]);
            h[i] = __fdividef(gv, 1.0f + __expf(-gv)) * __uint_as_float(u[b][i]);  // silu(g) * u
        }
        uint32_t packed[8];
        scales |= mx::quant_block(h, packed) << (8 * b);
        if (row_ok) {
            uint4 *dst = reinterpret_cast<uint4 *>(mp.hq + static_cast<size_t>(grow) * p.n_out + t.n_blk * 128 + c);
            dst[0] = make_uint4(packed[0], packed[1], packed[2], packed[3]);
            dst[1] = make_uint4(packed[4], packed[5], packed[6], packed[7]);
        }
    }
    if (row_ok) {
        const int ns = p.n_out / 128;
        const size_t atom = clamp_atom(static_cast<size_t>(rb) * ns + t.n_blk, mp.sfh_atoms);
        const size_t word = atom * 128 + ((grow - t.row0) & 31) * 4 + ((grow - t.row0) >> 5);
        reinterpret_cast<uint16_t *>(mp.sfh)[2 * word + half] = static_cast<uint16_t>(scales);
    }
}

// GEMM2 epilogue of one warp: 32 rows and half (128) of the tile's 256
// output columns.  Each thread owns one row; it loads its 128 accumulator
// values, releases the accumulator (`release`), then converts them to bf16
// 32 columns at a time.  A chunk whose 32 rows all belong to the group is
// staged in the warp's shared-memory buffer (64-byte swizzle) and written by
// one TMA store of full lines; one that crosses the group's end is written
// by masked 16-byte stores per row.
template <typename Release>
__device__ __forceinline__ void epilogue_plain_mx(const gg::Params &p, const CUtensorMap *tm_out, uint8_t *buf,
                                                  uint32_t tbase, const gg::Tile &t, int q, int half, int lane,
                                                  Release release) {
    const int wrow0 = t.row0 + q * 32;
    if (wrow0 >= t.grp_end) {  // warp-uniform: nothing of this warp's rows to store
        release();
        return;
    }
    const bool full = wrow0 + 31 < t.grp_end;
    const int grow = wrow0 + lane;
    const bool row_ok = grow < t.grp_end;
    uint32_t v[4][32];
#pragma unroll
    for (int j = 0; j < 4; ++j) tmem_ld_32x32b_x32(tbase + half * 128 + 32 * j, v[j]);
    tmem_ld_wait();
    release();
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const int col = t.n_blk * BN_ACC + half * 128 + 32 * j;
        if (col >= p.n_out) break;  // column tail (uniform)
        uint32_t packed[16];
#pragma unroll
        for (int i = 0; i < 16; ++i)
            packed[i] = gg::pack_bf16x2(__uint_as_float(v[j][2 * i]), __uint_as_float(v[j][2 * i + 1]));
        if (full) {
            if (lane == 0) bulk_wait_read<0>();  // the previous chunk's store has read the buffer
            __syncwarp();
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const int kk = k ^ ((lane >> 1) & 3);
                *reinterpret_cast<uint4 *>(buf + lane * 64 + kk * 16) =
                    make_uint4(packed[4 * k], packed[4 * k + 1], packed[4 * k + 2], packed[4 * k + 3]);
            }
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
                tma_store_2d_evict_first(tm_out, buf, col, wrow0, l2_policy_evict_first());
                bulk_commit();
            }
        } else if (row_ok) {
            gg::store_row32(p.out + static_cast<size_t>(grow) * p.n_out + col, packed);
        }
    }
}

template <bool SWIGLU>
__global__ void __launch_bounds__(Roles<SWIGLU>::THREADS, 1)
grouped_gemm_mx_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                       const __grid_constant__ CUtensorMap tmOut, const MxParams mp) {
    const gg::Params &p = mp.g;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + OFF_BARS);
    uint64_t *full = bars;
    uint64_t *empty = bars + STAGES;
    uint64_t *tfull = bars + 2 * STAGES;
    uint64_t *tempty = tfull + 1;
    uint64_t *drain = tfull + 2;
    uint32_t *s_tmem = reinterpret_cast<uint32_t *>(smem + OFF_TMEM);
    volatile int *s_abort = reinterpret_cast<volatile int *>(smem + OFF_ABORT);
    int *s_off = reinterpret_cast<int *>(smem + OFF_OFFS);
    int *s_end = reinterpret_cast<int *>(smem + OFF_ENDS);
    int *s_pre = reinterpret_cast<int *>(smem + OFF_PRE);
    int *s_mix = reinterpret_cast<int *>(smem + OFF_MIX);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int E = p.E;
    const int NT = p.NT;

    if (threadIdx.x == 0) {
        for (int i = 0; i < STAGES; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], 1);
        }
        mbar_init(tfull, 1);
        mbar_init(tempty, Roles<SWIGLU>::EPI_WARPS);
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
    if (warp == 2) gg::build_groups<BM>(p, lane, s_off, s_end, s_pre, s_mix);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();

    const uint32_t tmem_base = *s_tmem;
    const int total_tiles = s_pre[E];
    const int mix = *s_mix;
    const int KB = p.Kdim / BK;
    const size_t wrows_total = static_cast<size_t>(E) * p.w_rows;

    if (warp == 0) {
        if (lane == 0) {
            int armed_phase[STAGES];
#pragma unroll
            for (int i = 0; i < STAGES; ++i) armed_phase[i] = -1;
            uint32_t stage = 0, phase = 0;
            bool ok = true;
            for (int k = 0, tile = gg::round_position(0, blockIdx.x, gridDim.x, mix); ok && tile < total_tiles;
                 ++k, tile = gg::round_position(k, blockIdx.x, gridDim.x, mix)) {
                const gg::Tile t =
                    gg::decode_tile<BM, BAND>(gg::visit_order(tile, total_tiles, mix), s_pre, s_off, s_end, E, NT);
                const int rb = s_pre[t.e] / NT + t.m_blk;
                int brow0, brow1;
                if (SWIGLU) {
                    brow0 = t.e * p.w_rows + t.n_blk * (BN_ACC / 2);
                    brow1 = brow0 + p.n_out;  // the up half starts f rows later
                } else {
                    brow0 = t.e * p.w_rows + t.n_blk * BN_ACC;
                    brow1 = brow0 + BN_ACC / 2;
                }
                // a B block past the last weight row only feeds masked columns:
                // take any valid atom for it
                const size_t wb0 = static_cast<size_t>(brow0) / 128;
                const size_t wb1 = static_cast<size_t>(brow1) < wrows_total ? static_cast<size_t>(brow1) / 128 : wb0;
                for (int kb = 0; kb < KB; ++kb) {
                    if (!mbar_wait(&empty[stage], phase ^ 1u, s_abort, p.status, p.timeout_ns)) { ok = false; break; }
                    uint8_t *sa = smem + stage * STAGE;
                    uint8_t *sb = sa + A_BYTES;
                    uint8_t *ssf = sa + SF_OFF;
                    mbar_arrive_expect_tx(&full[stage], TX_BYTES);
                    tma_load_2d(sa, &tmA, &full[stage], kb * BK, t.row0);
                    tma_load_2d(sb, &tmB, &full[stage], kb * BK, brow0);
                    tma_load_2d(sb + B_BYTES / 2, &tmB, &full[stage], kb * BK, brow1);
                    bulk_load(ssf, mp.sfa + clamp_atom(static_cast<size_t>(rb) * KB + kb, mp.sfa_atoms) * 512, 512,
                              &full[stage]);
                    bulk_load(ssf + 512, mp.sfb + clamp_atom(wb0 * KB + kb, mp.sfb_atoms) * 512, 512, &full[stage]);
                    bulk_load(ssf + 1024, mp.sfb + clamp_atom(wb1 * KB + kb, mp.sfb_atoms) * 512, 512, &full[stage]);
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
            uint32_t stage = 0, phase = 0, acc_phase = 0;
            bool ok = true, issued = false;
            for (int k = 0, tile = gg::round_position(0, blockIdx.x, gridDim.x, mix); ok && tile < total_tiles;
                 ++k, tile = gg::round_position(k, blockIdx.x, gridDim.x, mix)) {
                if (!mbar_wait(tempty, acc_phase ^ 1u, s_abort, p.status, p.timeout_ns)) { ok = false; break; }
                tc_fence_after();
                for (int kb = 0; kb < KB; ++kb) {
                    if (!mbar_wait(&full[stage], phase, s_abort, p.status, p.timeout_ns)) { ok = false; break; }
                    tc_fence_after();
                    const uint32_t sa = smem_u32(smem + stage * STAGE);
                    const uint32_t t_sfa = tmem_base + SF_COL0 + stage * SF_SLOT;
                    const uint32_t t_sfb = t_sfa + 4;
                    tmem_cp_32x128b_warpx4(t_sfa, smem_desc_rows16(sa + SF_OFF));
                    tmem_cp_32x128b_warpx4(t_sfb, smem_desc_rows16(sa + SF_OFF + 512));
                    tmem_cp_32x128b_warpx4(t_sfb + 4, smem_desc_rows16(sa + SF_OFF + 1024));
                    const uint64_t adesc = smem_desc_kmajor_sw128(sa);
                    const uint64_t bdesc = smem_desc_kmajor_sw128(sa + A_BYTES);
#pragma unroll
                    for (int j = 0; j < BK / UMMA_K; ++j)
                        umma_mxf8(tmem_base, adesc + 2 * j, bdesc + 2 * j, idesc_mxf8(BM, BN_ACC, j), t_sfa, t_sfb,
                                  (kb | j) != 0);
                    issued = true;
                    umma_commit(&empty[stage]);
                    if (++stage == STAGES) { stage = 0; phase ^= 1u; }
                }
                if (!ok) break;
                umma_commit(tfull);
                acc_phase ^= 1u;
            }
            if (!ok && issued) {
                volatile int no_abort = 0;
                umma_commit(drain);
                mbar_wait(drain, 0, &no_abort, p.status, p.timeout_ns);
            }
        }
    } else {
        const int q = warp & 3;  // TMEM lane quarter this warp may access
        const int half = (warp - 2) / 4;  // which half of the tile's columns
        static_assert(Roles<SWIGLU>::EPI_WARPS * EPI_BUF <= EPI_BYTES, "epilogue staging");
        uint8_t *stage_buf = smem + OFF_EPI + (warp - 2) * EPI_BUF;
        uint32_t acc_phase = 0;
        for (int k = 0, tile = gg::round_position(0, blockIdx.x, gridDim.x, mix); tile < total_tiles;
             ++k, tile = gg::round_position(k, blockIdx.x, gridDim.x, mix)) {
            const gg::Tile t =
                gg::decode_tile<BM, BAND>(gg::visit_order(tile, total_tiles, mix), s_pre, s_off, s_end, E, NT);
            if (!mbar_wait(tfull, acc_phase, s_abort, p.status, p.timeout_ns)) break;
            tc_fence_after();
            const uint32_t tbase = tmem_base + (static_cast<uint32_t>(q * 32) << 16);
            // hands the accumulator back to the MMA thread (after this warp's
            // TMEM loads have completed)
            auto release = [&]() {
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(tempty);
            };
            if (SWIGLU) {
                epilogue_swiglu_mx(mp, tbase, t, q, half, lane, s_pre[t.e] / NT + t.m_blk, release);
            } else {
                epilogue_plain_mx(p, &tmOut, stage_buf, tbase, t, q, half, lane, release);
            }
            acc_phase ^= 1u;
        }
        if (lane == 0) bulk_wait_all();  // stores done before the CTA's shared memory goes away
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem_base, TMEM_COLS);
    }
}

// ======================================================================
// CTA-pair variant of GEMM2 (cluster of 2): 256-row tiles through
// cta_group::2 block-scaled MMAs (M = 256).  CTA r loads A rows row0 + 128 r
// .. + 127 and rows 128 r .. 128 r + 127 of the 256-row column block of W2,
// so each SM moves 32 KB of operands per 128-wide K slice instead of 48 KB.
// Scales: each CTA holds the scale atom of its own 128 A rows and both atoms
// of the 256 B rows (each CTA's half of D needs all B columns' scales), and
// the pair copy (tcgen05.cp.cta_group::2, issued by CTA 0) moves each CTA's
// atoms into its own TMEM.  Every copy of both CTAs -- the atoms too, through
// 2D tensor maps of 256-byte rows -- completes on CTA 0's full barrier; CTA
// 0's commits free both CTAs' stages and fill both accumulators.  The eight
// epilogue warps of each CTA hand CTA 0's accumulator back once their values
// are loaded.
// ======================================================================
constexpr int P_BM = 256;
constexpr int P_BAND = 8;
constexpr int P_STAGES = 5;
constexpr int P_A_BYTES = 128 * BK;
constexpr int P_B_BYTES = 128 * BK;
constexpr int P_SF_OFF = P_A_BYTES + P_B_BYTES;
constexpr int P_STAGE = 34816;  // 1024-aligned
constexpr int P_TX_BYTES = P_A_BYTES + P_B_BYTES + SF_BYTES;  // per CTA
static_assert(P_SF_OFF + SF_BYTES <= P_STAGE && P_STAGE % 1024 == 0, "pair stage layout");
static_assert(SF_COL0 + P_STAGES * SF_SLOT <= TMEM_COLS, "pair TMEM budget");
constexpr int P_OFF_EPI = P_STAGES * P_STAGE;
constexpr int P_OFF_BARS = P_OFF_EPI + EPI_BYTES;
constexpr int P_NUM_BARS = 2 * P_STAGES + 3;  // full, empty, tfull, tempty, drain
constexpr int P_OFF_TMEM = P_OFF_BARS + P_NUM_BARS * 8;
constexpr int P_OFF_ABORT = P_OFF_TMEM + 4;
constexpr int P_OFF_OFFS = P_OFF_ABORT + 4;
constexpr int P_OFF_ENDS = P_OFF_OFFS + MAX_E * 4;
constexpr int P_OFF_PRE = P_OFF_ENDS + MAX_E * 4;
constexpr int P_OFF_P128 = P_OFF_PRE + (MAX_E + 1) * 4;
constexpr int P_OFF_MIX = P_OFF_P128 + MAX_E * 4;
constexpr int P_SMEM_BYTES = P_OFF_MIX + 4 + 1024;
static_assert(P_SMEM_BYTES <= 227 * 1024, "shared memory budget");

// Per expert, the 128-row scale-atom blocks of the experts before it (A and h
// atoms are numbered by 128-row blocks of the expert groups); one warp.
__device__ __forceinline__ void atom_block_prefix(const gg::Params &p, int lane, int *s_p128) {
    int carry = 0;
    for (int base = 0; base < p.E; base += 32) {
        const int e = base + lane;
        int v = 0;
        if (e < p.E) {
            const int o0 = min(max(p.offsets[e], 0), p.TK);
            const int o1 = min(max(p.offsets[e + 1], o0), p.TK);
            v = (o1 - o0 + 127) / 128;
        }
        int incl = v;
#pragma unroll
        for (int sh = 1; sh < 32; sh <<= 1) {
            const int n = __shfl_up_sync(0xffffffffu, incl, sh);
            if (lane >= sh) incl += n;
        }
        if (e < p.E) s_p128[e] = carry + incl - v;
        carry += __shfl_sync(0xffffffffu, incl, 31);
    }
}

__global__ void __launch_bounds__(Roles<false>::THREADS, 1)
grouped_gemm_mx_pair_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                            const __grid_constant__ CUtensorMap tmOut, const __grid_constant__ CUtensorMap tmSFA,
                            const __grid_constant__ CUtensorMap tmSFB, const MxParams mp) {
    const gg::Params &p = mp.g;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + P_OFF_BARS);
    uint64_t *full = bars;                 // CTA 0: both CTAs' copies
    uint64_t *empty = bars + P_STAGES;     // both CTAs: CTA 0's commits
    uint64_t *tfull = bars + 2 * P_STAGES;  // both CTAs
    uint64_t *tempty = tfull + 1;          // CTA 0: the epilogue warps of both CTAs
    uint64_t *drain = tfull + 2;
    uint32_t *s_tmem = reinterpret_cast<uint32_t *>(smem + P_OFF_TMEM);
    volatile int *s_abort = reinterpret_cast<volatile int *>(smem + P_OFF_ABORT);
    int *s_off = reinterpret_cast<int *>(smem + P_OFF_OFFS);
    int *s_end = reinterpret_cast<int *>(smem + P_OFF_ENDS);
    int *s_pre = reinterpret_cast<int *>(smem + P_OFF_PRE);
    int *s_p128 = reinterpret_cast<int *>(smem + P_OFF_P128);
    int *s_mix = reinterpret_cast<int *>(smem + P_OFF_MIX);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int E = p.E;
    const int NT = p.NT;
    const uint32_t rank = cluster_ctarank();
    const int pair = blockIdx.x >> 1;
    const int npairs = gridDim.x >> 1;
    constexpr int EPI_WARPS = Roles<false>::EPI_WARPS;

    if (threadIdx.x == 0) {
        for (int i = 0; i < P_STAGES; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], 1);
        }
        mbar_init(tfull, 1);
        mbar_init(tempty, 2 * EPI_WARPS);
        mbar_init(drain, 1);
        *s_abort = 0;
        fence_mbar_init();
        tma_prefetch_desc(&tmA);
        tma_prefetch_desc(&tmB);
    }
    if (warp == 2) gg::build_groups<P_BM>(p, lane, s_off, s_end, s_pre, s_mix);
    if (warp == 3) atom_block_prefix(p, lane, s_p128);
    __syncthreads();
    cluster_sync();
    if (warp == 1) {
        tmem_alloc_pair(s_tmem, TMEM_COLS);
        tmem_relinquish_pair();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();

    const uint32_t tmem_base = *s_tmem;
    const int total_tiles = s_pre[E];
    const int mix = *s_mix;
    const int KB = p.Kdim / BK;
    const size_t wrows_total = static_cast<size_t>(E) * p.w_rows;
    const int half_row = 128 * static_cast<int>(rank);

    if (warp == 0) {
        if (lane == 0) {
            const uint32_t full0 = mapa_shared(smem_u32(&full[0]), 0);
            int armed_phase[P_STAGES];
#pragma unroll
            for (int i = 0; i < P_STAGES; ++i) armed_phase[i] = -1;
            uint32_t stage = 0, phase = 0;
            bool ok = true;
            for (int k = 0, tile = gg::round_position(0, pair, npairs, mix); ok && tile < total_tiles;
                 ++k, tile = gg::round_position(k, pair, npairs, mix)) {
                const gg::Tile t =
                    gg::decode_tile<P_BM, P_BAND>(gg::visit_order(tile, total_tiles, mix), s_pre, s_off, s_end, E, NT);
                const int a_row = t.row0 + half_row;
                const size_t rb = static_cast<size_t>(s_p128[t.e] + 2 * t.m_blk) + rank;
                // weight rows of the tile: the two 128-row halves of the 256-row column block
                const int g0 = t.e * p.w_rows + t.n_blk * BN_ACC;
                const int g1 = g0 + BN_ACC / 2;
                const int brow = rank == 0 ? g0 : g1;
                const size_t wb0 = static_cast<size_t>(g0) / 128;
                const size_t wb1 = static_cast<size_t>(g1) < wrows_total ? static_cast<size_t>(g1) / 128 : wb0;
                for (int kb = 0; kb < KB; ++kb) {
                    if (!mbar_wait<true>(&empty[stage], phase ^ 1u, s_abort, p.status, p.timeout_ns)) {
                        ok = false;
                        break;
                    }
                    uint8_t *sa = smem + stage * P_STAGE;
                    const uint32_t bar = full0 + 8u * stage;
                    if (rank == 0) mbar_arrive_expect_tx(&full[stage], 2 * P_TX_BYTES);
                    tma_load_2d_pair(sa, &tmA, bar, kb * BK, a_row);
                    tma_load_2d_pair(sa + P_A_BYTES, &tmB, bar, kb * BK, brow);
                    // scale atoms as 2 rows of 256 bytes
                    tma_load_2d_pair(sa + P_SF_OFF, &tmSFA, bar, 0,
                                     static_cast<int>(2 * clamp_atom(rb * KB + kb, mp.sfa_atoms)));
                    tma_load_2d_pair(sa + P_SF_OFF + 512, &tmSFB, bar, 0,
                                     static_cast<int>(2 * clamp_atom(wb0 * KB + kb, mp.sfb_atoms)));
                    tma_load_2d_pair(sa + P_SF_OFF + 1024, &tmSFB, bar, 0,
                                     static_cast<int>(2 * clamp_atom(wb1 * KB + kb, mp.sfb_atoms)));
                    armed_phase[stage] = static_cast<int>(phase);
                    if (++stage == P_STAGES) { stage = 0; phase ^= 1u; }
                }
            }
            if (!ok) {
                volatile int no_abort = 0;
                if (rank == 0) {
                    for (int i = 0; i < P_STAGES; ++i)
                        if (armed_phase[i] >= 0)
                            mbar_wait<true>(&full[i], static_cast<uint32_t>(armed_phase[i]), &no_abort, p.status,
                                            p.timeout_ns);
                } else {
                    // this CTA's copies signal CTA 0's barriers: give them time to land
                    const uint64_t t0 = global_timer_ns();
                    while (global_timer_ns() - t0 < 200000ull) __nanosleep(1000);
                }
            }
        }
    } else if (warp == 1) {
        if (lane == 0 && rank == 0) {
            uint32_t stage = 0, phase = 0, acc_phase = 0;
            bool ok = true, issued = false;
            for (int k = 0, tile = gg::round_position(0, pair, npairs, mix); ok && tile < total_tiles;
                 ++k, tile = gg::round_position(k, pair, npairs, mix)) {
                if (!mbar_wait<true>(tempty, acc_phase ^ 1u, s_abort, p.status, p.timeout_ns)) { ok = false; break; }
                tc_fence_after();
                for (int kb = 0; kb < KB; ++kb) {
                    if (!mbar_wait<true>(&full[stage], phase, s_abort, p.status, p.timeout_ns)) { ok = false; break; }
                    tc_fence_after();
                    const uint32_t sa = smem_u32(smem + stage * P_STAGE);
                    const uint32_t t_sfa = tmem_base + SF_COL0 + stage * SF_SLOT;
                    const uint32_t t_sfb = t_sfa + 4;
                    tmem_cp_32x128b_warpx4_pair(t_sfa, smem_desc_rows16(sa + P_SF_OFF));
                    tmem_cp_32x128b_warpx4_pair(t_sfb, smem_desc_rows16(sa + P_SF_OFF + 512));
                    tmem_cp_32x128b_warpx4_pair(t_sfb + 4, smem_desc_rows16(sa + P_SF_OFF + 1024));
                    const uint64_t adesc = smem_desc_kmajor_sw128(sa);
                    const uint64_t bdesc = smem_desc_kmajor_sw128(sa + P_A_BYTES);
#pragma unroll
                    for (int j = 0; j < BK / UMMA_K; ++j)
                        umma_mxf8_pair(tmem_base, adesc + 2 * j, bdesc + 2 * j, idesc_mxf8(P_BM, BN_ACC, j), t_sfa,
                                       t_sfb, (kb | j) != 0);
                    issued = true;
                    umma_commit_pair_multicast(&empty[stage], 0x3);
                    if (++stage == P_STAGES) { stage = 0; phase ^= 1u; }
                }
                if (!ok) break;
                umma_commit_pair_multicast(tfull, 0x3);
                acc_phase ^= 1u;
            }
            if (!ok && issued) {
                volatile int no_abort = 0;
                umma_commit_pair_multicast(drain, 0x1);
                mbar_wait<true>(drain, 0, &no_abort, p.status, p.timeout_ns);
            }
        }
    } else {
        const int q = warp & 3;
        const int half = (warp - 2) / 4;
        static_assert(EPI_WARPS * EPI_BUF <= EPI_BYTES, "epilogue staging");
        uint8_t *stage_buf = smem + P_OFF_EPI + (warp - 2) * EPI_BUF;
        const uint32_t tempty0 = mapa_shared(smem_u32(tempty), 0);
        uint32_t acc_phase = 0;
        for (int k = 0, tile = gg::round_position(0, pair, npairs, mix); tile < total_tiles;
             ++k, tile = gg::round_position(k, pair, npairs, mix)) {
            gg::Tile t =
                gg::decode_tile<P_BM, P_BAND>(gg::visit_order(tile, total_tiles, mix), s_pre, s_off, s_end, E, NT);
            if (!mbar_wait<true>(tfull, acc_phase, s_abort, p.status, p.timeout_ns)) break;
            tc_fence_after();
            const uint32_t tbase = tmem_base + (static_cast<uint32_t>(q * 32) << 16);
            t.row0 += half_row;  // this CTA's 128 rows
            // hands CTA 0's accumulator back once this warp's TMEM loads have
            // completed (a hand-over with no data in memory: CTA-scope release)
            auto release = [&]() {
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive_cluster_cta(tempty0);
            };
            epilogue_plain_mx(p, &tmOut, stage_buf, tbase, t, q, half, lane, release);
            acc_phase ^= 1u;
        }
        if (lane == 0) bulk_wait_all();
    }

    tc_fence_before();
    __syncthreads();
    cluster_sync();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc_pair(tmem_base, TMEM_COLS);
    }
}

}  // namespace gmx

namespace {

cudaLaunchConfig_t mx_pair_config(int grid, cudaStream_t stream, cudaLaunchAttribute *attr) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid, 1, 1);
    cfg.blockDim = dim3(gmx::Roles<false>::THREADS, 1, 1);
    cfg.dynamicSmemBytes = gmx::P_SMEM_BYTES;
    cfg.stream = stream;
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cfg;
}

int mx_max_pairs() {
    cudaLaunchAttribute attr[1];
    cudaLaunchConfig_t cfg = mx_pair_config(2, nullptr, attr);
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, gmx::grouped_gemm_mx_pair_kernel, &cfg) != cudaSuccess) return 0;
    return n;
}

}  // namespace

cudaError_t grouped_gemm_mx_setup(GemmLaunch *cfg) {
    cudaError_t e;
    if ((e = cudaFuncSetAttribute(gmx::grouped_gemm_mx_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  gmx::SMEM_BYTES)) != cudaSuccess)
        return e;
    if ((e = cudaFuncSetAttribute(gmx::grouped_gemm_mx_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  gmx::SMEM_BYTES)) != cudaSuccess)
        return e;
    if ((e = cudaFuncSetAttribute(gmx::grouped_gemm_mx_pair_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  gmx::P_SMEM_BYTES)) != cudaSuccess)
        return e;
    // every pair of the persistent kernel must be resident at once
    cfg->mx_pairs = std::min(mx_max_pairs(), cfg->num_sms / 2);
    cudaGetLastError();  // a failed query leaves 0 pairs: single-CTA kernels only
    return cudaSuccess;
}

cudaError_t launch_grouped_gemm_mx(bool swiglu, const uint8_t *A, const uint8_t *sfa, size_t sfa_bytes, int TK,
                                   int Kdim, const uint8_t *W, const uint8_t *sfw, size_t sfw_bytes, int E, int n_out,
                                   const int32_t *offsets, void *out, uint8_t *sfo, size_t sfo_bytes,
                                   const GemmLaunch &cfg, int *status, uint64_t timeout_ns, cudaStream_t stream) {
    const int w_rows = swiglu ? 2 * n_out : n_out;
    CUtensorMap tmA, tmB, tmOut;
    if (!make_tmap_u8(&tmA, A, static_cast<uint64_t>(TK), static_cast<uint64_t>(Kdim), gmx::BM))
        return cudaErrorInvalidValue;
    if (!make_tmap_u8(&tmB, W, static_cast<uint64_t>(E) * w_rows, static_cast<uint64_t>(Kdim), 128))
        return cudaErrorInvalidValue;
    if (swiglu) {
        tmOut = tmA;  // unused: GEMM1 stores h codes directly
    } else if (!make_tmap(&tmOut, out, static_cast<uint64_t>(TK), static_cast<uint64_t>(n_out), 32, 32,
                          CU_TENSOR_MAP_SWIZZLE_64B)) {
        return cudaErrorInvalidValue;
    }
    gmx::MxParams mp = {};  // comb.counters == nullptr: no fused combine
    gg::Params &p = mp.g;
    p.offsets = offsets;
    p.E = E;
    p.TK = TK;
    p.Kdim = Kdim;
    p.n_out = n_out;
    p.w_rows = w_rows;
    p.NT = swiglu ? n_out / (gg::BN_ACC / 2) : (n_out + gg::BN_ACC - 1) / gg::BN_ACC;
    p.out = swiglu ? nullptr : static_cast<__nv_bfloat16 *>(out);
    p.status = status;
    p.timeout_ns = timeout_ns;
    mp.sfa = sfa;
    mp.sfa_atoms = sfa_bytes / 512;
    mp.sfb = sfw;
    mp.sfb_atoms = sfw_bytes / 512;
    mp.hq = swiglu ? static_cast<uint8_t *>(out) : nullptr;
    mp.sfh = reinterpret_cast<uint32_t *>(sfo);
    mp.sfh_atoms = sfo_bytes / 512;
    if (mp.sfa_atoms == 0 || mp.sfb_atoms == 0 || (swiglu && mp.sfh_atoms == 0)) return cudaErrorInvalidValue;
    // GEMM2 on CTA pairs where the pair kernel's groups are large and the
    // reduction short.  Measured on GB300 against the single-CTA kernel (µs):
    // skew-shaped GEMM2 (Kdim 1536) 942-947 against 999-1006, Qwen-shaped
    // (768) 210-211 against 222, but Mixtral-shaped (14336) 704-705 against
    // 655-657, and GEMM1 level or 4-5% slower on every shape.
    if (!swiglu && Kdim < 4096 && grouped_gemm_use_pair(TK, E) && cfg.mx_pairs > 0) {
        // the scale atoms as rows of 256 bytes, two per atom, for 2D pair copies
        CUtensorMap tmSFA, tmSFB;
        if (!make_tmap_2d(&tmSFA, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, sfa, 2 * mp.sfa_atoms, 256, 2, 256,
                          CU_TENSOR_MAP_SWIZZLE_NONE) ||
            !make_tmap_2d(&tmSFB, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, sfw, 2 * mp.sfb_atoms, 256, 2, 256,
                          CU_TENSOR_MAP_SWIZZLE_NONE))
            return cudaErrorInvalidValue;
        cudaLaunchAttribute attr[1];
        cudaLaunchConfig_t lc = mx_pair_config(2 * cfg.mx_pairs, stream, attr);
        return cudaLaunchKernelEx(&lc, gmx::grouped_gemm_mx_pair_kernel, tmA, tmB, tmOut, tmSFA, tmSFB, mp);
    }
    if (swiglu)
        gmx::grouped_gemm_mx_kernel<true><<<cfg.num_sms, gmx::Roles<true>::THREADS, gmx::SMEM_BYTES, stream>>>(
            tmA, tmB, tmOut, mp);
    else
        gmx::grouped_gemm_mx_kernel<false><<<cfg.num_sms, gmx::Roles<false>::THREADS, gmx::SMEM_BYTES, stream>>>(
            tmA, tmB, tmOut, mp);
    return cudaGetLastError();
}

}  // namespace moe
