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
// for every row r of expert e's group offsets[e]..offsets[e+1]-1.  With
// BT = true (plain GEMM only) the weights are read as stored [E, K, N], i.e.
// out[r, n] = bf16( sum_k A[r,k] W[e,k,n] ): the layer backward's dgrad
// products dy_perm.W2[e] and da.W1[e] without transposing the weights.  The
// B tile then comes as MN-major 64 x 64 boxes and the MMAs read it MN-major.
//
// Design (both variants):
//  * Persistent over a device-side tile list.  Every CTA reads offsets[] (E+1
//    ints) and builds the tile prefix itself, so the host never sees a count
//    and the launch is the same for every routing.
//  * Accumulator tile: rows x 256 columns.  GEMM1 stacks the gate rows
//    n0..n0+127 and the up rows f+n0..f+n0+127 of W1[e] into one 256-column
//    B operand, so one MMA yields both SwiGLU halves of 128 output columns;
//    GEMM2 uses 256 consecutive rows of W2[e].  A tile that runs past its
//    group reads neighbouring rows (or TMA zero fill); the epilogue masks them.
//  * Warp roles: warp 0 = TMA producer, warp 1 = tcgen05.mma issuer (and TMEM
//    owner), warps 2..5 = epilogue (TMEM -> registers -> bf16 -> shared memory
//    -> TMA store of full lines; masked row stores where a warp's 32 rows
//    cross the end of the group).
//  * Shared-memory ring of bf16 tiles (64-wide K slices, 128-byte swizzle)
//    with full/empty mbarriers; two 256-column fp32 accumulators in TMEM (512
//    columns) so the epilogue of tile i overlaps the mainloop of tile i+1
//    (except after a single-CTA tile of two row blocks, which uses both).
//  * Tiles are ordered expert by expert; inside an expert, bands of row
//    blocks sweep all column blocks, so concurrent CTAs share each weight tile
//    through L2 and the band's activation rows stay L2-resident.
//  * Every wait is bounded: on expiry the kernel records a timeout, drains its
//    copies and MMAs, frees TMEM and returns.
//
// Single-CTA variant (grouped_gemm_kernel), used when groups are small (a
// few row blocks): tiles of up to two 128-row blocks of one group.  A tile
// with more than 128 rows left in its group takes both row blocks: per K
// slice two M=128 x N=256 MMAs share the B tile, one into each TMEM
// accumulator, so the SM moves 64 KB per slice for twice the work (its
// epilogue then runs after the mainloop, both accumulators being in use).  A
// tile with at most 128 rows takes one accumulator, and consecutive such
// tiles alternate, so their epilogues overlap the next mainloop.  3 stages of
// 64 KB.
//
// Fused permute (GATHER, single-CTA GEMM1 only; "Optimization 2" of the page:
// a naive dispatch writes and reads the tokens again): two more warps copy
// the A rows straight from the token matrix x, row r being x[src_tok[r]],
// with 16-byte cp.async into the same 128-byte-swizzled layout TMA writes.
// Each gathering lane arrives on the stage's full barrier once its copies
// have landed, beside the producer's transaction count for B; the MMA thread
// fences the async proxy before the tensor core reads the rows.  The MMAs
// see the same operand bytes as after a separate permute, so h is identical.
//
// CTA-pair variant (grouped_gemm_pair_kernel): clusters of 2 CTAs on 2 SMs
// share a 256-row tile through cta_group::2 MMAs (M=256 x N=256).  Each CTA
// loads its 128 A rows and half of the B columns (GEMM1: CTA 0 the gate rows,
// CTA 1 the up rows), so each SM moves 32 KB per K slice instead of 48 KB and
// the ring holds 6 stages.  The even CTA issues the MMAs; both CTAs' copies
// signal its full barrier, its commits free both CTAs' stages, and both CTAs'
// epilogues release its accumulator.
#include <algorithm>
#include <atomic>

#include "gemm_common.cuh"
#include "kernels.h"
#include "ptx.cuh"
#include "tmap.h"

namespace moe {
namespace gg {

constexpr int BK = 64;
constexpr int UMMA_K = 16;
constexpr int TMEM_COLS = 2 * BN_ACC;
constexpr int THREADS = 192;
constexpr int BOX_ROWS = 128;  // every K-major TMA box is 128 rows x 64 bf16
constexpr int GATHER_WARPS = 2;  // fused permute: the last two warps copy the A rows
constexpr int GATHER_ROWS = 128 / GATHER_WARPS / 4;  // rows of a 128-row block per gathering lane
// Epilogue warps of the single-CTA kernel: two per TMEM lane quarter, each
// owning half of the tile's columns (GEMM1: 64 of its 128 h columns; the
// plain GEMMs: 128 of 256) and storing through one staging buffer.  Tiles of
// two row blocks use both accumulators, so their epilogue runs between
// mainloops and its length counts in full.
template <bool SWIGLU>
__host__ __device__ constexpr int epi_warps() {
    return 8;
}
template <bool SWIGLU, bool GATHER>
__host__ __device__ constexpr int threads_of() {
    return 64 + 32 * epi_warps<SWIGLU>() + (GATHER ? 32 * GATHER_WARPS : 0);
}
constexpr int BT_BOX = 64 * 64 * 2;  // MN-major B box: 64 K rows x 64 columns

// single-CTA variant
constexpr int BM = 128;        // rows of one MMA and one accumulator
constexpr int TILE_ROWS = 2 * BM;
constexpr int BAND = 8;        // tiles per raster band
constexpr int STAGES = 3;
constexpr int A_BLOCK = BM * BK * 2;
constexpr int A_BYTES = 2 * A_BLOCK;
constexpr int B_BYTES = BN_ACC * BK * 2;
constexpr int STAGE_BYTES = A_BYTES + B_BYTES;

// CTA-pair variant (per CTA)
constexpr int P_BM = 256;      // rows of a pair tile (128 per CTA)
constexpr int P_BAND = 8;
constexpr int P_STAGES = 6;
constexpr int P_A_BYTES = 128 * BK * 2;
constexpr int P_B_BYTES = 128 * BK * 2;
constexpr int P_STAGE_BYTES = P_A_BYTES + P_B_BYTES;

// shared-memory layout after the ring: barriers, TMEM address, abort flag,
// group bounds and tile prefix

template <int NSTAGES, int STAGE>
struct Layout {
    static constexpr int TQ = queue_slots(NSTAGES);
    static_assert(TQ >= NSTAGES + 4, "tile queue shorter than the pipeline's lead");
    static constexpr int OFF_EPI = NSTAGES * STAGE;  // 1024-aligned: the ring is whole KBs
    static constexpr int OFF_BARS = OFF_EPI + EPI_BYTES;
    // full, empty, tfull[2], tempty[2], drain, qfull[TQ]
    static constexpr int NUM_BARS = 2 * NSTAGES + 5 + TQ;
    static constexpr int OFF_TMEM = OFF_BARS + NUM_BARS * 8;
    static constexpr int OFF_ABORT = OFF_TMEM + 4;
    static constexpr int OFF_OFFS = OFF_ABORT + 4;
    static constexpr int OFF_ENDS = OFF_OFFS + MAX_E * 4;
    static constexpr int OFF_PRE = OFF_ENDS + MAX_E * 4;
    static constexpr int OFF_MIX = OFF_PRE + (MAX_E + 1) * 4;
    static constexpr int OFF_TQ = OFF_MIX + 4;  // tile-queue slots
    static constexpr int USED = OFF_TQ + TQ * 4;
    static constexpr int BYTES = USED + 1024;  // slack for 1024-byte alignment
};
using L1 = Layout<STAGES, STAGE_BYTES>;
using L2 = Layout<P_STAGES, P_STAGE_BYTES>;
constexpr int SMEM_BYTES = L1::BYTES;
constexpr int P_SMEM_BYTES = L2::BYTES;
static_assert(SMEM_BYTES <= 227 * 1024 && P_SMEM_BYTES <= 227 * 1024, "shared memory budget");
static_assert(B_BYTES == (BN_ACC / 64) * BT_BOX && P_B_BYTES == 2 * BT_BOX, "MN-major B boxes fill the B slot");

// Fused permute: the GATHER_ROWS rows of a 128-row block starting at row0
// that this lane copies, as pointers to their token rows in x, and a bit per
// row that lies inside the group.  Lane l of gathering warp gw copies 16-byte
// chunk l % 8 of rows (128 / GATHER_WARPS) gw + 4 i + l / 8, so eight lanes
// move one whole 128-byte line.  Rows past the group's end are not copied: row i of A reaches only
// row i of the accumulator, which the epilogue masks, so whatever their
// slot holds cannot reach a stored value.  A token index outside [0, T) is
// clamped (outside the contract, but never read out of bounds).
__device__ __forceinline__ uint32_t gather_sources(const Params &p, int row0, int grp_end, int gw, int lane,
                                                   const __nv_bfloat16 *(&src)[GATHER_ROWS]) {
    uint32_t valid = 0;
#pragma unroll
    for (int i = 0; i < GATHER_ROWS; ++i) {
        const int row = row0 + 4 * GATHER_ROWS * gw + 4 * i + (lane >> 3);
        const int r = min(row, grp_end - 1);
        const int tok = min(max(p.gather_src[r], 0), p.gather_T - 1);
        src[i] = p.gather_x + static_cast<size_t>(tok) * p.Kdim + (lane & 7) * 8;
        valid |= (row < grp_end ? 1u : 0u) << i;
    }
    return valid;
}
// Copies K slice kb of those rows into a 128-row A block `slot` (128-byte
// swizzle: 16-byte chunk j of row r sits at chunk j ^ (r % 8) of its line).
__device__ __forceinline__ void gather_block(uint8_t *slot, const __nv_bfloat16 *const (&src)[GATHER_ROWS],
                                             uint32_t valid, int gw, int kb, int lane) {
    const int j = lane & 7;
#pragma unroll
    for (int i = 0; i < GATHER_ROWS; ++i) {
        const int r = 4 * GATHER_ROWS * gw + 4 * i + (lane >> 3);
        if (valid & (1u << i)) cp_async_16(slot + r * (BK * 2) + ((j ^ (r & 7)) << 4), src[i] + kb * BK);
    }
}

// ======================================================================
// single-CTA variant
// ======================================================================
template <bool SWIGLU, bool BT, bool GATHER, bool DYN>
__global__ void __launch_bounds__(threads_of<SWIGLU, GATHER>(), 1)
grouped_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                    const __grid_constant__ CUtensorMap tmOut, const __grid_constant__ CUtensorMap tmPre,
                    const Params p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + L1::OFF_BARS);
    uint64_t *full = bars;
    uint64_t *empty = bars + STAGES;
    uint64_t *tfull = bars + 2 * STAGES;
    uint64_t *tempty = bars + 2 * STAGES + 2;
    uint64_t *drain = bars + 2 * STAGES + 4;
    constexpr int TQ = L1::TQ;
    uint64_t *qfull = bars + 2 * STAGES + 5;
    volatile int *s_tq = reinterpret_cast<volatile int *>(smem + L1::OFF_TQ);
    uint32_t *s_tmem = reinterpret_cast<uint32_t *>(smem + L1::OFF_TMEM);
    volatile int *s_abort = reinterpret_cast<volatile int *>(smem + L1::OFF_ABORT);
    int *s_off = reinterpret_cast<int *>(smem + L1::OFF_OFFS);
    int *s_end = reinterpret_cast<int *>(smem + L1::OFF_ENDS);
    int *s_pre = reinterpret_cast<int *>(smem + L1::OFF_PRE);
    int *s_mix = reinterpret_cast<int *>(smem + L1::OFF_MIX);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int E = p.E;
    const int NT = p.NT;

    static_assert(!GATHER || (SWIGLU && !BT), "the fused permute feeds GEMM1 only");
    static_assert(!(GATHER && DYN), "the fused-permute kernel keeps the static order");
    if (threadIdx.x == 0) {
        for (int i = 0; i < STAGES; ++i) {
            // fused permute: + one cp.async arrival per gathering lane
            mbar_init(&full[i], GATHER ? 1 + 32 * GATHER_WARPS : 1);
            mbar_init(&empty[i], 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&tfull[i], 1);
            mbar_init(&tempty[i], epi_warps<SWIGLU>());
        }
        mbar_init(drain, 1);
        for (int i = 0; i < TQ; ++i) mbar_init(&qfull[i], 1);
        *s_abort = 0;
        fence_mbar_init();
        tma_prefetch_desc(&tmA);
        tma_prefetch_desc(&tmB);
    }
    if (warp == 1) {
        tmem_alloc(s_tmem, TMEM_COLS);
        tmem_relinquish();
    }
    if (warp == 2) build_groups<TILE_ROWS>(p, lane, s_off, s_end, s_pre, s_mix);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();

    const uint32_t tmem_base = *s_tmem;
    const int total_tiles = s_pre[E];
    const int mix = *s_mix;
    const int KB = p.Kdim / BK;

    if (warp == 0) {
        if (lane == 0) {
            int armed_phase[STAGES];
#pragma unroll
            for (int i = 0; i < STAGES; ++i) armed_phase[i] = -1;
            uint32_t stage = 0, phase = 0;
            // Tiles are handed to the other roles one ahead of this thread's
            // own loads, and drawn two ahead: tile k + 1 is published when tile
            // k's loads begin, and the position of tile k + 2 drawn then, its
            // latency hidden behind those loads.
            auto publish = [&](int k, int tile) {
                s_tq[k % TQ] = tile;
                mbar_arrive(&qfull[k % TQ]);
                return true;
            };
            // (static order, !DYN: every role computes the positions itself)
            int cur = DYN ? first_position(p, blockIdx.x, gridDim.x, mix) : round_position(0, blockIdx.x, gridDim.x, mix);
            cur = cur < total_tiles ? cur : -1;
            int nxt = (DYN && cur >= 0) ? next_position(p, 0, blockIdx.x, gridDim.x, mix) : total_tiles;
            bool ok = DYN ? publish(0, cur) : true;
            for (int k = 0; ok && cur >= 0; ++k) {
                const int tile = cur;
                if (DYN) {
                    cur = nxt < total_tiles ? nxt : -1;
                    if (!publish(k + 1, cur)) { ok = false; break; }
                    if (cur >= 0) nxt = next_position(p, k + 1, blockIdx.x, gridDim.x, mix);
                } else {
                    cur = round_position(k + 1, blockIdx.x, gridDim.x, mix);
                    cur = cur < total_tiles ? cur : -1;
                }
                const Tile t =
                    decode_tile<TILE_ROWS, BAND>(visit_order(tile, total_tiles, mix), s_pre, s_off, s_end, E, NT);
                const bool two = t.grp_end - t.row0 > BM;  // both row blocks of the tile hold rows
                static_assert(!(SWIGLU && BT), "the transposed-weight form is a plain GEMM");
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
                    mbar_arrive_expect_tx(&full[stage], (GATHER ? 0 : (two ? 2 : 1) * A_BLOCK) + B_BYTES);
                    if (!GATHER) {
                        tma_load_2d(sa, &tmA, &full[stage], kb * BK, t.row0);
                        if (two) tma_load_2d(sa + A_BLOCK, &tmA, &full[stage], kb * BK, t.row0 + BM);
                    }
                    if (BT) {
                        // W[e] rows kb*64.., columns of the 256-wide block in 64-wide boxes
                        const int krow = t.e * p.Kdim + kb * BK;
#pragma unroll
                        for (int j = 0; j < BN_ACC / 64; ++j)
                            tma_load_2d(sb + j * BT_BOX, &tmB, &full[stage], t.n_blk * BN_ACC + 64 * j, krow);
                    } else {
                        tma_load_2d(sb, &tmB, &full[stage], kb * BK, brow0);
                        tma_load_2d(sb + B_BYTES / 2, &tmB, &full[stage], kb * BK, brow1);
                    }
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
            constexpr uint32_t idesc = idesc_bf16_f32(BM, BN_ACC, false, BT);
            // acc: the accumulator the next tile starts in; ph[i]: parity of
            // accumulator i's next use.  A two-block tile takes acc and acc ^ 1
            // (in that order, as the epilogue drains them) and leaves acc as it
            // is; a one-block tile takes acc and moves it on.
            uint32_t stage = 0, phase = 0, acc = 0;
            uint32_t ph[2] = {0u, 0u};
            bool ok = true;
            bool issued = false;
            for (int k = 0; ok; ++k) {
                int tile;
                if (DYN) {
                    if (!mbar_wait(&qfull[k % TQ], (k / TQ) & 1u, s_abort, p.status, p.timeout_ns)) { ok = false; break; }
                    tile = s_tq[k % TQ];
                    if (tile < 0) break;
                } else {
                    tile = round_position(k, blockIdx.x, gridDim.x, mix);
                    if (tile >= total_tiles) break;
                }
                const Tile t =
                    decode_tile<TILE_ROWS, BAND>(visit_order(tile, total_tiles, mix), s_pre, s_off, s_end, E, NT);
                const bool two = t.grp_end - t.row0 > BM;
                const uint32_t a0 = acc, a1 = acc ^ 1u;
                if (!mbar_wait(&tempty[a0], ph[a0] ^ 1u, s_abort, p.status, p.timeout_ns)) { ok = false; break; }
                if (two && !mbar_wait(&tempty[a1], ph[a1] ^ 1u, s_abort, p.status, p.timeout_ns)) { ok = false; break; }
                tc_fence_after();
                const uint32_t d0 = tmem_base + a0 * BN_ACC;
                const uint32_t d1 = tmem_base + a1 * BN_ACC;
                for (int kb = 0; kb < KB; ++kb) {
                    if (!mbar_wait(&full[stage], phase, s_abort, p.status, p.timeout_ns)) { ok = false; break; }
                    if (GATHER) fence_proxy_async_smem();  // cp.async rows -> tensor-core reads
                    tc_fence_after();
                    const uint32_t sa = smem_u32(smem + stage * STAGE_BYTES);
                    const uint64_t adesc0 = smem_desc_kmajor_sw128(sa);
                    const uint64_t adesc1 = smem_desc_kmajor_sw128(sa + A_BLOCK);
                    const uint64_t bdesc = BT ? smem_desc_mnmajor_sw128(sa + A_BYTES, BT_BOX)
                                              : smem_desc_kmajor_sw128(sa + A_BYTES);
#pragma unroll
                    for (int j = 0; j < BK / UMMA_K; ++j) {
                        // advance 16 elements along K: 32 bytes inside a K-major swizzled
                        // row, 16 rows (2048 bytes) of an MN-major box
                        const uint64_t bj = bdesc + (BT ? 128 : 2) * j;
                        umma_bf16(d0, adesc0 + 2 * j, bj, idesc, (kb | j) != 0);
                        if (two) umma_bf16(d1, adesc1 + 2 * j, bj, idesc, (kb | j) != 0);
                    }
                    issued = true;
                    umma_commit(&empty[stage]);
                    if (++stage == STAGES) { stage = 0; phase ^= 1u; }
                }
                if (!ok) break;
                umma_commit(&tfull[a0]);
                ph[a0] ^= 1u;
                if (two) {
                    umma_commit(&tfull[a1]);
                    ph[a1] ^= 1u;
                } else {
                    acc = a1;
                }
            }
            if (!ok && issued) {
                volatile int no_abort = 0;
                umma_commit(drain);
                mbar_wait(drain, 0, &no_abort, p.status, p.timeout_ns);
            }
        }
    } else if (GATHER && warp >= 2 + epi_warps<SWIGLU>()) {
        // fused permute: this warp's 32 rows of each A block of every stage
        const int gw = warp - 2 - epi_warps<SWIGLU>();
        uint32_t stage = 0, phase = 0;
        bool ok = true;
        for (int k = 0; ok; ++k) {
            int tile;
            if (DYN) {
                if (!mbar_wait(&qfull[k % TQ], (k / TQ) & 1u, s_abort, p.status, p.timeout_ns)) break;
                tile = s_tq[k % TQ];
                if (tile < 0) break;
            } else {
                tile = round_position(k, blockIdx.x, gridDim.x, mix);
                if (tile >= total_tiles) break;
            }
            const Tile t =
                decode_tile<TILE_ROWS, BAND>(visit_order(tile, total_tiles, mix), s_pre, s_off, s_end, E, NT);
            const bool two = t.grp_end - t.row0 > BM;
            const __nv_bfloat16 *src0[GATHER_ROWS], *src1[GATHER_ROWS];
            const uint32_t v0 = gather_sources(p, t.row0, t.grp_end, gw, lane, src0);
            const uint32_t v1 = two ? gather_sources(p, t.row0 + BM, t.grp_end, gw, lane, src1) : 0u;
            for (int kb = 0; kb < KB; ++kb) {
                int got = 1;
                if (lane == 0) got = mbar_wait(&empty[stage], phase ^ 1u, s_abort, p.status, p.timeout_ns) ? 1 : 0;
                if (!__shfl_sync(0xffffffffu, got, 0)) { ok = false; break; }
                uint8_t *sa = smem + stage * STAGE_BYTES;
                if (v0) gather_block(sa, src0, v0, gw, kb, lane);
                if (v1) gather_block(sa + A_BLOCK, src1, v1, gw, kb, lane);
                cp_async_arrive_noinc(&full[stage]);
                if (++stage == STAGES) { stage = 0; phase ^= 1u; }
            }
        }
        cp_async_wait_all();  // this lane's copies have landed before the CTA's shared memory goes away
    } else {
        const int q = warp & 3;  // TMEM lane quarter this warp may access
        constexpr int NBUF = 1;  // staging buffers per epilogue warp
        static_assert(epi_warps<SWIGLU>() * NBUF * EPI_BUF == EPI_BYTES, "epilogue staging");
        // the two warps of a lane quarter split the tile's columns
        constexpr int SHARE = (SWIGLU ? BN_ACC / 2 : BN_ACC) / 2;
        const int c_begin = ((warp - 2) >> 2) * SHARE;
        const int c_end = c_begin + SHARE;
        uint8_t *stage = smem + L1::OFF_EPI + (warp - 2) * NBUF * EPI_BUF;
        uint32_t sbuf = 0;
        uint32_t acc = 0;
        uint32_t ph[2] = {0u, 0u};  // the MMA thread's accumulator order, mirrored
        bool ok = true;
        for (int k = 0; ok; ++k) {
            int tile;
            if (DYN) {
                if (!mbar_wait(&qfull[k % TQ], (k / TQ) & 1u, s_abort, p.status, p.timeout_ns)) break;
                tile = s_tq[k % TQ];
                if (tile < 0) break;
            } else {
                tile = round_position(k, blockIdx.x, gridDim.x, mix);
                if (tile >= total_tiles) break;
            }
            const Tile t =
                decode_tile<TILE_ROWS, BAND>(visit_order(tile, total_tiles, mix), s_pre, s_off, s_end, E, NT);
            const int nblk = t.grp_end - t.row0 > BM ? 2 : 1;
            if (SWIGLU && p.preact == nullptr && nblk == 2 && t.row0 + q * 32 < t.grp_end) {
                // GEMM1, two blocks: both accumulators go back before any store
                const uint32_t a0 = acc, a1 = acc ^ 1u;
                if (!mbar_wait(&tfull[a0], ph[a0], s_abort, p.status, p.timeout_ns)) break;
                tc_fence_after();
                const uint32_t tq = tmem_base + (static_cast<uint32_t>(q * 32) << 16);
                auto release_of = [&](uint32_t a) {
                    return [&, a]() {
                        tc_fence_before();
                        __syncwarp();
                        if (lane == 0) mbar_arrive(&tempty[a]);
                    };
                };
                auto wait1 = [&]() {
                    if (!mbar_wait(&tfull[a1], ph[a1], s_abort, p.status, p.timeout_ns)) return false;
                    tc_fence_after();
                    return true;
                };
                if (!epilogue_swiglu_early2(p, &tmOut, stage, sbuf, tq + a0 * BN_ACC, tq + a1 * BN_ACC, t.n_blk,
                                            t.row0 + q * 32, lane, t.grp_end, c_begin, wait1, release_of(a0),
                                            release_of(a1)))
                    break;
                ph[a0] ^= 1u;
                ph[a1] ^= 1u;
                continue;  // a tile of two blocks leaves acc as it is
            }
            for (int b = 0; b < nblk; ++b) {
                const uint32_t a = acc ^ static_cast<uint32_t>(b);
                if (!mbar_wait(&tfull[a], ph[a], s_abort, p.status, p.timeout_ns)) { ok = false; break; }
                tc_fence_after();
                const uint32_t tbase = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + a * BN_ACC;
                // hands accumulator a back to the MMA thread (after this warp's TMEM loads)
                auto release = [&]() {
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&tempty[a]);
                };
                if (SWIGLU && p.preact == nullptr) {
                    // GEMM1: the accumulator goes back once its values are loaded
                    epilogue_swiglu_early(p, &tmOut, stage, sbuf, tbase, t.n_blk, t.row0 + b * BM + q * 32, lane,
                                          t.grp_end, c_begin, release);
                } else {
                    epilogue_tile<SWIGLU, NBUF>(p, &tmOut, &tmPre, stage, sbuf, tbase, t.n_blk,
                                                t.row0 + b * BM + q * 32, lane, t.grp_end, c_begin, c_end);
                    release();
                }
                ph[a] ^= 1u;
            }
            if (nblk == 1) acc ^= 1u;
        }
        if (lane == 0) bulk_wait_all();  // stores done before the CTA's shared memory goes away
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem_base, TMEM_COLS);
    }
    if (threadIdx.x == 0) sched_retire(p);
}

// ======================================================================
// CTA-pair variant (cluster of 2)
// ======================================================================
template <bool SWIGLU, bool BT, bool DYN>
__global__ void __launch_bounds__(THREADS, 1)
grouped_gemm_pair_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                         const __grid_constant__ CUtensorMap tmOut, const __grid_constant__ CUtensorMap tmPre,
                         const Params p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + L2::OFF_BARS);
    uint64_t *full = bars;                       // used in CTA 0 only
    uint64_t *empty = bars + P_STAGES;           // both CTAs
    uint64_t *tfull = bars + 2 * P_STAGES;       // both CTAs
    uint64_t *tempty = bars + 2 * P_STAGES + 2;  // CTA 0 only: 4 warps x 2 CTAs arrive
    uint64_t *drain = bars + 2 * P_STAGES + 4;
    constexpr int TQ = L2::TQ;
    uint64_t *qfull = bars + 2 * P_STAGES + 5;   // both CTAs
    volatile int *s_tq = reinterpret_cast<volatile int *>(smem + L2::OFF_TQ);
    uint32_t *s_tmem = reinterpret_cast<uint32_t *>(smem + L2::OFF_TMEM);
    volatile int *s_abort = reinterpret_cast<volatile int *>(smem + L2::OFF_ABORT);
    int *s_off = reinterpret_cast<int *>(smem + L2::OFF_OFFS);
    int *s_end = reinterpret_cast<int *>(smem + L2::OFF_ENDS);
    int *s_pre = reinterpret_cast<int *>(smem + L2::OFF_PRE);
    int *s_mix = reinterpret_cast<int *>(smem + L2::OFF_MIX);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int E = p.E;
    const int NT = p.NT;
    const uint32_t rank = cluster_ctarank();  // 0 issues the MMAs
    const int pair = blockIdx.x >> 1;
    const int npairs = gridDim.x >> 1;

    if (threadIdx.x == 0) {
        for (int i = 0; i < P_STAGES; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&tfull[i], 1);
            mbar_init(&tempty[i], 8);
        }
        mbar_init(drain, 1);
        for (int i = 0; i < TQ; ++i) mbar_init(&qfull[i], 1);
        *s_abort = 0;
        fence_mbar_init();
        tma_prefetch_desc(&tmA);
        tma_prefetch_desc(&tmB);
    }
    if (warp == 2) build_groups<P_BM>(p, lane, s_off, s_end, s_pre, s_mix);
    __syncthreads();
    // both CTAs' barriers are initialised (and both CTAs are running) before
    // any copy, commit or arrive crosses the pair, and before the collective
    // TMEM allocation
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

    if (warp == 0) {
        if (lane == 0) {
            // both CTAs' copies signal CTA 0's full barriers
            const uint32_t full0 = mapa_shared(smem_u32(&full[0]), 0);
            int armed_phase[P_STAGES];
#pragma unroll
            for (int i = 0; i < P_STAGES; ++i) armed_phase[i] = -1;
            uint32_t stage = 0, phase = 0;
            bool ok = true;
            // CTA 0 decides the pair's tiles and writes each into both CTAs' queue
            const uint32_t tq_peer = mapa_shared(smem_u32(const_cast<int *>(s_tq)), 1);
            const uint32_t qfull_peer = mapa_shared(smem_u32(&qfull[0]), 1);
            // DYN: CTA 0 publishes tile k + 1 to both CTAs when its loads of
            // tile k begin, and draws the position of tile k + 2 then (see the
            // single-CTA kernel), so CTA 1 learns each tile well before its
            // stages free up.  Otherwise both CTAs follow the static order.
            auto publish = [&](int k, int tile) {
                s_tq[k % TQ] = tile;
                mbar_arrive(&qfull[k % TQ]);
                send_to_peer(tq_peer + 4u * (k % TQ), tile, qfull_peer + 8u * (k % TQ));
                return true;
            };
            int cur = -1, nxt = total_tiles;
            if (DYN && rank == 0) {
                cur = first_position(p, pair, npairs, mix);
                cur = cur < total_tiles ? cur : -1;
                nxt = cur >= 0 ? next_position(p, 0, pair, npairs, mix) : total_tiles;
                ok = publish(0, cur);
            }
            for (int k = 0; ok; ++k) {
                int tile;
                if (!DYN) {
                    // static order: both CTAs compute the pair's positions themselves
                    tile = round_position(k, pair, npairs, mix);
                    if (tile >= total_tiles) break;
                } else if (rank == 0) {
                    tile = cur;
                    if (tile < 0) break;
                    cur = nxt < total_tiles ? nxt : -1;
                    if (!publish(k + 1, cur)) { ok = false; break; }
                    if (cur >= 0) nxt = next_position(p, k + 1, pair, npairs, mix);
                } else {
                    if (!mbar_wait<true>(&qfull[k % TQ], (k / TQ) & 1u, s_abort, p.status, p.timeout_ns)) {
                        ok = false;
                        break;
                    }
                    tile = s_tq[k % TQ];
                    if (tile < 0) break;
                }
                const Tile t = decode_tile<P_BM, P_BAND>(visit_order(tile, total_tiles, mix), s_pre, s_off, s_end, E, NT);
                const int a_row = t.row0 + 128 * static_cast<int>(rank);
                // GEMM1: CTA 0 loads the gate rows, CTA 1 the up rows (f rows later);
                // GEMM2: CTA r loads rows 128r..128r+127 of the 256-row column block
                const int brow = SWIGLU ? t.e * p.w_rows + static_cast<int>(rank) * p.n_out + t.n_blk * (BN_ACC / 2)
                                        : t.e * p.w_rows + t.n_blk * BN_ACC + static_cast<int>(rank) * (BN_ACC / 2);
                for (int kb = 0; kb < KB; ++kb) {
                    if (!mbar_wait<true>(&empty[stage], phase ^ 1u, s_abort, p.status, p.timeout_ns)) { ok = false; break; }
                    uint8_t *sa = smem + stage * P_STAGE_BYTES;
                    uint8_t *sb = sa + P_A_BYTES;
                    if (rank == 0) mbar_arrive_expect_tx(&full[stage], 2 * P_STAGE_BYTES);
                    tma_load_2d_pair(sa, &tmA, full0 + 8u * stage, kb * BK, a_row);
                    if (BT) {
                        // CTA r: columns 128r..128r+127 of the 256-wide block, two 64-wide boxes
                        const int krow = t.e * p.Kdim + kb * BK;
                        const int n0 = t.n_blk * BN_ACC + static_cast<int>(rank) * (BN_ACC / 2);
                        tma_load_2d_pair(sb, &tmB, full0 + 8u * stage, n0, krow);
                        tma_load_2d_pair(sb + BT_BOX, &tmB, full0 + 8u * stage, n0 + 64, krow);
                    } else {
                        tma_load_2d_pair(sb, &tmB, full0 + 8u * stage, kb * BK, brow);
                    }
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
            constexpr uint32_t idesc = idesc_bf16_f32(P_BM, BN_ACC, false, BT);
            uint32_t stage = 0, phase = 0, acc = 0, acc_phase = 0;
            bool ok = true;
            bool issued = false;
            for (int k = 0; ok; ++k) {
                if (DYN) {
                    if (!mbar_wait(&qfull[k % TQ], (k / TQ) & 1u, s_abort, p.status, p.timeout_ns)) { ok = false; break; }
                    if (s_tq[k % TQ] < 0) break;
                } else if (round_position(k, pair, npairs, mix) >= total_tiles) {
                    break;
                }
                if (!mbar_wait<true>(&tempty[acc], acc_phase ^ 1u, s_abort, p.status, p.timeout_ns)) { ok = false; break; }
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + acc * BN_ACC;
                for (int kb = 0; kb < KB; ++kb) {
                    if (!mbar_wait<true>(&full[stage], phase, s_abort, p.status, p.timeout_ns)) { ok = false; break; }
                    tc_fence_after();
                    const uint32_t sa = smem_u32(smem + stage * P_STAGE_BYTES);
                    const uint64_t adesc = smem_desc_kmajor_sw128(sa);
                    const uint64_t bdesc = BT ? smem_desc_mnmajor_sw128(sa + P_A_BYTES, BT_BOX)
                                              : smem_desc_kmajor_sw128(sa + P_A_BYTES);
#pragma unroll
                    for (int j = 0; j < BK / UMMA_K; ++j)
                        umma_bf16_pair(d_tmem, adesc + 2 * j, bdesc + (BT ? 128 : 2) * j, idesc, (kb | j) != 0);
                    issued = true;
                    umma_commit_pair_multicast(&empty[stage], 0x3);
                    if (++stage == P_STAGES) { stage = 0; phase ^= 1u; }
                }
                if (!ok) break;
                umma_commit_pair_multicast(&tfull[acc], 0x3);
                acc ^= 1u;
                if (acc == 0) acc_phase ^= 1u;
            }
            if (!ok && issued) {
                volatile int no_abort = 0;
                umma_commit_pair_multicast(drain, 0x1);
                mbar_wait<true>(drain, 0, &no_abort, p.status, p.timeout_ns);
            }
        }
    } else {
        const int q = warp & 3;
        uint8_t *stage = smem + L2::OFF_EPI + (warp - 2) * 2 * EPI_BUF;
        uint32_t sbuf = 0;
        const uint32_t tempty0 = mapa_shared(smem_u32(&tempty[0]), 0);
        uint32_t acc = 0, acc_phase = 0;
        for (int k = 0;; ++k) {
            int tile;
            if (DYN) {
                if (!mbar_wait<true>(&qfull[k % TQ], (k / TQ) & 1u, s_abort, p.status, p.timeout_ns)) break;
                tile = s_tq[k % TQ];
                if (tile < 0) break;
            } else {
                tile = round_position(k, pair, npairs, mix);
                if (tile >= total_tiles) break;
            }
            const Tile t = decode_tile<P_BM, P_BAND>(visit_order(tile, total_tiles, mix), s_pre, s_off, s_end, E, NT);
            if (!mbar_wait<true>(&tfull[acc], acc_phase, s_abort, p.status, p.timeout_ns)) break;
            tc_fence_after();
            const uint32_t tbase = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + acc * BN_ACC;
            const int wrow0 = t.row0 + 128 * static_cast<int>(rank) + q * 32;
            epilogue_tile<SWIGLU>(p, &tmOut, &tmPre, stage, sbuf, tbase, t.n_blk, wrow0, lane, t.grp_end);
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive_cluster_cta(tempty0 + 8u * acc);
            acc ^= 1u;
            if (acc == 0) acc_phase ^= 1u;
        }
        if (lane == 0) bulk_wait_all();
    }

    tc_fence_before();
    __syncthreads();
    // neither CTA leaves (or frees TMEM) while its peer may still touch its
    // shared memory or tensor memory
    cluster_sync();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc_pair(tmem_base, TMEM_COLS);
    }
    if (threadIdx.x == 0) sched_retire(p);
}

}  // namespace gg

// ------------------------------------------------------------------ host side
namespace {

// Counters of the dynamic tile order (Params::sched), two ints per slot, in a
// library-owned table on every device that loads the library (zero at load;
// each launch leaves its slot at zero).  An eager launch takes the next slot
// of a ring of kEagerSlots, so only kernels of launches kEagerSlots apart
// could share one, and those are never in flight together.  A launch being
// captured into a CUDA graph takes a slot of its own that no later launch
// reuses: every replay of the graph uses it, and replays of one graph run one
// after another.  Once the captured slots are used up, captured launches fall
// back to the static order (sched == nullptr).
constexpr int kEagerSlots = 2048;
constexpr int kCapturedSlots = 14336;
__device__ int g_sched_slots[2 * (kEagerSlots + kCapturedSlots)];
constexpr int kMaxDev = 64;
std::atomic<uint32_t> g_eager_next[kMaxDev];
std::atomic<uint32_t> g_captured_next[kMaxDev];

int *sched_slot(const GemmLaunch &cfg, cudaStream_t stream) {
    if (cfg.sched_base == nullptr || cfg.device < 0 || cfg.device >= kMaxDev) return nullptr;
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(stream, &cs) != cudaSuccess) {
        cudaGetLastError();
        return nullptr;
    }
    if (cs == cudaStreamCaptureStatusActive) {
        const uint32_t i = g_captured_next[cfg.device].fetch_add(1, std::memory_order_relaxed);
        if (i >= static_cast<uint32_t>(kCapturedSlots)) return nullptr;
        return cfg.sched_base + 2 * (kEagerSlots + static_cast<int>(i));
    }
    const uint32_t i = g_eager_next[cfg.device].fetch_add(1, std::memory_order_relaxed) % kEagerSlots;
    return cfg.sched_base + 2 * static_cast<int>(i);
}

template <bool SWIGLU, bool BT, bool DYN>
cudaError_t launch_pair(const CUtensorMap &tmA, const CUtensorMap &tmB, const CUtensorMap &tmOut,
                        const CUtensorMap &tmPre, const gg::Params &p, int grid, cudaStream_t stream) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid, 1, 1);
    cfg.blockDim = dim3(gg::THREADS, 1, 1);
    cfg.dynamicSmemBytes = gg::P_SMEM_BYTES;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, gg::grouped_gemm_pair_kernel<SWIGLU, BT, DYN>, tmA, tmB, tmOut, tmPre, p);
}

template <bool SWIGLU>
int max_pairs() {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2, 1, 1);
    cfg.blockDim = dim3(gg::THREADS, 1, 1);
    cfg.dynamicSmemBytes = gg::P_SMEM_BYTES;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, gg::grouped_gemm_pair_kernel<SWIGLU, false, true>, &cfg) != cudaSuccess)
        return 0;
    return n;
}

}  // namespace

bool grouped_gemm_use_pair(int TK, int E) {
    // a 256-row pair tile pays off once the average group holds a few of them
    return static_cast<int64_t>(TK) >= static_cast<int64_t>(E) * 384;
}

bool grouped_gemm1_prefers_gather(int TK, int E, int f) {
    // The fused permute runs on the single-CTA kernel.  Where that kernel is
    // chosen anyway, the fusion only removes the permute's x_perm round trip.
    // Where the pair kernel would run, GEMM1 loses about 5-9% to the
    // single-CTA kernel, while the permute's share of GEMM1's time falls as
    // 1/f (its bytes are 4*TK*d, GEMM1's work 4*TK*d*f): measured on GB300,
    // the fusion wins at f = 768 and 1536 and loses at f = 14336.
    return !grouped_gemm_use_pair(TK, E) || f <= 4096;
}

cudaError_t launch_grouped_gemm(bool swiglu, const void *A, int TK, int Kdim, const void *W, int E, int n_out,
                                const int32_t *offsets, void *out, const GemmLaunch &cfg, int *status,
                                uint64_t timeout_ns, cudaStream_t stream, const CombineArgs *comb, bool b_trans,
                                void *preact, const GatherArgs *gather) {
    CUtensorMap tmA, tmB;
    if (b_trans && (swiglu || comb)) return cudaErrorInvalidValue;
    if (preact && !swiglu) return cudaErrorInvalidValue;
    if (gather && (!swiglu || b_trans || comb || gather->T < 1)) return cudaErrorInvalidValue;
    const int w_rows = swiglu ? 2 * n_out : n_out;
    // with the fused permute A is the token matrix [T, Kdim]; its rows are
    // copied by the gather warps and the map goes unused
    const uint64_t a_rows = gather ? static_cast<uint64_t>(gather->T) : static_cast<uint64_t>(TK);
    if (!make_tmap(&tmA, A, a_rows, static_cast<uint64_t>(Kdim), gg::BOX_ROWS, gg::BK))
        return cudaErrorInvalidValue;
    if (b_trans) {
        // W as stored: [E * Kdim, n_out], 64 x 64 boxes
        if (!make_tmap(&tmB, W, static_cast<uint64_t>(E) * Kdim, static_cast<uint64_t>(n_out), 64, 64))
            return cudaErrorInvalidValue;
    } else if (!make_tmap(&tmB, W, static_cast<uint64_t>(E) * w_rows, static_cast<uint64_t>(Kdim), gg::BOX_ROWS,
                          gg::BK)) {
        return cudaErrorInvalidValue;
    }
    CUtensorMap tmOut, tmPre;
    if (!make_tmap(&tmOut, out, static_cast<uint64_t>(TK), static_cast<uint64_t>(n_out), 32, 32,
                   CU_TENSOR_MAP_SWIZZLE_64B))
        return cudaErrorInvalidValue;
    // the pre-activations [TK, 2 n_out] (GEMM1 only); otherwise an unused copy of tmOut
    if (preact) {
        if (!make_tmap(&tmPre, preact, static_cast<uint64_t>(TK), 2 * static_cast<uint64_t>(n_out), 32, 32,
                       CU_TENSOR_MAP_SWIZZLE_64B))
            return cudaErrorInvalidValue;
    } else {
        tmPre = tmOut;
    }
    gg::Params p = {};
    if (comb && !swiglu) {
        p.comb.src_tok = comb->src_tok;
        p.comb.row_of = comb->row_of;
        p.comb.topk_w = comb->topk_w;
        p.comb.T = comb->T;
        p.comb.K = comb->K;
        p.comb.nb = (n_out + gg::BN_ACC - 1) / gg::BN_ACC;
        p.comb.counters = comb->counters;
        p.comb.y = static_cast<__nv_bfloat16 *>(comb->y);
    }
    p.offsets = offsets;
    p.E = E;
    p.TK = TK;
    p.Kdim = Kdim;
    p.n_out = n_out;
    p.w_rows = w_rows;
    p.NT = swiglu ? (n_out + gg::BN_ACC / 2 - 1) / (gg::BN_ACC / 2) : (n_out + gg::BN_ACC - 1) / gg::BN_ACC;
    p.out = static_cast<__nv_bfloat16 *>(out);
    p.preact = static_cast<__nv_bfloat16 *>(preact);
    p.status = status;
    p.timeout_ns = timeout_ns;
    const dim3 grid(cfg.num_sms);
    const int pairs = swiglu ? cfg.pairs_swiglu : cfg.pairs_plain;
    const bool use_pair = !gather && grouped_gemm_use_pair(TK, E) && pairs > 0;
    // Dynamic tile order (measured on GB300 against the static order):
    //  - the CTA-pair kernel with long reductions (Kdim >= 4096): 2-5% faster
    //    and half the DRAM traffic on the Mixtral shape (GEMM1 3.2 GB per
    //    launch against 2.48 GB algorithmic, from 6.1 GB);
    //  - the CTA-pair kernel with short ones: 5-10% slower (the Qwen- and
    //    skew-shaped GEMM2s, Kdim = 768 and 1536): per tile, CTA 0 must hand
    //    the tile to CTA 1, which the static order does not need;
    //  - the single-CTA kernel: 5% faster on the DSv3-shaped GEMM2, but 5%
    //    slower on its fused-permute GEMM1, which keeps the static order.
    p.sched = (gather || (use_pair && Kdim < 4096)) ? nullptr : sched_slot(cfg, stream);
    if (gather) {
        // the fused permute runs on the single-CTA kernel for every shape
        p.gather_src = gather->src_tok;
        p.gather_x = static_cast<const __nv_bfloat16 *>(A);
        p.gather_T = gather->T;
        gg::grouped_gemm_kernel<true, false, true, false>
            <<<grid, gg::threads_of<true, true>(), gg::SMEM_BYTES, stream>>>(tmA, tmB, tmOut, tmPre, p);
        return cudaGetLastError();
    }
    if (use_pair) {
        const int g = 2 * pairs;
        if (p.sched)
            return swiglu    ? launch_pair<true, false, true>(tmA, tmB, tmOut, tmPre, p, g, stream)
                   : b_trans ? launch_pair<false, true, true>(tmA, tmB, tmOut, tmPre, p, g, stream)
                             : launch_pair<false, false, true>(tmA, tmB, tmOut, tmPre, p, g, stream);
        return swiglu    ? launch_pair<true, false, false>(tmA, tmB, tmOut, tmPre, p, g, stream)
               : b_trans ? launch_pair<false, true, false>(tmA, tmB, tmOut, tmPre, p, g, stream)
                         : launch_pair<false, false, false>(tmA, tmB, tmOut, tmPre, p, g, stream);
    }
    auto single = [&](auto kernel) {
        kernel<<<grid, swiglu ? gg::threads_of<true, false>() : gg::threads_of<false, false>(), gg::SMEM_BYTES,
                 stream>>>(tmA, tmB, tmOut, tmPre, p);
        return cudaGetLastError();
    };
    if (p.sched)
        return swiglu    ? single(gg::grouped_gemm_kernel<true, false, false, true>)
               : b_trans ? single(gg::grouped_gemm_kernel<false, true, false, true>)
                         : single(gg::grouped_gemm_kernel<false, false, false, true>);
    return swiglu    ? single(gg::grouped_gemm_kernel<true, false, false, false>)
           : b_trans ? single(gg::grouped_gemm_kernel<false, true, false, false>)
                     : single(gg::grouped_gemm_kernel<false, false, false, false>);
}

cudaError_t grouped_gemm_setup(int num_sms, GemmLaunch *cfg) {
    cudaError_t e;
    const void *single[7] = {reinterpret_cast<const void *>(gg::grouped_gemm_kernel<true, false, false, false>),
                             reinterpret_cast<const void *>(gg::grouped_gemm_kernel<false, false, false, false>),
                             reinterpret_cast<const void *>(gg::grouped_gemm_kernel<false, true, false, false>),
                             reinterpret_cast<const void *>(gg::grouped_gemm_kernel<true, false, false, true>),
                             reinterpret_cast<const void *>(gg::grouped_gemm_kernel<false, false, false, true>),
                             reinterpret_cast<const void *>(gg::grouped_gemm_kernel<false, true, false, true>),
                             reinterpret_cast<const void *>(gg::grouped_gemm_kernel<true, false, true, false>)};
    const void *pair[6] = {reinterpret_cast<const void *>(gg::grouped_gemm_pair_kernel<true, false, false>),
                           reinterpret_cast<const void *>(gg::grouped_gemm_pair_kernel<false, false, false>),
                           reinterpret_cast<const void *>(gg::grouped_gemm_pair_kernel<false, true, false>),
                           reinterpret_cast<const void *>(gg::grouped_gemm_pair_kernel<true, false, true>),
                           reinterpret_cast<const void *>(gg::grouped_gemm_pair_kernel<false, false, true>),
                           reinterpret_cast<const void *>(gg::grouped_gemm_pair_kernel<false, true, true>)};
    for (int i = 0; i < 7; ++i)
        if ((e = cudaFuncSetAttribute(single[i], cudaFuncAttributeMaxDynamicSharedMemorySize, gg::SMEM_BYTES)) !=
            cudaSuccess)
            return e;
    for (int i = 0; i < 6; ++i)
        if ((e = cudaFuncSetAttribute(pair[i], cudaFuncAttributeMaxDynamicSharedMemorySize, gg::P_SMEM_BYTES)) !=
            cudaSuccess)
            return e;
    cfg->num_sms = num_sms;
    if ((e = cudaGetDevice(&cfg->device)) != cudaSuccess) return e;
    if ((e = cudaGetSymbolAddress(reinterpret_cast<void **>(&cfg->sched_base), g_sched_slots)) != cudaSuccess)
        return e;
    // every pair must be resident at once (the kernel is persistent): never
    // launch more pairs than fit, nor more CTAs than SMs
    cfg->pairs_swiglu = std::min(max_pairs<true>(), num_sms / 2);
    // (the transposed-weight form has the plain form's resources)
    cfg->pairs_plain = std::min(max_pairs<false>(), num_sms / 2);
    cudaGetLastError();  // a failed occupancy query leaves pairs = 0: single-CTA kernels only
    return cudaSuccess;
}

}  // namespace moe
