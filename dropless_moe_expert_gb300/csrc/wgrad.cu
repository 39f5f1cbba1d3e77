// Weight gradients of the grouped GEMMs: for every expert e,
//     D[e] = A[group e]^T . B[group e]    (M x N, fp32)
// i.e. dW2[e] = dy_perm[e]^T h[e] (M = d, N = f) and dW1[e] = da[e]^T x_perm[e]
// (M = 2f, N = d): a sum over the expert's own rows, a ragged reduction
// length per expert.
//
// The pages are about training with the grouped GEMM ("Optimization 1:
// Grouped GEMM" of "Accelerating dropless MoE training in JAX with NVIDIA
// Transformer Engine"); its weight gradients reduce over each expert's actual
// token rows, again without padding to a capacity.
//
// Operands are the activations as the forward and backward leave them: rows
// grouped by expert, A [TK, M] and B [TK, N] bf16, row-major.  The reduction
// runs along the rows, so both operands are MN-major: a stage holds 64 rows
// (K) of A's 128 columns and B's 256 columns as 64 x 64 TMA boxes (128-byte
// swizzle), and the MMAs read them with MN-major descriptors -- no transposed
// copy in memory.  Every expert has its own pair of tensor maps, copies of
// the host-encoded ones that a one-block kernel moves on the device to the
// group's first row and cuts to the group's row count (the host never sees
// the counts).  A group's K blocks then start at row 0 of its maps, and in
// its last block TMA fills the rows past the group with zeros, so they add
// nothing and no thread touches the staged tiles.
//
// Persistent kernels, one CTA per SM, over tiles (e, row block of D, 256-column
// block) of every expert, with two 256-column TMEM accumulators so a tile's
// epilogue (fp32 by TMA stores of 32 x 32 boxes) overlaps the next tile's
// mainloop.  Experts without rows get their tiles written as zeros.  Bounded
// waits as in the forward GEMMs.
//  * wgrad_kernel: 128-row tiles, tcgen05.mma M=128 N=256 K=16, a 3-stage
//    ring of 48 KB.
//  * wgrad_pair_kernel: clusters of 2 CTAs share 256-row tiles through
//    cta_group::2 MMAs (M=256): each CTA loads 128 columns of A and 128 of B
//    per stage (32 KB instead of 48 KB for the same MMA work per SM), 5
//    stages.  Both CTAs' copies complete on CTA 0's full barrier, and CTA
//    0 issues the MMAs.
#include <algorithm>

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
constexpr int STAGES = 3;
constexpr int MAX_E = 256;
constexpr int A_BYTES = BM * BK * 2;
constexpr int B_BYTES = BN * BK * 2;
constexpr int STAGE = A_BYTES + B_BYTES;
constexpr int TMEM_COLS = 2 * BN;
// epilogue staging: per epilogue warp two 32 x 32 fp32 boxes (128-byte swizzle)
constexpr int EPI_BUF = 32 * 32 * 4;
constexpr int OFF_EPI = STAGES * STAGE;
constexpr int OFF_BARS = OFF_EPI + 4 * 2 * EPI_BUF;
constexpr int NUM_BARS = 2 * STAGES + 5;  // full, empty, tfull[2], tempty[2], drain
constexpr int OFF_TMEM = OFF_BARS + NUM_BARS * 8;
constexpr int OFF_ABORT = OFF_TMEM + 4;
constexpr int OFF_GCNT = OFF_ABORT + 4;
constexpr int SMEM_BYTES = OFF_GCNT + MAX_E * 4 + 1024;
constexpr int BOX = 64 * 64 * 2;  // one 64-row x 64-column bf16 box
static_assert(A_BYTES == 2 * BOX && B_BYTES == 4 * BOX, "a stage is six boxes");
static_assert(SMEM_BYTES <= 227 * 1024, "shared memory budget");

// CTA-pair variant (per CTA)
constexpr int P_STAGES = 5;
constexpr int P_STAGE = 4 * BOX;  // 128 columns of A + 128 columns of B, 64 rows
constexpr int P_OFF_EPI = P_STAGES * P_STAGE;
constexpr int P_OFF_BARS = P_OFF_EPI + 4 * 2 * EPI_BUF;
constexpr int P_NUM_BARS = 2 * P_STAGES + 5;  // full (CTA 0), empty, tfull[2], tempty[2], drain
constexpr int P_OFF_TMEM = P_OFF_BARS + P_NUM_BARS * 8;
constexpr int P_OFF_ABORT = P_OFF_TMEM + 4;
constexpr int P_OFF_GCNT = P_OFF_ABORT + 4;
constexpr int P_SMEM_BYTES = P_OFF_GCNT + MAX_E * 4 + 1024;
static_assert(P_SMEM_BYTES <= 227 * 1024, "shared memory budget");

struct Params {
    const int32_t *offsets;  // [E+1]
    const CUtensorMap *maps; // [2E] per expert: A's rows, then B's rows of its group
    int E, TK, M, N, MT, NT;
    float *D;                // [E, M, N]
    int *status;
    uint64_t timeout_ns;
};

// Group row counts from offsets, clamped to [0, TK] as the per-expert maps
// are; one warp.
__device__ __forceinline__ void groups(const Params &p, int lane, int *s_gcnt) {
    for (int e = lane; e < p.E; e += 32) {
        const int o0 = min(max(p.offsets[e], 0), p.TK);
        const int o1 = min(max(p.offsets[e + 1], o0), p.TK);
        s_gcnt[e] = o1 - o0;
    }
}

struct Tile {
    int e, m0, n0;
};

// Tile -> (expert, first row of D, first column of D); p.MT row blocks of RB.
template <int RB>
__device__ __forceinline__ Tile decode(const Params &p, int tile) {
    Tile t;
    const int per = p.MT * p.NT;
    t.e = tile / per;
    const int rem = tile - t.e * per;
    // column blocks vary fastest: neighbouring CTAs share the A rows in L2
    t.m0 = (rem / p.NT) * RB;
    t.n0 = (rem % p.NT) * BN;
    return t;
}

// Per-expert tensor maps: maps[2e] and maps[2e+1] are tmA and tmB moved to
// the group's first row, with the group's row count as their extent (at
// least 1 row: an empty group's maps are never used but stay valid).  One
// thread per expert.
__global__ void __launch_bounds__(MAX_E)
wgrad_maps_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                  const uint16_t *A, const uint16_t *B, const int32_t *offsets, int E, int TK, int M, int N,
                  CUtensorMap *maps) {
    const int e = threadIdx.x;
    if (e >= E) return;
    const int o0 = min(max(offsets[e], 0), TK);
    const int o1 = min(max(offsets[e + 1], o0), TK);
    const int start = min(o0, TK - 1);
    const int rows = max(o1 - o0, 1);
    CUtensorMap *ma = maps + 2 * e;
    const uint4 *ta = reinterpret_cast<const uint4 *>(&tmA);
    const uint4 *tb = reinterpret_cast<const uint4 *>(&tmB);
    uint4 *da = reinterpret_cast<uint4 *>(ma);
    uint4 *db = reinterpret_cast<uint4 *>(ma + 1);
#pragma unroll
    for (int i = 0; i < static_cast<int>(sizeof(CUtensorMap) / 16); ++i) {
        da[i] = ta[i];
        db[i] = tb[i];
    }
    tmap_set_base(ma, A + static_cast<size_t>(start) * M);
    tmap_set_rows(ma, rows);
    tmap_set_base(ma + 1, B + static_cast<size_t>(start) * N);
    tmap_set_rows(ma + 1, rows);
    fence_tmap_release();
}

// One warp's 32 rows of a tile, 32 columns at a time: the fp32 values go to
// shared memory (128-byte swizzle: 16-byte chunk j of row i at j ^ (i & 7))
// and one TMA store writes the 32 x 32 box as full lines (L2 evict-first:
// the gradients are not read again here).  M and N are multiples of 32, so
// boxes are whole; a warp whose 32 rows lie past M stores nothing.  `zero`:
// the expert has no rows, the accumulator is not read.
__device__ __forceinline__ void epilogue(const Params &p, const CUtensorMap *tm_out, const Tile &t, uint32_t tbase,
                                         int q, int lane, bool zero, uint8_t *stage, uint32_t &sbuf) {
    const int m0 = t.m0 + q * 32;
    if (m0 >= p.M) return;  // warp-uniform
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
        uint8_t *buf = stage + sbuf * EPI_BUF;
        if (lane == 0) bulk_wait_read<1>();  // this buffer's store from two chunks ago has read it
        __syncwarp();
#pragma unroll
        for (int j = 0; j < 8; ++j)
            *reinterpret_cast<uint4 *>(buf + lane * 128 + ((j ^ (lane & 7)) << 4)) =
                make_uint4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]);
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
            tma_store_2d_evict_first(tm_out, buf, n, t.e * p.M + m0, l2_policy_evict_first());
            bulk_commit();
        }
        sbuf ^= 1u;
    }
}

__global__ void __launch_bounds__(THREADS, 1)
wgrad_kernel(const __grid_constant__ CUtensorMap tmD, const Params p) {
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
    int *s_gcnt = reinterpret_cast<int *>(smem + OFF_GCNT);

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
    }
    if (warp == 1) {
        tmem_alloc(s_tmem, TMEM_COLS);
        tmem_relinquish();
    }
    if (warp == 2) groups(p, lane, s_gcnt);
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
                const Tile t = decode<BM>(p, tile);
                const int KB = (s_gcnt[t.e] + BK - 1) / BK;
                const CUtensorMap *ma = p.maps + 2 * t.e;
                const CUtensorMap *mb = ma + 1;
                if (KB > 0) {
                    fence_tmap_acquire(ma);
                    fence_tmap_acquire(mb);
                }
                for (int kb = 0; kb < KB; ++kb) {
                    if (!mbar_wait(&empty[stage], phase ^ 1u, s_abort, p.status, p.timeout_ns)) { ok = false; break; }
                    uint8_t *sa = smem + stage * STAGE;
                    uint8_t *sb = sa + A_BYTES;
                    const int row = kb * BK;  // within the group: rows past it read TMA zero fill
                    mbar_arrive_expect_tx(&full[stage], STAGE);
                    // columns past M or N read TMA zero fill too
                    tma_load_2d(sa, ma, &full[stage], t.m0, row);
                    tma_load_2d(sa + BOX, ma, &full[stage], t.m0 + 64, row);
#pragma unroll
                    for (int j = 0; j < 4; ++j) tma_load_2d(sb + j * BOX, mb, &full[stage], t.n0 + 64 * j, row);
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
        // The whole warp follows the ring; lane 0 waits and issues.
        constexpr uint32_t idesc = idesc_bf16_f32(BM, BN, true, true);
        uint32_t stage = 0, phase = 0, acc = 0, acc_phase = 0;
        bool ok = true, issued = false;
        for (int tile = blockIdx.x; ok && tile < total; tile += gridDim.x) {
            const Tile t = decode<BM>(p, tile);
            const int cnt = s_gcnt[t.e];
            const int KB = (cnt + BK - 1) / BK;
            int w = 1;
            if (lane == 0) w = mbar_wait(&tempty[acc], acc_phase ^ 1u, s_abort, p.status, p.timeout_ns);
            if (!__shfl_sync(0xffffffffu, w, 0)) { ok = false; break; }
            tc_fence_after();
            const uint32_t d_tmem = tmem_base + acc * BN;
            for (int kb = 0; kb < KB; ++kb) {
                if (lane == 0) w = mbar_wait(&full[stage], phase, s_abort, p.status, p.timeout_ns);
                if (!__shfl_sync(0xffffffffu, w, 0)) { ok = false; break; }
                tc_fence_after();
                uint8_t *sa = smem + stage * STAGE;
                if (lane == 0) {
                    const uint32_t a_addr = smem_u32(sa);
                    const uint64_t adesc = smem_desc_mnmajor_sw128(a_addr, BOX);
                    const uint64_t bdesc = smem_desc_mnmajor_sw128(a_addr + A_BYTES, BOX);
#pragma unroll
                    for (int j = 0; j < BK / UMMA_K; ++j)  // 16 rows of K: 2048 bytes further
                        umma_bf16(d_tmem, adesc + 128 * j, bdesc + 128 * j, idesc, (kb | j) != 0);
                    umma_commit(&empty[stage]);
                }
                issued = true;
                __syncwarp();
                if (++stage == STAGES) { stage = 0; phase ^= 1u; }
            }
            if (!ok) break;
            if (lane == 0) umma_commit(&tfull[acc]);  // with no MMAs (empty expert) it arrives at once
            __syncwarp();
            acc ^= 1u;
            if (acc == 0) acc_phase ^= 1u;
        }
        if (!ok && issued && lane == 0) {
            volatile int no_abort = 0;
            umma_commit(drain);
            mbar_wait(drain, 0, &no_abort, p.status, p.timeout_ns);
        }
    } else {
        const int q = warp & 3;
        uint8_t *stage = smem + OFF_EPI + (warp - 2) * 2 * EPI_BUF;
        uint32_t sbuf = 0;
        uint32_t acc = 0, acc_phase = 0;
        for (int tile = blockIdx.x; tile < total; tile += gridDim.x) {
            const Tile t = decode<BM>(p, tile);
            if (!mbar_wait(&tfull[acc], acc_phase, s_abort, p.status, p.timeout_ns)) break;
            tc_fence_after();
            const uint32_t tbase = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + acc * BN;
            epilogue(p, &tmD, t, tbase, q, lane, s_gcnt[t.e] == 0, stage, sbuf);
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&tempty[acc]);
            acc ^= 1u;
            if (acc == 0) acc_phase ^= 1u;
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
// CTA-pair variant (cluster of 2): 256-row tiles, CTA r owns rows
// m0 + 128 r .. m0 + 128 r + 127 of D and supplies columns n0 + 128 r ..
// n0 + 128 r + 127 of B; CTA 0 issues the cta_group::2 MMAs.
// ======================================================================
__global__ void __launch_bounds__(THREADS, 1)
wgrad_pair_kernel(const __grid_constant__ CUtensorMap tmD, const Params p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + P_OFF_BARS);
    uint64_t *full = bars;                  // CTA 0: both CTAs' bytes
    uint64_t *empty = bars + P_STAGES;      // both CTAs: freed by CTA 0's MMA commits
    uint64_t *tfull = bars + 2 * P_STAGES;  // both CTAs
    uint64_t *tempty = tfull + 2;           // CTA 0: 4 epilogue warps x 2 CTAs
    uint64_t *drain = tfull + 4;
    uint32_t *s_tmem = reinterpret_cast<uint32_t *>(smem + P_OFF_TMEM);
    volatile int *s_abort = reinterpret_cast<volatile int *>(smem + P_OFF_ABORT);
    int *s_gcnt = reinterpret_cast<int *>(smem + P_OFF_GCNT);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint32_t rank = cluster_ctarank();
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
        *s_abort = 0;
        fence_mbar_init();
    }
    if (warp == 2) groups(p, lane, s_gcnt);
    __syncthreads();
    // both CTAs' barriers exist before anything crosses the pair, and before
    // the collective TMEM allocation
    cluster_sync();
    if (warp == 1) {
        tmem_alloc_pair(s_tmem, TMEM_COLS);
        tmem_relinquish_pair();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *s_tmem;
    const int total = p.E * p.MT * p.NT;
    const int half = static_cast<int>(rank) * 128;

    if (warp == 0) {
        if (lane == 0) {
            // both CTAs' copies signal CTA 0's full barriers
            const uint32_t full0 = mapa_shared(smem_u32(&full[0]), 0);
            int armed_phase[P_STAGES];
#pragma unroll
            for (int i = 0; i < P_STAGES; ++i) armed_phase[i] = -1;
            uint32_t stage = 0, phase = 0;
            bool ok = true;
            for (int tile = pair; ok && tile < total; tile += npairs) {
                const Tile t = decode<2 * BM>(p, tile);
                const int KB = (s_gcnt[t.e] + BK - 1) / BK;
                const CUtensorMap *ma = p.maps + 2 * t.e;
                const CUtensorMap *mb = ma + 1;
                if (KB > 0) {
                    fence_tmap_acquire(ma);
                    fence_tmap_acquire(mb);
                }
                for (int kb = 0; kb < KB; ++kb) {
                    if (!mbar_wait<true>(&empty[stage], phase ^ 1u, s_abort, p.status, p.timeout_ns)) {
                        ok = false;
                        break;
                    }
                    uint8_t *sa = smem + stage * P_STAGE;
                    const int row = kb * BK;  // within the group: rows past it read TMA zero fill
                    const uint32_t bar = full0 + 8u * stage;
                    if (rank == 0) mbar_arrive_expect_tx(&full[stage], 2 * P_STAGE);
                    // columns past M or N read TMA zero fill too
                    tma_load_2d_pair(sa, ma, bar, t.m0 + half, row);
                    tma_load_2d_pair(sa + BOX, ma, bar, t.m0 + half + 64, row);
                    tma_load_2d_pair(sa + 2 * BOX, mb, bar, t.n0 + half, row);
                    tma_load_2d_pair(sa + 3 * BOX, mb, bar, t.n0 + half + 64, row);
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
    } else if (warp == 1 && rank == 0) {
        // Waits for both CTAs' bytes and issues the MMAs; the whole warp
        // follows the ring, lane 0 waits and issues.
        constexpr uint32_t idesc = idesc_bf16_f32(2 * BM, BN, true, true);
        uint32_t stage = 0, phase = 0, acc = 0, acc_phase = 0;
        bool ok = true, issued = false;
        for (int tile = pair; ok && tile < total; tile += npairs) {
            const Tile t = decode<2 * BM>(p, tile);
            const int cnt = s_gcnt[t.e];
            const int KB = (cnt + BK - 1) / BK;
            int w = 1;
            if (lane == 0) w = mbar_wait<true>(&tempty[acc], acc_phase ^ 1u, s_abort, p.status, p.timeout_ns);
            if (!__shfl_sync(0xffffffffu, w, 0)) { ok = false; break; }
            tc_fence_after();
            const uint32_t d_tmem = tmem_base + acc * BN;
            for (int kb = 0; kb < KB; ++kb) {
                if (lane == 0) w = mbar_wait<true>(&full[stage], phase, s_abort, p.status, p.timeout_ns);
                if (!__shfl_sync(0xffffffffu, w, 0)) { ok = false; break; }
                tc_fence_after();
                uint8_t *sa = smem + stage * P_STAGE;
                if (lane == 0) {
                    const uint32_t a_addr = smem_u32(sa);
                    const uint64_t adesc = smem_desc_mnmajor_sw128(a_addr, BOX);
                    const uint64_t bdesc = smem_desc_mnmajor_sw128(a_addr + 2 * BOX, BOX);
#pragma unroll
                    for (int j = 0; j < BK / UMMA_K; ++j)
                        umma_bf16_pair(d_tmem, adesc + 128 * j, bdesc + 128 * j, idesc, (kb | j) != 0);
                    umma_commit_pair_multicast(&empty[stage], 0x3);
                }
                issued = true;
                __syncwarp();
                if (++stage == P_STAGES) { stage = 0; phase ^= 1u; }
            }
            if (!ok) break;
            if (lane == 0) umma_commit_pair_multicast(&tfull[acc], 0x3);
            __syncwarp();
            acc ^= 1u;
            if (acc == 0) acc_phase ^= 1u;
        }
        if (!ok && issued && lane == 0) {
            volatile int no_abort = 0;
            umma_commit_pair_multicast(drain, 0x1);
            mbar_wait<true>(drain, 0, &no_abort, p.status, p.timeout_ns);
        }
    } else if (warp == 1) {
        // CTA 1's MMA warp has no role after the allocation
    } else {
        const int q = warp & 3;
        uint8_t *stage = smem + P_OFF_EPI + (warp - 2) * 2 * EPI_BUF;
        uint32_t sbuf = 0;
        const uint32_t tempty0 = mapa_shared(smem_u32(&tempty[0]), 0);
        uint32_t acc = 0, acc_phase = 0;
        for (int tile = pair; tile < total; tile += npairs) {
            Tile t = decode<2 * BM>(p, tile);
            if (!mbar_wait<true>(&tfull[acc], acc_phase, s_abort, p.status, p.timeout_ns)) break;
            tc_fence_after();
            const uint32_t tbase = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + acc * BN;
            t.m0 += half;  // this CTA's 128 rows of the tile
            epilogue(p, &tmD, t, tbase, q, lane, s_gcnt[t.e] == 0, stage, sbuf);
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
}

}  // namespace wg

namespace {

cudaLaunchConfig_t pair_config(int grid, cudaStream_t stream, cudaLaunchAttribute *attr) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid, 1, 1);
    cfg.blockDim = dim3(wg::THREADS, 1, 1);
    cfg.dynamicSmemBytes = wg::P_SMEM_BYTES;
    cfg.stream = stream;
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cfg;
}

}  // namespace

cudaError_t wgrad_setup(GemmLaunch *cfg) {
    cudaError_t e;
    if ((e = cudaFuncSetAttribute(wg::wgrad_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, wg::SMEM_BYTES)) !=
        cudaSuccess)
        return e;
    if ((e = cudaFuncSetAttribute(wg::wgrad_pair_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  wg::P_SMEM_BYTES)) != cudaSuccess)
        return e;
    // every pair of the persistent kernel must be resident at once
    cudaLaunchAttribute attr[1];
    cudaLaunchConfig_t lc = pair_config(2, nullptr, attr);
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, wg::wgrad_pair_kernel, &lc) != cudaSuccess) n = 0;
    cudaGetLastError();  // a failed query leaves 0 pairs: single-CTA kernel only
    cfg->wgrad_pairs = std::min(n, cfg->num_sms / 2);
    return cudaSuccess;
}

cudaError_t launch_wgrad(const uint16_t *A, const uint16_t *B, int M, int N, const int32_t *offsets, int E, int TK,
                         float *D, void *maps, const GemmLaunch &lc, int *status, uint64_t timeout_ns,
                         cudaStream_t stream) {
    CUtensorMap tmA, tmB, tmD;
    if (M % 64 != 0 || N % 64 != 0 || TK < 1 || E < 1 || E > wg::MAX_E) return cudaErrorInvalidValue;
    if (reinterpret_cast<uintptr_t>(maps) % 128 != 0) return cudaErrorInvalidValue;
    // A [TK, M] and B [TK, N] with 64-row x 64-column boxes
    if (!make_tmap(&tmA, A, static_cast<uint64_t>(TK), static_cast<uint64_t>(M), 64, 64)) return cudaErrorInvalidValue;
    if (!make_tmap(&tmB, B, static_cast<uint64_t>(TK), static_cast<uint64_t>(N), 64, 64)) return cudaErrorInvalidValue;
    // D as [E * M, N] fp32, 32 x 32 boxes of 128-byte rows
    if (!make_tmap_2d(&tmD, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, D, static_cast<uint64_t>(E) * M,
                      static_cast<uint64_t>(N), 32, 32, CU_TENSOR_MAP_SWIZZLE_128B))
        return cudaErrorInvalidValue;
    // the per-expert maps first (same stream: the GEMM reads them after)
    wg::wgrad_maps_kernel<<<1, wg::MAX_E, 0, stream>>>(tmA, tmB, A, B, offsets, E, TK, M, N,
                                                       static_cast<CUtensorMap *>(maps));
    cudaError_t err = cudaGetLastError();
    if (err != cudaSuccess) return err;
    wg::Params p = {};
    p.offsets = offsets;
    p.maps = static_cast<const CUtensorMap *>(maps);
    p.E = E;
    p.TK = TK;
    p.M = M;
    p.N = N;
    // CTA pairs for D blocks of 256 rows, when D has that many and the
    // groups are long (the forward GEMMs' rule): on groups of 128 rows on
    // average the pair measured slower (each tile's K loop is a few blocks)
    const bool use_pair = lc.wgrad_pairs > 0 && M >= 2 * wg::BM && grouped_gemm_use_pair(TK, E);
    const int rb = use_pair ? 2 * wg::BM : wg::BM;
    p.MT = (M + rb - 1) / rb;
    p.NT = (N + wg::BN - 1) / wg::BN;
    p.D = D;
    p.status = status;
    p.timeout_ns = timeout_ns;
    if (use_pair) {
        cudaLaunchAttribute attr[1];
        cudaLaunchConfig_t cfg = pair_config(2 * lc.wgrad_pairs, stream, attr);
        return cudaLaunchKernelEx(&cfg, wg::wgrad_pair_kernel, tmD, p);
    }
    wg::wgrad_kernel<<<lc.num_sms, wg::THREADS, wg::SMEM_BYTES, stream>>>(tmD, p);
    return cudaGetLastError();
}

}  // namespace moe
