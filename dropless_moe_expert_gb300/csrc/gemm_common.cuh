// Pieces shared by the bf16 and the MXFP8 grouped GEMMs: the parameters,
// the device-side tile scheduler over ragged expert groups and the bf16
// epilogue (TMEM -> registers -> bf16 -> shared memory -> TMA store).
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include "ptx.cuh"

namespace moe {
namespace gg {

constexpr int BN_ACC = 256;   // accumulator columns of one tile
constexpr int MAX_E = 256;

// Epilogue staging for TMA stores: per epilogue warp two 32-row x 32-column
// bf16 buffers (2 KB each, 64-byte swizzle).
constexpr int EPI_WARPS = 4;
constexpr int EPI_BUF = 32 * 32 * 2;
constexpr int EPI_BYTES = EPI_WARPS * 2 * EPI_BUF;

// GEMM2 with the combine fused into its epilogue (counters == nullptr: not
// fused).  counters [T, nb] count, per token and 256-column block of y, the
// token's rows already stored; they are zero at launch.
struct Combine {
    const int32_t *src_tok;   // [TK] token of each row
    const int32_t *row_of;    // [T, K]
    const float *topk_w;      // [T, K]
    int T, K, nb;
    int *counters;
    __nv_bfloat16 *y;         // [T, n_out]
};

struct Params {
    const int32_t *offsets;  // [E+1] device
    int E;
    int TK;         // rows of the activation matrix
    int Kdim;       // reduction length (d for GEMM1, f for GEMM2)
    int n_out;      // output columns (f for GEMM1, d for GEMM2)
    int w_rows;     // weight rows per expert (2f or d)
    int NT;         // column blocks per row block
    __nv_bfloat16 *out;  // [TK, n_out]
    __nv_bfloat16 *preact;  // GEMM1 only, nullable: [TK, 2 n_out] gate | up pre-activations, bf16
    int *status;
    uint64_t timeout_ns;
    // Dynamic tile order (nullable: static round-robin): two ints, zero at
    // launch, shared by every CTA of the launch -- [0] the next ticket, [1]
    // the CTAs done; the last CTA to finish sets both back to zero.
    int *sched;
    Combine comb;
    // GEMM1 with the permute fused into its operand load (single-CTA kernel
    // only): row r of A is gather_x[gather_src[r], :], gather_x [gather_T, Kdim]
    const int32_t *gather_src;
    const __nv_bfloat16 *gather_x;
    int gather_T;
};

struct Tile {
    int e, m_blk, n_blk, row0, grp_end;
};

// Group bounds [s_off[e], s_end[e]), clamped to [0, TK] so that no content of
// offsets[] can send a store out of bounds, and the per-expert tile prefix
// s_pre (tiles of experts < e) for row blocks of RB rows.  One warp.
//
// Also decides the visit order (s_mix): when the largest group holds more
// than 4x the average, heavy and light groups' tiles are interleaved.
template <int RB>
__device__ __forceinline__ void build_groups(const Params &p, int lane, int *s_off, int *s_end, int *s_pre,
                                             int *s_mix) {
    int carry = 0, cmax = 0, csum = 0;
    for (int base = 0; base < p.E; base += 32) {
        const int e = base + lane;
        int v = 0;
        if (e < p.E) {
            const int o0 = min(max(p.offsets[e], 0), p.TK);
            const int o1 = min(max(p.offsets[e + 1], o0), p.TK);
            s_off[e] = o0;
            s_end[e] = o1;
            v = ((o1 - o0 + RB - 1) / RB) * p.NT;
            cmax = max(cmax, o1 - o0);
            csum += o1 - o0;
        }
#pragma unroll
        for (int s = 1; s < 32; s <<= 1) {
            const int n = __shfl_up_sync(0xffffffffu, v, s);
            if (lane >= s) v += n;
        }
        if (e < p.E) s_pre[e + 1] = carry + v;
        carry += __shfl_sync(0xffffffffu, v, 31);
    }
#pragma unroll
    for (int s = 16; s >= 1; s >>= 1) {
        cmax = max(cmax, __shfl_xor_sync(0xffffffffu, cmax, s));
        csum += __shfl_xor_sync(0xffffffffu, csum, s);
    }
    if (lane == 0) {
        s_pre[0] = 0;
        *s_mix = static_cast<int64_t>(cmax) * p.E > 4ll * csum ? 1 : 0;
    }
}

template <int RB, int NBAND>
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
    const int MT = (g1 - g0 + RB - 1) / RB;
    const int band = local / (NBAND * NT);
    const int within = local - band * NBAND * NT;
    const int mb0 = band * NBAND;
    const int bm = min(NBAND, MT - mb0);
    t.n_blk = within / bm;
    t.m_blk = mb0 + (within - t.n_blk * bm);
    t.row0 = g0 + t.m_blk * RB;
    t.grp_end = g1;
    return t;
}

// Order in which the persistent CTAs visit the tile list.  Under a skewed
// load (mix), positions alternate between the front and the back of the list,
// so every wave mixes tiles of the experts at both ends: the heavy groups'
// tiles, whose weight tiles are shared by many row blocks and so are bounded
// by the tensor pipe, run beside the light groups' tiles, which only stream
// weights.  A bijection of [0, N); neighbours in each half stay neighbours,
// so tiles that share operands through L2 still run together.
__device__ __forceinline__ int visit_order(int p, int N, int mix) {
    return mix ? ((p & 1) ? N - 1 - (p >> 1) : (p >> 1)) : p;
}

// Position of round k for worker c of G: rounds cover consecutive blocks of
// G positions.  Under the interleaved order (mix) the workers sweep them in
// alternating direction, so a worker alternates between even and odd
// positions (the two ends of the list); otherwise every round keeps the same
// direction, which keeps the tiles in flight at one time (and their shared
// operands in L2) close together even when workers drift apart.
__device__ __forceinline__ int round_position(int k, int c, int G, int mix) {
    return k * G + ((mix && (k & 1)) ? G - 1 - c : c);
}

// ------------------------------------------------------------ tile queue
// The producer thread decides the CTA's (or CTA pair's) next tile and hands it
// to the CTA's other roles through a ring of shared-memory slots: slot j % Q
// holds the j-th tile, and its `full` barrier takes the producer's arrival
// after the store.  The next tile is the static round-robin position
// (Params::sched == nullptr) or a ticket drawn from the launch's global
// counter: a CTA that finishes early then takes the next tile in visit order,
// so no worker falls behind the others by more than a tile, and the tiles in
// flight stay a contiguous window of the visit order (neighbours share
// operands in L2).  A slot holds -1 after the last tile.
//
// No reader frees its slot: the pipeline itself bounds how far the producer
// can run ahead of every reader.  The producer publishes tile k + 1 when it
// starts loading tile k's stages, which needs the stages of S ring positions
// earlier to have been consumed by the MMAs, so the MMAs are at most S tiles
// behind (S stages of one slice each in the worst case); the MMAs of tile m
// need the accumulator of tile m - 2 drained, so the epilogue is at most two
// tiles behind them; the loaders of the other operand (gather warps, the
// second CTA of a pair) complete the MMAs' stages, so they are within S
// stages of the producer.  At most S + 3 published tiles are unread at any
// time, and a ring of Q >= S + 4 slots is never overwritten before it is read.
__host__ __device__ constexpr int queue_slots(int stages) { return stages + 4 <= 8 ? 8 : 16; }

// First position (round 0) of worker c of G.
__device__ __forceinline__ int first_position(const Params &p, int c, int G, int mix) {
    return p.sched ? atomicAdd(p.sched, 1) : round_position(0, c, G, mix);
}
// Position of round k + 1, drawn while round k's tile is being loaded.
__device__ __forceinline__ int next_position(const Params &p, int k, int c, int G, int mix) {
    return p.sched ? atomicAdd(p.sched, 1) : round_position(k + 1, c, G, mix);
}
// End of the launch for a CTA (one thread, after the CTA's last use of the
// counter): the last of the launch's CTAs resets it for the next launch,
// which stream order places after this one.
__device__ __forceinline__ void sched_retire(const Params &p) {
    if (!p.sched) return;
    __threadfence();
    if (atomicAdd(p.sched + 1, 1) == static_cast<int>(gridDim.x) - 1) {
        atomicExch(p.sched, 0);
        atomicExch(p.sched + 1, 0);
        __threadfence();
    }
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<const uint32_t *>(&v);
}

__device__ __forceinline__ void store_row32(__nv_bfloat16 *dst_row, const uint32_t (&packed)[16]) {
    uint4 *dst = reinterpret_cast<uint4 *>(dst_row);
#pragma unroll
    for (int i = 0; i < 4; ++i) dst[i] = make_uint4(packed[4 * i], packed[4 * i + 1], packed[4 * i + 2], packed[4 * i + 3]);
}

__device__ __forceinline__ void fma_bf16x8(float (&acc)[8], float w, const uint4 &v) {
    const uint32_t q[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        acc[2 * i] = __fmaf_rn(w, __uint_as_float(q[i] << 16), acc[2 * i]);
        acc[2 * i + 1] = __fmaf_rn(w, __uint_as_float(q[i] & 0xffff0000u), acc[2 * i + 1]);
    }
}

// Fused combine, after this warp's 32 rows of y_perm (its columns of block
// n_blk) are stored; `parts` warps share those rows, each storing its share
// of the block's columns.  Each row's lane makes its stores visible and
// counts the row for its token; the lane that brings the count to K * parts
// holds the token's last row (and share) in this column block, and the warp
// then forms
//   y[t, cols] = bf16( sum_{k=0..K-1} w[t,k] * y_perm[row_of[t,k], cols] )
// (fp32 fused multiply-add in ascending k, the unfused combine's
// arithmetic) from the K stored rows, 8 columns per lane.  Which row comes
// last does not change the sum, so the result is deterministic.
__device__ __forceinline__ void combine_arrive(const Params &p, int n_blk, int grow, bool row_ok, int lane,
                                               int parts) {
    const Combine &cb = p.comb;
    __threadfence();  // this row's stores before its count
    int tok = -1;
    bool last = false;
    if (row_ok) {
        tok = cb.src_tok[grow];
        if (tok >= 0 && tok < cb.T)
            last = atomicAdd(&cb.counters[static_cast<size_t>(tok) * cb.nb + n_blk], 1) == cb.K * parts - 1;
    }
    unsigned m = __ballot_sync(0xffffffffu, last);
    if (m == 0) return;
    __threadfence();  // the token's other rows, seen through the count, before reading them
    const int n0 = n_blk * BN_ACC + 8 * lane;
    while (m) {
        const int j = __ffs(m) - 1;
        m &= m - 1;
        const int t = __shfl_sync(0xffffffffu, tok, j);
        if (n0 >= p.n_out) continue;
        float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
        // up to 8 of the token's rows in flight, then added in ascending k
        for (int k0 = 0; k0 < cb.K; k0 += 8) {
            uint4 v[8];
            float w[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const int k = k0 + i;
                v[i] = make_uint4(0, 0, 0, 0);
                w[i] = 0.0f;
                if (k < cb.K) {
                    const int r = cb.row_of[static_cast<size_t>(t) * cb.K + k];
                    w[i] = cb.topk_w[static_cast<size_t>(t) * cb.K + k];
                    if (r >= 0 && r < p.TK)  // else outside the contract
                        v[i] = __ldcg(reinterpret_cast<const uint4 *>(p.out + static_cast<size_t>(r) * p.n_out + n0));
                }
            }
#pragma unroll
            for (int i = 0; i < 8; ++i)
                if (k0 + i < cb.K) fma_bf16x8(acc, w[i], v[i]);
        }
        uint32_t q[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) q[i] = pack_bf16x2(acc[2 * i], acc[2 * i + 1]);
        *reinterpret_cast<uint4 *>(cb.y + static_cast<size_t>(t) * p.n_out + n0) = make_uint4(q[0], q[1], q[2], q[3]);
    }
}

// One 32-column chunk of a warp's 32 rows, 16 words of packed bf16 pairs per
// lane, into dst (row length ld, tensor map tm) at column col.  When all 32
// rows belong to the group (`full`) the chunk is staged in the warp's buffer
// `sbuf` of NBUF (64-byte swizzle) and written by one TMA store of full lines;
// otherwise each lane whose row lies in the group stores its 64 bytes.
template <int NBUF>
__device__ __forceinline__ void put_chunk32(const CUtensorMap *tm, __nv_bfloat16 *dst, int ld, int col,
                                            const uint32_t (&packed)[16], bool full, bool row_ok, int grow,
                                            int wrow0, int lane, uint8_t *stage, uint32_t &sbuf) {
    if (full) {
        uint8_t *buf = stage + sbuf * EPI_BUF;
        if (lane == 0) bulk_wait_read<NBUF - 1>();  // this buffer's store from NBUF chunks ago has read it
        __syncwarp();
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int jj = j ^ ((lane >> 1) & 3);
            *reinterpret_cast<uint4 *>(buf + lane * 64 + jj * 16) =
                make_uint4(packed[4 * j], packed[4 * j + 1], packed[4 * j + 2], packed[4 * j + 3]);
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
            // the output is not read again by this kernel: let L2 evict it
            // before the operand tiles that other CTAs still share
            tma_store_2d_evict_first(tm, buf, col, wrow0, l2_policy_evict_first());
            bulk_commit();
        }
        sbuf = (sbuf + 1 == NBUF) ? 0u : sbuf + 1;
    } else if (row_ok) {
        store_row32(dst + static_cast<size_t>(grow) * ld + col, packed);
    }
}

// silu(g) * u of 32 gate and up accumulator values, as 16 packed bf16 pairs
__device__ __forceinline__ void swiglu32(const uint32_t (&g)[32], const uint32_t (&u)[32], uint32_t (&packed)[16]) {
#pragma unroll
    for (int i = 0; i < 16; ++i) {
        float h2[2];
#pragma unroll
        for (int k = 0; k < 2; ++k) {
            const float gv = __uint_as_float(g[2 * i + k]);
            const float uv = __uint_as_float(u[2 * i + k]);
            h2[k] = __fdividef(gv, 1.0f + __expf(-gv)) * uv;  // silu(g) * u
        }
        packed[i] = pack_bf16x2(h2[0], h2[1]);
    }
}

// Epilogue of one accumulator for one warp: 32 TMEM lanes = 32 output rows
// wrow0..wrow0+31 (this thread's row is wrow0 + lane), tbase points at the
// warp's lane quarter of the accumulator.  The warp covers output columns
// [c_begin, c_end) of the tile (all of them, or half where two warps share a
// lane quarter).  Each 32-column chunk is converted to bf16 and, when all 32
// rows belong to the group, staged in shared memory (64-byte swizzle) and
// written by one TMA store of full lines; a slice that crosses the group's
// end falls back to masked 16-byte stores per row.  `sbuf` cycles through
// the warp's NBUF staging buffers across chunks and tiles.
template <bool SWIGLU, int NBUF = 2>
__device__ __forceinline__ void epilogue_tile(const Params &p, const CUtensorMap *tm_out, const CUtensorMap *tm_pre,
                                              uint8_t *stage, uint32_t &sbuf, uint32_t tbase, int n_blk, int wrow0,
                                              int lane, int grp_end, int c_begin = 0,
                                              int c_end = SWIGLU ? BN_ACC / 2 : BN_ACC) {
    if (wrow0 >= grp_end) return;  // whole slice outside the group (warp-uniform)
    const bool full = wrow0 + 31 < grp_end;
    const int grow = wrow0 + lane;
    const bool row_ok = grow < grp_end;
    if (!SWIGLU && p.comb.counters != nullptr) {
        // fused combine: rows stored directly (generic proxy), so that a fence
        // orders them before the token's count
#pragma unroll 1
        for (int c = c_begin; c < c_end; c += 64) {
            const int col = n_blk * BN_ACC + c;
            if (col >= p.n_out) break;  // column tail (uniform)
            uint32_t v[2][32];
            tmem_ld_32x32b_x32(tbase + c, v[0]);
            tmem_ld_32x32b_x32(tbase + c + 32, v[1]);
            tmem_ld_wait();
#pragma unroll
            for (int hlf = 0; hlf < 2; ++hlf) {
                if (col + 32 * hlf >= p.n_out) break;
                uint32_t packed[16];
#pragma unroll
                for (int i = 0; i < 16; ++i)
                    packed[i] = pack_bf16x2(__uint_as_float(v[hlf][2 * i]), __uint_as_float(v[hlf][2 * i + 1]));
                if (row_ok) store_row32(p.out + static_cast<size_t>(grow) * p.n_out + col + 32 * hlf, packed);
            }
        }
        combine_arrive(p, n_blk, grow, row_ok, lane, BN_ACC / (c_end - c_begin));
        return;
    }
    constexpr int NCOL = SWIGLU ? BN_ACC / 2 : BN_ACC;
    // 32 columns of the warp's 32 rows into `dst` (row length ld, its tensor
    // map `tm`) at column col
    auto put = [&](const CUtensorMap *tm, __nv_bfloat16 *dst, int ld, int col, const uint32_t (&packed)[16]) {
        put_chunk32<NBUF>(tm, dst, ld, col, packed, full, row_ok, grow, wrow0, lane, stage, sbuf);
    };
    auto emit = [&](int c, const uint32_t (&packed)[16]) {
        const int col = n_blk * NCOL + c;
        if (col >= p.n_out) return;  // column tail (uniform)
        put(tm_out, p.out, p.n_out, col, packed);
    };
    if (SWIGLU) {
#pragma unroll 1
        for (int c = c_begin; c < c_end; c += 32) {
            uint32_t g[32], u[32];
            tmem_ld_32x32b_x32(tbase + c, g);
            tmem_ld_32x32b_x32(tbase + BN_ACC / 2 + c, u);
            tmem_ld_wait();
            uint32_t packed[16];
            swiglu32(g, u, packed);
            emit(c, packed);
            const int col = n_blk * NCOL + c;
            if (p.preact != nullptr && col < p.n_out) {
                // the pre-activations the backward needs, rounded to bf16
#pragma unroll
                for (int i = 0; i < 16; ++i)
                    packed[i] = pack_bf16x2(__uint_as_float(g[2 * i]), __uint_as_float(g[2 * i + 1]));
                put(tm_pre, p.preact, 2 * p.n_out, col, packed);
#pragma unroll
                for (int i = 0; i < 16; ++i)
                    packed[i] = pack_bf16x2(__uint_as_float(u[2 * i]), __uint_as_float(u[2 * i + 1]));
                put(tm_pre, p.preact, 2 * p.n_out, p.n_out + col, packed);
            }
        }
    } else {
        // two 32-column loads per wait, so TMEM latency is paid 4 times per tile, not 8
#pragma unroll 1
        for (int c = c_begin; c < c_end; c += 64) {
            uint32_t v[2][32];
            tmem_ld_32x32b_x32(tbase + c, v[0]);
            tmem_ld_32x32b_x32(tbase + c + 32, v[1]);
            tmem_ld_wait();
#pragma unroll
            for (int hlf = 0; hlf < 2; ++hlf) {
                uint32_t packed[16];
#pragma unroll
                for (int i = 0; i < 16; ++i)
                    packed[i] = pack_bf16x2(__uint_as_float(v[hlf][2 * i]), __uint_as_float(v[hlf][2 * i + 1]));
                emit(c + 32 * hlf, packed);
            }
        }
    }
}

// GEMM1 epilogue of one warp that hands its accumulator back early: 32 rows
// and the 64 h columns [c_begin, c_begin + 64) of the tile, two 32-column
// chunks.  The first chunk's gate and up values are loaded and turned into
// h, the second chunk's are loaded, and then the accumulator is released
// (`release`: fence, warp sync, arrive) before the second chunk's h is
// formed and both chunks are stored.  The same arithmetic and stores as
// epilogue_tile<true> without pre-activations, so h is bit-identical.
template <typename Release>
__device__ __forceinline__ void epilogue_swiglu_early(const Params &p, const CUtensorMap *tm_out, uint8_t *stage,
                                                      uint32_t &sbuf, uint32_t tbase, int n_blk, int wrow0, int lane,
                                                      int grp_end, int c_begin, Release release) {
    if (wrow0 >= grp_end) {  // whole slice outside the group (warp-uniform)
        release();
        return;
    }
    const bool full = wrow0 + 31 < grp_end;
    const int grow = wrow0 + lane;
    const bool row_ok = grow < grp_end;
    constexpr int NCOL = BN_ACC / 2;
    uint32_t g[32], u[32], h0[16], h1[16];
    tmem_ld_32x32b_x32(tbase + c_begin, g);
    tmem_ld_32x32b_x32(tbase + NCOL + c_begin, u);
    tmem_ld_wait();
    swiglu32(g, u, h0);
    tmem_ld_32x32b_x32(tbase + c_begin + 32, g);
    tmem_ld_32x32b_x32(tbase + NCOL + c_begin + 32, u);
    tmem_ld_wait();
    release();
    swiglu32(g, u, h1);
    const int col = n_blk * NCOL + c_begin;
    if (col < p.n_out) put_chunk32<1>(tm_out, p.out, p.n_out, col, h0, full, row_ok, grow, wrow0, lane, stage, sbuf);
    if (col + 32 < p.n_out)
        put_chunk32<1>(tm_out, p.out, p.n_out, col + 32, h1, full, row_ok, grow, wrow0, lane, stage, sbuf);
}

// silu(g) * u of 16 gate and up accumulator values into 8 packed bf16 pairs
// (the first or second half of a 32-column chunk's packed words)
__device__ __forceinline__ void swiglu16(const uint32_t (&g)[16], const uint32_t (&u)[16], uint32_t *packed) {
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        float h2[2];
#pragma unroll
        for (int k = 0; k < 2; ++k) {
            const float gv = __uint_as_float(g[2 * i + k]);
            const float uv = __uint_as_float(u[2 * i + k]);
            h2[k] = __fdividef(gv, 1.0f + __expf(-gv)) * uv;  // silu(g) * u
        }
        packed[i] = pack_bf16x2(h2[0], h2[1]);
    }
}

// GEMM1 epilogue of one warp over a tile of two row blocks (accumulators at
// tb0 and tb1, rows wrow0 and wrow0 + 128): the 64 h columns [c_begin,
// c_begin + 64) of each block are formed 16 columns at a time and kept in
// registers, each accumulator is released once its last values are loaded,
// and only then are the four 32-column chunks stored.  Both accumulators go
// back before any store.  The arithmetic and stores are epilogue_tile<true>'s
// without pre-activations, so h is bit-identical.  Returns false if the wait
// for block 1's accumulator gave up.
template <typename Wait, typename Release>
__device__ __forceinline__ bool epilogue_swiglu_early2(const Params &p, const CUtensorMap *tm_out, uint8_t *stage,
                                                       uint32_t &sbuf, uint32_t tb0, uint32_t tb1, int n_blk,
                                                       int wrow0, int lane, int grp_end, int c_begin, Wait wait1,
                                                       Release release0, Release release1) {
    constexpr int NCOL = BN_ACC / 2;
    uint32_t h[4][16];
    // the 64 columns of one block, 16 at a time; `release` after the last load
    auto block = [&](uint32_t tb, uint32_t(*hb)[16], Release release) {
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            uint32_t g[16], u[16];
            tmem_ld_32x32b_x16(tb + c_begin + 16 * j, g);
            tmem_ld_32x32b_x16(tb + NCOL + c_begin + 16 * j, u);
            tmem_ld_wait();
            if (j == 3) release();
            swiglu16(g, u, &hb[j >> 1][8 * (j & 1)]);
        }
    };
    block(tb0, h, release0);  // block 0: its rows start inside the group
    if (!wait1()) return false;
    if (wrow0 + 128 < grp_end) block(tb1, h + 2, release1);
    else release1();
    const int col = n_blk * NCOL + c_begin;
#pragma unroll
    for (int b = 0; b < 2; ++b) {
        const int wr = wrow0 + 128 * b;
        if (wr >= grp_end) break;  // warp-uniform
        const bool full = wr + 31 < grp_end;
        const int grow = wr + lane;
        const bool row_ok = grow < grp_end;
        if (col < p.n_out)
            put_chunk32<1>(tm_out, p.out, p.n_out, col, h[2 * b], full, row_ok, grow, wr, lane, stage, sbuf);
        if (col + 32 < p.n_out)
            put_chunk32<1>(tm_out, p.out, p.n_out, col + 32, h[2 * b + 1], full, row_ok, grow, wr, lane, stage, sbuf);
    }
    return true;
}

}  // namespace gg
}  // namespace moe
