/*
 * moe.h -- C ABI of a dropless Mixture-of-Experts SwiGLU FFN layer on one
 * NVIDIA GB300 (sm_103a): the forward (bf16, and MXFP8 expert matmuls) and the
 * backward of a training step.
 *
 * The operation follows "Accelerating dropless MoE training in JAX with NVIDIA
 * Transformer Engine":
 *   - introduction: a learned router activates the Top-K experts per token;
 *   - "How is dropless MoE different from capacity-based MoE?": every token is
 *     processed by its chosen experts whatever the load (no drop, no padding);
 *   - "What specialized optimizations are needed for dropless MoE?": per-expert
 *     token counts are data dependent and must stay invisible to the CPU, so
 *     that CUDA graphs work without recompiling;
 *   - Figure 3 caption: dispatch moves tokens to their experts, the grouped MLP
 *     runs two grouped GEMMs over the variable-length groups, combine restores
 *     the original token order;
 *   - "Optimization 1: Grouped GEMM": all expert matmuls in one kernel call,
 *     each with its actual token count, computing only valid-token rows; a
 *     device-to-host copy of the counts would break CUDA graphs.
 *
 * Notation: T tokens, d model dim, E experts, K experts per token, f expert
 * FFN dim, TK = T*K.  Layouts are row-major and dense:
 *   x      [T, d]      bf16        token activations
 *   Wr     [d, E]      fp32        router weights;  bias [E] fp32 (nullable)
 *   logits [T, E]      fp32
 *   W1     [E, 2f, d]  bf16        rows 0..f-1 gate, rows f..2f-1 up (out x in)
 *   W2     [E, d, f]   bf16        (out x in)
 *   topk_idx [T, K] int32, topk_w [T, K] fp32   (descending logit; equal
 *                                   logits -> lower expert index)
 *   counts [E], offsets [E+1] int32 (offsets[E] = TK)
 *   row_of [T, K] int32: row of x_perm holding token t's k-th choice
 *   src_tok [TK] int32: token held by each row of x_perm
 *   x_perm, y_perm [TK, d] bf16, h [TK, f] bf16: rows grouped by expert,
 *                                   ascending token index inside a group
 *   y      [T, d]      bf16        layer output
 * bf16 buffers are passed as uint16_t* (bit patterns).
 *
 * Conventions for every entry point:
 *   - All pointers except those of *_host calls are device pointers owned by
 *     the caller.  The library allocates no memory and performs no
 *     host<->device copy, except the *_host calls (stated there).  It keeps
 *     two small tables of its own in static device memory on every GPU that
 *     loads it: the device status word, and 128 KB of counters through which
 *     the CTAs of one bf16 grouped-GEMM launch hand out its tiles in order
 *     (dynamic scheduling).  Each launch takes a counter slot on the host:
 *     eager launches from a ring of 2048 (so only launches 2048 apart could
 *     share one, and those are never in flight together), launches captured
 *     into a CUDA graph a slot of their own, kept for every replay (the
 *     replays of one graph run one after another; a capture instantiated
 *     twice must not run both instances at once).  After 14336 captured
 *     launches, later captures use a static tile order instead.
 *   - Calls are asynchronous on `stream` and never synchronize; no value flows
 *     from device to host, so a sequence of calls can be captured in a CUDA
 *     graph and replayed for any routing.  (The first call on a device also
 *     sets kernel attributes; make it once before capturing.)
 *   - Arguments are checked on the host before anything is launched; a bad
 *     argument returns an error and launches nothing.  Sizes: T >= 1,
 *     1 <= K <= E <= 256, K <= 16, d and f multiples of 64, T*K < 2^31.
 *     bf16 matrices must be 16-byte aligned; fp32/int32 arrays 4-byte aligned.
 *   - Device-side waits are bounded (about one second).  A kernel whose wait
 *     expires records MOE_ERR_DEVICE_TIMEOUT in a device status word, drains
 *     its own copies, frees its tensor memory and returns; read the word with
 *     moe_device_status() (synchronous) or moe_last_device_status() (on a
 *     stream, capture-safe).
 *   - Inputs are assumed finite; NaN or Inf logits are outside the contract.
 */
#ifndef MOE_GB300_H
#define MOE_GB300_H

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    MOE_OK = 0,
    MOE_ERR_INVALID_ARG = 1,    /* null/misaligned pointer, size out of range    */
    MOE_ERR_UNSUPPORTED = 2,    /* sizes the kernels do not cover (E>256, ...)   */
    MOE_ERR_WORKSPACE = 3,      /* workspace smaller than *_workspace_size()     */
    MOE_ERR_CUDA = 4,           /* a CUDA runtime/driver call or launch failed   */
    MOE_ERR_DEVICE_TIMEOUT = 5  /* a bounded device-side wait expired            */
} moe_status_t;

/* Static, human-readable name of a status code. */
const char *moe_status_string(int status);

/* ABI version: 100 * major + minor. */
int moe_abi_version(void);

/* Step a0 -- router logits (introduction: the learned router).
 * logits[t,e] = fp32 dot product of x[t,:] and Wr[:,e], + bias[e] (if bias
 * is not NULL).  Computed on the tensor cores with exact products: Wr is
 * split exactly into three bf16 pieces (hi + mid + lo == Wr), every
 * bf16 x bf16 product is exact in fp32, and the 3d products are summed in
 * fp32 in the tensor core's order (not index order).  The logits are
 * deterministic for a given shape and device, and within fp32 summation
 * error of the exact dot product.
 * `workspace` (16-byte aligned, moe_router_workspace_size(d, E) bytes)
 * receives the split weights [3][E][d] bf16; 2 kernel launches.  */
size_t moe_router_workspace_size(int d, int E);
moe_status_t moe_router_logits(const uint16_t *x, const float *Wr, const float *bias,
                               int T, int d, int E, float *logits,
                               void *workspace, size_t workspace_bytes, cudaStream_t stream);

/* Steps a1 + a2 -- top-K softmax routing, expert histogram, offsets and the
 * stable dispatch order (introduction: Top-K experts; "What specialized
 * optimizations are needed for dropless MoE?": counts stay on the device).
 *   topk_idx[t,:]: the K largest logits of token t, descending, equal logits
 *                  in ascending expert order (-0.0 equals +0.0);
 *   topk_w[t,k]  : exp(l_k - l_0) / sum_j exp(l_j - l_0) over the K selected;
 *   counts, offsets (exclusive scan, E+1 entries), row_of, src_tok as above.
 * Every output is bit-deterministic.  `workspace` must hold
 * moe_route_workspace_size(T, E, K) bytes (4-byte aligned): two int32
 * tables of [ceil(T / 64), E].  */
size_t moe_route_workspace_size(int T, int E, int K);
moe_status_t moe_route(const float *logits, int T, int E, int K,
                       int32_t *topk_idx, float *topk_w, int32_t *counts, int32_t *offsets,
                       int32_t *row_of, int32_t *src_tok,
                       void *workspace, size_t workspace_bytes, cudaStream_t stream);

/* moe_route without a workspace argument, for callers that cannot allocate
 * device memory where they route: an inference-engine plugin whose enqueue
 * step must not allocate, or a runtime that owns all device memory in a
 * fixed pool and forbids any other allocation.  The page has no counterpart: this is
 * a packaging variant of moe_route, with identical outputs.
 *   - Scratch lives in a library-owned static device array of
 *     MOE_ROUTE_STATIC_MAX_SCRATCH_BYTES (1 MiB) on every GPU that loads
 *     the library, held until the process exits.  Sizes whose scratch,
 *     moe_route_workspace_size(T, E, K), exceeds it return
 *     MOE_ERR_UNSUPPORTED with nothing launched (e.g. E = 256 allows up to
 *     32768 tokens).
 *   - The call allocates and frees nothing.  Its first call on a device looks
 *     up the array's device address (cudaGetSymbolAddress) with that device
 *     current; make that first call before any stream capture.
 *   - Every call shares the one array and leaves its contents behind; nothing
 *     in it needs to start at zero.  Calls whose kernels overlap on the GPU
 *     (several streams, or several host threads) race on it: serialize them.
 *   - Kernel launches of this call are not counted by moe_launch_count(). */
#define MOE_ROUTE_STATIC_MAX_SCRATCH_BYTES (1024u * 1024u)
moe_status_t moe_route_static(const float *logits, int T, int E, int K,
                              int32_t *topk_idx, float *topk_w, int32_t *counts, int32_t *offsets,
                              int32_t *row_of, int32_t *src_tok, cudaStream_t stream);

/* Step a3 -- permute (local part of dispatch, Figure 3 caption):
 * x_perm[row_of[t,k], :] = x[t, :] for every (t, k).  */
moe_status_t moe_permute(const uint16_t *x, const int32_t *row_of, int T, int K, int d,
                         uint16_t *x_perm, cudaStream_t stream);

/* Steps a4 + a5 -- the grouped MLP ("Optimization 1: Grouped GEMM"; Figure 3
 * caption: two grouped GEMMs over the variable-length groups).  For each
 * expert e and each row r in offsets[e]..offsets[e+1]-1:
 *   g = x_perm[r] . W1[e, 0:f]^T,  u = x_perm[r] . W1[e, f:2f]^T  (fp32 accumulate)
 *   h[r] = bf16(silu(g) * u)                                    (GEMM1 epilogue)
 *   y_perm[r] = bf16(h[r] . W2[e]^T)                            (fp32 accumulate)
 * The kernels read `offsets` on the device; empty experts cost nothing and
 * their weights are not read.  `h` is caller-owned scratch [TK, f].  */
moe_status_t moe_grouped_mlp(const uint16_t *x_perm, const int32_t *offsets, int E, int TK,
                             int d, int f, const uint16_t *W1, const uint16_t *W2,
                             uint16_t *h, uint16_t *y_perm, cudaStream_t stream);
/* The two halves of moe_grouped_mlp, one kernel launch each. */
moe_status_t moe_grouped_gemm1_swiglu(const uint16_t *x_perm, const int32_t *offsets, int E,
                                      int TK, int d, int f, const uint16_t *W1, uint16_t *h,
                                      cudaStream_t stream);
moe_status_t moe_grouped_gemm2(const uint16_t *h, const int32_t *offsets, int E, int TK,
                               int d, int f, const uint16_t *W2, uint16_t *y_perm,
                               cudaStream_t stream);
/* GEMM1 that also stores the pre-activations for a backward pass:
 * preact [TK, 2f] bf16 (caller-owned, 16-byte aligned), row r holding
 * bf16(g) in columns 0..f-1 and bf16(u) in columns f..2f-1, rows grouped by
 * expert like h.  One kernel launch.  */
moe_status_t moe_grouped_gemm1_swiglu_preact(const uint16_t *x_perm, const int32_t *offsets,
                                             int E, int TK, int d, int f, const uint16_t *W1,
                                             uint16_t *h, uint16_t *preact, cudaStream_t stream);

/* Steps a3 + a4 in one kernel (the permute fused into GEMM1's operand load;
 * "Optimization 2": a naive dispatch reads and writes the tokens again).
 * Computes h exactly as moe_permute followed by moe_grouped_gemm1_swiglu
 * (bit-identical), without x_perm: row r of expert e's group is read as
 * x[src_tok[r], :] (x [T, d] bf16, src_tok [TK] from moe_route).  It runs the
 * single-CTA kernel for every shape, so on shapes whose average group holds
 * 384 rows or more it is slower than the unfused pair; on the small-group
 * shapes it trades the permute's x_perm round trip for row gathers.
 * src_tok values outside [0, T) are outside the contract (they are clamped,
 * never read out of bounds).  One kernel launch.  */
moe_status_t moe_grouped_gemm1_swiglu_gather(const uint16_t *x, const int32_t *src_tok,
                                             const int32_t *offsets, int T, int E, int TK, int d,
                                             int f, const uint16_t *W1, uint16_t *h,
                                             cudaStream_t stream);

/* Steps a5 + a6 in one kernel (the combine fused into GEMM2's epilogue;
 * "Optimization 2": a naive dispatch/combine reads and writes the data many
 * times, TE fuses them into one pipeline).  Computes y exactly as
 * moe_grouped_gemm2 followed by moe_unpermute (bit-identical): each stored
 * row of y_perm (scratch [TK, d]) is counted per token and 256-column block
 * in `counters`, and the row that completes a token's K rows forms y for
 * that block from the K stored rows, fp32 in ascending k.  No floating-point
 * atomics: the result does not depend on which row comes last.
 * `counters` holds moe_combine_counters_size(T, d) bytes and is zeroed by
 * the call (cudaMemsetAsync on `stream`).  TK must equal T * K.  */
size_t moe_combine_counters_size(int T, int d);
moe_status_t moe_grouped_gemm2_combine(const uint16_t *h, const int32_t *offsets, int E, int TK, int d,
                                       int f, const uint16_t *W2, const int32_t *src_tok,
                                       const int32_t *row_of, const float *topk_w, int T, int K,
                                       uint16_t *y_perm, int32_t *counters, size_t counters_bytes,
                                       uint16_t *y, cudaStream_t stream);

/* Step a6 -- unpermute + combine (Figure 3 caption: restore token order):
 * y[t,:] = bf16( sum_{k=0..K-1} topk_w[t,k] * y_perm[row_of[t,k], :] ),
 * fp32 accumulation in ascending k.  */
moe_status_t moe_unpermute(const uint16_t *y_perm, const int32_t *row_of, const float *topk_w,
                           int T, int K, int d, uint16_t *y, cudaStream_t stream);

/* The whole layer, a0..a6 in order on `stream` (9 kernel launches, or 8
 * when the permute is fused into GEMM1).
 * `workspace` (16-byte aligned, moe_forward_workspace_size() bytes) holds
 * every intermediate; moe_forward_views() gives their byte offsets so that a
 * caller can inspect them after the call.  Whether moe_forward fuses the
 * permute into GEMM1 (moe_grouped_gemm1_swiglu_gather; the region x_perm is
 * then left unwritten, and every other output is bit-identical) is decided
 * on the sizes alone, so it is the same for every routing:
 * moe_forward_fuses_permute() returns 1 for the shapes where it does, which
 * are those whose grouped GEMMs run single-CTA tiles (average group under
 * 384 rows) and those with f <= 4096, where the permute's round trip costs
 * more than the CTA-pair kernel saves.  moe_forward_train never fuses it:
 * the backward reads x_perm.  */
int moe_forward_fuses_permute(int T, int d, int E, int K, int f);
size_t moe_forward_workspace_size(int T, int d, int E, int K, int f);
typedef struct {
    size_t logits, topk_idx, topk_w, counts, offsets, row_of, src_tok, route_ws,
           router_ws, x_perm, h, y_perm, x_dev, y_dev, total;
} moe_forward_layout_t;
moe_status_t moe_forward_views(int T, int d, int E, int K, int f, moe_forward_layout_t *layout);
moe_status_t moe_forward(const uint16_t *x, const float *Wr, const float *bias,
                         const uint16_t *W1, const uint16_t *W2, int T, int d, int E, int K,
                         int f, uint16_t *y, void *workspace, size_t workspace_bytes,
                         cudaStream_t stream);
/* moe_forward for training: GEMM1 also stores the pre-activations into
 * `preact` [T*K, 2f] bf16 (see moe_grouped_gemm1_swiglu_preact; nullable, then
 * identical to moe_forward), which moe_backward then reads instead of
 * recomputing them.  Same 9 launches.  */
moe_status_t moe_forward_train(const uint16_t *x, const float *Wr, const float *bias,
                               const uint16_t *W1, const uint16_t *W2, int T, int d, int E, int K,
                               int f, uint16_t *y, void *workspace, size_t workspace_bytes,
                               uint16_t *preact, cudaStream_t stream);

/* moe_forward with the activations in HOST memory (pinned memory makes the
 * copies asynchronous): copies x_host [T, d] bf16 into the workspace,
 * runs the layer, copies y back to y_host [T, d] bf16, all on `stream`.
 * The weights stay device pointers.  y_host is valid after the stream
 * has been synchronized.  */
moe_status_t moe_forward_host(const uint16_t *x_host, const float *Wr, const float *bias,
                              const uint16_t *W1, const uint16_t *W2, int T, int d, int E,
                              int K, int f, uint16_t *y_host, void *workspace,
                              size_t workspace_bytes, cudaStream_t stream);

/* moe_forward over a sequence of n_batches batches in HOST memory, with the
 * copies overlapped: batch i's host->device copy and batch i-1's
 * device->host copy run on two copy streams of the call while the layer of
 * batch i-1 / i runs on `stream` (double-buffered device copies of x and y).
 * x_hosts[i], y_hosts[i]: [T, d] bf16 host buffers (pinned, or the copies
 * are not asynchronous), which may repeat; y_hosts[i] is written from batch
 * i.  `workspace` (256-byte aligned) holds
 * moe_forward_host_pipelined_workspace_size() bytes: the layer's workspace
 * (moe_forward_views) followed by the second x and y buffers.  All of the
 * call's work -- every copy included -- is complete when `stream` is.
 * 9 kernel launches per batch.  */
size_t moe_forward_host_pipelined_workspace_size(int T, int d, int E, int K, int f);
moe_status_t moe_forward_host_pipelined(const uint16_t *const *x_hosts, uint16_t *const *y_hosts,
                                        int n_batches, const float *Wr, const float *bias,
                                        const uint16_t *W1, const uint16_t *W2, int T, int d, int E,
                                        int K, int f, void *workspace, size_t workspace_bytes,
                                        cudaStream_t stream);

/* ---------------------------------------------------------------------------
 * MXFP8 path ("Optimization 1: Grouped GEMM": on Blackwell the expert
 * matmuls run with MXFP8 block scaling, fed by grouped quantisation).
 * Format: E4M3 element codes (uint8), one scale byte s (value 2^(s-127)) per
 * 32 consecutive elements along the reduction dimension; s is the smallest
 * power of two with 448 * 2^(s-127) >= the block's largest magnitude, and
 * each code is the element / 2^(s-127) rounded to nearest E4M3, ties to
 * even.  Scales are stored as 512-byte atoms of 128 rows x 128 columns
 * (4 blocks), byte (row % 32) * 16 + ((row % 128) / 32) * 4 + block.
 * Requires d and f to be multiples of 128.  Codes and scale buffers are
 * 16-byte aligned device memory owned by the caller.
 * ------------------------------------------------------------------------ */

/* Quantises a row-major bf16 matrix [rows, K] (K a multiple of 128) along K:
 * codes [rows, K]; scale atoms for row block rb = row / 128 and column slice
 * ks = k / 128 at byte offset (rb * (K / 128) + ks) * 512 of `scales`, which
 * must hold moe_mxfp8_scales_size(rows, K) bytes.  The expert weights are
 * quantised with this once: W1 as [E * 2f, d], W2 as [E * d, f].  */
size_t moe_mxfp8_scales_size(int rows, int K);
moe_status_t moe_mxfp8_quantize(const uint16_t *src, int rows, int K, uint8_t *codes, uint8_t *scales,
                                cudaStream_t stream);

/* Scale atoms of the permuted activations [TK, K] (rows grouped by expert
 * by `offsets`): the rows of each expert group are cut into 128-row blocks
 * from the group's first row; block b of expert e is row block
 * rb = sum_{e'<e} ceil(count[e'] / 128) + b.  Size bound: */
size_t moe_mxfp8_act_scales_size(int TK, int E, int K);

/* Step a3 with quantisation: every token row of x [T, d] bf16 is quantised
 * once and its codes written to the K rows of xq_perm [TK, d] it occupies
 * (row_of), with its scales into those rows' atoms of `sfa`.  */
moe_status_t moe_permute_mxfp8(const uint16_t *x, const int32_t *topk_idx, const int32_t *row_of,
                               const int32_t *offsets, int T, int K, int d, int E, uint8_t *xq_perm,
                               uint8_t *sfa, size_t sfa_bytes, cudaStream_t stream);

/* Steps a4 and a5 in MXFP8.  GEMM1: h = silu(x.W1g^T) * (x.W1u^T) from the
 * dequantised operands with fp32 accumulation, then quantised along f into
 * hq [TK, f] and the atoms `sfh` (grouped layout).  GEMM2: y_perm [TK, d]
 * bf16 = hq.W2q^T (fp32 accumulation).  W1s / W2s are the weight scales from
 * moe_mxfp8_quantize.  */
moe_status_t moe_grouped_gemm1_swiglu_mxfp8(const uint8_t *xq_perm, const uint8_t *sfa, size_t sfa_bytes,
                                            const int32_t *offsets, int E, int TK, int d, int f,
                                            const uint8_t *W1q, const uint8_t *W1s, uint8_t *hq, uint8_t *sfh,
                                            size_t sfh_bytes, cudaStream_t stream);
moe_status_t moe_grouped_gemm2_mxfp8(const uint8_t *hq, const uint8_t *sfh, size_t sfh_bytes,
                                     const int32_t *offsets, int E, int TK, int d, int f, const uint8_t *W2q,
                                     const uint8_t *W2s, uint16_t *y_perm, cudaStream_t stream);

/* The whole layer with MXFP8 expert matmuls (router, routing and combine as
 * in moe_forward; 9 kernel launches), weights pre-quantised by
 * moe_mxfp8_quantize.  */
size_t moe_forward_mxfp8_workspace_size(int T, int d, int E, int K, int f);
typedef struct {
    size_t logits, topk_idx, topk_w, counts, offsets, row_of, src_tok, route_ws, router_ws,
           xq_perm, sfa, hq, sfh, y_perm, total;
} moe_forward_mxfp8_layout_t;
moe_status_t moe_forward_mxfp8_views(int T, int d, int E, int K, int f, moe_forward_mxfp8_layout_t *layout);
moe_status_t moe_forward_mxfp8(const uint16_t *x, const float *Wr, const float *bias, const uint8_t *W1q,
                               const uint8_t *W1s, const uint8_t *W2q, const uint8_t *W2s, int T, int d,
                               int E, int K, int f, uint16_t *y, void *workspace, size_t workspace_bytes,
                               cudaStream_t stream);
/* The same over n_batches host batches with overlapped copies (see
 * moe_forward_host_pipelined): the layer's MXFP8 workspace followed by two x
 * and two y buffers.  */
size_t moe_forward_mxfp8_host_pipelined_workspace_size(int T, int d, int E, int K, int f);
moe_status_t moe_forward_mxfp8_host_pipelined(const uint16_t *const *x_hosts, uint16_t *const *y_hosts,
                                              int n_batches, const float *Wr, const float *bias,
                                              const uint8_t *W1q, const uint8_t *W1s,
                                              const uint8_t *W2q, const uint8_t *W2s, int T, int d,
                                              int E, int K, int f, void *workspace,
                                              size_t workspace_bytes, cudaStream_t stream);

/* ---------------------------------------------------------------------------
 * Backward of the layer (the pages are about MoE training; they give no
 * backward formula, so these are the gradients of the forward's definition
 * for an output gradient dy: no gradient through the choice of the K
 * experts, softmax over the K selected logits).
 *   dx [T, d] bf16; dWr [d, E], dbias [E], dW1 [E, 2f, d], dW2 [E, d, f]
 *   fp32 (every expert's entries written, zeros for experts without tokens).
 * `fwd_workspace` is the workspace of a moe_forward_train call on the same
 * x and weights (it holds the routing, x_perm, h and y_perm the backward
 * reuses), or of a moe_forward call on sizes for which
 * moe_forward_fuses_permute() is 0 (elsewhere moe_forward leaves x_perm
 * unwritten: run moe_permute into its x_perm region first);
 * `preact` (nullable) the pre-activations a moe_forward_train call saved --
 * when null they are computed again (one more grouped GEMM, into the
 * workspace region `a`); `workspace` (128-byte aligned) holds
 * moe_backward_workspace_size() bytes of scratch (moe_backward_views() gives
 * its regions; `tmaps` holds 256 bytes per expert of tensor maps that the
 * weight-gradient GEMMs build on the device, one pair per expert group).  The dgrad GEMMs run on the
 * forward's grouped GEMM reading W1 and W2 as stored (MN-major operands),
 * the weight gradients on a grouped GEMM whose reduction runs over each
 * expert's own rows, read from the grouped activations in place.  All sums
 * have a fixed order: the gradients are deterministic.  13 kernel launches
 * (14 without `preact`).  */
size_t moe_backward_workspace_size(int T, int d, int E, int K, int f);
typedef struct {
    size_t dw, dl, dl_row, dy_perm, dh, a, da, dx_perm, WrT, rw_part, tmaps, total;
} moe_backward_layout_t;
moe_status_t moe_backward_views(int T, int d, int E, int K, int f, moe_backward_layout_t *layout);
moe_status_t moe_backward(const uint16_t *x, const float *Wr, const float *bias, const uint16_t *W1,
                          const uint16_t *W2, int T, int d, int E, int K, int f, const uint16_t *dy,
                          const void *fwd_workspace, size_t fwd_workspace_bytes,
                          const uint16_t *preact, uint16_t *dx, float *dWr, float *dbias,
                          float *dW1, float *dW2, void *workspace,
                          size_t workspace_bytes, cudaStream_t stream);

/* Reads and clears the device status word of the current device (0 = OK, or
 * a moe_status_t a kernel recorded).  Synchronous: call outside capture. */
moe_status_t moe_device_status(int *status_out);

/* The same read, asynchronous and capture-safe ("What specialized
 * optimizations are needed for dropless MoE?": no value may cross to the CPU
 * inside a captured step, so that CUDA graphs work): one kernel on `stream`
 * copies the device status word of the current device into the caller's
 * device word `dev_status_word` (int32, 4-byte aligned, caller-owned) and
 * clears the status word, atomically.  Queued after a layer's kernels on the
 * same stream, it reports what they recorded (0, or MOE_ERR_DEVICE_TIMEOUT);
 * it can be captured into a CUDA graph with them and replayed.  The status
 * word is shared by every stream of the device, so a read also reports and
 * clears what kernels of other streams recorded before it ran.  Returns
 * MOE_ERR_INVALID_ARG for a null or misaligned pointer (nothing launched),
 * MOE_ERR_CUDA if the launch fails.  One kernel launch.  */
moe_status_t moe_last_device_status(int32_t *dev_status_word, cudaStream_t stream);

/* Exercises the failure path of the device-side waits: launches one kernel
 * whose single wait can never complete.  After limit_ns (1 us .. 1 s) it
 * gives up, records MOE_ERR_DEVICE_TIMEOUT in the device status word (read
 * it with moe_device_status()) and returns; the CUDA context stays usable.
 * Returns MOE_OK when the launch succeeded.  */
moe_status_t moe_check_bounded_wait(uint64_t limit_ns, cudaStream_t stream);

/* Number of kernels this library has launched in this process. */
uint64_t moe_launch_count(void);

#ifdef __cplusplus
}
#endif
#endif /* MOE_GB300_H */
