"""MXFP8 oracle of the dropless MoE layer forward -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU legs may
use it; it shares no code with the CUDA library and never imports it.

Source page: "Accelerating dropless MoE training in JAX with NVIDIA Transformer
Engine", "Optimization 1: Grouped GEMM" (last paragraph): on Blackwell the
grouped GEMM path also runs the expert matmuls with MXFP8 block scaling, fed
by grouped quantisation kernels.  The page names the format only; the format
itself and the readings taken here:
  * MXFP8 E4M3: every block of 32 consecutive elements along the reduction
    dimension shares one power-of-two scale X = 2^e, stored as an unsigned
    8-bit exponent code e + 127 (UE8M0); each element is stored as an FP8
    E4M3 value (1 sign, 4 exponent bits with bias 7, 3 mantissa bits,
    subnormals, largest finite 448, no infinities, S.1111.111 is NaN).
  * the scale of a block: the smallest power of two with 448 X >= amax, so
    that no element of the block saturates (for amax = m 2^E, 1 <= m < 2:
    e = E - 8, or E - 7 when m > 1.75); a block of zeros gets e = -127;
  * elements: V / X rounded to the nearest E4M3 value, ties to even
    mantissa; the sign of a zero is kept;
  * which tensors are quantised: the token activations (blocks along d), W1
    (blocks along d), the SwiGLU output h (blocks along f) and W2 (blocks
    along f).  Accumulation is exact here (fp64), the router and the
    combine are the same as in the bf16 oracle, and y_perm is the fp64
    product of the dequantised h and W2.
Pins: ``tests/test_oracle_mxfp8.py``.
"""
from __future__ import annotations

import numpy as np

from .moe_oracle import combine, dispatch_order, expert_counts, router_logits_fp32, silu, topk_route

E4M3_MAX = 448.0
BLOCK = 32


def e4m3_decode(codes) -> np.ndarray:
    """Values of E4M3 codes (uint8) as fp64; NaN for S.1111.111."""
    c = np.asarray(codes, np.uint8).astype(np.int64)
    sign = np.where(c & 0x80, -1.0, 1.0)
    exp = (c >> 3) & 0xF
    man = c & 0x7
    mag = np.where(exp == 0, man * 2.0 ** -9, (8 + man) * 2.0 ** (exp - 10))
    mag = np.where((exp == 0xF) & (man == 0x7), np.nan, mag)
    return sign * mag


def e4m3_round(v) -> np.ndarray:
    """v (fp64) rounded to the nearest E4M3 value, ties to even, saturating at
    +-448; the sign of zero is kept."""
    v = np.asarray(v, np.float64)
    a = np.abs(v)
    _, ex = np.frexp(a)                     # a = f 2^ex, 0.5 <= f < 1
    k = np.maximum(ex - 1, -6)              # binade of a; below 2^-6 the subnormal spacing
    step = np.ldexp(1.0, k - 3)             # 3 mantissa bits
    q = np.minimum(np.rint(a / step) * step, E4M3_MAX)
    return np.copysign(q, v)


def e4m3_encode(q) -> np.ndarray:
    """Codes of E4M3 values (exactly representable, as from e4m3_round)."""
    q = np.asarray(q, np.float64)
    a = np.abs(q)
    _, ex = np.frexp(a)
    k = ex - 1
    normal = a >= 2.0 ** -6
    kk = np.where(normal, k, -6)
    exp_field = np.where(normal, k + 7, 0)
    man = np.where(normal, np.ldexp(a, -kk) * 8 - 8, np.ldexp(a, 9))
    man = np.rint(man).astype(np.int64)
    assert np.all((man >= 0) & (man < 8)), "value not representable in E4M3"
    code = (np.signbit(q).astype(np.int64) << 7) | (exp_field.astype(np.int64) << 3) | man
    return code.astype(np.uint8)


def mx_scale_exponent(amax) -> np.ndarray:
    """e of the block scale 2^e: the smallest power of two with 448 2^e >= amax."""
    amax = np.asarray(amax, np.float64)
    f, ex = np.frexp(amax)                  # amax = (2f) 2^(ex-1), 1 <= 2f < 2
    e = (ex - 1) - 8 + (2.0 * f > 1.75)
    e = np.where(amax < 2.0 ** -126, -127, e)   # zero (or below the fp32 normal range)
    return np.clip(e, -127, 127).astype(np.int64)


def _mx_quantize_rows(V):
    """mx_quantize of a 2-D block of rows [R, K]."""
    R, K = V.shape
    blocks = V.reshape(R, K // BLOCK, BLOCK)
    e = mx_scale_exponent(np.max(np.abs(blocks), axis=-1))
    X = np.ldexp(1.0, e)[..., None]
    q = e4m3_round(blocks / X)
    return e4m3_encode(q).reshape(R, K), (e + 127).astype(np.uint8), (q * X).reshape(R, K)


def mx_quantize(V):
    """Blocks of 32 along the last axis of V [..., K] (K a multiple of 32).
    Returns (codes uint8 [..., K], scale codes uint8 [..., K/32], dequantised
    fp64 [..., K]).  Every block lies within one row, so the rows are taken a
    few thousand elements' worth at a time (the same values; only the size of
    numpy's temporaries changes)."""
    V = np.asarray(V, np.float64)
    K = V.shape[-1]
    assert K % BLOCK == 0
    lead = V.shape[:-1]
    V2 = V.reshape(-1, K)
    R = V2.shape[0]
    codes = np.empty((R, K), np.uint8)
    scales = np.empty((R, K // BLOCK), np.uint8)
    deq = np.empty((R, K), np.float64)
    step = max(1, (1 << 20) // max(K, 1))
    for r0 in range(0, R, step):
        r1 = min(R, r0 + step)
        codes[r0:r1], scales[r0:r1], deq[r0:r1] = _mx_quantize_rows(V2[r0:r1])
    return codes.reshape(V.shape), scales.reshape(lead + (K // BLOCK,)), deq.reshape(V.shape)


def mx_dequantize(codes, scale_codes) -> np.ndarray:
    """Inverse of mx_quantize for valid codes: value = E4M3(code) * 2^(s - 127)."""
    c = np.asarray(codes, np.uint8)
    K = c.shape[-1]
    s = np.asarray(scale_codes, np.uint8).astype(np.int64) - 127
    vals = e4m3_decode(c).reshape(c.shape[:-1] + (K // BLOCK, BLOCK))
    return (vals * np.ldexp(1.0, s)[..., None]).reshape(c.shape)


def expert_ffn_mxfp8(x_rows, W1d_e, W2d_e):
    """One expert's MXFP8 SwiGLU FFN on a few of its token rows, for checks at
    full size.  x_rows [n, d] (bf16 values), W1d_e [2f, d] and W2d_e [d, f]
    the expert's dequantised MXFP8 weights (mx_quantize(...)[2]).  A row's
    result depends only on its own token and the expert: the token row is
    quantised in blocks of 32 along d, h = silu(g) * u in fp64 from the
    dequantised operands, h quantised in blocks of 32 along f, and
    y_perm = dequantised h times W2d_e^T in fp64.  Returns a dict with xq, xs,
    h, hq, hs, hd and y_perm."""
    f = np.asarray(W1d_e).shape[0] // 2
    xq, xs, xd = mx_quantize(np.asarray(x_rows, np.float32))
    a = xd @ np.asarray(W1d_e, np.float64).T
    h = silu(a[:, :f]) * a[:, f:]
    hq, hs, hd = mx_quantize(h)
    y_perm = hd @ np.asarray(W2d_e, np.float64).T
    return dict(xq=xq, xs=xs, h=h, hq=hq, hs=hs, hd=hd, y_perm=y_perm)


def forward_mxfp8_tokens(x_rows, L_rows, K: int, expert_weights):
    """y with MXFP8 expert matmuls for a few tokens, from their own fp32
    logits L_rows [n, E] and activations x_rows [n, d]; expert_weights(e) ->
    (W1d_e, W2d_e) dequantised.  Returns (idx, w, per-slot results
    [n][K] of expert_ffn_mxfp8 for one row, y [n, d])."""
    idx, w = topk_route(L_rows, K)
    n = idx.shape[0]
    slots = [[None] * K for _ in range(n)]
    for e in sorted(set(int(v) for v in np.asarray(idx).ravel())):
        W1d_e, W2d_e = expert_weights(e)
        at = [(i, k) for i in range(n) for k in range(K) if idx[i, k] == e]
        res = expert_ffn_mxfp8(np.asarray(x_rows)[[i for i, _ in at]], W1d_e, W2d_e)
        for j, (i, k) in enumerate(at):
            slots[i][k] = {name: val[j] for name, val in res.items()}
    y = np.zeros((n, np.asarray(x_rows).shape[1]))
    for i in range(n):
        for k in range(K):
            y[i] += w[i, k] * slots[i][k]["y_perm"]
    return idx, w, slots, y


def forward_mxfp8(x, Wr, bias, W1, W2, K: int, nthreads: int | None = None):
    """The layer with MXFP8 expert matmuls, step by step; returns every
    intermediate.  x [T,d], Wr [d,E], bias [E] or None, W1 [E,2f,d] and
    W2 [E,d,f] (bf16 values as fp32)."""
    x = np.asarray(x, np.float32)
    W1 = np.asarray(W1, np.float64)
    W2 = np.asarray(W2, np.float64)
    E, two_f, d = W1.shape
    f = two_f // 2
    L = router_logits_fp32(x, Wr, bias, nthreads)
    idx, w = topk_route(L, K)
    counts, offsets = expert_counts(idx, E)
    src_tok, row_of = dispatch_order(idx, E)
    xq, xs, xd = mx_quantize(x)
    _, _, W1d = mx_quantize(W1)
    _, _, W2d = mx_quantize(W2)
    TK = src_tok.shape[0]
    x_perm = xd[src_tok]
    h = np.zeros((TK, f))
    for e in range(E):
        r0, r1 = offsets[e], offsets[e + 1]
        if r1 > r0:
            a = x_perm[r0:r1] @ W1d[e].T
            h[r0:r1] = silu(a[:, :f]) * a[:, f:]
    hq, hs, hd = mx_quantize(h)
    y_perm = np.zeros((TK, d))
    for e in range(E):
        r0, r1 = offsets[e], offsets[e + 1]
        if r1 > r0:
            y_perm[r0:r1] = hd[r0:r1] @ W2d[e].T
    y = combine(y_perm, row_of, w)
    return dict(logits=L, idx=idx, w=w, counts=counts, offsets=offsets, src_tok=src_tok, row_of=row_of,
                xq=xq, xs=xs, x_perm=x_perm, h=h, hq=hq, hs=hs, hd=hd, y_perm=y_perm, y=y)
