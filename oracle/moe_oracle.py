"""Oracle for the dropless MoE layer forward -- TEST INFRASTRUCTURE ONLY.

Plain, slow, obviously correct CPU implementation of what the layer computes.
Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline
and reference legs may import it.  It shares no code with the CUDA library
and never imports it.

Source page: "Accelerating dropless MoE training in JAX with NVIDIA Transformer
Engine".  Passages followed:
  * introduction -- a learned router picks the Top-K experts of each token;
  * "How is dropless MoE different from capacity-based MoE?" -- every token is
    processed by the experts it chose, whatever the load: no drop, no padding;
  * Figure 3 caption -- dispatch moves tokens to their experts, the grouped MLP
    runs two grouped GEMMs over the variable-length groups, combine reverses
    the exchange and restores the original token order;
  * "Optimization 1: Grouped GEMM" -- each expert's matmul uses its actual
    token count and only rows holding valid tokens are computed.

Readings where the page is silent (the page never names softmax, SwiGLU or
the row order inside a group):
  * gate weights: softmax over the K selected logits (they sum to 1);
  * selection order: descending logit, equal logits -> lower expert index,
    -0.0 equals +0.0 (IEEE comparison);
  * rows of an expert group: ascending token index (a stable counting sort of
    the token-major (t, k) list by expert);
  * expert FFN: SwiGLU, W1 rows 0..f-1 = gate (silu applied), rows f..2f-1 =
    up, silu(z) = z / (1 + exp(-z)), then W2 maps f -> d;
  * combine: y[t] = sum over k = 0..K-1 (ascending) of w[t,k] * y_row.

Precision: the router logits are fp32 by definition (``router_fp32.c``,
which fixes their rounding exactly); everything after them -- gate weights,
the two expert matmuls, SwiGLU and the combine -- is fp64 with no
intermediate rounding.  Pins: ``tests/test_oracle.py``.
"""
from __future__ import annotations

import ctypes
import os

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB = None


def _lib():
    global _LIB
    if _LIB is None:
        path = os.path.join(_HERE, "liboracle_router.so")
        if not os.path.exists(path):
            from . import build as _b
            _b.build()
        lib = ctypes.CDLL(path)
        lib.oracle_router_logits_fp32.restype = None
        lib.oracle_router_logits_fp32.argtypes = [
            ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
            ctypes.c_int64, ctypes.c_int64, ctypes.c_int64, ctypes.c_void_p, ctypes.c_int]
        _LIB = lib
    return _LIB


def host_threads() -> int:
    return len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else (os.cpu_count() or 1)


# --------------------------------------------------------------------------
# a0: router logits
# --------------------------------------------------------------------------
def router_logits_fp32(x, Wr, bias=None, nthreads: int | None = None) -> np.ndarray:
    """fp32 logits L[T,E]: index-ordered fused multiply-add chain, then + bias.

    x: [T,d] values exactly representable in fp32 (the layer's bf16 tokens);
    Wr: [d,E] fp32; bias: [E] fp32 or None.  (Introduction: the learned
    router that picks the Top-K experts.)
    """
    x = np.ascontiguousarray(x, dtype=np.float32)
    Wr = np.ascontiguousarray(Wr, dtype=np.float32)
    T, d = x.shape
    d2, E = Wr.shape
    assert d == d2
    L = np.empty((T, E), dtype=np.float32)
    b = None if bias is None else np.ascontiguousarray(bias, dtype=np.float32)
    _lib().oracle_router_logits_fp32(
        x.ctypes.data, Wr.ctypes.data, None if b is None else b.ctypes.data,
        T, d, E, L.ctypes.data, nthreads or host_threads())
    return L


def router_logits_fp64(x, Wr, bias=None) -> np.ndarray:
    """Exact-as-fp64 logits x.Wr + bias, used only to bound the fp32 ones."""
    L = np.asarray(x, np.float64) @ np.asarray(Wr, np.float64)
    if bias is not None:
        L = L + np.asarray(bias, np.float64)[None, :]
    return L


# --------------------------------------------------------------------------
# a1: top-K selection and gate weights
# --------------------------------------------------------------------------
def topk_route(L, K: int):
    """Per token the K largest logits (descending; equal -> lower expert index)
    and their softmax weights in fp64.  Returns (idx [T,K] int32, w [T,K] f64).

    The stable sort of -L keeps equal logits in ascending expert order, and
    numpy's comparison treats -0.0 and +0.0 as equal.
    """
    L = np.asarray(L, dtype=np.float32)
    T, E = L.shape
    assert 1 <= K <= E
    order = np.argsort(-L, axis=1, kind="stable")[:, :K]
    top = np.take_along_axis(L, order, axis=1).astype(np.float64)
    z = np.exp(top - top[:, :1])
    w = z / z.sum(axis=1, keepdims=True)
    return order.astype(np.int32), w


# --------------------------------------------------------------------------
# a2: histogram, offsets, stable dispatch order
# --------------------------------------------------------------------------
def expert_counts(idx, E: int):
    """counts[e] = number of (t, k) routed to e; offsets = exclusive scan (E+1)."""
    counts = np.bincount(np.asarray(idx).ravel(), minlength=E).astype(np.int64)
    offsets = np.zeros(E + 1, dtype=np.int64)
    offsets[1:] = np.cumsum(counts)
    return counts, offsets


def dispatch_order(idx, E: int):
    """Stable counting sort of the token-major list of (t, k) by expert.

    Returns src_tok [TK] (token held by row r) and row_of [T,K] (row that holds
    token t's k-th choice).  Rows of expert e are offsets[e]..offsets[e+1]-1,
    in ascending token order.
    """
    idx = np.asarray(idx)
    T, K = idx.shape
    flat = idx.ravel()                            # pair p = t*K + k
    rows = np.argsort(flat, kind="stable")        # row r holds pair rows[r]
    src_tok = (rows // K).astype(np.int64)
    row_of = np.empty(T * K, dtype=np.int64)
    row_of[rows] = np.arange(T * K)
    return src_tok, row_of.reshape(T, K)


# --------------------------------------------------------------------------
# a3..a6: permute, expert SwiGLU FFN, combine
# --------------------------------------------------------------------------
def permute(x, src_tok):
    """Dispatch on one device: x_perm[r] = x[src_tok[r]] (Figure 3 caption)."""
    return np.asarray(x)[np.asarray(src_tok)]


def silu(z):
    return z / (1.0 + np.exp(-z))


def expert_ffn(X, W1e, W2e):
    """One expert's SwiGLU FFN on rows X [n,d] in fp64.

    a = X W1e^T (2f), gate g = a[:, :f], up u = a[:, f:], h = silu(g) * u,
    y = h W2e^T.  Returns (h [n,f], y [n,d]).
    """
    X = np.asarray(X, np.float64)
    W1e = np.asarray(W1e, np.float64)
    W2e = np.asarray(W2e, np.float64)
    f = W1e.shape[0] // 2
    a = X @ W1e.T
    h = silu(a[:, :f]) * a[:, f:]
    return h, h @ W2e.T


def grouped_mlp(x_perm, offsets, W1, W2, weight_fn=None):
    """The grouped MLP: for each expert e, its FFN over rows
    offsets[e]..offsets[e+1]-1 with the group's actual row count ("Optimization
    1: Grouped GEMM").  Empty groups do nothing.  ``weight_fn(e)`` may return
    (W1e, W2e) for callers that keep the weights elsewhere."""
    TK = x_perm.shape[0]
    E = len(offsets) - 1
    h = y = None
    for e in range(E):
        r0, r1 = int(offsets[e]), int(offsets[e + 1])
        if r1 == r0:
            continue
        W1e, W2e = (W1[e], W2[e]) if weight_fn is None else weight_fn(e)
        he, ye = expert_ffn(x_perm[r0:r1], W1e, W2e)
        if h is None:
            h = np.zeros((TK, he.shape[1]), np.float64)
            y = np.zeros((TK, ye.shape[1]), np.float64)
        h[r0:r1] = he
        y[r0:r1] = ye
    return h, y


def combine(y_perm, row_of, w):
    """Combine on one device: y[t] = sum_k w[t,k] * y_perm[row_of[t,k]],
    k ascending, fp64 (Figure 3 caption: restore the original token order)."""
    y_perm = np.asarray(y_perm, np.float64)
    row_of = np.asarray(row_of)
    w = np.asarray(w, np.float64)
    T, K = row_of.shape
    y = np.zeros((T, y_perm.shape[1]), np.float64)
    for k in range(K):
        y += w[:, k:k + 1] * y_perm[row_of[:, k]]
    return y


def forward(x, Wr, bias, W1, W2, K: int, nthreads: int | None = None):
    """The whole layer, step by step; returns every intermediate.

    x [T,d] (bf16 values as fp32), Wr [d,E] fp32, bias [E] fp32 or None,
    W1 [E,2f,d], W2 [E,d,f] (bf16 values as fp32 or fp64).
    """
    x = np.asarray(x, np.float32)
    E = np.asarray(Wr).shape[1]
    L = router_logits_fp32(x, Wr, bias, nthreads)
    idx, w = topk_route(L, K)
    counts, offsets = expert_counts(idx, E)
    src_tok, row_of = dispatch_order(idx, E)
    x_perm = permute(x, src_tok)
    h, y_perm = grouped_mlp(x_perm, offsets, W1, W2)
    y = combine(y_perm, row_of, w)
    return dict(logits=L, idx=idx, w=w, counts=counts, offsets=offsets,
                src_tok=src_tok, row_of=row_of, x_perm=x_perm, h=h, y_perm=y_perm, y=y)


def forward_tokens(tokens, x_rows, L_rows, K: int, expert_weights):
    """y for a few tokens straight from the definition, for checks at full size.

    tokens: their indices (for bookkeeping only); x_rows [n,d] and L_rows [n,E]
    their activations and fp32 logits; expert_weights(e) -> (W1e, W2e).  A
    token's output depends only on its own logits and its K experts, so no other
    token is needed.  Returns (idx, w, h [n,K,f], y_rows [n,K,d], y [n,d]).
    """
    idx, w = topk_route(L_rows, K)
    n = len(tokens)
    cache = {}
    hs, ys = [None] * n, [None] * n
    for e in sorted(set(int(v) for v in np.asarray(idx).ravel())):
        cache[e] = expert_weights(e)
        for i in range(n):
            for k in range(K):
                if idx[i, k] == e:
                    he, ye = expert_ffn(np.asarray(x_rows[i:i + 1], np.float64), *cache[e])
                    if hs[i] is None:
                        hs[i] = np.zeros((K, he.shape[1]))
                        ys[i] = np.zeros((K, ye.shape[1]))
                    hs[i][k] = he[0]
                    ys[i][k] = ye[0]
        del cache[e]
    h = np.stack(hs)
    yk = np.stack(ys)
    y = np.zeros((n, yk.shape[2]))
    for k in range(K):
        y += w[:, k:k + 1] * yk[:, k]
    return idx, w, h, yk, y
