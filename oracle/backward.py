"""Backward of the dropless MoE layer -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU legs may
use it; it shares no code with the CUDA library and never imports it.

The pages are about MoE training ("Accelerating dropless MoE training in JAX
with NVIDIA Transformer Engine", introduction: the MoE layer inside a training
step) but give no backward formula; the gradients below are those of the
forward's definition (oracle/moe_oracle.py) for a loss whose gradient with
respect to the layer output is dy, i.e. loss = sum(dy * y).  Readings:
  * the top-K selection is piecewise constant in the logits: no gradient
    flows through the choice of experts, only through the K gate weights;
  * gate weights are a softmax over the K selected logits, so
    dl_k = w_k (dw_k - sum_j w_j dw_j) for the selected experts and 0 for
    the others;
  * silu'(g) = s + g s (1 - s) with s = sigmoid(g).
Everything is fp64 with no intermediate rounding.  Pins (central finite
differences of ``forward_fp64`` and closed forms): tests/test_oracle_backward.py.
"""
from __future__ import annotations

import numpy as np

from .moe_oracle import combine, dispatch_order, expert_counts, router_logits_fp64, silu


def forward_fp64(x, Wr, bias, W1, W2, K: int):
    """The layer's forward in fp64 throughout (router included), for finite
    differences: y [T, d]."""
    x = np.asarray(x, np.float64)
    W1 = np.asarray(W1, np.float64)
    W2 = np.asarray(W2, np.float64)
    E, two_f, _ = W1.shape
    f = two_f // 2
    L = router_logits_fp64(x, Wr, bias)
    # top-K and softmax in fp64 (topk_route rounds the logits to fp32, the
    # layer's contract, which would quantise finite differences)
    idx = np.argsort(-L, axis=1, kind="stable")[:, :K].astype(np.int32)
    top = np.take_along_axis(L, idx, axis=1)
    z = np.exp(top - top[:, :1])
    w = z / z.sum(axis=1, keepdims=True)
    _, offsets = expert_counts(idx, E)
    src_tok, row_of = dispatch_order(idx, E)
    x_perm = x[src_tok]
    y_perm = np.zeros((len(src_tok), x.shape[1]))
    for e in range(E):
        r0, r1 = offsets[e], offsets[e + 1]
        if r1 > r0:
            a = x_perm[r0:r1] @ W1[e].T
            y_perm[r0:r1] = (silu(a[:, :f]) * a[:, f:]) @ W2[e].T
    return combine(y_perm, row_of, w)


def backward(x, Wr, bias, W1, W2, K: int, dy, routing):
    """Gradients of sum(dy * y) for the routing given (``routing``: a dict
    with idx, w, offsets, src_tok, row_of, e.g. the output of
    oracle.forward).  Returns dx [T,d], dWr [d,E], dbias [E], dW1 [E,2f,d],
    dW2 [E,d,f] and the intermediates dw [T,K], dy_perm, dh, da, dx_perm
    (rows grouped by expert) and dL [T,E]."""
    x = np.asarray(x, np.float64)
    Wr = np.asarray(Wr, np.float64)
    W1 = np.asarray(W1, np.float64)
    W2 = np.asarray(W2, np.float64)
    dy = np.asarray(dy, np.float64)
    idx, w = np.asarray(routing["idx"]), np.asarray(routing["w"], np.float64)
    offsets, src_tok, row_of = routing["offsets"], routing["src_tok"], routing["row_of"]
    T, d = x.shape
    E, two_f, _ = W1.shape
    f = two_f // 2
    TK = len(src_tok)
    x_perm = x[src_tok]

    # expert FFNs, forward again in fp64 (pre-activations, h, y rows)
    a = np.zeros((TK, two_f))
    h = np.zeros((TK, f))
    y_perm = np.zeros((TK, d))
    for e in range(E):
        r0, r1 = offsets[e], offsets[e + 1]
        if r1 > r0:
            a[r0:r1] = x_perm[r0:r1] @ W1[e].T
            h[r0:r1] = silu(a[r0:r1, :f]) * a[r0:r1, f:]
            y_perm[r0:r1] = h[r0:r1] @ W2[e].T

    # combine: y[t] = sum_k w[t,k] y_perm[row_of[t,k]]
    dw = np.einsum("tkc,tc->tk", y_perm[row_of], dy)
    dy_perm = np.zeros((TK, d))
    dy_perm[row_of] = w[:, :, None] * dy[:, None, :]

    # experts: y_row = h W2^T, h = silu(g) u, (g, u) = x_row W1^T
    dh = np.zeros((TK, f))
    da = np.zeros((TK, two_f))
    dx_perm = np.zeros((TK, d))
    dW1 = np.zeros_like(W1)
    dW2 = np.zeros_like(W2)
    for e in range(E):
        r0, r1 = offsets[e], offsets[e + 1]
        if r1 == r0:
            continue
        g, u = a[r0:r1, :f], a[r0:r1, f:]
        s = 1.0 / (1.0 + np.exp(-g))
        dh[r0:r1] = dy_perm[r0:r1] @ W2[e]
        dW2[e] = dy_perm[r0:r1].T @ h[r0:r1]
        da[r0:r1, :f] = dh[r0:r1] * u * (s + g * s * (1.0 - s))
        da[r0:r1, f:] = dh[r0:r1] * g * s
        dx_perm[r0:r1] = da[r0:r1] @ W1[e]
        dW1[e] = da[r0:r1].T @ x_perm[r0:r1]

    # router: w = softmax over the K selected logits, L = x Wr + bias
    dl = w * (dw - np.sum(w * dw, axis=1, keepdims=True))
    dL = np.zeros((T, E))
    np.put_along_axis(dL, idx, dl, axis=1)
    dbias = dL.sum(axis=0)
    dWr = x.T @ dL

    dx = dL @ Wr.T
    for k in range(K):
        dx += dx_perm[row_of[:, k]]
    return dict(dx=dx, dWr=dWr, dbias=dbias, dW1=dW1, dW2=dW2, dw=dw, dy_perm=dy_perm, dh=dh, da=da,
                dx_perm=dx_perm, dL=dL, a=a, h=h, y_perm=y_perm)


def backward_sampled(x, Wr, bias, W1, W2, K: int, dy, routing, dW1_at=(), dW2_at=(), dx_at=()):
    """Selected elements of backward()'s gradients, each evaluated from the
    same definitions with only the rows it needs, for checks at sizes where
    the full backward is too slow: dW1[e, i, j] for (e, i, j) in dW1_at,
    dW2[e, i, j] for (e, i, j) in dW2_at and dx[t] for t in dx_at.

    With every value comes S, the sum of the magnitudes of its terms carried
    through each intermediate that is itself a sum (dh from |dy_perm|·|W2|,
    the two terms of silu' separately, dw from |dy|·|y_perm|, dl from the
    softmax's terms), for an error bound that scales with the terms rather
    than with a result that cancels.  fp64; W1, W2 may be given in fp32.
    Returns dict(dW1=[(value, S)], dW2=[...], dx=[(row [d], S row [d])])."""
    x = np.asarray(x, np.float64)
    Wr = np.asarray(Wr, np.float64)
    dy = np.asarray(dy, np.float64)
    idx, w = np.asarray(routing["idx"]), np.asarray(routing["w"], np.float64)
    offsets, src_tok, row_of = routing["offsets"], routing["src_tok"], routing["row_of"]
    E, two_f, d = W1.shape
    f = two_f // 2
    # the slot k of each row r: row_of[t, k] = r
    slot = np.zeros(len(src_tok), np.int64)
    for k in range(K):
        slot[row_of[:, k]] = k

    def group(e):
        rows = np.arange(offsets[e], offsets[e + 1])
        toks = src_tok[rows]
        return toks, w[toks, slot[rows]]            # the tokens of the group and their gate weights

    out = dict(dW1=[], dW2=[], dx=[])
    for e, i, j in dW2_at:                           # dW2[e, i, j] = sum_r dy_perm[r, i] h[r, j]
        toks, wr = group(e)
        g = x[toks] @ np.asarray(W1[e][j], np.float64)
        u = x[toks] @ np.asarray(W1[e][f + j], np.float64)
        h = silu(g) * u
        dyp = wr * dy[toks, i]
        out["dW2"].append((float(np.sum(dyp * h)), float(np.sum(np.abs(dyp) * np.abs(h)))))
    for e, i, j in dW1_at:                           # dW1[e, i, j] = sum_r da[r, i] x_perm[r, j]
        toks, wr = group(e)
        c = i % f                                    # the feature of the gate (i < f) or up (i >= f) row
        g = x[toks] @ np.asarray(W1[e][c], np.float64)
        u = x[toks] @ np.asarray(W1[e][f + c], np.float64)
        s = 1.0 / (1.0 + np.exp(-g))
        dyp = wr[:, None] * dy[toks]                 # dy_perm rows [n, d]
        w2c = np.asarray(W2[e][:, c], np.float64)
        dh = dyp @ w2c
        dh_mag = np.abs(dyp) @ np.abs(w2c)
        if i < f:
            da = dh * u * (s + g * s * (1.0 - s))
            da_mag = dh_mag * np.abs(u) * (np.abs(s) + np.abs(g * s * (1.0 - s)))
        else:
            da = dh * g * s
            da_mag = dh_mag * np.abs(g * s)
        xj = x[toks, j]
        out["dW1"].append((float(np.sum(da * xj)), float(np.sum(da_mag * np.abs(xj)))))
    expert_cache = {}

    def expert(e):                                   # an expert's weights in fp64, converted once
        if e not in expert_cache:
            expert_cache[e] = (np.asarray(W1[e], np.float64), np.asarray(W2[e], np.float64))
        return expert_cache[e]

    for t in dx_at:                                  # dx[t] = sum_k dx_perm[row_of[t,k]] + sum_k dl[t,k] Wr[:, idx[t,k]]
        dxt = np.zeros(d)
        sdx = np.zeros(d)
        dw = np.zeros(K)
        dw_mag = np.zeros(K)
        for k in range(K):
            e = int(idx[t, k])
            W1e, W2e = expert(e)
            a = W1e @ x[t]
            g, u = a[:f], a[f:]
            s = 1.0 / (1.0 + np.exp(-g))
            h = silu(g) * u
            yp = W2e @ h
            dw[k] = float(dy[t] @ yp)
            dw_mag[k] = float(np.abs(dy[t]) @ np.abs(yp))
            dyp = w[t, k] * dy[t]
            dh = W2e.T @ dyp
            dh_mag = np.abs(W2e.T) @ np.abs(dyp)
            da = np.concatenate([dh * u * (s + g * s * (1.0 - s)), dh * g * s])
            da_mag = np.concatenate([dh_mag * np.abs(u) * (np.abs(s) + np.abs(g * s * (1.0 - s))),
                                     dh_mag * np.abs(g * s)])
            dxt += da @ W1e
            sdx += da_mag @ np.abs(W1e)
        wt = w[t]
        dl = wt * (dw - np.sum(wt * dw))
        dl_mag = wt * (dw_mag + np.sum(wt * dw_mag))
        for k in range(K):
            e = int(idx[t, k])
            dxt += dl[k] * Wr[:, e]
            sdx += dl_mag[k] * np.abs(Wr[:, e])
        out["dx"].append((dxt, sdx))
    return out
