"""Pins of the backward oracle (oracle/backward.py), on CPU: central finite
differences of the fp64 forward for every kind of input (token activations,
gate and up rows of W1, W2, router weights and bias), and closed forms (the
softmax's shift invariance, no router gradient at K = 1, experts without
tokens get no weight gradient)."""
import numpy as np
import pytest

import oracle
from oracle import moe_oracle as mo


def _case(T=14, d=16, E=5, K=2, f=12, seed=0):
    g = np.random.default_rng(seed)
    x = g.standard_normal((T, d))
    Wr = g.standard_normal((d, E)) / np.sqrt(d)
    bias = g.standard_normal(E) * 0.5
    W1 = g.standard_normal((E, 2 * f, d)) / np.sqrt(d)
    W2 = g.standard_normal((E, d, f)) / np.sqrt(f)
    dy = g.standard_normal((T, d))
    return x, Wr, bias, W1, W2, K, dy


def _routing(x, Wr, bias, K):
    E = Wr.shape[1]
    L = mo.router_logits_fp64(x, Wr, bias)
    idx = np.argsort(-L, axis=1, kind="stable")[:, :K]
    top = np.take_along_axis(L, idx, axis=1)
    z = np.exp(top - top[:, :1])
    w = z / z.sum(axis=1, keepdims=True)
    _, offsets = mo.expert_counts(idx, E)
    src_tok, row_of = mo.dispatch_order(idx, E)
    srt = np.sort(L, axis=1)[:, ::-1]
    margin = np.min(srt[:, :K] - srt[:, 1:K + 1]) if K < E else np.inf
    return dict(idx=idx, w=w, offsets=offsets, src_tok=src_tok, row_of=row_of), margin


def _loss(args, dy):
    return float(np.sum(dy * oracle.forward_fp64(*args)))


def _fd(args, dy, which, index, eps=1e-6):
    a = [np.array(v, np.float64, copy=True) if isinstance(v, np.ndarray) else v for v in args]
    a[which][index] += eps
    lp = _loss(a, dy)
    a[which][index] -= 2 * eps
    lm = _loss(a, dy)
    return (lp - lm) / (2 * eps)


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_gradients_match_finite_differences(seed):
    x, Wr, bias, W1, W2, K, dy = _case(seed=seed)
    r, margin = _routing(x, Wr, bias, K)
    assert margin > 1e-4                       # no selection changes within the step
    gr = oracle.backward(x, Wr, bias, W1, W2, K, dy, r)
    args = [x, Wr, bias, W1, W2, K]
    g = np.random.default_rng(seed + 100)
    f = W1.shape[1] // 2
    checks = []
    for _ in range(6):
        checks.append((0, (g.integers(x.shape[0]), g.integers(x.shape[1])), gr["dx"]))
        checks.append((1, (g.integers(Wr.shape[0]), g.integers(Wr.shape[1])), gr["dWr"]))
        checks.append((4, tuple(g.integers(s) for s in W2.shape), gr["dW2"]))
    for e in range(W1.shape[0]):
        checks.append((2, (e,), gr["dbias"]))
        checks.append((3, (e, g.integers(f), g.integers(W1.shape[2])), gr["dW1"]))           # gate row
        checks.append((3, (e, f + g.integers(f), g.integers(W1.shape[2])), gr["dW1"]))       # up row
    for which, index, grad in checks:
        num = _fd(args, dy, which, index)
        assert abs(num - grad[index]) <= 1e-6 * (1 + abs(num)), (which, index, num, grad[index])


def test_softmax_shift_invariance():
    x, Wr, bias, W1, W2, K, dy = _case(K=3, seed=4)
    r, _ = _routing(x, Wr, bias, K)
    gr = oracle.backward(x, Wr, bias, W1, W2, K, dy, r)
    # adding a constant to all logits of a token changes nothing
    assert abs(gr["dbias"].sum()) < 1e-10
    assert np.max(np.abs(gr["dWr"].sum(axis=1))) < 1e-10
    assert np.max(np.abs(gr["dL"].sum(axis=1))) < 1e-12


def test_top1_has_no_router_gradient():
    x, Wr, bias, W1, W2, _, dy = _case(K=1, seed=5)
    r, _ = _routing(x, Wr, bias, 1)
    gr = oracle.backward(x, Wr, bias, W1, W2, 1, dy, r)
    assert np.all(gr["dWr"] == 0) and np.all(gr["dbias"] == 0)
    assert np.allclose(gr["dx"], gr["dx_perm"][r["row_of"][:, 0]], rtol=0, atol=0)


def test_unused_expert_gets_no_weight_gradient():
    x, Wr, bias, W1, W2, K, dy = _case(seed=6)
    bias = bias.copy()
    bias[3] = -50.0                              # expert 3 is never chosen
    r, _ = _routing(x, Wr, bias, K)
    assert r["offsets"][4] == r["offsets"][3]
    gr = oracle.backward(x, Wr, bias, W1, W2, K, dy, r)
    assert np.all(gr["dW1"][3] == 0) and np.all(gr["dW2"][3] == 0)
    assert np.all(gr["dWr"][:, 3] == 0) and gr["dbias"][3] == 0


def test_forward_fp64_matches_forward():
    x, Wr, bias, W1, W2, K, _ = _case(seed=7)
    y64 = oracle.forward_fp64(x, Wr, bias, W1, W2, K)
    y = oracle.forward(x.astype(np.float32), Wr.astype(np.float32), bias.astype(np.float32), W1, W2, K)["y"]
    assert np.allclose(y64, y, rtol=1e-5, atol=1e-5)


@pytest.mark.parametrize("K", [1, 2, 3])
def test_sampled_elements_equal_the_full_backward(K):
    """backward_sampled() evaluates single elements from the definitions with
    only the rows they need; on a case small enough for backward() every
    sampled element must equal it, and each S must bound its |value|."""
    args = _case(T=40, d=16, E=5, K=K, f=12, seed=7)
    x, Wr, bias, W1, W2, K_, dy = args
    routing, _ = _routing(x, Wr, bias, K_)
    full = oracle.backward(x, Wr, bias, W1, W2, K_, dy, routing)
    f = W1.shape[1] // 2
    dW1_at = [(e, i, j) for e in range(5) for i in (0, f - 1, f, 2 * f - 1) for j in (0, 15)]
    dW2_at = [(e, i, j) for e in range(5) for i in (0, 15) for j in (0, f - 1)]
    dx_at = [0, 17, 39]
    got = oracle.backward_sampled(x, Wr, bias, W1, W2, K_, dy, routing, dW1_at, dW2_at, dx_at)
    for (e, i, j), (v, S) in zip(dW1_at, got["dW1"]):
        assert v == pytest.approx(full["dW1"][e, i, j], rel=1e-10, abs=1e-12)
        assert S >= abs(v) - 1e-12
    for (e, i, j), (v, S) in zip(dW2_at, got["dW2"]):
        assert v == pytest.approx(full["dW2"][e, i, j], rel=1e-10, abs=1e-12)
        assert S >= abs(v) - 1e-12
    for t, (v, S) in zip(dx_at, got["dx"]):
        np.testing.assert_allclose(v, full["dx"][t], rtol=1e-10, atol=1e-12)
        assert np.all(S >= np.abs(v) - 1e-12)
