"""Pins of the oracle against things other than itself (CPU only).

Each check is chosen so that a plausible mistake in the oracle -- a dropped
term, a wrong sign, a swapped SwiGLU half, a transposed operand, an unstable
sort, a wrong tie rule -- fails at least one of them:

* router logits: bit-exact against exact rational arithmetic rounded to fp32
  step by step (brute force on tiny inputs), and within the textbook
  forward-error bound of an fp32 dot product against fp64;
* top-K: brute force over all C(E, K) subsets, the pairwise selection rule,
  hand-worked ties and signed zeros;
* gate weights: K = E equals the library softmax, K = 1 gives 1, shift
  invariance;
* dispatch order: a brute-force double loop, invariants (bijection, zero
  drops, ascending tokens per group);
* FFN and combine: a hand-worked example with closed-form values, a dense
  reference that runs every expert on every token and masks, special cases
  (E = 1, identity permute/combine, linearity), perturbation of every input.
"""
import itertools
import json
import math
import os
from fractions import Fraction

import numpy as np
import pytest
import scipy.special

import oracle
from workloads import make_tokens, make_weights, shape

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ---------------------------------------------------------------- helpers
def _round_f32(q: Fraction) -> float:
    """Round an exact rational to the nearest fp32 value, ties to even."""
    if q == 0:
        return 0.0
    s = -1 if q < 0 else 1
    a = abs(q)
    e = a.numerator.bit_length() - a.denominator.bit_length()
    if Fraction(2) ** e > a:
        e -= 1
    while Fraction(2) ** (e + 1) <= a:
        e += 1
    ulp_exp = max(e - 23, -149)
    ulp = Fraction(2) ** ulp_exp
    m = a / ulp
    n = m.numerator // m.denominator
    rem = m - n
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and n % 2 == 1):
        n += 1
    return s * float(n * ulp)


def _fma_chain_exact(x, Wr, bias):
    T, d = x.shape
    E = Wr.shape[1]
    out = np.zeros((T, E), np.float32)
    for t in range(T):
        for e in range(E):
            acc = 0.0
            for i in range(d):
                acc = _round_f32(Fraction(float(x[t, i])) * Fraction(float(Wr[i, e])) + Fraction(acc))
            if bias is not None:
                acc = _round_f32(Fraction(acc) + Fraction(float(bias[e])))
            out[t, e] = acc
    return out


def _bf16_values(a):
    import torch
    return torch.from_numpy(np.ascontiguousarray(a, np.float32)).to(torch.bfloat16).float().numpy()


def _small_layer(T, d, E, K, f, seed=0, bias_scale=0.5):
    rng = np.random.default_rng(seed)
    x = _bf16_values(rng.standard_normal((T, d)))
    Wr = (rng.standard_normal((d, E)) / math.sqrt(d)).astype(np.float32)
    bias = (bias_scale * rng.standard_normal(E)).astype(np.float32)
    W1 = _bf16_values(rng.standard_normal((E, 2 * f, d)) / math.sqrt(d))
    W2 = _bf16_values(rng.standard_normal((E, d, f)) / math.sqrt(f))
    return x, Wr, bias, W1, W2


# ---------------------------------------------------------------- a0 router logits
def test_round_f32_helper_matches_numpy_on_doubles():
    # the exact rounding helper agrees with numpy's own fp64 -> fp32 rounding
    rng = np.random.default_rng(1)
    for v in rng.standard_normal(2000) * 10.0 ** rng.integers(-40, 38, 2000):
        assert _round_f32(Fraction(float(v))) == float(np.float32(v))


def test_router_fp32_bit_exact_vs_rational_fma_chain():
    rng = np.random.default_rng(2)
    for T, d, E in [(3, 5, 4), (2, 17, 3), (4, 9, 1)]:
        x = _bf16_values(rng.standard_normal((T, d)))
        Wr = rng.standard_normal((d, E)).astype(np.float32) / np.float32(3.0)
        bias = rng.standard_normal(E).astype(np.float32)
        got = oracle.router_logits_fp32(x, Wr, bias)
        want = _fma_chain_exact(x, Wr, bias)
        assert np.array_equal(got.view(np.uint32), want.view(np.uint32)) or np.array_equal(got, want)


def test_router_fp32_fma_differs_from_separate_rounding():
    # chain: acc = -(1 + 2^-11) exactly, then fma(a, a, acc) with a = 1 + 2^-12:
    # a^2 - (1 + 2^-11) = 2^-24 exactly; rounding a^2 first would give 0
    a = np.float32(1.0 + 2.0 ** -12)
    x = np.array([[1.0, a]], np.float32)
    Wr = np.array([[np.float32(-(1.0 + 2.0 ** -11))], [a]], np.float32)
    got = oracle.router_logits_fp32(x, Wr, None)[0, 0]
    assert got == np.float32(2.0 ** -24)


def test_router_fp32_within_dot_product_error_bound():
    rng = np.random.default_rng(3)
    T, d, E = 64, 1024, 32
    x = _bf16_values(rng.standard_normal((T, d)))
    Wr = (rng.standard_normal((d, E)) / math.sqrt(d)).astype(np.float32)
    bias = rng.standard_normal(E).astype(np.float32)
    L32 = oracle.router_logits_fp32(x, Wr, bias).astype(np.float64)
    L64 = oracle.router_logits_fp64(x, Wr, bias)
    u = 2.0 ** -24
    n = d + 1
    gamma = n * u / (1 - n * u)
    bound = gamma * (np.abs(x.astype(np.float64)) @ np.abs(Wr.astype(np.float64)) + np.abs(bias)[None, :])
    assert np.all(np.abs(L32 - L64) <= bound)
    # and the fp64 logits are the plain matrix product (transposition check)
    t, e = 5, 7
    assert L64[t, e] == pytest.approx(sum(float(x[t, i]) * float(Wr[i, e]) for i in range(d)) + float(bias[e]), rel=1e-12, abs=1e-12)


def test_router_bias_is_added():
    x, Wr, bias, *_ = _small_layer(4, 8, 5, 2, 8)
    a = oracle.router_logits_fp32(x, Wr, None)
    b = oracle.router_logits_fp32(x, Wr, bias)
    assert np.allclose(b - a, bias[None, :], atol=1e-6)


# ---------------------------------------------------------------- a1 top-K
def _brute_topk(row, K):
    E = len(row)
    best, best_key = None, None
    for sub in itertools.combinations(range(E), K):
        # sum of the subset's logits; ties between subsets go to the
        # lexicographically smallest sorted index tuple
        key = (sum(float(row[e]) for e in sub), tuple(-e for e in sub))
        if best_key is None or key > best_key:
            best, best_key = sub, key
    return set(best)


def test_topk_matches_brute_force_subsets():
    rng = np.random.default_rng(4)
    for trial in range(60):
        E = int(rng.integers(1, 9))
        K = int(rng.integers(1, E + 1))
        T = 8
        # coarse values make ties frequent
        L = rng.integers(-3, 4, size=(T, E)).astype(np.float32) * np.float32(0.5)
        idx, w = oracle.topk_route(L, K)
        for t in range(T):
            assert set(idx[t].tolist()) == _brute_topk(L[t], K)
            # order: descending value, equal values in ascending index
            for k in range(K - 1):
                a, b = idx[t, k], idx[t, k + 1]
                assert L[t, a] > L[t, b] or (L[t, a] == L[t, b] and a < b)
            # pairwise rule against every unselected expert
            sel = set(idx[t].tolist())
            for s_ in sel:
                for u_ in set(range(E)) - sel:
                    assert L[t, s_] > L[t, u_] or (L[t, s_] == L[t, u_] and s_ < u_)


def test_topk_hand_worked_ties_and_signed_zero():
    L = np.array([[1.0, 1.0, 0.0, 1.0],          # three-way tie -> 0, 1 then 3
                  [-0.0, 0.0, -1.0, 0.0],        # -0 == +0 -> lowest indices 0, 1
                  [0.0, -0.0, 2.0, -0.0],        # 2 first, then zeros by index
                  [-5.0, -4.0, -3.0, -2.0]], np.float32)
    idx, w = oracle.topk_route(L, 3)
    assert idx.tolist() == [[0, 1, 3], [0, 1, 3], [2, 0, 1], [3, 2, 1]]
    assert np.allclose(w[0], 1 / 3) and np.allclose(w[1], 1 / 3)
    e = math.exp
    assert w[2].tolist() == pytest.approx([1 / (1 + 2 * e(-2)), e(-2) / (1 + 2 * e(-2)), e(-2) / (1 + 2 * e(-2))])
    assert w[3].tolist() == pytest.approx([1 / (1 + e(-1) + e(-2)), e(-1) / (1 + e(-1) + e(-2)), e(-2) / (1 + e(-1) + e(-2))])


def test_gate_weights_special_cases():
    rng = np.random.default_rng(5)
    L = rng.standard_normal((50, 6)).astype(np.float32)
    idx, w = oracle.topk_route(L, 6)            # K = E: the full softmax, permuted
    full = scipy.special.softmax(L.astype(np.float64), axis=1)
    assert np.allclose(w, np.take_along_axis(full, idx, 1), rtol=1e-13, atol=0)
    idx1, w1 = oracle.topk_route(L, 1)          # K = 1: weight 1 on the argmax
    assert np.all(w1 == 1.0) and np.array_equal(idx1[:, 0], np.argmax(L, axis=1))
    idx3, w3 = oracle.topk_route(L, 3)
    assert np.allclose(w3.sum(1), 1.0, atol=1e-12)
    # softmax over the selected logits is invariant to a common shift
    _, w3s = oracle.topk_route(L + np.float32(4.0), 3)
    assert np.allclose(w3, w3s, atol=1e-6)
    # and equals the full softmax renormalised over the top-K
    ren = np.take_along_axis(full, idx3, 1)
    assert np.allclose(w3, ren / ren.sum(1, keepdims=True), rtol=1e-12)


def test_equal_logits_route_to_first_k():
    T, E, K = 9, 6, 4
    idx, w = oracle.topk_route(np.zeros((T, E), np.float32), K)
    assert np.all(idx == np.arange(K)[None, :]) and np.allclose(w, 1 / K)
    counts, offsets = oracle.expert_counts(idx, E)
    assert counts.tolist() == [T] * K + [0] * (E - K)


# ---------------------------------------------------------------- a2 dispatch
def test_dispatch_matches_brute_force_loops_and_invariants():
    rng = np.random.default_rng(6)
    for T, E, K in [(1, 1, 1), (5, 3, 2), (40, 8, 3), (33, 16, 16), (64, 7, 1)]:
        L = rng.standard_normal((T, E)).astype(np.float32)
        idx, _ = oracle.topk_route(L, K)
        counts, offsets = oracle.expert_counts(idx, E)
        src_tok, row_of = oracle.dispatch_order(idx, E)
        # brute force: walk experts, then tokens in order
        rows = []
        for e in range(E):
            for t in range(T):
                for k in range(K):
                    if idx[t, k] == e:
                        rows.append((t, k))
        assert src_tok.tolist() == [t for t, _ in rows]
        for r, (t, k) in enumerate(rows):
            assert row_of[t, k] == r
        assert counts.sum() == T * K and offsets[0] == 0 and offsets[-1] == T * K
        assert np.all(np.diff(offsets) >= 0) and np.array_equal(np.diff(offsets), counts)
        assert sorted(row_of.ravel().tolist()) == list(range(T * K))      # bijection, zero drops
        for t in range(T):
            assert len(set(idx[t].tolist())) == K
            for k in range(K):
                r = row_of[t, k]
                assert src_tok[r] == t and offsets[idx[t, k]] <= r < offsets[idx[t, k] + 1]
        for e in range(E):
            grp = src_tok[offsets[e]:offsets[e + 1]]
            assert np.all(np.diff(grp) > 0)                                # ascending tokens


# ---------------------------------------------------------------- FFN / combine
def _sigma(z):
    return 1.0 / (1.0 + math.exp(-z))


def test_hand_worked_example():
    with open(os.path.join(GOLDEN, "worked_example_T2_E3_K2.json")) as fh:
        g = json.load(fh)
    x = np.array(g["x"], np.float32)
    out = oracle.forward(x, np.array(g["Wr"], np.float32), np.array(g["bias"], np.float32),
                         np.array(g["W1"]), np.array(g["W2"]), g["shape"]["K"])
    s = _sigma
    assert out["logits"].tolist() == [[2.0, 1.5, 0.0], [0.0, 1.5, 3.0]]
    assert out["idx"].tolist() == [[0, 1], [2, 1]]
    assert np.allclose(out["w"], [[s(0.5), 1 - s(0.5)], [s(1.5), 1 - s(1.5)]], rtol=1e-14, atol=0)
    assert out["counts"].tolist() == [1, 2, 1] and out["offsets"].tolist() == [0, 1, 3, 4]
    assert out["src_tok"].tolist() == [0, 0, 1, 1] and out["row_of"].tolist() == [[0, 1], [3, 2]]
    assert out["h"][:, 0].tolist() == pytest.approx([s(1), 0.0, 2 * s(2), -3 * s(-1)], rel=1e-14)
    y0 = [s(0.5) * s(1), 2 * s(0.5) * s(1)]
    y1 = [s(1.5) * (-1.5 * s(-1)) + (1 - s(1.5)) * 2 * s(2),
          s(1.5) * (-3 * s(-1)) + (1 - s(1.5)) * (-2 * s(2))]
    assert np.allclose(out["y"], [y0, y1], rtol=1e-14, atol=0)


def test_silu_closed_forms():
    assert oracle.silu(np.float64(0.0)) == 0.0
    z = np.linspace(-8, 8, 33)
    assert np.allclose(oracle.silu(z) - oracle.silu(-z), z, rtol=0, atol=1e-14)   # odd part is z/2 * 2
    assert np.allclose(oracle.silu(np.array([40.0])), [40.0], rtol=1e-15)
    assert np.allclose(oracle.silu(np.array([1e-8])), [0.5e-8], rtol=1e-7)


def _dense_masked(x, Wr, bias, W1, W2, K, L):
    """Every expert on every token, then a [T, E] weight mask (zero for the
    unselected experts).  Uses einsum over whole weight tensors: a different
    formulation from the oracle's permute / per-group / combine path."""
    f = W1.shape[1] // 2
    idx, w = oracle.topk_route(L, K)
    T, E = L.shape
    m = np.zeros((T, E))
    np.put_along_axis(m, idx, w, axis=1)
    a = np.einsum("td,ejd->tej", x.astype(np.float64), W1.astype(np.float64))
    g, u = a[..., :f], a[..., f:]
    hh = g * scipy.special.expit(g) * u
    ye = np.einsum("tej,eoj->teo", hh, W2.astype(np.float64))
    return np.einsum("te,teo->to", m, ye)


@pytest.mark.parametrize("T,d,E,K,f", [(16, 8, 4, 2, 4), (40, 16, 8, 3, 8), (9, 8, 1, 1, 6), (12, 8, 5, 5, 4)])
def test_forward_equals_dense_masked_reference(T, d, E, K, f):
    x, Wr, bias, W1, W2 = _small_layer(T, d, E, K, f, seed=T + E)
    out = oracle.forward(x, Wr, bias, W1, W2, K)
    ref = _dense_masked(x, Wr, bias, W1, W2, K, out["logits"])
    assert np.allclose(out["y"], ref, rtol=1e-12, atol=1e-13)


def test_single_expert_is_dense_swiglu_ffn():
    x, Wr, bias, W1, W2 = _small_layer(10, 8, 1, 1, 6, seed=9)
    out = oracle.forward(x, Wr, bias, W1, W2, 1)
    assert np.all(out["w"] == 1.0) and np.array_equal(out["src_tok"], np.arange(10))
    f = 6
    g = x.astype(np.float64) @ W1[0, :f].T.astype(np.float64)
    u = x.astype(np.float64) @ W1[0, f:].T.astype(np.float64)
    ref = (g * scipy.special.expit(g) * u) @ W2[0].T.astype(np.float64)
    assert np.allclose(out["y"], ref, rtol=1e-12, atol=1e-13)


def test_permute_then_combine_is_identity():
    rng = np.random.default_rng(7)
    T, d, E, K = 30, 5, 6, 3
    L = rng.standard_normal((T, E)).astype(np.float32)
    x = rng.standard_normal((T, d))
    idx, w = oracle.topk_route(L, K)
    src_tok, row_of = oracle.dispatch_order(idx, E)
    xp = oracle.permute(x, src_tok)
    # an identity expert: weights sum to 1, so combine returns x
    assert np.allclose(oracle.combine(xp, row_of, w), x, atol=1e-13)
    one_hot = np.zeros_like(w)
    one_hot[:, 0] = 1.0
    assert np.array_equal(oracle.combine(xp, row_of, one_hot), x)


def test_linearity_in_up_half_and_w2():
    x, Wr, bias, W1, W2 = _small_layer(20, 8, 4, 2, 4, seed=11)
    f = 4
    base = oracle.forward(x, Wr, bias, W1, W2, 2)["y"]
    W1b = W1.copy()
    W1b[:, f:] *= 2.0
    assert np.allclose(oracle.forward(x, Wr, bias, W1b, W2, 2)["y"], 2 * base, rtol=1e-12)
    assert np.allclose(oracle.forward(x, Wr, bias, W1, 3 * W2, 2)["y"], 3 * base, rtol=1e-12)
    W1c = W1.copy()
    W1c[:, :f] *= 2.0                                    # the gate half is not linear
    assert not np.allclose(oracle.forward(x, Wr, bias, W1c, W2, 2)["y"], 2 * base, rtol=1e-3)


def test_every_input_is_consumed():
    x, Wr, bias, W1, W2 = _small_layer(64, 8, 8, 2, 4, seed=12, bias_scale=1.0)
    f = 4
    base = oracle.forward(x, Wr, bias, W1, W2, 2)["y"]
    variants = []
    b2 = bias.copy(); b2[int(np.argmax(bias))] -= 10.0; variants.append((x, Wr, b2, W1, W2))
    g2 = W1.copy(); g2[:, :f] *= -1.0; variants.append((x, Wr, bias, g2, W2))
    u2 = W1.copy(); u2[:, f:] += 0.25; variants.append((x, Wr, bias, u2, W2))
    w2 = W2.copy(); w2[:, 0, :] += 1.0; variants.append((x, Wr, bias, W1, w2))
    r2 = Wr.copy(); r2[0, :] *= -5.0; variants.append((x, r2, bias, W1, W2))
    for args in variants:
        assert not np.allclose(oracle.forward(*args, 2)["y"], base)


def test_forward_tokens_agrees_with_forward():
    s = shape("tiny")
    wts = make_weights(s, seed=0, device="cpu")
    x = make_tokens(s, seed=0, device="cpu").float().numpy()
    W1 = wts.W1.float().numpy()
    W2 = wts.W2.float().numpy()
    out = oracle.forward(x, wts.Wr.numpy(), wts.bias.numpy(), W1, W2, s.K)
    toks = np.array([0, 17, 255])
    idx, w, h, yk, y = oracle.forward_tokens(toks, x[toks], out["logits"][toks], s.K, lambda e: (W1[e], W2[e]))
    assert np.array_equal(idx, out["idx"][toks])
    assert np.allclose(y, out["y"][toks], rtol=1e-12, atol=1e-14)
    for i, t in enumerate(toks):
        for k in range(s.K):
            assert np.allclose(h[i, k], out["h"][out["row_of"][t, k]], rtol=1e-12, atol=1e-14)


def test_workload_generators_shapes_and_distributions():
    s = shape("tiny")
    wts = make_weights(s, seed=0)
    assert tuple(wts.W1.shape) == (s.E, 2 * s.f, s.d) and tuple(wts.W2.shape) == (s.E, s.d, s.f)
    assert abs(float(wts.W1.float().std()) - 1 / math.sqrt(s.d)) < 0.01 / math.sqrt(s.d) * 5
    x = make_tokens(s, seed=0)
    assert abs(float(x.float().std()) - 1.0) < 0.02
    # re-drawing x with another seed keeps the weights and changes the routing
    x2 = make_tokens(s, seed=1)
    assert not np.array_equal(x.float().numpy(), x2.float().numpy())
    sk = make_weights(dict(T=64, d=64, E=64, K=6, f=64, bias="skew"), seed=0)
    assert float(sk.bias[0]) == 3.0 and np.all(sk.bias.numpy()[48:] == -30.0)
