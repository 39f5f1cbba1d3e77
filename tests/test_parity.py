"""GPU parity: the CUDA layer, called through the C ABI, against the oracle.

Small cases compare every intermediate on every element; the full-size
workloads compare the routing of all tokens bit-exactly and the outputs of
sampled tokens, which the oracle computes one by one.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from workloads import LayerWeights, Shape, make_tokens, make_weights, random_shape_cases, shape

from _helpers import W_TOL, check_output, check_rounded, compare_small, run_layer, to_np

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _to_dev(w: LayerWeights):
    return LayerWeights(*(t.to(DEV) for t in (w.Wr, w.bias, w.W1, w.W2)))


def _cpu_case(s: Shape, seed=0, bias_std=0.5):
    w = make_weights(s, seed=seed, device="cpu")
    if s.bias == "zero" and bias_std:
        g = np.random.default_rng(seed + 17)
        w.bias = torch.from_numpy((bias_std * g.standard_normal(s.E)).astype(np.float32))
    x = make_tokens(s, seed=seed, device="cpu")
    return x.to(DEV), _to_dev(w)


def test_tiny_config_all_intermediates():
    s = shape("tiny")
    x, w = _cpu_case(s, bias_std=0)
    compare_small(x, w, s.K)


@pytest.mark.parametrize("s", random_shape_cases(), ids=lambda s: f"T{s.T}_d{s.d}_E{s.E}_K{s.K}_f{s.f}")
def test_random_small_shapes(s):
    x, w = _cpu_case(s, seed=s.T)
    compare_small(x, w, s.K)


def test_single_expert_single_token():
    s = Shape(T=1, d=64, E=1, K=1, f=64)
    x, w = _cpu_case(s)
    compare_small(x, w, 1)


def test_all_experts_per_token():
    s = Shape(T=70, d=128, E=6, K=6, f=128)
    x, w = _cpu_case(s, seed=3)
    compare_small(x, w, s.K)


def test_maximum_experts_and_k():
    s = Shape(T=200, d=64, E=256, K=16, f=64)
    x, w = _cpu_case(s, seed=4)
    compare_small(x, w, s.K)


@pytest.mark.parametrize("K", [1, 2])
def test_every_token_to_one_expert(K):
    s = Shape(T=600, d=128, E=8, K=K, f=192)
    x, w = _cpu_case(s, seed=5)
    w.bias = torch.zeros(8, device=DEV)
    w.bias[3] = 50.0            # expert 3 wins every token: one long group, 7 empty
    compare_small(x, w, K)


def test_equal_logits_route_to_first_k_experts():
    s = Shape(T=300, d=64, E=16, K=4, f=64)
    x, w = _cpu_case(s, seed=6)
    w.Wr.zero_()
    w.bias.zero_()              # every logit is +0.0: experts 0..3 for every token
    _, v, _ = run_layer(x, w, s.K)
    assert np.all(to_np(v["topk_idx"]) == np.arange(4)[None, :])
    assert np.allclose(to_np(v["topk_w"]), 0.25)
    compare_small(x, w, s.K)


def test_many_empty_experts_and_ragged_groups():
    s = Shape(T=130, d=192, E=256, K=2, f=128)
    x, w = _cpu_case(s, seed=7)
    w.bias = torch.tensor([-1.1 * math.log(e + 1) for e in range(256)], device=DEV)
    _, v, _ = run_layer(x, w, s.K)
    assert (to_np(v["counts"]) == 0).sum() > 100
    compare_small(x, w, s.K)


def test_route_ties_and_signed_zeros_direct():
    import dropless_moe_expert_gb300 as moe
    g = np.random.default_rng(8)
    T, E, K = 777, 40, 5
    L = (g.integers(-3, 4, size=(T, E)) * 0.5).astype(np.float32)     # many exact ties
    zeros = g.random((T, E)) < 0.2
    L[zeros] = np.where(g.random(zeros.sum()) < 0.5, -0.0, 0.0).astype(np.float32)
    r = moe.route(torch.from_numpy(L).to(DEV), K)
    torch.cuda.synchronize()
    idx, wref = oracle.topk_route(L, K)
    counts, offsets = oracle.expert_counts(idx, E)
    src_tok, row_of = oracle.dispatch_order(idx, E)
    assert np.array_equal(to_np(r.topk_idx), idx)
    assert np.max(np.abs(to_np(r.topk_w) - wref)) <= W_TOL
    assert np.array_equal(to_np(r.counts), counts)
    assert np.array_equal(to_np(r.offsets), offsets)
    assert np.array_equal(to_np(r.row_of), row_of)
    assert np.array_equal(to_np(r.src_tok), src_tok)


def test_step_by_step_api_matches_single_call():
    import dropless_moe_expert_gb300 as moe
    s = Shape(T=517, d=320, E=16, K=4, f=448)
    x, w = _cpu_case(s, seed=9)
    y_one, _, _ = run_layer(x, w, s.K)
    L = moe.router_logits(x, w.Wr, w.bias)
    r = moe.route(L, s.K)
    xp = moe.permute(x, r.row_of)
    h, yp = moe.grouped_mlp(xp, r.offsets, w.W1, w.W2)
    y = moe.unpermute(yp, r.row_of, r.topk_w)
    torch.cuda.synchronize()
    assert torch.equal(y.view(torch.int16), y_one.view(torch.int16))


def test_host_buffers_entry_point():
    import dropless_moe_expert_gb300 as moe
    s = Shape(T=300, d=256, E=8, K=2, f=256)
    x, w = _cpu_case(s, seed=10)
    y_dev, _, _ = run_layer(x, w, s.K)
    xh = x.cpu().pin_memory()
    yh = moe.forward_host(xh, w.Wr, w.bias, w.W1, w.W2, s.K)
    torch.cuda.synchronize()
    assert torch.equal(yh.view(torch.int16), y_dev.cpu().view(torch.int16))


# ---------------------------------------------------------------- full size
def _sample_tokens(T, v, K, n=24, seed=0):
    g = np.random.default_rng(seed)
    toks = set(g.choice(T, size=min(n, T), replace=False).tolist()) | {0, T - 1}
    # add tokens of the most and least loaded non-empty experts
    counts = to_np(v["counts"])
    src = v["src_tok"]
    offs = to_np(v["offsets"])
    nz = np.nonzero(counts)[0]
    for e in (nz[np.argmax(counts[nz])], nz[np.argmin(counts[nz])]):
        toks.add(int(src[offs[e]].item()))
        toks.add(int(src[offs[e + 1] - 1].item()))
    return np.array(sorted(toks))


@pytest.mark.parametrize("name", ["mixtral", "dsv3", "qwen", "skew"])
def test_full_size_workload(name):
    s = shape(name)
    torch.manual_seed(0)
    w = make_weights(s, seed=0, device=DEV)
    x = make_tokens(s, seed=0, device=DEV)
    y, v, layer = run_layer(x, w, s.K)

    # routing of every token, bit-exact
    xs = to_np(x)
    L = oracle.router_logits_fp32(xs, to_np(w.Wr), to_np(w.bias))
    assert np.array_equal(to_np(v["logits"]).view(np.uint32), L.view(np.uint32)), "logits"
    idx, wref = oracle.topk_route(L, s.K)
    counts, offsets = oracle.expert_counts(idx, s.E)
    src_tok, row_of = oracle.dispatch_order(idx, s.E)
    assert np.array_equal(to_np(v["topk_idx"]), idx)
    assert np.max(np.abs(to_np(v["topk_w"]) - wref)) <= W_TOL
    assert np.array_equal(to_np(v["counts"]), counts)
    assert np.array_equal(to_np(v["offsets"]), offsets)
    assert np.array_equal(to_np(v["row_of"]), row_of)
    assert np.array_equal(to_np(v["src_tok"]), src_tok)
    # every permuted row is its token's row (checked on the device, bit patterns)
    st = torch.from_numpy(src_tok).to(DEV)
    assert torch.equal(v["x_perm"].view(torch.int16), x.view(torch.int16)[st])
    del st

    # sampled tokens through the oracle, one by one
    toks = _sample_tokens(s.T, v, s.K)
    W1, W2 = w.W1, w.W2
    ridx, rw, rh, ryk, ry = oracle.forward_tokens(
        toks, xs[toks], L[toks], s.K, lambda e: (to_np(W1[e]), to_np(W2[e])))
    assert np.array_equal(ridx, idx[toks])
    rows = torch.from_numpy(row_of[toks].reshape(-1)).to(DEV)
    h_rows = to_np(v["h"][rows]).reshape(len(toks), s.K, s.f)
    yp_rows = to_np(v["y_perm"][rows]).reshape(len(toks), s.K, s.d)
    check_rounded(h_rows, rh, "h (sampled rows)")
    check_output(yp_rows, ryk, "y_perm (sampled rows)")
    r = check_output(to_np(y[torch.from_numpy(toks).to(DEV)]), ry, "y (sampled tokens)")
    # every output row was written and is finite
    assert bool(torch.isfinite(y.float()).all())
    print(f"{name}: sampled {len(toks)} tokens rel_l2={r[0]:.2e} max/rms={r[1]:.2e}; "
          f"experts with no token: {(counts == 0).sum()}, largest group {counts.max()}")
