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

from _helpers import (W_TOL, check_dispatch_valid, check_logits, check_output, check_rounded, check_routing,
                      check_stratified_rows, compare_small, run_layer, to_np, weight_tol)

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


# Medium shapes on which every CTA (or CTA pair) of the persistent grouped
# GEMMs takes several tiles, compared element by element (every row of h,
# y_perm and y): the pair kernel's accumulator alternation, phase flips and
# epilogue overlap across tiles, and the single-CTA kernel's two-block tiles
# over several waves.  Tiles per launch (GEMM1 / GEMM2) are about:
#   pair, mild skew          540 / 270 on 76 pairs
#   pair, interleaved order  440 / 220 on 76 pairs (one expert holds ~T rows)
#   single-CTA, two-block    380 / 380 on 152 CTAs (groups of 204..332 rows)
#   single-CTA, interleaved  670 / 330 on 152 CTAs (Zipf-skewed groups)
#   pair, long reductions    ~300 / ~130 on 76 pairs (d = 4096 and f = 4160:
#                            both GEMMs take the dynamic tile order)
MEDIUM_CASES = [
    Shape(T=8192, d=1024, E=8, K=2, f=1024, bias="normal_0.5"),
    Shape(T=4096, d=512, E=64, K=6, f=512, bias="skew"),
    Shape(T=8192, d=1024, E=64, K=2, f=512, bias="zero"),
    Shape(T=2048, d=512, E=128, K=8, f=512, bias="zipf_1.1"),
    Shape(T=1024, d=4096, E=3, K=2, f=4160, bias="normal_0.5"),
]


@pytest.mark.parametrize("s", MEDIUM_CASES, ids=lambda s: f"T{s.T}_d{s.d}_E{s.E}_K{s.K}_f{s.f}_{s.bias}")
def test_medium_multi_tile_shapes(s):
    x, w = _cpu_case(s, seed=s.T + s.E, bias_std=0)
    TK = s.T * s.K
    pair = TK >= 384 * s.E     # the grouped GEMMs' host-side choice of variant
    _, v, _ = run_layer(x, w, s.K)
    counts = to_np(v["counts"])
    rb = 256
    tiles1 = int(np.sum((counts + rb - 1) // rb)) * ((s.f + 127) // 128)
    workers = 76 if pair else 152
    assert tiles1 >= 2 * workers, f"{tiles1} GEMM1 tiles do not give each worker several"
    r = compare_small(x, w, s.K)
    print(f"{'pair' if pair else 'single'}: {tiles1} GEMM1 tiles, y rel_l2={r[0]:.2e} max/rms={r[1]:.2e}, "
          f"largest group {counts.max()}, empty {(counts == 0).sum()}")


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


@pytest.mark.parametrize("E,T", [(8, 300), (64, 300), (200, 300), (200, 16000), (64, 20000), (20, 40000)])
def test_router_one_hot_tokens_are_exact(E, T):
    """x[t] = 2^s e_i makes the dot product a single product: the logits must
    be exactly fp32(2^s Wr[i, e]) + bias[e], which holds only if all three
    bf16 pieces of Wr are added back exactly and each lands on its expert.
    T = 16000 takes 128-column expert tiles (two MMAs per K step); T = 20000
    and 40000 take tiles of two 128-token blocks (more than one wave of
    one-block tiles), the last one partial or with its second block past T."""
    import dropless_moe_expert_gb300 as moe
    d = 256
    g = np.random.default_rng(E)
    Wr = (g.standard_normal((d, E)) / math.sqrt(d)).astype(np.float32)
    bias = g.standard_normal(E).astype(np.float32)
    x = np.zeros((T, d), np.float32)
    i = (np.arange(T) * 7) % d
    scale = np.float32(2.0) ** (np.arange(T) % 5 - 2).astype(np.float32)
    x[np.arange(T), i] = scale
    xt = torch.from_numpy(x).to(torch.bfloat16).to(DEV)
    L = to_np(moe.router_logits(xt, torch.from_numpy(Wr).to(DEV), torch.from_numpy(bias).to(DEV)))
    torch.cuda.synchronize()
    ref = (scale[:, None] * Wr[i]).astype(np.float32) + bias[None, :]
    assert np.array_equal(L.view(np.uint32), ref.view(np.uint32))
    L0 = to_np(moe.router_logits(xt, torch.from_numpy(Wr).to(DEV), None))
    assert np.array_equal(L0.view(np.uint32), (scale[:, None] * Wr[i]).astype(np.float32).view(np.uint32))


# expert tiles of 32, 64 and (at least 120 token tiles) 128 columns, the last
# two with a partial tile; tiles of two 128-token blocks (the last two)
@pytest.mark.parametrize("s", [Shape(T=1000, d=512, E=8, K=2, f=64), Shape(T=300, d=1024, E=256, K=8, f=64),
                               Shape(T=129, d=64, E=100, K=4, f=64), Shape(T=16000, d=128, E=128, K=8, f=64),
                               Shape(T=15400, d=256, E=130, K=2, f=64), Shape(T=20000, d=256, E=64, K=2, f=64),
                               Shape(T=40000, d=128, E=20, K=2, f=64)],
                         ids=lambda s: f"T{s.T}_d{s.d}_E{s.E}")
def test_router_logits_bound_and_deterministic(s):
    import dropless_moe_expert_gb300 as moe
    x, w = _cpu_case(s, seed=11)
    L1 = moe.router_logits(x, w.Wr, w.bias)
    L2 = moe.router_logits(x, w.Wr, w.bias)
    torch.cuda.synchronize()
    assert torch.equal(L1.view(torch.int32), L2.view(torch.int32))
    err = check_logits(to_np(L1), to_np(x), to_np(w.Wr), to_np(w.bias))[0]
    print(f"router T={s.T} d={s.d} E={s.E}: max error / scale {err:.2e}")


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


@pytest.mark.parametrize("s", [Shape(T=517, d=320, E=16, K=4, f=448), Shape(T=2048, d=256, E=4, K=1, f=256),
                               Shape(T=1024, d=256, E=2, K=2, f=4160)],
                         ids=["single_cta", "pair_small_f", "pair_large_f"])
def test_forward_permute_choice_is_bit_identical(s):
    """moe_forward fuses the permute into GEMM1 on some shapes (sizes alone
    decide); its output equals the unfused step-by-step path's bit for bit
    either way, and the training forward (which keeps x_perm) gives the same y."""
    import dropless_moe_expert_gb300 as moe
    x, w = _cpu_case(s, seed=12)
    fused = moe.forward_fuses_permute(s.T, s.d, s.E, s.K, s.f)
    TK = s.T * s.K
    assert fused == ((TK < 384 * s.E) or s.f <= 4096)
    y_one, v, layer = run_layer(x, w, s.K)
    L = moe.router_logits(x, w.Wr, w.bias)
    r = moe.route(L, s.K)
    y = moe.unpermute(moe.grouped_gemm2(moe.grouped_gemm1_swiglu(moe.permute(x, r.row_of), r.offsets, w.W1),
                                        r.offsets, w.W2), r.row_of, r.topk_w)
    y_train = torch.empty_like(y)
    layer(x, out=y_train, save_preact=True)
    torch.cuda.synchronize()
    assert torch.equal(y.view(torch.int16), y_one.view(torch.int16))
    assert torch.equal(y_train.view(torch.int16), y_one.view(torch.int16))
    assert torch.equal(layer.views(s.T)["x_perm"].view(torch.int16), x.view(torch.int16)[r.src_tok.long()])


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
    import dropless_moe_expert_gb300 as moe
    s = shape(name)
    torch.manual_seed(0)
    w = make_weights(s, seed=0, device=DEV)
    x = make_tokens(s, seed=0, device=DEV)
    y, v, layer = run_layer(x, w, s.K)

    # logits of every token against fp64
    xs = to_np(x)
    Wr, bias = to_np(w.Wr), to_np(w.bias)
    lerr, scale, L64 = check_logits(to_np(v["logits"]), xs, Wr, bias)
    # routing given identical fp32 logits: the GPU route kernel on the
    # oracle's logits, every output bit-exact
    L = oracle.router_logits_fp32(xs, Wr, bias)
    idx, wref = oracle.topk_route(L, s.K)
    counts, offsets = oracle.expert_counts(idx, s.E)
    src_tok, row_of = oracle.dispatch_order(idx, s.E)
    r = moe.route(torch.from_numpy(L).to(DEV), s.K)
    torch.cuda.synchronize()
    assert np.array_equal(to_np(r.topk_idx), idx)
    assert np.max(np.abs(to_np(r.topk_w) - wref)) <= W_TOL
    assert np.array_equal(to_np(r.counts), counts)
    assert np.array_equal(to_np(r.offsets), offsets)
    assert np.array_equal(to_np(r.row_of), row_of)
    assert np.array_equal(to_np(r.src_tok), src_tok)
    del r
    # the layer's own routing (from its logits) against the oracle's
    gidx = to_np(v["topk_idx"])
    same = check_routing(gidx, idx, L64, scale, s.K)
    dw = np.abs(to_np(v["topk_w"]) - wref).max(axis=1)
    assert np.all(dw[same] <= weight_tol(scale, gidx)[same]), "topk_w"
    if same.all():
        assert np.array_equal(to_np(v["counts"]), counts)
        assert np.array_equal(to_np(v["offsets"]), offsets)
        assert np.array_equal(to_np(v["row_of"]), row_of)
        assert np.array_equal(to_np(v["src_tok"]), src_tok)
    else:
        check_dispatch_valid(v, s.T, s.K, s.E)
    # every permuted row is its token's row (checked on the device, bit
    # patterns), where the layer wrote x_perm rather than fusing the permute
    if not moe.forward_fuses_permute(s.T, s.d, s.E, s.K, s.f):
        st = v["src_tok"].long()
        assert torch.equal(v["x_perm"].view(torch.int16), x.view(torch.int16)[st])
        del st

    # one row of every 128-row slice of every live group, and each group's
    # first and last rows, from the definition
    nrows, nexp = check_stratified_rows(v["h"], v["y_perm"], v["row_of"], xs, idx, offsets, src_tok, same,
                                        w.W1, w.W2)

    # sampled tokens through the oracle, one by one
    toks = _sample_tokens(s.T, v, s.K)
    toks = toks[same[toks]]
    W1, W2 = w.W1, w.W2
    ridx, rw, rh, ryk, ry = oracle.forward_tokens(
        toks, xs[toks], L[toks], s.K, lambda e: (to_np(W1[e]), to_np(W2[e])))
    assert np.array_equal(ridx, idx[toks])
    rows = torch.from_numpy(to_np(v["row_of"])[toks].reshape(-1)).to(DEV)
    h_rows = to_np(v["h"][rows]).reshape(len(toks), s.K, s.f)
    yp_rows = to_np(v["y_perm"][rows]).reshape(len(toks), s.K, s.d)
    check_rounded(h_rows, rh, "h (sampled rows)")
    check_output(yp_rows, ryk, "y_perm (sampled rows)")
    r = check_output(to_np(y[torch.from_numpy(toks).to(DEV)]), ry, "y (sampled tokens)")
    # every output row was written and is finite
    assert bool(torch.isfinite(y.float()).all())
    print(f"{name}: logits err/scale {lerr:.2e}, tokens routed differently (near ties) {int((~same).sum())}; "
          f"stratified rows {nrows} of {nexp} experts; "
          f"sampled {len(toks)} tokens rel_l2={r[0]:.2e} max/rms={r[1]:.2e}; "
          f"experts with no token: {(counts == 0).sum()}, largest group {counts.max()}")
