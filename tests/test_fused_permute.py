"""GEMM1 with the permute fused into its operand load ("Optimization 2":
a naive dispatch writes the tokens out grouped and reads them back) against
the oracle, and against the unfused permute + GEMM1 it replaces.

Small and medium shapes compare every row of h with the oracle's
(oracle.forward, the per-element bf16 bound of the parity tests); the
full-size DeepSeek-V3- and Qwen-shaped layers, the small-group workloads this
path is meant for, compare one row of every 128-row slice of every live
expert group, and each group's first and last rows, with the expert FFN
evaluated from the definition, and so do the skew- and Mixtral-shaped layers,
whose large groups the unfused path runs on the CTA-pair kernel.  Every case
also checks that h is bit for bit the unfused path's, since both feed the
tensor cores the same bytes."""
import numpy as np
import pytest
import torch

import oracle
from workloads import Shape, make_tokens, make_weights, random_shape_cases, shape

from _helpers import check_logits, check_rounded, check_routing, check_stratified_rows, to_np

pytestmark = pytest.mark.gpu
DEV = "cuda"

CASES = random_shape_cases() + [
    Shape(T=200, d=64, E=256, K=16, f=64),                            # K = 16, E = 256
    Shape(T=130, d=192, E=256, K=2, f=128, bias="zipf_1.1"),          # > 100 empty experts
    Shape(T=2048, d=512, E=128, K=8, f=512, bias="zipf_1.1"),         # several tiles per CTA, two-block tiles
    Shape(T=4096, d=512, E=8, K=2, f=256, bias="normal_0.5"),         # pair-sized groups on the single-CTA kernel
    Shape(T=8192, d=512, E=8, K=2, f=1024, bias="normal_0.5"),        # pair-sized groups, several tiles per CTA
    Shape(T=4096, d=512, E=16, K=2, f=256, bias="zipf_1.1"),          # pair-sized, empty and <= 128-row groups
    Shape(T=4096, d=4096, E=4, K=2, f=1024, bias="normal_0.5"),       # pair-sized groups, 4096-deep reduction
]


def _routed(s, seed, device=DEV):
    import dropless_moe_expert_gb300 as moe
    w = make_weights(s, seed=seed, device=device)
    x = make_tokens(s, seed=seed, device=device)
    L = moe.router_logits(x, w.Wr, w.bias)
    r = moe.route(L, s.K)
    return w, x, L, r


@pytest.mark.parametrize("s", CASES, ids=lambda s: f"T{s.T}_d{s.d}_E{s.E}_K{s.K}_f{s.f}_{s.bias}")
def test_fused_permute_against_oracle(s):
    import dropless_moe_expert_gb300 as moe
    w, x, L, r = _routed(s, seed=s.T + 1)
    h = torch.full((s.T * s.K, s.f), float("nan"), dtype=torch.bfloat16, device=DEV)
    moe.grouped_gemm1_swiglu_gather(x, r.src_tok, r.offsets, w.W1, h=h)
    h_unfused = moe.grouped_gemm1_swiglu(moe.permute(x, r.row_of), r.offsets, w.W1)
    torch.cuda.synchronize()
    assert moe.device_status() == 0
    assert torch.equal(h.view(torch.int16), h_unfused.view(torch.int16)), "fused permute differs from unfused"
    xs, Wr, bias = to_np(x), to_np(w.Wr), to_np(w.bias)
    ref = oracle.forward(xs, Wr, bias, to_np(w.W1), to_np(w.W2), s.K)
    _, scale, L64 = check_logits(to_np(L), xs, Wr, bias)
    same = check_routing(to_np(r.topk_idx), ref["idx"], L64, scale, s.K)
    rg = to_np(r.row_of)[same].ravel()
    ro = ref["row_of"][same].ravel()
    check_rounded(to_np(h)[rg], ref["h"][ro], "h (fused permute)")


def test_fused_permute_repeated_calls_and_token_clamp():
    """Two calls give the same bits; token indices outside [0, T) (outside
    the contract) are clamped to valid rows instead of being read out of
    bounds, and every output row stays finite."""
    import dropless_moe_expert_gb300 as moe
    s = Shape(T=517, d=320, E=16, K=4, f=448)
    w, x, _, r = _routed(s, seed=3)
    a = moe.grouped_gemm1_swiglu_gather(x, r.src_tok, r.offsets, w.W1)
    b = moe.grouped_gemm1_swiglu_gather(x, r.src_tok, r.offsets, w.W1)
    bad = r.src_tok.clone()
    bad[::7] = s.T + 1000
    bad[1::7] = -5
    c = moe.grouped_gemm1_swiglu_gather(x, bad, r.offsets, w.W1)
    torch.cuda.synchronize()
    assert moe.device_status() == 0
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))
    assert bool(torch.isfinite(c.float()).all())


@pytest.mark.parametrize("name", ["dsv3", "qwen", "skew", "mixtral"])
def test_fused_permute_full_size_sampled_rows(name):
    import dropless_moe_expert_gb300 as moe
    s = shape(name)
    w, x, L, r = _routed(s, seed=0)
    h = moe.grouped_gemm1_swiglu_gather(x, r.src_tok, r.offsets, w.W1)
    h_unfused = moe.grouped_gemm1_swiglu(moe.permute(x, r.row_of), r.offsets, w.W1)
    torch.cuda.synchronize()
    assert moe.device_status() == 0
    assert torch.equal(h.view(torch.int16), h_unfused.view(torch.int16)), "fused permute differs from unfused"
    del h_unfused
    xs, Wr, bias = to_np(x), to_np(w.Wr), to_np(w.bias)
    Lo = oracle.router_logits_fp32(xs, Wr, bias)
    idx, _ = oracle.topk_route(Lo, s.K)
    _, offsets = oracle.expert_counts(idx, s.E)
    src_tok, _ = oracle.dispatch_order(idx, s.E)
    _, scale, L64 = check_logits(to_np(L), xs, Wr, bias)
    same = check_routing(to_np(r.topk_idx), idx, L64, scale, s.K)
    nrows, nexp = check_stratified_rows(h, None, r.row_of, xs, idx, offsets, src_tok, same, w.W1, w.W2)
    assert bool(torch.isfinite(h.float()).all())
    print(f"{name}: fused permute h, {nrows} stratified rows of {nexp} experts within the bf16 bound")
