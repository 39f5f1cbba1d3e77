"""GEMM2 with the combine fused into its epilogue ("Optimization 2": dispatch
and combine fused into one pipeline) must give y bit for bit equal to the
unfused GEMM2 + combine: the token's last stored row forms y from the K
stored rows in ascending k, so the order in which rows arrive cannot show.
Its y is also compared with the oracle's (tolerances and routing rule of the
parity tests) on every case below and on a Mixtral-like medium layer whose
CTA pairs each take several tiles.
Shapes cover K = 1, K = 16, E = 256, ragged groups, empty experts, a d with a
half column block (d % 256 = 128), both GEMM variants (single-CTA and
CTA-pair), repeated calls (the counters are re-zeroed each call) and a
full-size skew-shaped layer."""
import numpy as np
import pytest
import torch

import oracle
from workloads import Shape, make_tokens, make_weights, shape

from _helpers import check_logits, check_output, check_routing, to_np

pytestmark = pytest.mark.gpu
DEV = "cuda"

CASES = [
    Shape(T=7, d=64, E=3, K=2, f=128),
    Shape(T=300, d=256, E=64, K=8, f=128),
    Shape(T=129, d=128, E=256, K=8, f=64),
    Shape(T=1000, d=384, E=8, K=1, f=320),
    Shape(T=517, d=320, E=16, K=4, f=448, bias="skew"),
    Shape(T=200, d=64, E=256, K=16, f=64),
    Shape(T=2048, d=384, E=4, K=2, f=256),      # CTA-pair variant, half column block
    Shape(T=4096, d=512, E=8, K=2, f=256, bias="normal_0.5"),
    Shape(T=8192, d=1024, E=8, K=2, f=1024, bias="normal_0.5"),   # Mixtral-like, several tiles per pair
]


def _layer_inputs(s, seed):
    import dropless_moe_expert_gb300 as moe
    w = make_weights(s, seed=seed, device=DEV)
    x = make_tokens(s, seed=seed, device=DEV)
    L = moe.router_logits(x, w.Wr, w.bias)
    r = moe.route(L, s.K)
    xp = moe.permute(x, r.row_of)
    h = moe.grouped_gemm1_swiglu(xp, r.offsets, w.W1)
    return x, w, L, r, h


def _check_against_oracle(s, x, w, L, r, y):
    """y of the fused path against the oracle's forward on the same inputs,
    for the tokens both sides route identically (normally all)."""
    xs, Wr, bias = to_np(x), to_np(w.Wr), to_np(w.bias)
    ref = oracle.forward(xs, Wr, bias, to_np(w.W1), to_np(w.W2), s.K)
    _, scale, L64 = check_logits(to_np(L), xs, Wr, bias)
    same = check_routing(to_np(r.topk_idx), ref["idx"], L64, scale, s.K)
    return check_output(to_np(y)[same], ref["y"][same], "y (fused combine)")


def _check(s, seed, repeats=2, against_oracle=True):
    import dropless_moe_expert_gb300 as moe
    x, w, L, r, h = _layer_inputs(s, seed)
    ref = moe.unpermute(moe.grouped_gemm2(h, r.offsets, w.W2), r.row_of, r.topk_w)
    for _ in range(repeats):
        y = torch.full_like(ref, float("nan"))
        moe.grouped_gemm2_combine(h, r, w.W2, out=y)
        torch.cuda.synchronize()
        assert moe.device_status() == 0
        assert torch.equal(y.view(torch.int16), ref.view(torch.int16)), "fused combine differs from unfused"
    if against_oracle:
        _check_against_oracle(s, x, w, L, r, y)


@pytest.mark.parametrize("s", CASES, ids=lambda s: f"T{s.T}_d{s.d}_E{s.E}_K{s.K}_f{s.f}")
def test_fused_combine_equals_unfused(s):
    _check(s, seed=s.T)


def test_fused_combine_full_size_skew():
    # (the unfused path it equals is compared with the oracle at this size
    # in the parity tests)
    _check(shape("skew"), seed=0, repeats=3, against_oracle=False)


def test_fused_combine_rejects_inconsistent_sizes():
    import dropless_moe_expert_gb300 as moe
    L = moe.lib
    fake = 1 << 20
    # TK != T * K
    assert L.moe_grouped_gemm2_combine(fake, fake, 8, 100, 64, 64, fake, fake, fake, fake, 8, 2, fake, fake,
                                       1 << 20, fake, None) == 1
    # counters too small
    assert L.moe_grouped_gemm2_combine(fake, fake, 8, 16, 64, 64, fake, fake, fake, fake, 8, 2, fake, fake,
                                       4, fake, None) == 3
    assert moe.lib.moe_combine_counters_size(8192, 4096) == 8192 * 16 * 4
