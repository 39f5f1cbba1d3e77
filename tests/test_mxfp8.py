"""GPU parity of the MXFP8 path against the MXFP8 oracle (oracle/mxfp8.py).

Integer work is bit-exact: the E4M3 codes and scale bytes of the weight
quantiser and of the fused permute + quantise (both sides quantise the same
bf16 values).  h is computed in fp32 on the GPU and in fp64 by the oracle
before each is quantised, so the GPU's dequantised h is checked against the
oracle's unquantised h within the E4M3 rounding bound of its block (half an
ulp: 2^-4 relative in the normal range, 2^-10 of the block scale below it,
with the scale allowed to be one binade above the oracle's).  y_perm and y
have the bf16 path's tolerances against the oracle's MXFP8 forward.  Routing
follows the rules of the bf16 tests (each side routes on its own fp32
logits)."""
import numpy as np
import pytest
import torch

import oracle
from workloads import Shape, make_tokens, make_weights

from _helpers import (check_logits, check_mx_rounded, check_output, check_rounded, check_routing, to_np,
                      unpack_group_atoms, unpack_plain_atoms)

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.mark.parametrize("R,K", [(300, 256), (128, 128), (1, 384), (257, 512)])
def test_quantize_matches_oracle_bit_for_bit(R, K):
    import dropless_moe_expert_gb300 as moe
    g = torch.Generator().manual_seed(R + K)
    x = torch.randn(R, K, generator=g) * torch.exp(3 * torch.randn(R, 1, generator=g))
    x[0, :32] = 0.0                                   # a block of zeros
    x[0, 32:64] = torch.linspace(-14.0, 14.0, 32)     # amax 14 = 1.75 * 2^3: lands exactly on 448
    if K >= 128:
        x[0, 64:96] = 0.5
        x[0, 64] = 1.796875                           # mantissa above 1.75: one binade up
    x = x.to(torch.bfloat16)
    codes, sf = moe.mxfp8_quantize(x.to(DEV))
    torch.cuda.synchronize()
    rc, rs, _ = oracle.mx_quantize(x.float().numpy())
    assert np.array_equal(codes.cpu().numpy(), rc)
    assert np.array_equal(unpack_plain_atoms(sf.cpu().numpy(), R, K), rs)


CASES = [
    Shape(T=256, d=128, E=8, K=2, f=256),
    Shape(T=300, d=256, E=64, K=8, f=128),
    Shape(T=1000, d=384, E=8, K=1, f=384),
    Shape(T=517, d=256, E=16, K=4, f=512, bias="normal_0.5"),
    Shape(T=129, d=128, E=256, K=8, f=128),
    Shape(T=2048, d=256, E=4, K=1, f=256),     # groups of several 128-row blocks
    Shape(T=1500, d=128, E=3, K=2, f=640, bias="skew"),
    Shape(T=300, d=256, E=4, K=2, f=1664),     # GEMM2 reduction long enough for 256-column tiles
]


def _run(s, seed):
    import dropless_moe_expert_gb300 as moe
    w = make_weights(s, seed=seed, device="cpu")
    x = make_tokens(s, seed=seed, device="cpu")
    wd = [t.to(DEV) for t in (w.Wr, w.bias, w.W1, w.W2)]
    layer = moe.MoELayerMXFP8(*wd, s.K, s.T)
    layer.workspace.fill_(0xFF)
    y = layer(x.to(DEV))
    torch.cuda.synchronize()
    assert moe.device_status() == 0
    return x, w, y, layer


@pytest.mark.parametrize("s", CASES, ids=lambda s: f"T{s.T}_d{s.d}_E{s.E}_K{s.K}_f{s.f}")
def test_layer_matches_mxfp8_oracle(s):
    x, w, y, layer = _run(s, seed=s.T)
    v = layer.views(s.T)
    xs, Wr, bias = x.float().numpy(), w.Wr.numpy(), w.bias.numpy()
    ref = oracle.forward_mxfp8(xs, Wr, bias, w.W1.float().numpy(), w.W2.float().numpy(), s.K)
    _, scale, L64 = check_logits(to_np(v["logits"]), xs, Wr, bias)
    same = check_routing(to_np(v["topk_idx"]), ref["idx"], L64, scale, s.K)
    offs = to_np(v["offsets"])
    rg = to_np(v["row_of"])[same].ravel()      # GPU rows of the equally routed tokens
    ro = ref["row_of"][same].ravel()           # the oracle's rows of the same (token, slot)
    tok = np.repeat(np.nonzero(same)[0], s.K)
    # permute + quantise: codes and scales bit-exact
    xq = to_np(v["xq_perm"])
    assert np.array_equal(xq[rg], ref["xq"][tok])
    sfa = unpack_group_atoms(to_np(v["sfa"]), offs, s.d)
    assert np.array_equal(sfa[rg], ref["xs"][tok])
    # h: dequantised GPU h against the oracle's unquantised h
    hs = unpack_group_atoms(to_np(v["sfh"]), offs, s.f)
    hd = oracle.mx_dequantize(to_np(v["hq"]), hs)[rg]
    h = ref["h"][ro]
    check_mx_rounded(hd, h, ref["hs"][ro])
    codes_equal = np.mean(to_np(v["hq"])[rg] == ref["hq"][ro])
    check_output(to_np(v["y_perm"])[rg], ref["y_perm"][ro], "y_perm")
    r = check_output(to_np(y)[same], ref["y"][same], "y")
    y_bf16 = oracle.forward(xs, Wr, bias, w.W1.float().numpy(), w.W2.float().numpy(), s.K)["y"]
    q_err = np.linalg.norm(to_np(y)[same] - y_bf16[same]) / np.linalg.norm(y_bf16[same])
    print(f"{s}: h codes equal {codes_equal:.5f}; y rel_l2 {r[0]:.2e} vs the MXFP8 oracle, "
          f"{q_err:.2e} vs the bf16 oracle")


def test_gemm2_pairs_over_device_h_against_oracle():
    """GEMM2 of pair-sized groups with a short reduction, which runs on the
    CTA-pair MXFP8 kernel with several tiles per pair: y_perm against the
    fp64 product of the device's own dequantised h and the oracle's
    dequantised W2, every element within the bf16 rounding bound.  Taking the
    device's h isolates GEMM2 from the few h codes that round to the other
    side of an E4M3 step, which the whole-layer check meets at this size."""
    s = Shape(T=8192, d=1024, E=8, K=2, f=512, bias="normal_0.5")
    _, w, _, layer = _run(s, seed=s.T)
    v = layer.views(s.T)
    offs = to_np(v["offsets"]).astype(np.int64)
    hd = oracle.mx_dequantize(to_np(v["hq"]), unpack_group_atoms(to_np(v["sfh"]), offs, s.f))
    ref = np.zeros((s.T * s.K, s.d))
    for e in range(s.E):
        lo, hi = int(offs[e]), int(offs[e + 1])
        if hi > lo:
            _, _, W2d = oracle.mx_quantize(w.W2[e].float().numpy())
            ref[lo:hi] = hd[lo:hi] @ W2d.T
    check_rounded(to_np(v["y_perm"]), ref, "y_perm (MXFP8 GEMM2 over the device's h)")


def test_step_by_step_api_matches_single_call():
    import dropless_moe_expert_gb300 as moe
    s = CASES[3]
    x, w, y_one, layer = _run(s, seed=7)
    xd = x.to(DEV)
    L = moe.router_logits(xd, layer.Wr, layer.bias)
    r = moe.route(L, s.K)
    xq, sfa = moe.permute_mxfp8(xd, r)
    hq, sfh = moe.grouped_gemm1_swiglu_mxfp8(xq, sfa, r.offsets, layer.W1q, layer.W1s)
    yp = moe.grouped_gemm2_mxfp8(hq, sfh, r.offsets, layer.W2q, layer.W2s)
    y = moe.unpermute(yp, r.row_of, r.topk_w)
    torch.cuda.synchronize()
    assert torch.equal(y.view(torch.int16), y_one.view(torch.int16))


def test_rejects_dims_not_multiple_of_128():
    import dropless_moe_expert_gb300 as moe
    assert moe.lib.moe_forward_mxfp8_workspace_size(64, 192, 8, 2, 256) == 0
    assert moe.lib.moe_forward_mxfp8_workspace_size(64, 256, 8, 2, 192) == 0
    assert moe.mxfp8_scales_size(10, 64) == 0


@pytest.mark.parametrize("s", [Shape(T=1500, d=128, E=16, K=2, f=256, bias="skew"), "qwen"],
                         ids=["skew_small", "qwen_full"])
def test_graph_replays_match_eager(s):
    """The MXFP8 layer captured once in a CUDA graph and replayed on re-seeded
    tokens: each replay is bitwise equal to an eager call on the same tokens
    (no routing-dependent value frozen at capture), with different routings."""
    import dropless_moe_expert_gb300 as moe
    from workloads import shape
    s = shape(s)
    w = make_weights(s, seed=0, device=DEV)
    wd = (w.Wr, w.bias, w.W1, w.W2)
    layer = moe.MoELayerMXFP8(*wd, s.K, s.T)
    eager = moe.MoELayerMXFP8(*wd, s.K, s.T)
    x_static = make_tokens(s, seed=0, device=DEV)
    y_static = torch.empty_like(x_static)
    layer(x_static, out=y_static)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        layer(x_static, out=y_static)
    counts = []
    for seed in (1, 2, 3):
        x = make_tokens(s, seed=seed, device=DEV)
        x_static.copy_(x)
        layer.workspace.fill_(0xFF)
        y_static.fill_(float("nan"))
        graph.replay()
        y_eager = eager(x)
        torch.cuda.synchronize()
        assert moe.device_status() == 0
        assert torch.equal(y_static.view(torch.int16), y_eager.view(torch.int16)), f"replay seed {seed}"
        counts.append(tuple(layer.views(s.T)["counts"].cpu().tolist()))
    assert len(set(counts)) == len(counts), "replays should see different routings"


@pytest.mark.parametrize("s", [
    Shape(T=100, d=4096, E=8, K=2, f=128),                       # fewer tokens than warps: the chunks split evenly
    Shape(T=7000, d=640, E=16, K=3, f=128),                      # one round of whole tokens, then a split tail;
                                                                 # a 128-column last chunk
    Shape(T=13000, d=1152, E=64, K=2, f=128, bias="zipf_1.1"),   # two rounds, a tail, empty experts
], ids=lambda s: f"T{s.T}_d{s.d}_E{s.E}_K{s.K}")
def test_permute_quantise_every_row_bit_exact(s):
    """The quantising permute hands a grid of warps whole tokens in rounds
    while every warp still gets one, then splits the remaining tokens'
    512-column chunks into equal runs.  Every row of x_perm (codes and scale
    bytes) is compared with the oracle's quantisation of the token it came
    from, placed by the GPU's own routing; on a 152-SM GB300 the shapes take
    zero, one and two rounds before the split tail."""
    import dropless_moe_expert_gb300 as moe
    w = make_weights(s, seed=5, device=DEV)
    x = make_tokens(s, seed=5, device=DEV)
    r = moe.route(moe.router_logits(x, w.Wr, w.bias), s.K)
    xq, sfa = moe.permute_mxfp8(x, r)
    torch.cuda.synchronize()
    assert moe.device_status() == 0
    codes, scales, _ = oracle.mx_quantize(to_np(x))
    row_of = to_np(r.row_of).astype(np.int64)
    tok = np.repeat(np.arange(s.T), s.K)
    rows = row_of.ravel()
    assert np.array_equal(np.sort(rows), np.arange(s.T * s.K))
    assert np.array_equal(to_np(xq)[rows], codes[tok])
    assert np.array_equal(unpack_group_atoms(to_np(sfa), to_np(r.offsets), s.d, rows), scales[tok])
