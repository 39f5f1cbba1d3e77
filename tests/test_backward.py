"""GPU parity of the layer backward against the backward oracle
(oracle/backward.py), on cases where both sides route every token the same
way (asserted).

Tolerance.  The GPU keeps dy_perm, dh, the recomputed pre-activations g and
u, da and dx_perm in bf16 (each rounding within 2^-9 relative) with fp32
accumulation; the oracle is fp64 throughout.  Each gradient element is a sum
of products, so its error is bounded by a small multiple of the sum of the
terms' magnitudes: |d| <= 2^-5 * S + 1e-6 max(S), with S computed from the
oracle's magnitudes carried through each intermediate that is a sum (e.g.
S = |da|^T |x_perm| per expert for dW1, where |da| is formed from dh's terms
|dy_perm| |W2[e]| and the terms of silu' taken separately), which leaves
about 3x over the five bf16 roundings on the way; plus relative L2
<= 1e-2 over the whole tensor.  Also: dw and dl, zero gradients of experts
without tokens, and that two calls give identical bits (every sum has a
fixed order)."""
import numpy as np
import pytest
import torch

import oracle
from workloads import Shape, make_tokens, make_weights

from _helpers import check_logits, check_routing, run_layer, to_np

pytestmark = pytest.mark.gpu
DEV = "cuda"

CASES = [
    Shape(T=256, d=128, E=8, K=2, f=256),
    Shape(T=300, d=256, E=64, K=8, f=128),
    Shape(T=1000, d=192, E=8, K=1, f=320),
    Shape(T=517, d=320, E=16, K=4, f=448, bias="normal_0.5"),
    Shape(T=129, d=128, E=256, K=8, f=64),
    Shape(T=2048, d=256, E=4, K=2, f=256),       # CTA-pair dgrad and weight-gradient GEMMs, long groups
    Shape(T=600, d=128, E=8, K=2, f=192, bias="skew"),
    # long groups: CTA-pair weight gradients, with partial 256-row blocks of D
    # (d = 320, 2f = 384) and partial 256-column blocks
    Shape(T=1500, d=320, E=2, K=1, f=192),
    Shape(T=3000, d=128, E=4, K=2, f=384, bias="skew"),
    # degenerate cases: one token; one expert (a dense FFN, no router gradient);
    # K = E (every expert on every token); the smallest widths
    Shape(T=1, d=128, E=4, K=2, f=64),
    Shape(T=200, d=128, E=1, K=1, f=128),
    Shape(T=64, d=64, E=8, K=8, f=64),
    # K = E fixes every group at T rows: groups ending exactly on a 64-row K
    # block, and groups with a single row in their last block (single-CTA
    # kernels; then CTA pairs, TK >= 384 E)
    Shape(T=128, d=128, E=2, K=2, f=128),
    Shape(T=129, d=128, E=2, K=2, f=128),
    Shape(T=449, d=256, E=2, K=2, f=256),
    # K values without a specialised input-gradient kernel (3) and with one (6)
    Shape(T=300, d=128, E=16, K=3, f=128),
    Shape(T=257, d=192, E=12, K=6, f=128),
]


def check_bounded(gpu, ref, S, what):
    gpu = np.asarray(gpu, np.float64)
    ref = np.asarray(ref, np.float64)
    assert np.all(np.isfinite(gpu)), f"{what}: non-finite values"
    nr = np.linalg.norm(ref)
    r = np.linalg.norm(gpu - ref) / (nr if nr > 0 else 1.0)
    assert r <= 1e-2, f"{what}: relative L2 {r:.3e}"
    bound = 2.0 ** -5 * S + 1e-6 * (S.max() if S.size else 0.0)
    excess = np.abs(gpu - ref) - bound
    if not np.all(excess <= 0):
        bad = np.argwhere(excess > 0)
        worst = tuple(np.unravel_index(np.argmax(excess), excess.shape))
        print(f"{what}: {len(bad)} beyond; worst at {worst}: gpu {gpu[worst]:.5g} ref {ref[worst]:.5g} "
              f"S {S[worst]:.5g}; first bad {bad[:5].tolist()}")
    assert np.all(excess <= 0), f"{what}: {int((excess > 0).sum())} elements beyond the bound"
    return r, float(np.max(np.abs(gpu - ref) / np.maximum(bound, 1e-30)))


def _magnitudes(xs, Wr, W1, W2, dy, fwd, ref):
    """Sums of the absolute terms behind each gradient element, carried
    through every intermediate that is itself a sum or a cancelling
    expression: dh's terms |dy_perm| |W2[e]|, and the terms of
    silu'(g) = s + g s (1 - s) separately (near its root, g ~ -1.28, dg is
    tiny while its rounding error is not), and for the router dw's terms
    |dy| |y_perm| and the softmax's terms separately."""
    offsets, row_of, src_tok = fwd["offsets"], fwd["row_of"], fwd["src_tok"]
    E = W1.shape[0]
    f = W1.shape[1] // 2
    ax = np.abs(xs.astype(np.float64))
    xp = ax[src_tok]
    g, u = ref["a"][:, :f], ref["a"][:, f:]
    sg = 1.0 / (1.0 + np.exp(-g))
    # dh = dy_perm W2[e] is itself a sum: its error scales with |dy_perm| |W2[e]|
    adh = np.zeros_like(ref["dh"])
    for e in range(E):
        r0, r1 = offsets[e], offsets[e + 1]
        if r1 > r0:
            adh[r0:r1] = np.abs(ref["dy_perm"][r0:r1]) @ np.abs(W2[e].astype(np.float64))
    da_mag = np.concatenate([adh * np.abs(u) * (sg + np.abs(g) * sg * (1.0 - sg)), adh * np.abs(g) * sg], axis=1)
    S = {}
    S["dW2"] = np.zeros(W2.shape)
    S["dW1"] = np.zeros(W1.shape)
    for e in range(E):
        r0, r1 = offsets[e], offsets[e + 1]
        if r1 > r0:
            S["dW2"][e] = np.abs(ref["dy_perm"][r0:r1]).T @ np.abs(ref["h"][r0:r1])
            S["dW1"][e] = da_mag[r0:r1].T @ xp[r0:r1]
    aW1 = np.abs(W1.astype(np.float64))
    sxp = np.zeros_like(ref["dx_perm"])
    for e in range(E):
        r0, r1 = offsets[e], offsets[e + 1]
        if r1 > r0:
            sxp[r0:r1] = da_mag[r0:r1] @ aW1[e]
    # dw = <dy, y_perm[r]> is a sum, dl = w (dw - sum_j w_j dw_j) cancels:
    # dl's magnitude from dw's terms and the softmax terms separately
    S["dw"] = np.einsum("tkc,tc->tk", np.abs(ref["y_perm"])[row_of], np.abs(dy.astype(np.float64)))
    w = np.asarray(fwd["w"], np.float64)
    dl_mag = w * (S["dw"] + np.sum(w * S["dw"], axis=1, keepdims=True))
    dL_mag = np.zeros_like(ref["dL"])
    np.put_along_axis(dL_mag, np.asarray(fwd["idx"]), dl_mag, axis=1)
    S["dx"] = dL_mag @ np.abs(Wr.astype(np.float64)).T
    for k in range(row_of.shape[1]):
        S["dx"] += sxp[row_of[:, k]]
    S["dWr"] = ax.T @ dL_mag
    S["dbias"] = dL_mag.sum(axis=0)
    return S


def _case(s, seed):
    w = make_weights(s, seed=seed, device="cpu")
    x = make_tokens(s, seed=seed, device="cpu")
    g = np.random.default_rng(seed + 5)
    dy = torch.from_numpy(g.standard_normal((s.T, s.d)).astype(np.float32)).to(torch.bfloat16)
    return x, w, dy


@pytest.mark.parametrize("save", [False, True], ids=["recompute", "saved_preact"])
@pytest.mark.parametrize("s", CASES, ids=lambda s: f"T{s.T}_d{s.d}_E{s.E}_K{s.K}_f{s.f}")
def test_backward_matches_oracle(s, save):
    import dropless_moe_expert_gb300 as moe
    x, w, dy = _case(s, seed=s.T + 1)
    wd = type(w)(*(t.to(DEV) for t in (w.Wr, w.bias, w.W1, w.W2)))
    xd = x.to(DEV)
    y, v, layer = run_layer(xd, wd, s.K)
    if save:
        # the same forward again, GEMM1 storing its pre-activations
        layer.preact = None
        y2 = layer(xd, save_preact=True)
        assert layer.preact is not None
        assert torch.equal(y2.view(torch.int16), y.view(torch.int16))
    grads = layer.backward(xd, dy.to(DEV))
    grads2 = layer.backward(xd, dy.to(DEV))
    torch.cuda.synchronize()
    assert moe.device_status() == 0
    for k in grads:
        assert torch.equal(grads[k].view(torch.int16) if grads[k].dtype == torch.bfloat16 else grads[k],
                           grads2[k].view(torch.int16) if grads2[k].dtype == torch.bfloat16 else grads2[k]), k
    xs, Wr, bias = x.float().numpy(), w.Wr.numpy(), w.bias.numpy()
    W1, W2 = w.W1.float().numpy(), w.W2.float().numpy()
    fwd = oracle.forward(xs, Wr, bias, W1, W2, s.K)
    _, scale, L64 = check_logits(to_np(v["logits"]), xs, Wr, bias)
    same = check_routing(to_np(v["topk_idx"]), fwd["idx"], L64, scale, s.K)
    assert same.all(), "pick a case whose routing is decided on both sides"
    dyn = dy.float().numpy()
    ref = oracle.backward(xs, Wr, bias, W1, W2, s.K, dyn, fwd)
    S = _magnitudes(xs, Wr, W1, W2, dyn, fwd, ref)
    bv = layer.backward_views(s.T)
    report = {}
    report["dw"] = check_bounded(to_np(bv["dw"]), ref["dw"], S["dw"], "dw")
    for name in ("dx", "dW1", "dW2"):
        report[name] = check_bounded(to_np(grads[name]), ref[name], S[name], name)
    if s.K > 1:
        for name in ("dWr", "dbias"):
            report[name] = check_bounded(to_np(grads[name]), ref[name], S[name], name)
    else:
        assert not grads["dWr"].any() and not grads["dbias"].any()
    # experts without tokens: zero weight gradients
    empty = np.nonzero(np.diff(fwd["offsets"]) == 0)[0]
    for e in empty:
        assert not grads["dW1"][int(e)].any() and not grads["dW2"][int(e)].any()
    print(s, {k: f"rel {v[0]:.1e}, worst/bound {v[1]:.2f}" for k, v in report.items()})


@pytest.mark.parametrize("s", [CASES[0], CASES[4], CASES[5]], ids=lambda s: f"T{s.T}_d{s.d}_E{s.E}_K{s.K}_f{s.f}")
def test_saved_preact_matches_recomputed(s):
    """GEMM1's stored pre-activations against the backward's own recompute
    (a plain grouped GEMM over the 2f stacked rows): the same bf16 rounding
    of fp32 sums over the same K slices, so at most one bf16 step apart;
    every row written (the buffer starts as NaN)."""
    import dropless_moe_expert_gb300 as moe
    x, w, dy = _case(s, seed=s.T + 2)
    wd = type(w)(*(t.to(DEV) for t in (w.Wr, w.bias, w.W1, w.W2)))
    xd = x.to(DEV)
    _, _, layer = run_layer(xd, wd, s.K)
    layer.backward(xd, dy.to(DEV))              # recompute path: fills the region `a`
    a = layer.backward_views(s.T)["a"].float().clone()
    layer._preact_buf = torch.full((s.T * s.K * 2 * s.f,), float("nan"), dtype=torch.bfloat16, device=DEV)
    layer(xd, save_preact=True)
    torch.cuda.synchronize()
    assert moe.device_status() == 0
    pre = layer.preact.float()
    assert torch.isfinite(pre).all()
    diff = (pre - a).abs()
    assert (diff <= 2.0 ** -7 * a.abs() + 1e-30).all()
    print(s, f"bit-identical fraction {(pre == a).float().mean().item():.6f}")
