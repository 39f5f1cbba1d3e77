"""GPU parity of the layer backward at the full workload sizes, on sampled
gradient elements: the training step (moe_forward_train, then moe_backward)
runs on the device; the oracle routes on its own fp32 logits and evaluates
the sampled elements of dW1, dW2 and dx from the definitions
(oracle.backward_sampled, pinned to oracle.backward on small cases).  The
samples come from experts whose groups are routed identically on both sides
(every token of the group decided beyond the logits' error band) and from
such tokens; each element must lie within 2^-5 of the sum of its terms'
magnitudes, plus 1e-6 of the largest such sum (the bound of the small-shape
backward tests)."""
import numpy as np
import pytest
import torch

import oracle
from workloads import make_tokens, make_weights, shape

from _helpers import check_logits, check_routing, to_np

pytestmark = pytest.mark.gpu
DEV = "cuda"


class _Experts:
    """A device weight tensor [E, ...] seen by the oracle one expert at a time
    (copied to the host in fp32 when first touched)."""

    def __init__(self, t):
        self.t = t
        self.shape = tuple(t.shape)
        self.cache = {}

    def __getitem__(self, e):
        e = int(e)
        if e not in self.cache:
            self.cache[e] = self.t[e].float().cpu().numpy()
        return self.cache[e]


def _bounded(got, ref, S, Smax, what):
    got = np.asarray(got, np.float64)
    bound = 2.0 ** -5 * np.asarray(S) + 1e-6 * Smax
    err = np.abs(got - np.asarray(ref))
    assert np.all(np.isfinite(got)), what
    worst = float(np.max(err / bound))
    assert worst <= 1.0, f"{what}: worst error / bound {worst:.3f}"
    return worst


@pytest.mark.parametrize("name", ["mixtral", "qwen", "dsv3"])
def test_full_size_backward_sampled(name):
    import dropless_moe_expert_gb300 as moe
    s = shape(name)
    T, d, E, K, f = s.T, s.d, s.E, s.K, s.f
    w = make_weights(s, seed=0, device=DEV)
    x = make_tokens(s, seed=0, device=DEV)
    g = torch.Generator(device=DEV)
    g.manual_seed(11)
    dy = torch.randn((T, d), generator=g, device=DEV).to(torch.bfloat16)
    layer = moe.MoELayer(w.Wr, w.bias, w.W1, w.W2, K, T)
    layer(x, save_preact=True)
    grads = layer.backward(x, dy)
    torch.cuda.synchronize()
    assert moe.device_status() == 0
    v = layer.views(T)

    # the oracle's routing, from its own fp32 logits
    xs, Wr, bias = to_np(x), to_np(w.Wr), to_np(w.bias)
    _, scale, L64 = check_logits(to_np(v["logits"]), xs, Wr, bias)
    L = oracle.router_logits_fp32(xs, Wr, bias)
    idx, wref = oracle.topk_route(L, K)
    counts, offsets = oracle.expert_counts(idx, E)
    src_tok, row_of = oracle.dispatch_order(idx, E)
    routing = dict(idx=idx, w=wref, offsets=offsets, src_tok=src_tok, row_of=row_of)
    same = check_routing(to_np(v["topk_idx"]), idx, L64, scale, K)
    # experts whose groups hold the same tokens on both sides
    gpu_offs = to_np(v["offsets"])
    ok_e = [e for e in range(E) if counts[e] > 0 and gpu_offs[e] == offsets[e] and gpu_offs[e + 1] == offsets[e + 1]
            and same[src_tok[offsets[e]:offsets[e + 1]]].all()]
    assert ok_e, "no expert routed identically on both sides"
    by_size = sorted(ok_e, key=lambda e: counts[e])
    experts = sorted({by_size[0], by_size[len(by_size) // 2], by_size[-1]})

    rng = np.random.default_rng(3)
    dW1_at = [(e, i, j) for e in experts for i, j in
              [(0, 0), (f - 1, d - 1), (f, 1), (2 * f - 1, d // 2),
               (int(rng.integers(2 * f)), int(rng.integers(d)))]]
    dW2_at = [(e, i, j) for e in experts for i, j in
              [(0, 0), (d - 1, f - 1), (int(rng.integers(d)), int(rng.integers(f)))]]
    cand = np.nonzero(same)[0]
    dx_at = sorted({int(cand[0]), int(cand[-1]), int(rng.choice(cand))})

    ref = oracle.backward_sampled(xs, Wr, bias, _Experts(w.W1), _Experts(w.W2), K, to_np(dy), routing, dW1_at,
                                  dW2_at, dx_at)
    dW1 = grads["dW1"]
    dW2 = grads["dW2"]
    g1 = np.array([dW1[e, i, j].item() for e, i, j in dW1_at])
    g2 = np.array([dW2[e, i, j].item() for e, i, j in dW2_at])
    r1 = np.array([v_ for v_, _ in ref["dW1"]])
    S1 = np.array([s_ for _, s_ in ref["dW1"]])
    r2 = np.array([v_ for v_, _ in ref["dW2"]])
    S2 = np.array([s_ for _, s_ in ref["dW2"]])
    worst = {"dW1": _bounded(g1, r1, S1, S1.max(), "dW1"), "dW2": _bounded(g2, r2, S2, S2.max(), "dW2")}
    gdx = to_np(grads["dx"][torch.tensor(dx_at, device=DEV)])
    rdx = np.stack([v_ for v_, _ in ref["dx"]])
    Sdx = np.stack([s_ for _, s_ in ref["dx"]])
    worst["dx"] = _bounded(gdx, rdx, Sdx, Sdx.max(), "dx")
    # experts without tokens get exactly zero weight gradients
    for e in np.nonzero(counts == 0)[0][:3]:
        assert not dW1[int(e)].any() and not dW2[int(e)].any()
    print(f"{name}: experts {experts} (rows {[int(counts[e]) for e in experts]}), tokens {dx_at}; "
          f"worst error / bound {worst}")
