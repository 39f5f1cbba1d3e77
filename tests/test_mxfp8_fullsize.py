"""GPU parity of the MXFP8 layer forward at the full workload sizes, on
sampled rows.  The whole layer runs on the device; the oracle routes on its
own fp32 logits (every logit is checked against fp64 and the routing with
the rules of the bf16 tests), quantises the touched experts' weights on the
host and evaluates sampled rows of each touched expert one by one
(oracle.expert_ffn_mxfp8) and a few whole tokens
(oracle.forward_mxfp8_tokens), both pinned to oracle.forward_mxfp8 on small
cases.  The experts touched: every expert of the first identically routed
token, and the most and the least loaded non-empty expert.  Checks:
  * the device's weight codes and scale bytes of those experts, bit-exact;
  * the permuted, quantised token rows (codes and scale bytes), bit-exact;
  * h within half an E4M3 ulp of its block (check_mx_rounded);
  * y_perm of the sampled rows and y of the tokens whose experts are all
    touched, with the bf16 path's output tolerances."""
import numpy as np
import pytest
import torch

import oracle
from workloads import make_tokens, make_weights, shape

from _helpers import (check_logits, check_mx_rounded, check_output, check_routing, to_np, unpack_group_atoms,
                      unpack_plain_atoms)

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _atoms_of(buf, e, rows_per_expert, K):
    """Scale atoms of expert e's rows of a weight quantised as one plain
    matrix [E * rows_per_expert, K] (rows_per_expert a multiple of 128)."""
    n = (rows_per_expert // 128) * (K // 128) * 512
    return buf[e * n:(e + 1) * n].cpu().numpy()


@pytest.mark.parametrize("name", ["mixtral", "dsv3", "qwen", "skew"])
def test_full_size_mxfp8_sampled(name):
    import dropless_moe_expert_gb300 as moe
    s = shape(name)
    T, d, E, K, f = s.T, s.d, s.E, s.K, s.f
    w = make_weights(s, seed=0, device=DEV)
    x = make_tokens(s, seed=0, device=DEV)
    layer = moe.MoELayerMXFP8(w.Wr, w.bias, w.W1, w.W2, K, T)
    layer.workspace.fill_(0xFF)
    y = torch.full_like(x, float("nan"))
    layer(x, out=y)
    torch.cuda.synchronize()
    assert moe.device_status() == 0
    assert bool(torch.isfinite(y.float()).all())
    v = layer.views(T)

    xs, Wr, bias = to_np(x), to_np(w.Wr), to_np(w.bias)
    _, scale, L64 = check_logits(to_np(v["logits"]), xs, Wr, bias)
    L = oracle.router_logits_fp32(xs, Wr, bias)
    idx, _ = oracle.topk_route(L, K)
    same = check_routing(to_np(v["topk_idx"]), idx, L64, scale, K)
    offs = to_np(v["offsets"]).astype(np.int64)
    src = to_np(v["src_tok"]).astype(np.int64)
    row_of = to_np(v["row_of"]).astype(np.int64)
    counts = np.diff(offs)
    nz = np.nonzero(counts)[0]
    tok0 = int(np.nonzero(same)[0][0])
    experts = sorted(set(idx[tok0].tolist()) | {int(nz[np.argmax(counts[nz])]), int(nz[np.argmin(counts[nz])])})

    deq = {}

    def expert_weights(e):
        """The oracle's dequantised weights of expert e; its codes and scale
        bytes are checked against the device's on the way."""
        if e not in deq:
            c1, s1, W1d = oracle.mx_quantize(to_np(w.W1[e]))
            assert np.array_equal(layer.W1q[e].cpu().numpy(), c1), f"W1 codes of expert {e}"
            assert np.array_equal(unpack_plain_atoms(_atoms_of(layer.W1s, e, 2 * f, d), 2 * f, d), s1), \
                f"W1 scales of expert {e}"
            c2, s2, W2d = oracle.mx_quantize(to_np(w.W2[e]))
            assert np.array_equal(layer.W2q[e].cpu().numpy(), c2), f"W2 codes of expert {e}"
            assert np.array_equal(unpack_plain_atoms(_atoms_of(layer.W2s, e, d, f), d, f), s2), \
                f"W2 scales of expert {e}"
            deq[e] = (W1d, W2d)
        return deq[e]

    sfa = to_np(v["sfa"])
    sfh = to_np(v["sfh"])
    g = np.random.default_rng(7)
    n_rows = 0
    for e in experts:
        r0, r1 = int(offs[e]), int(offs[e + 1])
        rows = set(range(r0, min(r1, r0 + 4))) | set(range(max(r0, r1 - 4), r1))
        rows |= set(g.integers(r0, r1, 8).tolist())
        rows |= {int(row_of[tok0, k]) for k in range(K) if idx[tok0, k] == e}
        rows = np.array(sorted(r for r in rows if same[src[r]]))
        tok = src[rows]
        ref = oracle.expert_ffn_mxfp8(xs[tok], *expert_weights(e))
        rt = torch.from_numpy(rows).to(DEV)
        assert np.array_equal(to_np(v["xq_perm"][rt]), ref["xq"]), f"x codes, expert {e}"
        assert np.array_equal(unpack_group_atoms(sfa, offs, d, rows), ref["xs"]), f"x scales, expert {e}"
        hd = oracle.mx_dequantize(to_np(v["hq"][rt]), unpack_group_atoms(sfh, offs, f, rows))
        check_mx_rounded(hd, ref["h"], ref["hs"], f"h, expert {e}")
        check_output(to_np(v["y_perm"][rt]), ref["y_perm"], f"y_perm, expert {e}")
        n_rows += len(rows)

    # whole tokens whose K experts were all touched (the first one at least)
    cand = np.nonzero(same & np.isin(idx, experts).all(axis=1))[0]
    toks = np.unique(np.concatenate([[tok0], cand[:15]]))
    ridx, _, _, ry = oracle.forward_mxfp8_tokens(xs[toks], L[toks], K, expert_weights)
    assert np.array_equal(ridx, idx[toks])
    r = check_output(to_np(y[torch.from_numpy(toks).to(DEV)]), ry, "y (sampled tokens)")
    print(f"{name}: experts {experts}, {n_rows} sampled rows, {len(toks)} tokens y rel_l2={r[0]:.2e} "
          f"max/rms={r[1]:.2e}, tokens routed differently (near ties) {int((~same).sum())}")
