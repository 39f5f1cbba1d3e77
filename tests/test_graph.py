"""The whole layer captured once in a CUDA graph and replayed with re-drawn
tokens (hence new routings, new group sizes, new empty experts): every replay
must match the oracle, so no routing-dependent value was frozen at capture
("What specialized optimizations are needed for dropless MoE?": shapes the
CPU cannot see; "Optimization 1: Grouped GEMM": no device-to-host copy)."""
import numpy as np
import pytest
import torch

import dropless_moe_expert_gb300 as moe
import oracle
from workloads import Shape, make_tokens, make_weights

from _helpers import check_logits, check_output, check_routing, to_np, weight_tol

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("s", [
    Shape(T=256, d=128, E=8, K=2, f=256),
    Shape(T=2048, d=256, E=64, K=6, f=192, bias="skew"),
    Shape(T=1000, d=128, E=256, K=8, f=128, bias="zipf_1.1"),
], ids=["tiny", "skew_small", "zipf_small"])
def test_graph_replay_with_new_routing(s):
    w = make_weights(s, seed=0, device="cpu")
    wd = [t.cuda() for t in (w.Wr, w.bias, w.W1, w.W2)]
    layer = moe.MoELayer(*wd, s.K, s.T)
    x_static = make_tokens(s, seed=0, device="cpu").cuda()
    y_static = torch.empty_like(x_static)
    layer(x_static, out=y_static)          # first call on the device: set-up outside capture
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        layer(x_static, out=y_static)
    seen_counts = []
    for seed in (1, 2, 3, 4):
        xc = make_tokens(s, seed=seed, device="cpu")
        x_static.copy_(xc)
        layer.workspace.fill_(0xFF)
        y_static.fill_(float("nan"))
        graph.replay()
        torch.cuda.synchronize()
        assert moe.device_status() == 0
        v = layer.views(s.T)
        xs = xc.float().numpy()
        _, scale, L64 = check_logits(to_np(v["logits"]), xs, w.Wr.numpy(), w.bias.numpy())
        ref = oracle.forward(xs, w.Wr.numpy(), w.bias.numpy(), w.W1.float().numpy(), w.W2.float().numpy(), s.K)
        idx = to_np(v["topk_idx"])
        same = check_routing(idx, ref["idx"], L64, scale, s.K)
        dw = np.abs(to_np(v["topk_w"]) - ref["w"]).max(axis=1)
        assert np.all(dw[same] <= weight_tol(scale, idx)[same])
        if same.all():
            assert np.array_equal(to_np(v["offsets"]), ref["offsets"])
            assert np.array_equal(to_np(v["row_of"]), ref["row_of"])
        check_output(to_np(y_static)[same], ref["y"][same], f"y (replay seed {seed})")
        seen_counts.append(tuple(ref["counts"].tolist()))
    assert len(set(seen_counts)) == len(seen_counts), "replays should see different routings"
