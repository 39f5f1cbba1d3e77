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


@pytest.mark.parametrize("name", ["small", "dsv3", "mixtral"])
def test_training_step_graph_replays_match_eager(name):
    """The training step -- moe_forward_train (saving the pre-activations) then
    moe_backward -- captured once and replayed with new tokens and output
    gradients: the gradients equal an eager run's bit for bit (the backward
    reads every count on the device too, and rebuilds its per-expert tensor
    maps on the device every replay).  At a small shape and at the full
    DSv3- and Mixtral-shaped workloads (single-CTA and CTA-pair kernels)."""
    from workloads import shape
    s = Shape(T=300, d=256, E=16, K=4, f=128, bias="normal_0.5") if name == "small" else shape(name)
    w = make_weights(s, seed=0, device="cuda")
    wd = [w.Wr, w.bias, w.W1, w.W2]
    layer = moe.MoELayer(*wd, s.K, s.T)
    x_static = make_tokens(s, seed=0, device="cuda")
    dy_static = torch.randn((s.T, s.d), device="cuda").to(torch.bfloat16)
    y_static = torch.empty_like(x_static)
    layer(x_static, out=y_static, save_preact=True)   # set-up (buffers, library state) outside capture
    grads = layer.backward(x_static, dy_static)
    ws = layer.bw_workspace
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        layer(x_static, out=y_static, save_preact=True)
        layer.backward(x_static, dy_static, grads=grads, workspace=ws)
    eager = moe.MoELayer(*wd, s.K, s.T)
    for seed in (1, 2, 3):
        x_new = make_tokens(s, seed=seed, device="cuda")
        g = torch.Generator(device="cuda").manual_seed(seed)
        dy_new = torch.randn((s.T, s.d), device="cuda", generator=g).to(torch.bfloat16)
        x_static.copy_(x_new)
        dy_static.copy_(dy_new)
        for t in grads.values():
            t.fill_(float("nan"))
        graph.replay()
        y_e = eager(x_new, save_preact=True)
        g_e = eager.backward(x_new, dy_new)
        torch.cuda.synchronize()
        assert moe.device_status() == 0
        assert torch.equal(y_static.view(torch.int16), y_e.view(torch.int16))
        for k in g_e:
            a, b = grads[k], g_e[k]
            if a.dtype == torch.bfloat16:
                a, b = a.view(torch.int16), b.view(torch.int16)
            assert torch.equal(a, b), (seed, k)


def test_full_size_skew_graph_replays_match_eager():
    """The skew workload at full size (T=32768, d=4096, E=64, K=6, f=1536):
    one captured graph replayed on re-seeded tokens, each replay bitwise equal
    to an eager call on the same tokens (the eager layer is checked against
    the oracle at this size in test_parity.py), with different routings."""
    from workloads import shape
    s = shape("skew")
    w = make_weights(s, seed=0, device="cuda")
    layer = moe.MoELayer(w.Wr, w.bias, w.W1, w.W2, s.K, s.T)
    eager = moe.MoELayer(w.Wr, w.bias, w.W1, w.W2, s.K, s.T)
    x_static = make_tokens(s, seed=0, device="cuda")
    y_static = torch.empty_like(x_static)
    layer(x_static, out=y_static)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        layer(x_static, out=y_static)
    counts = []
    for seed in (1, 2, 3):
        x = make_tokens(s, seed=seed, device="cuda")
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
