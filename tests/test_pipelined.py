"""GPU tests of the pipelined host runners (moe_forward_host_pipelined,
moe_forward_mxfp8_host_pipelined): every batch's output equals, bit for bit,
the device forward of the same input, whatever the overlap of copies and
compute -- including host buffers that repeat across batches, so that a
buffer reused before its previous copy finished would show."""
import pytest
import torch

from workloads import Shape, make_tokens, make_weights

pytestmark = pytest.mark.gpu
DEV = "cuda"
S = Shape(T=300, d=256, E=16, K=4, f=128, bias="normal_0.5")


def _setup(seed=3):
    w = make_weights(S, seed=0, device=DEV)
    xs = [make_tokens(S, seed=seed + i, device="cpu").pin_memory() for i in range(5)]
    return w, xs


@pytest.mark.parametrize("n", [1, 2, 5])
def test_pipelined_matches_forward(n):
    import dropless_moe_expert_gb300 as moe
    w, xs = _setup()
    xs = xs[:n]
    ys = [torch.full((S.T, S.d), float("nan"), dtype=torch.bfloat16).pin_memory() for _ in range(n)]
    moe.forward_host_pipelined(xs, ys, w.Wr, w.bias, w.W1, w.W2, S.K)
    torch.cuda.synchronize()
    assert moe.device_status() == 0
    for x, y in zip(xs, ys):
        ref = moe.forward(x.to(DEV), w.Wr, w.bias, w.W1, w.W2, S.K).cpu()
        assert torch.equal(y.view(torch.int16), ref.view(torch.int16))


def test_pipelined_repeated_host_buffers():
    import dropless_moe_expert_gb300 as moe
    w, xs = _setup(seed=11)
    xa, xb = xs[0], xs[1]
    ya, yb = (torch.empty((S.T, S.d), dtype=torch.bfloat16).pin_memory() for _ in range(2))
    yc = torch.empty((S.T, S.d), dtype=torch.bfloat16).pin_memory()
    # batches a, b, a, b, b: the last write of ya comes from xa, of yb and yc from xb
    moe.forward_host_pipelined([xa, xb, xa, xb, xb], [ya, yb, ya, yb, yc], w.Wr, w.bias, w.W1, w.W2, S.K)
    torch.cuda.synchronize()
    ra = moe.forward(xa.to(DEV), w.Wr, w.bias, w.W1, w.W2, S.K).cpu()
    rb = moe.forward(xb.to(DEV), w.Wr, w.bias, w.W1, w.W2, S.K).cpu()
    assert torch.equal(ya.view(torch.int16), ra.view(torch.int16))
    assert torch.equal(yb.view(torch.int16), rb.view(torch.int16))
    assert torch.equal(yc.view(torch.int16), rb.view(torch.int16))


def test_pipelined_mxfp8_matches_forward():
    import dropless_moe_expert_gb300 as moe
    w, xs = _setup(seed=21)
    layer = moe.MoELayerMXFP8(w.Wr, w.bias, w.W1, w.W2, S.K, S.T)
    ys = [torch.empty((S.T, S.d), dtype=torch.bfloat16).pin_memory() for _ in xs]
    moe.forward_mxfp8_host_pipelined(xs, ys, w.Wr, w.bias, layer.W1q, layer.W1s, layer.W2q, layer.W2s, S.K)
    torch.cuda.synchronize()
    assert moe.device_status() == 0
    for x, y in zip(xs, ys):
        ref = layer(x.to(DEV)).cpu()
        assert torch.equal(y.view(torch.int16), ref.view(torch.int16))


def test_pipelined_full_size_skew():
    """The skew workload at full size (T=32768, d=4096: 268 MB of x and of y
    per batch), three batches: each equal to the device forward bit for bit."""
    import dropless_moe_expert_gb300 as moe
    from workloads import shape
    s = shape("skew")
    w = make_weights(s, seed=0, device=DEV)
    xs = [make_tokens(s, seed=40 + i, device=DEV).cpu().pin_memory() for i in range(3)]
    ys = [torch.full((s.T, s.d), float("nan"), dtype=torch.bfloat16).pin_memory() for _ in xs]
    moe.forward_host_pipelined(xs, ys, w.Wr, w.bias, w.W1, w.W2, s.K)
    torch.cuda.synchronize()
    assert moe.device_status() == 0
    for x, y in zip(xs, ys):
        ref = moe.forward(x.to(DEV), w.Wr, w.bias, w.W1, w.W2, s.K).cpu()
        assert torch.equal(y.view(torch.int16), ref.view(torch.int16))
