"""The grouped GEMMs' dynamic tile order under concurrency.

The CTAs of one grouped-GEMM launch hand out its tiles through a counter in
a library-owned table; each launch takes a slot of its own (eager launches
from a ring, launches captured into a graph a slot kept for every replay).
Whatever runs beside a launch, its output must be what it is alone: here
two layers run on two streams at once, eagerly and as two captured graphs
replayed side by side, and every output is compared bit for bit with the
same layer run alone.  The shapes take the dynamic order in both GEMMs (a
CTA-pair shape with d and f >= 4096) or in GEMM2 (a single-CTA shape)."""
import pytest
import torch

from workloads import Shape, make_tokens, make_weights

pytestmark = pytest.mark.gpu
DEV = "cuda"

CASES = [
    Shape(T=1024, d=4096, E=3, K=2, f=4160, bias="normal_0.5"),   # pair kernel, dynamic order in both GEMMs
    Shape(T=2048, d=512, E=128, K=8, f=512, bias="zipf_1.1"),     # single-CTA, dynamic order in GEMM2
]


def _layer(s, seed):
    import dropless_moe_expert_gb300 as moe
    w = make_weights(s, seed=seed, device=DEV)
    return moe.MoELayer(w.Wr, w.bias, w.W1, w.W2, s.K, s.T)


@pytest.mark.parametrize("s", CASES, ids=lambda s: f"T{s.T}_d{s.d}_E{s.E}_K{s.K}_f{s.f}")
def test_two_streams_eager_and_two_graphs_side_by_side(s):
    import dropless_moe_expert_gb300 as moe
    la, lb = _layer(s, 1), _layer(s, 2)
    xa = [make_tokens(s, seed=10 + i, device=DEV) for i in range(3)]
    xb = [make_tokens(s, seed=20 + i, device=DEV) for i in range(3)]
    # each layer alone, one call after the other
    ref_a = [la(x).clone() for x in xa]
    ref_b = [lb(x).clone() for x in xb]
    torch.cuda.synchronize()

    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    s1.wait_stream(torch.cuda.current_stream())
    s2.wait_stream(torch.cuda.current_stream())
    # eager, both streams at once
    ya, yb = [], []
    for i in range(3):
        with torch.cuda.stream(s1):
            ya.append(la(xa[i]))
        with torch.cuda.stream(s2):
            yb.append(lb(xb[i]))
    torch.cuda.synchronize()
    assert moe.device_status() == 0
    for i in range(3):
        assert torch.equal(ya[i].view(torch.int16), ref_a[i].view(torch.int16)), f"eager, stream 1, call {i}"
        assert torch.equal(yb[i].view(torch.int16), ref_b[i].view(torch.int16)), f"eager, stream 2, call {i}"

    # two captured graphs, replayed side by side on the two streams
    xa_g, xb_g = xa[0].clone(), xb[0].clone()
    ya_g = torch.empty_like(ref_a[0])
    yb_g = torch.empty_like(ref_b[0])
    ga, gb = torch.cuda.CUDAGraph(), torch.cuda.CUDAGraph()
    with torch.cuda.graph(ga, stream=s1):
        la(xa_g, out=ya_g)
    with torch.cuda.graph(gb, stream=s2):
        lb(xb_g, out=yb_g)
    torch.cuda.synchronize()
    for i in range(3):
        xa_g.copy_(xa[i])
        xb_g.copy_(xb[i])
        torch.cuda.synchronize()
        with torch.cuda.stream(s1):
            ga.replay()
        with torch.cuda.stream(s2):
            gb.replay()
        torch.cuda.synchronize()
        assert moe.device_status() == 0
        assert torch.equal(ya_g.view(torch.int16), ref_a[i].view(torch.int16)), f"graph A, replay {i}"
        assert torch.equal(yb_g.view(torch.int16), ref_b[i].view(torch.int16)), f"graph B, replay {i}"
    # and the eager path still right after the captures
    y = la(xa[2])
    torch.cuda.synchronize()
    assert torch.equal(y.view(torch.int16), ref_a[2].view(torch.int16))
