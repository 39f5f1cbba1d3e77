"""Failure detection without a GPU fault.

Host side: bad arguments come back as status codes with nothing launched
(tests/test_abi.py).  Device side: every wait in the kernels is bounded; here
a kernel whose wait can never complete runs out its short limit, records
MOE_ERR_DEVICE_TIMEOUT in the device status word, and returns, after which the
same context still runs the layer correctly."""
import time

import pytest
import torch

import dropless_moe_expert_gb300 as moe
from workloads import Shape, make_tokens, make_weights

from _helpers import check_output, to_np

pytestmark = pytest.mark.gpu

MOE_ERR_DEVICE_TIMEOUT = 5


def test_bounded_wait_times_out_and_reports():
    assert moe.device_status() == 0
    t0 = time.perf_counter()
    moe.check_bounded_wait(limit_ns=2_000_000)      # 2 ms
    torch.cuda.synchronize()
    waited = time.perf_counter() - t0
    assert moe.device_status() == MOE_ERR_DEVICE_TIMEOUT
    assert moe.device_status() == 0                 # reading clears the word
    assert waited < 5.0


def test_context_usable_after_timeout():
    import oracle
    moe.check_bounded_wait(limit_ns=1_000_000)
    torch.cuda.synchronize()
    assert moe.device_status() == MOE_ERR_DEVICE_TIMEOUT
    s = Shape(T=64, d=128, E=4, K=2, f=128)
    w = make_weights(s, seed=3, device="cpu")
    x = make_tokens(s, seed=3, device="cpu")
    y = moe.forward(x.cuda(), w.Wr.cuda(), w.bias.cuda(), w.W1.cuda(), w.W2.cuda(), s.K)
    torch.cuda.synchronize()
    assert moe.device_status() == 0
    ref = oracle.forward(x.float().numpy(), w.Wr.numpy(), w.bias.numpy(), w.W1.float().numpy(),
                         w.W2.float().numpy(), s.K)
    check_output(to_np(y), ref["y"])


def test_status_read_inside_a_captured_graph():
    """The capture-safe status read: a graph holding a wait that times out
    and then moe_last_device_status reports MOE_ERR_DEVICE_TIMEOUT in the
    caller's device word on every replay, with no synchronous read; a graph
    holding only the read, replayed next, reports 0 (the word was cleared)."""
    assert moe.device_status() == 0
    word = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    clean = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        moe.last_device_status(clean)          # the per-device set-up happens outside capture
    s.synchronize()
    g_wait, g_read = torch.cuda.CUDAGraph(), torch.cuda.CUDAGraph()
    with torch.cuda.graph(g_wait, stream=s):
        moe.check_bounded_wait(limit_ns=2_000_000)
        moe.last_device_status(word)
    with torch.cuda.graph(g_read, stream=s):
        moe.last_device_status(clean)
    for _ in range(2):
        word.fill_(-1)
        clean.fill_(-1)
        g_wait.replay()
        g_read.replay()
        torch.cuda.synchronize()
        assert int(word.item()) == MOE_ERR_DEVICE_TIMEOUT
        assert int(clean.item()) == 0
    assert moe.device_status() == 0


def test_bounded_wait_rejects_out_of_range_limits():
    with pytest.raises(moe.MoEError):
        moe.check_bounded_wait(limit_ns=10)
    with pytest.raises(moe.MoEError):
        moe.check_bounded_wait(limit_ns=5_000_000_000)
