"""moe_route_static, the routing entry point that allocates nothing, against
moe_route, the one that takes a caller-provided workspace.

Callers such as an inference-engine plugin (no allocation in its enqueue
step), or a runtime that owns all device memory in a fixed pool and forbids
any other allocation, cannot hand the library a workspace; moe_route_static
keeps its scratch in a fixed library-owned device array instead.  Its outputs must
be those of moe_route, on two calls in a row (the second call finds the
first call's scratch contents and must not depend on them).  This file is
collected last so that a stop at the first failure has run every other test.
"""
import ctypes

import numpy as np
import pytest
import torch

import dropless_moe_expert_gb300 as moe

from _helpers import to_np

pytestmark = pytest.mark.gpu

P, I = ctypes.c_void_p, ctypes.c_int


def _static_fn():
    lib = ctypes.CDLL(moe.build.lib_path())
    fn = lib.moe_route_static
    fn.restype = I
    fn.argtypes = [P, I, I, I, P, P, P, P, P, P, P]
    return fn


def _route_static(fn, logits, K):
    T, E = logits.shape
    dev = logits.device
    out = dict(topk_idx=torch.full((T, K), -7, dtype=torch.int32, device=dev),
               topk_w=torch.full((T, K), float("nan"), device=dev),
               counts=torch.full((E,), -7, dtype=torch.int32, device=dev),
               offsets=torch.full((E + 1,), -7, dtype=torch.int32, device=dev),
               row_of=torch.full((T, K), -7, dtype=torch.int32, device=dev),
               src_tok=torch.full((T * K,), -7, dtype=torch.int32, device=dev))
    st = fn(logits.data_ptr(), T, E, K, out["topk_idx"].data_ptr(), out["topk_w"].data_ptr(),
            out["counts"].data_ptr(), out["offsets"].data_ptr(), out["row_of"].data_ptr(),
            out["src_tok"].data_ptr(), torch.cuda.current_stream().cuda_stream)
    assert st == 0, moe.lib.moe_status_string(st).decode()
    return out


def _same_as_route(got, ref):
    assert np.array_equal(to_np(got["topk_idx"]), to_np(ref.topk_idx))
    # the same kernels on the same logits: the gate weights agree bit for bit
    assert np.array_equal(to_np(got["topk_w"]).view(np.uint32), to_np(ref.topk_w).view(np.uint32))
    assert np.array_equal(to_np(got["counts"]), to_np(ref.counts))
    assert np.array_equal(to_np(got["offsets"]), to_np(ref.offsets))
    assert np.array_equal(to_np(got["row_of"]), to_np(ref.row_of))
    assert np.array_equal(to_np(got["src_tok"]), to_np(ref.src_tok))


@pytest.mark.parametrize("T,E,K", [(8192, 8, 2), (4096, 256, 8), (1000, 64, 6), (1, 1, 1)])
def test_route_static_matches_route_on_two_calls(T, E, K):
    fn = _static_fn()
    g = torch.Generator(device="cuda")
    g.manual_seed(T + E + K)
    first = torch.randn((T, E), generator=g, device="cuda")
    second = torch.randn((T, E), generator=g, device="cuda")
    second[:, 0] += 3.0           # a different, skewed routing for the second call
    for logits in (first, second):
        got = _route_static(fn, logits, K)
        ref = moe.route(logits, K)
        torch.cuda.synchronize()
        _same_as_route(got, ref)


def test_route_static_rejects_sizes_beyond_its_scratch():
    fn = _static_fn()
    # 513 chunks of 64 tokens x 256 experts x 2 tables x 4 bytes > 1 MiB
    T, E, K = 64 * 513, 256, 8
    assert moe.route_workspace_size(T, E, K) > 1024 * 1024
    assert moe.route_workspace_size(64 * 512, E, K) == 1024 * 1024
    # inputs and outputs of the call's full sizes, so that a regression of
    # the size check shows up as a wrong status below, not as kernels
    # reading and writing past the ends of undersized stand-in buffers
    logits = torch.randn((T, E), device="cuda")
    out = dict(topk_idx=torch.full((T, K), -7, dtype=torch.int32, device="cuda"),
               topk_w=torch.zeros((T, K), device="cuda"),
               counts=torch.full((E,), -7, dtype=torch.int32, device="cuda"),
               offsets=torch.full((E + 1,), -7, dtype=torch.int32, device="cuda"),
               row_of=torch.full((T, K), -7, dtype=torch.int32, device="cuda"),
               src_tok=torch.full((T * K,), -7, dtype=torch.int32, device="cuda"))
    torch.cuda.synchronize()
    st = fn(logits.data_ptr(), T, E, K, out["topk_idx"].data_ptr(), out["topk_w"].data_ptr(),
            out["counts"].data_ptr(), out["offsets"].data_ptr(), out["row_of"].data_ptr(),
            out["src_tok"].data_ptr(), torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    assert st == 2                                          # MOE_ERR_UNSUPPORTED
    # nothing was launched: every output still holds its fill value
    assert bool((out["counts"] == -7).all()) and bool((out["row_of"] == -7).all())
