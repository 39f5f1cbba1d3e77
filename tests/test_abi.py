"""The C ABI: the library loads, exports every symbol include/moe.h declares,
and rejects bad arguments on the host before anything is launched (so these
run without a GPU)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "moe.h")


@pytest.fixture(scope="module")
def moe():
    import __graft_entry__
    __graft_entry__.build()
    import dropless_moe_expert_gb300 as m
    return m


def _declared():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(moe_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = _declared()
    for n in ["moe_router_logits", "moe_router_workspace_size", "moe_route", "moe_permute", "moe_grouped_mlp",
              "moe_unpermute",
              "moe_route_workspace_size", "moe_status_string", "moe_forward", "moe_device_status",
              "moe_last_device_status"]:
        assert n in names


def test_library_exports_every_declared_symbol(moe):
    lib = ctypes.CDLL(moe.build.lib_path())
    missing = [n for n in _declared() if not hasattr(lib, n)]
    assert not missing, missing


def test_status_strings(moe):
    for code in range(6):
        s = moe.lib.moe_status_string(code).decode()
        assert s.startswith("MOE_")
    assert moe.lib.moe_status_string(99).decode() == "unknown moe_status_t"
    assert moe.lib.moe_abi_version() == 403


def test_workspace_sizes(moe):
    # two int32 [chunks, E] tables, 64 tokens per chunk
    assert moe.route_workspace_size(64, 8, 2) == 1 * 8 * 2 * 4
    assert moe.route_workspace_size(65, 8, 2) == 2 * 8 * 2 * 4
    assert moe.route_workspace_size(32768, 64, 6) == 512 * 64 * 2 * 4
    v = moe.forward_views(8192, 4096, 8, 2, 14336)
    TK = 8192 * 2
    assert v["h"] - v["x_perm"] >= TK * 4096 * 2 and v["y_perm"] - v["h"] >= TK * 14336 * 2
    offs = [v[k] for k in ("logits", "topk_idx", "topk_w", "counts", "offsets", "row_of", "src_tok",
                           "route_ws", "router_ws", "x_perm", "h", "y_perm", "x_dev", "y_dev", "total")]
    assert v["x_perm"] - v["router_ws"] >= moe.router_workspace_size(4096, 8)
    assert offs == sorted(offs) and all(o % 256 == 0 for o in offs)
    assert moe.forward_workspace_size(8192, 4096, 8, 2, 14336) == v["total"]
    assert moe.forward_workspace_size(8, 100, 8, 2, 64) == 0      # d not a multiple of 64
    # three bf16 pieces of Wr, [3][E][d]
    assert moe.router_workspace_size(7168, 256) == 3 * 256 * 7168 * 2
    assert moe.router_workspace_size(100, 8) == 0 and moe.router_workspace_size(64, 257) == 0


FAKE = 1 << 20  # a 16-byte aligned non-null address; never dereferenced (rejected first)


@pytest.mark.parametrize("args,code", [
    # T, d, E, K, f
    ((0, 64, 8, 2, 64), 1),       # T < 1
    ((8, 64, 8, 9, 64), 1),       # K > E
    ((8, 64, 8, 0, 64), 1),       # K < 1
    ((8, 64, 300, 2, 64), 2),     # E > 256
    ((8, 64, 32, 17, 64), 2),     # K > 16
    ((8, 96, 8, 2, 64), 2),       # d % 64
    ((8, 64, 8, 2, 96), 2),       # f % 64
])
def test_forward_rejects_bad_shapes(moe, args, code):
    T, d, E, K, f = args
    r = moe.lib.moe_forward(FAKE, FAKE, None, FAKE, FAKE, T, d, E, K, f, FAKE, FAKE, 1 << 40, None)
    assert r == code


def test_null_and_misaligned_pointers_rejected(moe):
    L = moe.lib
    # the fused-permute GEMM1: null, misaligned and bad sizes
    assert L.moe_grouped_gemm1_swiglu_gather(None, FAKE, FAKE, 8, 8, 16, 64, 64, FAKE, FAKE, None) == 1
    assert L.moe_grouped_gemm1_swiglu_gather(FAKE + 2, FAKE, FAKE, 8, 8, 16, 64, 64, FAKE, FAKE, None) == 1
    assert L.moe_grouped_gemm1_swiglu_gather(FAKE, FAKE, FAKE, 0, 8, 16, 64, 64, FAKE, FAKE, None) == 1
    assert L.moe_grouped_gemm1_swiglu_gather(FAKE, FAKE, FAKE, 8, 8, 16, 96, 64, FAKE, FAKE, None) == 2
    # the status read checks its pointer before it touches CUDA
    assert L.moe_last_device_status(None, None) == 1
    assert L.moe_last_device_status(FAKE + 2, None) == 1
    assert L.moe_forward(None, FAKE, None, FAKE, FAKE, 8, 64, 8, 2, 64, FAKE, FAKE, 1 << 40, None) == 1
    assert L.moe_forward(FAKE + 2, FAKE, None, FAKE, FAKE, 8, 64, 8, 2, 64, FAKE, FAKE, 1 << 40, None) == 1
    assert L.moe_router_logits(FAKE, FAKE, None, 8, 64, 8, None, FAKE, 1 << 20, None) == 1
    assert L.moe_router_logits(FAKE + 8, FAKE, None, 8, 64, 8, FAKE, FAKE, 1 << 20, None) == 1
    assert L.moe_router_logits(FAKE, FAKE, None, 8, 64, 8, FAKE, None, 1 << 20, None) == 1
    assert L.moe_router_logits(FAKE, FAKE, None, 8, 64, 8, FAKE, FAKE + 8, 1 << 20, None) == 1
    assert L.moe_permute(FAKE, FAKE, 8, 2, 64, FAKE + 4, None) == 1
    assert L.moe_unpermute(FAKE, FAKE, None, 8, 2, 64, FAKE, None) == 1
    assert L.moe_grouped_mlp(FAKE, FAKE, 8, 16, 64, 64, FAKE, None, FAKE, FAKE, None) == 1
    assert L.moe_grouped_gemm1_swiglu(FAKE, FAKE, 8, 16, 64, 64, FAKE, FAKE + 1, None) == 1
    assert L.moe_device_status(None) == 1
    assert L.moe_forward_views(8, 64, 8, 2, 64, None) == 1


def test_route_workspace_too_small(moe):
    L = moe.lib
    need = moe.router_workspace_size(128, 16)
    assert L.moe_router_logits(FAKE, FAKE, None, 8, 128, 16, FAKE, FAKE, need - 16, None) == 3
    need = moe.route_workspace_size(1000, 16, 4)
    r = L.moe_route(FAKE, 1000, 16, 4, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, need - 4, None)
    assert r == 3
    r = L.moe_forward(FAKE, FAKE, None, FAKE, FAKE, 64, 64, 8, 2, 64, FAKE, FAKE, 1024, None)
    assert r == 3


def test_mxfp8_entry_points_reject_bad_arguments(moe):
    L = moe.lib
    assert moe.mxfp8_scales_size(300, 256) == 3 * 2 * 512          # 3 row blocks x 2 K slices
    assert moe.mxfp8_act_scales_size(1000, 8, 256) == (8 + 8) * 2 * 512
    assert L.moe_mxfp8_quantize(FAKE, 8, 192, FAKE, FAKE, None) == 2          # K % 128
    assert L.moe_mxfp8_quantize(FAKE + 8, 8, 256, FAKE, FAKE, None) == 1      # misaligned
    assert L.moe_permute_mxfp8(FAKE, FAKE, FAKE, FAKE, 8, 2, 192, 8, FAKE, FAKE, 1 << 30, None) == 2
    assert L.moe_permute_mxfp8(FAKE, FAKE, FAKE, FAKE, 8, 2, 256, 8, FAKE, FAKE, 16, None) == 3
    assert L.moe_grouped_gemm1_swiglu_mxfp8(FAKE, FAKE, 1 << 30, FAKE, 8, 16, 256, 192, FAKE, FAKE, FAKE, FAKE,
                                           1 << 30, None) == 2                # f % 128
    assert L.moe_grouped_gemm2_mxfp8(None, FAKE, 1 << 30, FAKE, 8, 16, 256, 256, FAKE, FAKE, FAKE, None) == 1
    assert L.moe_forward_mxfp8(FAKE, FAKE, None, FAKE, FAKE, FAKE, FAKE, 64, 256, 8, 2, 256, FAKE, FAKE, 16,
                               None) == 3
    v = moe.forward_mxfp8_views(8192, 4096, 8, 2, 14336)
    assert v["hq"] - v["xq_perm"] >= 8192 * 2 * 4096
    assert list(v.values()) == sorted(v.values())


def test_pipelined_host_runners_reject_bad_arguments(moe):
    import ctypes
    L = moe.lib
    one = (ctypes.c_void_p * 1)(FAKE)
    nul = (ctypes.c_void_p * 1)(None)
    n = L.moe_forward_host_pipelined_workspace_size(64, 64, 8, 2, 64)
    assert n >= L.moe_forward_workspace_size(64, 64, 8, 2, 64) + 2 * 64 * 64 * 2
    args = (FAKE, None, FAKE, FAKE, 64, 64, 8, 2, 64)
    assert L.moe_forward_host_pipelined(one, one, 0, *args, FAKE, n, None) == 1       # no batch
    assert L.moe_forward_host_pipelined(nul, one, 1, *args, FAKE, n, None) == 1       # null batch pointer
    assert L.moe_forward_host_pipelined(None, one, 1, *args, FAKE, n, None) == 1
    assert L.moe_forward_host_pipelined(one, one, 1, *args, FAKE + 16, n, None) == 1  # workspace alignment
    assert L.moe_forward_host_pipelined(one, one, 1, *args, FAKE, n - 1, None) == 3
    assert L.moe_forward_host_pipelined(one, one, 1, FAKE, None, FAKE, FAKE, 64, 64, 8, 2, 60, FAKE, n,
                                        None) == 2                                     # f % 64
    m = L.moe_forward_mxfp8_host_pipelined_workspace_size(64, 256, 8, 2, 256)
    assert m >= L.moe_forward_mxfp8_workspace_size(64, 256, 8, 2, 256) + 4 * 64 * 256 * 2
    assert L.moe_forward_mxfp8_host_pipelined_workspace_size(64, 192, 8, 2, 256) == 0
    mx = (FAKE, None, FAKE, FAKE, FAKE, FAKE, 64, 256, 8, 2, 256)
    assert L.moe_forward_mxfp8_host_pipelined(one, one, 0, *mx, FAKE, m, None) == 1
    assert L.moe_forward_mxfp8_host_pipelined(one, one, 1, *mx, FAKE, m - 1, None) == 3


def test_backward_entry_points_reject_bad_arguments(moe):
    import ctypes
    L = moe.lib
    T, d, E, K, f = 64, 128, 8, 2, 64
    nb = L.moe_backward_workspace_size(T, d, E, K, f)
    nf = L.moe_forward_workspace_size(T, d, E, K, f)
    assert nb > 0 and L.moe_backward_workspace_size(T, 96, E, K, f) == 0   # d % 64
    # layout: ordered regions, each large enough
    lay = moe._LayoutBW()
    assert L.moe_backward_views(T, d, E, K, f, ctypes.byref(lay)) == 0
    offs = [getattr(lay, n) for n, _ in moe._LayoutBW._fields_]
    assert offs == sorted(offs) and offs[-1] == nb
    TK = T * K
    assert lay.dy_perm - lay.dl_row >= TK * 4 and lay.da - lay.a >= TK * 2 * f * 2
    assert lay.rw_part - lay.WrT >= d * E * 4
    assert lay.total - lay.tmaps >= 256 * E and lay.tmaps % 128 == 0   # two 128-byte tensor maps per expert

    def bwd(*, x=FAKE, Wr=FAKE, W1=FAKE, dy=FAKE, fws=FAKE, fbytes=nf, pre=None, dx=FAKE, dWr=FAKE, ws=FAKE,
            wbytes=nb, f_=f):
        return L.moe_backward(x, Wr, None, W1, FAKE, T, d, E, K, f_, dy, fws, fbytes, pre, dx, dWr, FAKE, FAKE,
                              FAKE, ws, wbytes, None)
    assert bwd(x=None) == 1 and bwd(dy=None) == 1 and bwd(fws=None) == 1 and bwd(dx=None) == 1
    assert bwd(W1=FAKE + 8) == 1          # 16-byte alignment
    assert bwd(Wr=FAKE + 2) == 1          # 4-byte alignment
    assert bwd(pre=FAKE + 8) == 1         # saved pre-activations: 16-byte alignment
    assert bwd(ws=FAKE + 16) == 1         # workspace: 128-byte alignment (the tensor maps in it)
    assert bwd(f_=60) == 2                # f % 64
    assert bwd(fbytes=nf - 1) == 3 and bwd(wbytes=nb - 1) == 3
    # the training forward and GEMM1 with saved pre-activations
    assert L.moe_forward_train(FAKE, FAKE, None, FAKE, FAKE, T, d, E, K, f, FAKE, FAKE, nf, FAKE + 8, None) == 1
    assert L.moe_forward_train(FAKE, FAKE, None, FAKE, FAKE, T, d, E, K, f, FAKE, FAKE, nf - 1, FAKE, None) == 3
    assert L.moe_grouped_gemm1_swiglu_preact(FAKE, FAKE, E, TK, d, f, FAKE, FAKE, None, None) == 1
    assert L.moe_grouped_gemm1_swiglu_preact(FAKE, FAKE, E, TK, d, 96, FAKE, FAKE, FAKE, None) == 2


def test_no_launch_happened(moe):
    # every call above was rejected on the host
    assert moe.launch_count() == 0


def test_package_refuses_cpu_tensors(moe):
    import torch
    x = torch.zeros(4, 64, dtype=torch.bfloat16)
    Wr = torch.zeros(64, 8)
    with pytest.raises(ValueError, match="CUDA"):
        moe.router_logits(x, Wr)
