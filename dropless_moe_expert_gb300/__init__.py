"""Dropless MoE SwiGLU layer forward on one GB300 -- Python binding.

Thin ctypes binding over the C ABI in ``include/moe.h`` (library
``libmoe_gb300.so`` built in-tree by ``build.py``).  Functions carry the C
names without the ``moe_`` prefix, take torch tensors (device memory only,
any stream), check dtypes/shapes/contiguity, and pass raw pointers plus the
current CUDA stream.  Every step of the layer runs in the library's kernels;
there is no fallback: if the library is missing, importing this package
raises.
"""
from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass

import torch

from . import build as _build

__all__ = [
    "MoEError", "lib", "router_logits", "router_workspace_size", "route", "route_workspace_size", "permute",
    "grouped_mlp",
    "grouped_gemm1_swiglu", "grouped_gemm2", "unpermute", "forward", "forward_workspace_size",
    "forward_views", "forward_host", "device_status", "last_device_status", "launch_count", "MoELayer",
    "mxfp8_quantize", "mxfp8_scales_size", "mxfp8_act_scales_size", "permute_mxfp8",
    "grouped_gemm1_swiglu_mxfp8", "grouped_gemm2_mxfp8", "forward_mxfp8", "forward_mxfp8_views", "MoELayerMXFP8",
    "grouped_gemm2_combine", "grouped_gemm1_swiglu_gather", "last_device_status", "forward_fuses_permute",
]

_HERE = os.path.dirname(os.path.abspath(__file__))
_STATUS = {0: "MOE_OK", 1: "MOE_ERR_INVALID_ARG", 2: "MOE_ERR_UNSUPPORTED", 3: "MOE_ERR_WORKSPACE",
           4: "MOE_ERR_CUDA", 5: "MOE_ERR_DEVICE_TIMEOUT"}


class MoEError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        msg = lib.moe_status_string(code).decode() if _LIB is not None else _STATUS.get(code, str(code))
        super().__init__(f"{where}: {msg}")


class _Layout(ctypes.Structure):
    _fields_ = [(n, ctypes.c_size_t) for n in (
        "logits", "topk_idx", "topk_w", "counts", "offsets", "row_of", "src_tok", "route_ws",
        "router_ws", "x_perm", "h", "y_perm", "x_dev", "y_dev", "total")]


class _LayoutBW(ctypes.Structure):
    _fields_ = [(n, ctypes.c_size_t) for n in (
        "dw", "dl", "dl_row", "dy_perm", "dh", "a", "da", "dx_perm", "WrT", "rw_part", "tmaps", "total")]


class _LayoutMX(ctypes.Structure):
    _fields_ = [(n, ctypes.c_size_t) for n in (
        "logits", "topk_idx", "topk_w", "counts", "offsets", "row_of", "src_tok", "route_ws", "router_ws",
        "xq_perm", "sfa", "hq", "sfh", "y_perm", "total")]


def _load():
    path = _build.lib_path()
    if not os.path.exists(path):
        raise ImportError(
            f"{path} is missing: build the CUDA library first "
            "(python -c 'import __graft_entry__ as g; g.build()')")
    L = ctypes.CDLL(path)
    P, I, S, U64 = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t, ctypes.c_uint64
    sig = {
        "moe_status_string": (ctypes.c_char_p, [I]),
        "moe_abi_version": (I, []),
        "moe_launch_count": (U64, []),
        "moe_router_workspace_size": (S, [I, I]),
        "moe_router_logits": (I, [P, P, P, I, I, I, P, P, S, P]),
        "moe_route_workspace_size": (S, [I, I, I]),
        "moe_route": (I, [P, I, I, I, P, P, P, P, P, P, P, S, P]),
        "moe_permute": (I, [P, P, I, I, I, P, P]),
        "moe_grouped_mlp": (I, [P, P, I, I, I, I, P, P, P, P, P]),
        "moe_grouped_gemm1_swiglu": (I, [P, P, I, I, I, I, P, P, P]),
        "moe_grouped_gemm1_swiglu_preact": (I, [P, P, I, I, I, I, P, P, P, P]),
        "moe_grouped_gemm1_swiglu_gather": (I, [P, P, P, I, I, I, I, I, P, P, P]),
        "moe_grouped_gemm2": (I, [P, P, I, I, I, I, P, P, P]),
        "moe_unpermute": (I, [P, P, P, I, I, I, P, P]),
        "moe_forward_workspace_size": (S, [I, I, I, I, I]),
        "moe_forward_fuses_permute": (I, [I, I, I, I, I]),
        "moe_forward_views": (I, [I, I, I, I, I, ctypes.POINTER(_Layout)]),
        "moe_forward": (I, [P, P, P, P, P, I, I, I, I, I, P, P, S, P]),
        "moe_forward_train": (I, [P, P, P, P, P, I, I, I, I, I, P, P, S, P, P]),
        "moe_forward_host_pipelined_workspace_size": (S, [I, I, I, I, I]),
        "moe_forward_host_pipelined": (I, [P, P, I, P, P, P, P, I, I, I, I, I, P, S, P]),
        "moe_forward_mxfp8_host_pipelined_workspace_size": (S, [I, I, I, I, I]),
        "moe_forward_mxfp8_host_pipelined": (I, [P, P, I, P, P, P, P, P, P, I, I, I, I, I, P, S, P]),
        "moe_forward_host": (I, [P, P, P, P, P, I, I, I, I, I, P, P, S, P]),
        "moe_mxfp8_scales_size": (S, [I, I]),
        "moe_mxfp8_quantize": (I, [P, I, I, P, P, P]),
        "moe_mxfp8_act_scales_size": (S, [I, I, I]),
        "moe_permute_mxfp8": (I, [P, P, P, P, I, I, I, I, P, P, S, P]),
        "moe_grouped_gemm1_swiglu_mxfp8": (I, [P, P, S, P, I, I, I, I, P, P, P, P, S, P]),
        "moe_grouped_gemm2_mxfp8": (I, [P, P, S, P, I, I, I, I, P, P, P, P]),
        "moe_forward_mxfp8_workspace_size": (S, [I, I, I, I, I]),
        "moe_forward_mxfp8_views": (I, [I, I, I, I, I, ctypes.POINTER(_LayoutMX)]),
        "moe_forward_mxfp8": (I, [P, P, P, P, P, P, P, I, I, I, I, I, P, P, S, P]),
        "moe_backward_workspace_size": (S, [I, I, I, I, I]),
        "moe_backward_views": (I, [I, I, I, I, I, ctypes.POINTER(_LayoutBW)]),
        "moe_backward": (I, [P, P, P, P, P, I, I, I, I, I, P, P, S, P, P, P, P, P, P, P, S, P]),
        "moe_combine_counters_size": (S, [I, I]),
        "moe_grouped_gemm2_combine": (I, [P, P, I, I, I, I, P, P, P, P, I, I, P, P, S, P, P]),
        "moe_device_status": (I, [ctypes.POINTER(I)]),
        "moe_last_device_status": (I, [P, P]),
        "moe_check_bounded_wait": (I, [U64, P]),
    }
    for name, (res, args) in sig.items():
        fn = getattr(L, name)
        fn.restype = res
        fn.argtypes = args
    return L


_LIB = _load()
lib = _LIB


# ------------------------------------------------------------------ helpers
def _stream(stream=None) -> int:
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream


def _ptr(t) -> int | None:
    return None if t is None else t.data_ptr()


def _check(code: int, where: str):
    if code != 0:
        raise MoEError(code, where)


def _need(t, dtype, shape, name):
    if t is None:
        raise ValueError(f"{name} is required")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor (the library has no CPU path)")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return t


def _empty(shape, dtype, like):
    return torch.empty(shape, dtype=dtype, device=like.device)


# ------------------------------------------------------------------ a0
def router_workspace_size(d, E) -> int:
    return int(lib.moe_router_workspace_size(d, E))


def router_logits(x, Wr, bias=None, out=None, workspace=None, stream=None):
    """logits[T,E] fp32 = x[t,:] . Wr[:,e] + bias[e]: exact products (Wr split
    into three bf16 pieces) summed in fp32 on the tensor cores."""
    T, d = x.shape
    E = Wr.shape[1]
    _need(x, torch.bfloat16, (T, d), "x")
    _need(Wr, torch.float32, (d, E), "Wr")
    if bias is not None:
        _need(bias, torch.float32, (E,), "bias")
    out = _empty((T, E), torch.float32, x) if out is None else _need(out, torch.float32, (T, E), "logits")
    nbytes = router_workspace_size(d, E)
    if nbytes == 0:
        raise MoEError(2, "moe_router_workspace_size")
    if workspace is None:
        workspace = _empty((nbytes,), torch.uint8, x)
    _check(lib.moe_router_logits(_ptr(x), _ptr(Wr), _ptr(bias), T, d, E, _ptr(out), _ptr(workspace),
                                 workspace.numel(), _stream(stream)), "moe_router_logits")
    return out


# ------------------------------------------------------------------ a1 + a2
@dataclass
class Routing:
    topk_idx: torch.Tensor   # [T, K] int32
    topk_w: torch.Tensor     # [T, K] fp32
    counts: torch.Tensor     # [E] int32
    offsets: torch.Tensor    # [E+1] int32
    row_of: torch.Tensor     # [T, K] int32
    src_tok: torch.Tensor    # [TK] int32


def route_workspace_size(T: int, E: int, K: int) -> int:
    return int(lib.moe_route_workspace_size(T, E, K))


def route(logits, K: int, workspace=None, stream=None) -> Routing:
    T, E = logits.shape
    _need(logits, torch.float32, (T, E), "logits")
    i32 = torch.int32
    r = Routing(_empty((T, K), i32, logits), _empty((T, K), torch.float32, logits), _empty((E,), i32, logits),
                _empty((E + 1,), i32, logits), _empty((T, K), i32, logits), _empty((T * K,), i32, logits))
    nbytes = route_workspace_size(T, E, K)
    if workspace is None:
        workspace = _empty((max(nbytes, 4),), torch.uint8, logits)
    _check(lib.moe_route(_ptr(logits), T, E, K, _ptr(r.topk_idx), _ptr(r.topk_w), _ptr(r.counts),
                         _ptr(r.offsets), _ptr(r.row_of), _ptr(r.src_tok), _ptr(workspace),
                         workspace.numel() * workspace.element_size(), _stream(stream)), "moe_route")
    return r


# ------------------------------------------------------------------ a3
def permute(x, row_of, out=None, stream=None):
    """x_perm[row_of[t,k]] = x[t]."""
    T, d = x.shape
    K = row_of.shape[1]
    _need(x, torch.bfloat16, (T, d), "x")
    _need(row_of, torch.int32, (T, K), "row_of")
    out = _empty((T * K, d), torch.bfloat16, x) if out is None else _need(out, torch.bfloat16, (T * K, d), "x_perm")
    _check(lib.moe_permute(_ptr(x), _ptr(row_of), T, K, d, _ptr(out), _stream(stream)), "moe_permute")
    return out


# ------------------------------------------------------------------ a4 + a5
def _mlp_shapes(x_perm, offsets, W1=None, W2=None):
    TK, d = x_perm.shape
    E = offsets.shape[0] - 1
    f = W1.shape[1] // 2 if W1 is not None else W2.shape[2]
    return TK, d, E, f


def grouped_gemm1_swiglu(x_perm, offsets, W1, h=None, preact=None, stream=None):
    """h [TK, f]; with ``preact`` ([TK, 2f] bf16) the pre-activations are stored too."""
    TK, d, E, f = _mlp_shapes(x_perm, offsets, W1=W1)
    _need(x_perm, torch.bfloat16, (TK, d), "x_perm")
    _need(offsets, torch.int32, (E + 1,), "offsets")
    _need(W1, torch.bfloat16, (E, 2 * f, d), "W1")
    h = _empty((TK, f), torch.bfloat16, x_perm) if h is None else _need(h, torch.bfloat16, (TK, f), "h")
    if preact is None:
        _check(lib.moe_grouped_gemm1_swiglu(_ptr(x_perm), _ptr(offsets), E, TK, d, f, _ptr(W1), _ptr(h),
                                            _stream(stream)), "moe_grouped_gemm1_swiglu")
    else:
        _need(preact, torch.bfloat16, (TK, 2 * f), "preact")
        _check(lib.moe_grouped_gemm1_swiglu_preact(_ptr(x_perm), _ptr(offsets), E, TK, d, f, _ptr(W1), _ptr(h),
                                                   _ptr(preact), _stream(stream)), "moe_grouped_gemm1_swiglu_preact")
    return h


def grouped_gemm1_swiglu_gather(x, src_tok, offsets, W1, h=None, stream=None):
    """GEMM1 + SwiGLU with the permute fused into its operand load: row r of
    expert e's group is read as x[src_tok[r]]; h [TK, f] equals
    grouped_gemm1_swiglu(permute(x, row_of), offsets, W1) bit for bit."""
    T, d = x.shape
    TK = src_tok.shape[0]
    E = offsets.shape[0] - 1
    f = W1.shape[1] // 2
    _need(x, torch.bfloat16, (T, d), "x")
    _need(src_tok, torch.int32, (TK,), "src_tok")
    _need(offsets, torch.int32, (E + 1,), "offsets")
    _need(W1, torch.bfloat16, (E, 2 * f, d), "W1")
    h = _empty((TK, f), torch.bfloat16, x) if h is None else _need(h, torch.bfloat16, (TK, f), "h")
    _check(lib.moe_grouped_gemm1_swiglu_gather(_ptr(x), _ptr(src_tok), _ptr(offsets), T, E, TK, d, f, _ptr(W1),
                                               _ptr(h), _stream(stream)), "moe_grouped_gemm1_swiglu_gather")
    return h


def grouped_gemm2(h, offsets, W2, y_perm=None, stream=None):
    TK, f = h.shape
    E = offsets.shape[0] - 1
    d = W2.shape[1]
    _need(h, torch.bfloat16, (TK, f), "h")
    _need(offsets, torch.int32, (E + 1,), "offsets")
    _need(W2, torch.bfloat16, (E, d, f), "W2")
    y_perm = _empty((TK, d), torch.bfloat16, h) if y_perm is None else _need(y_perm, torch.bfloat16, (TK, d), "y_perm")
    _check(lib.moe_grouped_gemm2(_ptr(h), _ptr(offsets), E, TK, d, f, _ptr(W2), _ptr(y_perm), _stream(stream)),
           "moe_grouped_gemm2")
    return y_perm


def grouped_mlp(x_perm, offsets, W1, W2, h=None, y_perm=None, stream=None):
    TK, d, E, f = _mlp_shapes(x_perm, offsets, W1=W1)
    _need(x_perm, torch.bfloat16, (TK, d), "x_perm")
    _need(offsets, torch.int32, (E + 1,), "offsets")
    _need(W1, torch.bfloat16, (E, 2 * f, d), "W1")
    _need(W2, torch.bfloat16, (E, d, f), "W2")
    h = _empty((TK, f), torch.bfloat16, x_perm) if h is None else _need(h, torch.bfloat16, (TK, f), "h")
    y_perm = _empty((TK, d), torch.bfloat16, x_perm) if y_perm is None else _need(y_perm, torch.bfloat16, (TK, d), "y_perm")
    _check(lib.moe_grouped_mlp(_ptr(x_perm), _ptr(offsets), E, TK, d, f, _ptr(W1), _ptr(W2), _ptr(h), _ptr(y_perm),
                               _stream(stream)), "moe_grouped_mlp")
    return h, y_perm


# ------------------------------------------------------------------ a6
def unpermute(y_perm, row_of, topk_w, out=None, stream=None):
    """y[t] = bf16(sum_k topk_w[t,k] * y_perm[row_of[t,k]]), fp32 accumulate."""
    T, K = row_of.shape
    d = y_perm.shape[1]
    _need(y_perm, torch.bfloat16, (T * K, d), "y_perm")
    _need(row_of, torch.int32, (T, K), "row_of")
    _need(topk_w, torch.float32, (T, K), "topk_w")
    out = _empty((T, d), torch.bfloat16, y_perm) if out is None else _need(out, torch.bfloat16, (T, d), "y")
    _check(lib.moe_unpermute(_ptr(y_perm), _ptr(row_of), _ptr(topk_w), T, K, d, _ptr(out), _stream(stream)),
           "moe_unpermute")
    return out


def grouped_gemm2_combine(h, r: "Routing", W2, out=None, y_perm=None, counters=None, stream=None):
    """GEMM2 with the combine fused into its epilogue: y [T, d] bf16, equal
    bit for bit to unpermute(grouped_gemm2(h)).  y_perm and counters are
    scratch (allocated when not given)."""
    TK, f = h.shape
    E, d, _ = W2.shape
    T, K = r.row_of.shape
    _need(h, torch.bfloat16, (TK, f), "h")
    _need(W2, torch.bfloat16, (E, d, f), "W2")
    if y_perm is None:
        y_perm = _empty((TK, d), torch.bfloat16, h)
    if counters is None:
        counters = _empty((max(1, int(lib.moe_combine_counters_size(T, d)) // 4),), torch.int32, h)
    out = _empty((T, d), torch.bfloat16, h) if out is None else _need(out, torch.bfloat16, (T, d), "y")
    _check(lib.moe_grouped_gemm2_combine(_ptr(h), _ptr(r.offsets), E, TK, d, f, _ptr(W2), _ptr(r.src_tok),
                                         _ptr(r.row_of), _ptr(r.topk_w), T, K, _ptr(y_perm), _ptr(counters),
                                         counters.numel() * 4, _ptr(out), _stream(stream)),
           "moe_grouped_gemm2_combine")
    return out


# ------------------------------------------------------------------ whole layer
def forward_workspace_size(T, d, E, K, f) -> int:
    return int(lib.moe_forward_workspace_size(T, d, E, K, f))


def forward_views(T, d, E, K, f) -> dict:
    lay = _Layout()
    _check(lib.moe_forward_views(T, d, E, K, f, ctypes.byref(lay)), "moe_forward_views")
    return {n: getattr(lay, n) for n, _ in _Layout._fields_}


def _weights_check(x, Wr, bias, W1, W2, K):
    T, d = x.shape
    E = Wr.shape[1]
    f = W1.shape[1] // 2
    _need(Wr, torch.float32, (d, E), "Wr")
    if bias is not None:
        _need(bias, torch.float32, (E,), "bias")
    _need(W1, torch.bfloat16, (E, 2 * f, d), "W1")
    _need(W2, torch.bfloat16, (E, d, f), "W2")
    return T, d, E, f


def forward(x, Wr, bias, W1, W2, K: int, out=None, workspace=None, stream=None, preact=None):
    """The whole layer in one C-ABI call (9 kernel launches, no host sync).
    With ``preact`` ([T*K, 2f] bf16) GEMM1 also stores the pre-activations
    for a backward pass (moe_forward_train)."""
    T, d, E, f = _weights_check(x, Wr, bias, W1, W2, K)
    _need(x, torch.bfloat16, (T, d), "x")
    nbytes = forward_workspace_size(T, d, E, K, f)
    if nbytes == 0:
        raise MoEError(2, "moe_forward_workspace_size")
    if workspace is None:
        workspace = _empty((nbytes,), torch.uint8, x)
    out = _empty((T, d), torch.bfloat16, x) if out is None else _need(out, torch.bfloat16, (T, d), "y")
    if preact is None:
        _check(lib.moe_forward(_ptr(x), _ptr(Wr), _ptr(bias), _ptr(W1), _ptr(W2), T, d, E, K, f, _ptr(out),
                               _ptr(workspace), workspace.numel(), _stream(stream)), "moe_forward")
    else:
        _need(preact, torch.bfloat16, (T * K, 2 * f), "preact")
        _check(lib.moe_forward_train(_ptr(x), _ptr(Wr), _ptr(bias), _ptr(W1), _ptr(W2), T, d, E, K, f, _ptr(out),
                                     _ptr(workspace), workspace.numel(), _ptr(preact), _stream(stream)),
               "moe_forward_train")
    return out


def forward_host(x_host, Wr, bias, W1, W2, K: int, y_host=None, workspace=None, stream=None):
    """The layer with activations in host memory (pinned for async copies):
    x_host [T,d] bf16 (CPU) -> y_host [T,d] bf16 (CPU).  Copies happen on the
    stream inside the C call; synchronize the stream before reading y_host."""
    if x_host.is_cuda or x_host.dtype != torch.bfloat16 or not x_host.is_contiguous():
        raise ValueError("x_host must be a contiguous CPU bf16 tensor")
    T, d = x_host.shape
    _, _, E, f = _weights_check(x_host, Wr, bias, W1, W2, K)
    nbytes = forward_workspace_size(T, d, E, K, f)
    if workspace is None:
        workspace = torch.empty((nbytes,), dtype=torch.uint8, device=W1.device)
    if y_host is None:
        y_host = torch.empty((T, d), dtype=torch.bfloat16, pin_memory=x_host.is_pinned())
    _check(lib.moe_forward_host(_ptr(x_host), _ptr(Wr), _ptr(bias), _ptr(W1), _ptr(W2), T, d, E, K, f,
                                _ptr(y_host), _ptr(workspace), workspace.numel(), _stream(stream)),
           "moe_forward_host")
    return y_host


def _host_batches(x_hosts, y_hosts, T, d):
    """Pointer arrays of the host batches (checked: contiguous CPU bf16 [T, d])."""
    if len(x_hosts) != len(y_hosts) or not x_hosts:
        raise ValueError("x_hosts and y_hosts must be non-empty and of equal length")
    for t in list(x_hosts) + list(y_hosts):
        if t.is_cuda or t.dtype != torch.bfloat16 or not t.is_contiguous() or tuple(t.shape) != (T, d):
            raise ValueError("host batches must be contiguous CPU bf16 [T, d] tensors")
    xp = (ctypes.c_void_p * len(x_hosts))(*[t.data_ptr() for t in x_hosts])
    yp = (ctypes.c_void_p * len(y_hosts))(*[t.data_ptr() for t in y_hosts])
    return xp, yp


def forward_host_pipelined(x_hosts, y_hosts, Wr, bias, W1, W2, K: int, workspace=None, stream=None):
    """The layer over a list of host batches (pinned [T,d] bf16 CPU tensors;
    entries may repeat), y_hosts[i] written from x_hosts[i]; host<->device
    copies overlap the compute of neighbouring batches.  Synchronize the
    stream before reading y_hosts."""
    T, d = x_hosts[0].shape
    _, _, E, f = _weights_check(x_hosts[0], Wr, bias, W1, W2, K)
    xp, yp = _host_batches(x_hosts, y_hosts, T, d)
    nbytes = int(lib.moe_forward_host_pipelined_workspace_size(T, d, E, K, f))
    if nbytes == 0:
        raise MoEError(2, "moe_forward_host_pipelined_workspace_size")
    if workspace is None:
        workspace = torch.empty((nbytes,), dtype=torch.uint8, device=W1.device)
    _check(lib.moe_forward_host_pipelined(xp, yp, len(x_hosts), _ptr(Wr), _ptr(bias), _ptr(W1), _ptr(W2), T, d, E,
                                          K, f, _ptr(workspace), workspace.numel(), _stream(stream)),
           "moe_forward_host_pipelined")
    return y_hosts


def forward_mxfp8_host_pipelined(x_hosts, y_hosts, Wr, bias, W1q, W1s, W2q, W2s, K: int, workspace=None,
                                 stream=None):
    """forward_host_pipelined with the MXFP8 expert matmuls (weights quantised)."""
    T, d = x_hosts[0].shape
    E, two_f, _ = W1q.shape
    f = two_f // 2
    xp, yp = _host_batches(x_hosts, y_hosts, T, d)
    nbytes = int(lib.moe_forward_mxfp8_host_pipelined_workspace_size(T, d, E, K, f))
    if nbytes == 0:
        raise MoEError(2, "moe_forward_mxfp8_host_pipelined_workspace_size")
    if workspace is None:
        workspace = torch.empty((nbytes,), dtype=torch.uint8, device=W1q.device)
    _check(lib.moe_forward_mxfp8_host_pipelined(xp, yp, len(x_hosts), _ptr(Wr), _ptr(bias), _ptr(W1q), _ptr(W1s),
                                                _ptr(W2q), _ptr(W2s), T, d, E, K, f, _ptr(workspace),
                                                workspace.numel(), _stream(stream)),
           "moe_forward_mxfp8_host_pipelined")
    return y_hosts


def device_status() -> int:
    v = ctypes.c_int(0)
    _check(lib.moe_device_status(ctypes.byref(v)), "moe_device_status")
    return v.value


def last_device_status(out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """Queues a read-and-clear of the device status word on the stream into
    ``out`` (one int32 on the device, allocated when None), without
    synchronizing: capture-safe.  Read ``out`` after the stream has run."""
    if out is None:
        out = torch.empty((1,), dtype=torch.int32, device="cuda")
    if out.dtype != torch.int32 or not out.is_cuda or out.numel() < 1:
        raise ValueError("out must be an int32 CUDA tensor with at least one element")
    _check(lib.moe_last_device_status(out.data_ptr(), _stream(stream)), "moe_last_device_status")
    return out


def check_bounded_wait(limit_ns: int = 2_000_000, stream=None) -> None:
    """Launches a kernel whose only wait never completes; it times out after
    limit_ns and records MOE_ERR_DEVICE_TIMEOUT (see device_status())."""
    _check(lib.moe_check_bounded_wait(limit_ns, _stream(stream)), "moe_check_bounded_wait")


def forward_fuses_permute(T: int, d: int, E: int, K: int, f: int) -> bool:
    """True when moe_forward fuses the permute into GEMM1 for these sizes
    (then its workspace region x_perm is left unwritten)."""
    return bool(lib.moe_forward_fuses_permute(T, d, E, K, f))


def launch_count() -> int:
    return int(lib.moe_launch_count())


class MoELayer:
    """Holds one layer's weights and a persistent workspace; ``__call__(x)``
    runs the forward with one C call.  Intermediates can be read back with
    ``views()`` after a call (they live in the workspace)."""

    def __init__(self, Wr, bias, W1, W2, K: int, T_max: int):
        self.Wr, self.bias, self.W1, self.W2, self.K = Wr, bias, W1, W2, K
        self.d = W1.shape[2]
        self.E = Wr.shape[1]
        self.f = W1.shape[1] // 2
        self.T_max = T_max
        n = forward_workspace_size(T_max, self.d, self.E, K, self.f)
        if n == 0:
            raise MoEError(2, "moe_forward_workspace_size")
        self.workspace = torch.empty((n,), dtype=torch.uint8, device=W1.device)
        self._preact_buf = None
        self.preact = None

    def __call__(self, x, out=None, stream=None, save_preact=False):
        """y = layer(x).  ``save_preact``: also keep GEMM1's pre-activations
        ([T*K, 2f] bf16, held by the layer) for the next backward(), which
        then skips recomputing them."""
        if x.shape[0] > self.T_max:
            raise ValueError("more tokens than the workspace was sized for")
        pre = None
        if save_preact:
            n = x.shape[0] * self.K * 2 * self.f
            if self._preact_buf is None or self._preact_buf.numel() < n:
                self._preact_buf = torch.empty((self.T_max * self.K * 2 * self.f,), dtype=torch.bfloat16,
                                               device=x.device)
            pre = self._preact_buf[:n].view(x.shape[0] * self.K, 2 * self.f)
        self.preact = pre
        # moe_forward may fuse the permute into GEMM1 and leave x_perm
        # unwritten; the training forward (save_preact) always writes it
        self._x_perm_written = save_preact or not forward_fuses_permute(x.shape[0], self.d, self.E, self.K, self.f)
        return forward(x, self.Wr, self.bias, self.W1, self.W2, self.K, out=out, workspace=self.workspace,
                       stream=stream, preact=pre)

    def backward(self, x, dy, grads=None, workspace=None, stream=None):
        """Gradients of sum(dy * y) for the last call (same x): dict of dx
        [T,d] bf16 and dWr, dbias, dW1, dW2 (fp32, shaped like the weights).
        Uses the pre-activations the last call saved, if it did."""
        T, d = x.shape
        pre = self.preact if self.preact is not None and self.preact.shape[0] == T * self.K else None
        _need(x, torch.bfloat16, (T, d), "x")
        _need(dy, torch.bfloat16, (T, d), "dy")
        n = int(lib.moe_backward_workspace_size(T, d, self.E, self.K, self.f))
        if n == 0:
            raise MoEError(2, "moe_backward_workspace_size")
        if workspace is None:
            workspace = torch.empty((n,), dtype=torch.uint8, device=x.device)
        if not getattr(self, "_x_perm_written", True):
            # the last forward fused the permute: write the grouped rows the
            # backward reads (one permute kernel)
            v = self.views(T)
            permute(x, v["row_of"], out=v["x_perm"], stream=stream)
            self._x_perm_written = True
        if grads is None:
            f32 = dict(dtype=torch.float32, device=x.device)
            grads = dict(dx=torch.empty((T, d), dtype=torch.bfloat16, device=x.device),
                         dWr=torch.empty(self.Wr.shape, **f32), dbias=torch.empty((self.E,), **f32),
                         dW1=torch.empty(self.W1.shape, **f32), dW2=torch.empty(self.W2.shape, **f32))
        _check(lib.moe_backward(_ptr(x), _ptr(self.Wr), _ptr(self.bias), _ptr(self.W1), _ptr(self.W2), T, d, self.E,
                                self.K, self.f, _ptr(dy), _ptr(self.workspace), self.workspace.numel(),
                                _ptr(pre), _ptr(grads["dx"]), _ptr(grads["dWr"]), _ptr(grads["dbias"]), _ptr(grads["dW1"]),
                                _ptr(grads["dW2"]), _ptr(workspace), workspace.numel(), _stream(stream)),
               "moe_backward")
        self.bw_workspace = workspace
        return grads

    def backward_views(self, T: int) -> dict:
        """Typed views of the backward's intermediates (after backward())."""
        lay = _LayoutBW()
        _check(lib.moe_backward_views(T, self.d, self.E, self.K, self.f, ctypes.byref(lay)), "moe_backward_views")
        ws = self.bw_workspace
        TK = T * self.K

        def v(name, n, dtype, shape):
            off = getattr(lay, name)
            return ws[off:off + n * torch.tensor([], dtype=dtype).element_size()].view(dtype).view(shape)

        return dict(dw=v("dw", TK, torch.float32, (T, self.K)), dl=v("dl", TK, torch.float32, (T, self.K)),
                    dy_perm=v("dy_perm", TK * self.d, torch.bfloat16, (TK, self.d)),
                    dh=v("dh", TK * self.f, torch.bfloat16, (TK, self.f)),
                    a=v("a", TK * 2 * self.f, torch.bfloat16, (TK, 2 * self.f)),
                    da=v("da", TK * 2 * self.f, torch.bfloat16, (TK, 2 * self.f)),
                    dx_perm=v("dx_perm", TK * self.d, torch.bfloat16, (TK, self.d)))

    def views(self, T: int) -> dict:
        """Typed tensor views of the intermediates of the last call with T tokens."""
        lay = forward_views(T, self.d, self.E, self.K, self.f)
        ws = self.workspace
        K, E, d, f = self.K, self.E, self.d, self.f
        TK = T * K

        def v(name, n, dtype, shape):
            return ws[lay[name]:lay[name] + n * torch.tensor([], dtype=dtype).element_size()].view(dtype).view(shape)

        return dict(
            logits=v("logits", T * E, torch.float32, (T, E)),
            topk_idx=v("topk_idx", TK, torch.int32, (T, K)),
            topk_w=v("topk_w", TK, torch.float32, (T, K)),
            counts=v("counts", E, torch.int32, (E,)),
            offsets=v("offsets", E + 1, torch.int32, (E + 1,)),
            row_of=v("row_of", TK, torch.int32, (T, K)),
            src_tok=v("src_tok", TK, torch.int32, (TK,)),
            x_perm=v("x_perm", TK * d, torch.bfloat16, (TK, d)),
            h=v("h", TK * f, torch.bfloat16, (TK, f)),
            y_perm=v("y_perm", TK * d, torch.bfloat16, (TK, d)),
        )


# ------------------------------------------------------------------ MXFP8 path
def mxfp8_scales_size(rows: int, K: int) -> int:
    return int(lib.moe_mxfp8_scales_size(rows, K))


def mxfp8_act_scales_size(TK: int, E: int, K: int) -> int:
    return int(lib.moe_mxfp8_act_scales_size(TK, E, K))


def mxfp8_quantize(src, stream=None):
    """bf16 [..., K] (K a multiple of 128) -> (codes uint8 [..., K], scale
    atoms uint8 [moe_mxfp8_scales_size(rows, K)]), rows = src.numel() / K."""
    if not src.is_cuda or src.dtype != torch.bfloat16 or not src.is_contiguous():
        raise ValueError("src must be a contiguous CUDA bf16 tensor")
    K = src.shape[-1]
    rows = src.numel() // K
    n = mxfp8_scales_size(rows, K)
    if n == 0:
        raise MoEError(2, "moe_mxfp8_scales_size")
    codes = torch.empty(src.shape, dtype=torch.uint8, device=src.device)
    scales = torch.empty((n,), dtype=torch.uint8, device=src.device)
    _check(lib.moe_mxfp8_quantize(_ptr(src), rows, K, _ptr(codes), _ptr(scales), _stream(stream)),
           "moe_mxfp8_quantize")
    return codes, scales


def permute_mxfp8(x, r: "Routing", stream=None):
    """(xq_perm uint8 [TK, d], sfa scale atoms) of the routed tokens."""
    T, d = x.shape
    K = r.topk_idx.shape[1]
    E = r.counts.shape[0]
    _need(x, torch.bfloat16, (T, d), "x")
    n = mxfp8_act_scales_size(T * K, E, d)
    if n == 0:
        raise MoEError(2, "moe_mxfp8_act_scales_size")
    xq = torch.empty((T * K, d), dtype=torch.uint8, device=x.device)
    sfa = torch.empty((n,), dtype=torch.uint8, device=x.device)
    _check(lib.moe_permute_mxfp8(_ptr(x), _ptr(r.topk_idx), _ptr(r.row_of), _ptr(r.offsets), T, K, d, E, _ptr(xq),
                                 _ptr(sfa), sfa.numel(), _stream(stream)), "moe_permute_mxfp8")
    return xq, sfa


def grouped_gemm1_swiglu_mxfp8(xq, sfa, offsets, W1q, W1s, stream=None):
    """(hq uint8 [TK, f], sfh scale atoms)."""
    TK, d = xq.shape
    E, two_f, _ = W1q.shape
    f = two_f // 2
    n = mxfp8_act_scales_size(TK, E, f)
    hq = torch.empty((TK, f), dtype=torch.uint8, device=xq.device)
    sfh = torch.empty((n,), dtype=torch.uint8, device=xq.device)
    _check(lib.moe_grouped_gemm1_swiglu_mxfp8(_ptr(xq), _ptr(sfa), sfa.numel(), _ptr(offsets), E, TK, d, f,
                                              _ptr(W1q), _ptr(W1s), _ptr(hq), _ptr(sfh), sfh.numel(),
                                              _stream(stream)), "moe_grouped_gemm1_swiglu_mxfp8")
    return hq, sfh


def grouped_gemm2_mxfp8(hq, sfh, offsets, W2q, W2s, out=None, stream=None):
    """y_perm bf16 [TK, d]."""
    TK, f = hq.shape
    E, d, _ = W2q.shape
    out = _empty((TK, d), torch.bfloat16, hq) if out is None else _need(out, torch.bfloat16, (TK, d), "y_perm")
    _check(lib.moe_grouped_gemm2_mxfp8(_ptr(hq), _ptr(sfh), sfh.numel(), _ptr(offsets), E, TK, d, f, _ptr(W2q),
                                       _ptr(W2s), _ptr(out), _stream(stream)), "moe_grouped_gemm2_mxfp8")
    return out


def forward_mxfp8_views(T, d, E, K, f) -> dict:
    lay = _LayoutMX()
    _check(lib.moe_forward_mxfp8_views(T, d, E, K, f, ctypes.byref(lay)), "moe_forward_mxfp8_views")
    return {n: getattr(lay, n) for n, _ in _LayoutMX._fields_}


def forward_mxfp8(x, Wr, bias, W1q, W1s, W2q, W2s, K: int, out=None, workspace=None, stream=None):
    """The whole layer with MXFP8 expert matmuls in one C-ABI call."""
    T, d = x.shape
    E, two_f, _ = W1q.shape
    f = two_f // 2
    _need(x, torch.bfloat16, (T, d), "x")
    _need(Wr, torch.float32, (d, E), "Wr")
    if bias is not None:
        _need(bias, torch.float32, (E,), "bias")
    _need(W1q, torch.uint8, (E, 2 * f, d), "W1q")
    _need(W2q, torch.uint8, (E, d, f), "W2q")
    nbytes = int(lib.moe_forward_mxfp8_workspace_size(T, d, E, K, f))
    if nbytes == 0:
        raise MoEError(2, "moe_forward_mxfp8_workspace_size")
    if workspace is None:
        workspace = _empty((nbytes,), torch.uint8, x)
    out = _empty((T, d), torch.bfloat16, x) if out is None else _need(out, torch.bfloat16, (T, d), "y")
    _check(lib.moe_forward_mxfp8(_ptr(x), _ptr(Wr), _ptr(bias), _ptr(W1q), _ptr(W1s), _ptr(W2q), _ptr(W2s), T, d,
                                 E, K, f, _ptr(out), _ptr(workspace), workspace.numel(), _stream(stream)),
           "moe_forward_mxfp8")
    return out


class MoELayerMXFP8:
    """A layer whose expert weights are quantised to MXFP8 once at
    construction; ``__call__(x)`` runs the MXFP8 forward with one C call."""

    def __init__(self, Wr, bias, W1, W2, K: int, T_max: int):
        self.Wr, self.bias, self.K = Wr, bias, K
        self.E, two_f, self.d = W1.shape
        self.f = two_f // 2
        self.W1q, self.W1s = mxfp8_quantize(W1)
        self.W2q, self.W2s = mxfp8_quantize(W2)
        self.T_max = T_max
        n = int(lib.moe_forward_mxfp8_workspace_size(T_max, self.d, self.E, K, self.f))
        if n == 0:
            raise MoEError(2, "moe_forward_mxfp8_workspace_size")
        self.workspace = torch.empty((n,), dtype=torch.uint8, device=W1.device)

    def __call__(self, x, out=None, stream=None):
        if x.shape[0] > self.T_max:
            raise ValueError("more tokens than the workspace was sized for")
        return forward_mxfp8(x, self.Wr, self.bias, self.W1q, self.W1s, self.W2q, self.W2s, self.K, out=out,
                             workspace=self.workspace, stream=stream)

    def views(self, T: int) -> dict:
        """Typed views of the intermediates of the last call with T tokens."""
        lay = forward_mxfp8_views(T, self.d, self.E, self.K, self.f)
        ws = self.workspace
        K, E, d, f = self.K, self.E, self.d, self.f
        TK = T * K

        def v(name, n, dtype, shape):
            return ws[lay[name]:lay[name] + n * torch.tensor([], dtype=dtype).element_size()].view(dtype).view(shape)

        return dict(
            logits=v("logits", T * E, torch.float32, (T, E)),
            topk_idx=v("topk_idx", TK, torch.int32, (T, K)),
            topk_w=v("topk_w", TK, torch.float32, (T, K)),
            counts=v("counts", E, torch.int32, (E,)),
            offsets=v("offsets", E + 1, torch.int32, (E + 1,)),
            row_of=v("row_of", TK, torch.int32, (T, K)),
            src_tok=v("src_tok", TK, torch.int32, (TK,)),
            xq_perm=v("xq_perm", TK * d, torch.uint8, (TK, d)),
            sfa=ws[lay["sfa"]:lay["hq"]],
            hq=v("hq", TK * f, torch.uint8, (TK, f)),
            sfh=ws[lay["sfh"]:lay["y_perm"]],
            y_perm=v("y_perm", TK * d, torch.bfloat16, (TK, d)),
        )
