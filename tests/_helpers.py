"""Shared helpers of the GPU parity tests: run the CUDA layer through the C
ABI and compare it with the oracle.

Tolerances (floating point): logits bit-exact (both sides follow the same
fp32 FMA chain); gate weights |dw| <= 1e-6 (fp32 exp and divide against
fp64); layer output y and y_perm: relative L2 <= 1e-2 and max |dy| <= 5e-2 x
RMS of the oracle's values.  h = bf16(silu(g) * u) is heavy-tailed (products
of two Gaussians), so a bound relative to its RMS would be set by a few
outliers; its error is instead bounded per element by its own rounding:
fp32 accumulation and silu are exact to ~1e-6 relative and the bf16 store
adds at most 2^-9 relative, so |dh| <= 2^-8 |h_ref| + 1e-3 RMS(h_ref) (twice
the rounding bound plus a small absolute floor), besides relative L2 <= 1e-2.  Integer outputs (indices, counts, offsets, dispatch
order, the permuted rows) are bit-exact.
"""
import numpy as np
import torch

import dropless_moe_expert_gb300 as moe
import oracle

W_TOL = 1e-6
REL_L2 = 1e-2
MAX_ABS_RMS = 5e-2


def rel_l2(a, b):
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    nb = np.linalg.norm(b)
    return np.linalg.norm(a - b) / (nb if nb > 0 else 1.0)


def check_output(y_gpu, y_ref, what="y"):
    y_gpu = np.asarray(y_gpu, np.float64)
    y_ref = np.asarray(y_ref, np.float64)
    assert np.all(np.isfinite(y_gpu)), f"{what}: non-finite values (unwritten rows?)"
    r = rel_l2(y_gpu, y_ref)
    rms = np.sqrt(np.mean(y_ref ** 2))
    mx = np.max(np.abs(y_gpu - y_ref)) if y_ref.size else 0.0
    assert r <= REL_L2, f"{what}: relative L2 {r:.3e} > {REL_L2}"
    assert mx <= MAX_ABS_RMS * rms, f"{what}: max abs {mx:.3e} > {MAX_ABS_RMS} x RMS {rms:.3e}"
    return r, mx / rms if rms > 0 else 0.0


def check_rounded(h_gpu, h_ref, what="h"):
    """Per-element bound for a value computed in fp32 and stored as bf16."""
    h_gpu = np.asarray(h_gpu, np.float64)
    h_ref = np.asarray(h_ref, np.float64)
    assert np.all(np.isfinite(h_gpu)), f"{what}: non-finite values (unwritten rows?)"
    r = rel_l2(h_gpu, h_ref)
    assert r <= REL_L2, f"{what}: relative L2 {r:.3e} > {REL_L2}"
    rms = np.sqrt(np.mean(h_ref ** 2))
    bound = 2.0 ** -8 * np.abs(h_ref) + 1e-3 * rms
    excess = np.abs(h_gpu - h_ref) - bound
    assert np.all(excess <= 0), f"{what}: {np.sum(excess > 0)} elements beyond the bf16 rounding bound"
    return r


def run_layer(x, w, K, fill_nan=True):
    """Runs the whole layer with moe.MoELayer on the tensors' device; the
    workspace is filled with 0xFF bytes first (NaN in bf16 and fp32, -1 in
    int32) so that any row a kernel fails to write shows up."""
    T = x.shape[0]
    layer = moe.MoELayer(w.Wr, w.bias, w.W1, w.W2, K, T)
    if fill_nan:
        layer.workspace.fill_(0xFF)
    y = torch.full_like(x, float("nan"))
    layer(x, out=y)
    torch.cuda.synchronize()
    assert moe.device_status() == 0
    return y, layer.views(T), layer


def to_np(t):
    if t.dtype == torch.bfloat16:
        return t.float().cpu().numpy()
    return t.cpu().numpy()


def oracle_inputs(x, w):
    return (to_np(x), to_np(w.Wr), to_np(w.bias), to_np(w.W1), to_np(w.W2))


def compare_small(x, w, K):
    """Full comparison of every intermediate on a case the oracle runs whole."""
    y, v, _ = run_layer(x, w, K)
    xs, Wr, bias, W1, W2 = oracle_inputs(x, w)
    ref = oracle.forward(xs, Wr, bias, W1, W2, K)
    L = to_np(v["logits"])
    assert np.array_equal(L.view(np.uint32), ref["logits"].view(np.uint32)), "logits not bit-exact"
    assert np.array_equal(to_np(v["topk_idx"]), ref["idx"]), "topk_idx"
    assert np.max(np.abs(to_np(v["topk_w"]) - ref["w"])) <= W_TOL, "topk_w"
    assert np.array_equal(to_np(v["counts"]), ref["counts"]), "counts"
    assert np.array_equal(to_np(v["offsets"]), ref["offsets"]), "offsets"
    assert np.array_equal(to_np(v["row_of"]), ref["row_of"]), "row_of"
    assert np.array_equal(to_np(v["src_tok"]), ref["src_tok"]), "src_tok"
    xp = v["x_perm"].view(torch.int16).cpu().numpy()
    assert np.array_equal(xp, x.view(torch.int16).cpu().numpy()[ref["src_tok"]]), "x_perm"
    check_rounded(to_np(v["h"]), ref["h"], "h")
    check_output(to_np(v["y_perm"]), ref["y_perm"], "y_perm")
    return check_output(to_np(y), ref["y"], "y")
