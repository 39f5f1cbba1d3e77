"""Shared helpers of the GPU parity tests: run the CUDA layer through the C
ABI and compare it with the oracle.

Router logits: the GPU sums exact products in fp32 in the tensor core's
order, the oracle in index order; both are fp32 roundings of the same dot
product.  The GPU's are checked elementwise against fp64:
|dL| <= LOGIT_TOL x (sum_i |x_i Wr_ie| + |bias_e|).  The oracle's own fp32
logits obey the same bound.

Routing ("bit-exact given identical fp32 logits"): the GPU route kernel fed
with the oracle's fp32 logits must reproduce the oracle's routing bit for
bit (tests that call moe.route directly).  Through the whole layer, each
side routes on its own fp32 logits: every token whose top-K selection and
order are decided by fp64 margins wider than twice the logits' error bound
must be routed identically; a token inside that band has two correct
answers, and the GPU's must be a valid one (its experts rank as selected
within the bound).  Outputs are then compared for the tokens both sides
routed identically (normally all of them).

Other tolerances: gate weights |dw| <= 1e-6 from identical logits (fp32 exp
and divide against fp64), plus half the logits' error bound through the
layer; layer output y and y_perm: relative L2 <= 1e-2 and max |dy| <= 5e-2 x
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

import oracle

W_TOL = 1e-6
LOGIT_TOL = 1e-5
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


def logit_scale(x, Wr, bias):
    """sum_i |x_i Wr_ie| + |bias_e| in fp64: the scale of the logits' error bound."""
    sc = np.abs(np.asarray(x, np.float64)) @ np.abs(np.asarray(Wr, np.float64))
    if bias is not None:
        sc = sc + np.abs(np.asarray(bias, np.float64))[None, :]
    return sc


def check_logits(L_gpu, x, Wr, bias):
    """|L_gpu - L_fp64| <= LOGIT_TOL x scale, elementwise.  Returns the worst
    ratio, the scale and the fp64 logits."""
    L_gpu = np.asarray(L_gpu, np.float64)
    assert np.all(np.isfinite(L_gpu)), "logits: non-finite values"
    L64 = oracle.router_logits_fp64(x, Wr, bias)
    scale = logit_scale(x, Wr, bias)
    ratio = np.abs(L_gpu - L64) / np.maximum(scale, 1e-30)
    worst = float(ratio.max()) if ratio.size else 0.0
    assert worst <= LOGIT_TOL, f"logits: error {worst:.3e} x scale > {LOGIT_TOL}"
    return worst, scale, L64


def decided_tokens(L64, scale, K):
    """Tokens whose top-K selection and order are the same for every pair of
    logit vectors within LOGIT_TOL x scale of L64: each gap between
    consecutive ranks 0..K exceeds twice the band on both sides."""
    E = L64.shape[1]
    m = min(K + 1, E)
    order = np.argsort(-L64, axis=1, kind="stable")[:, :m]
    Ls = np.take_along_axis(L64, order, 1)
    band = 2 * LOGIT_TOL * np.take_along_axis(scale, order, 1)
    if m < 2:
        return np.ones(L64.shape[0], bool)
    return np.all(Ls[:, :-1] - Ls[:, 1:] > band[:, :-1] + band[:, 1:], axis=1)


def check_routing(idx_gpu, idx_ref, L64, scale, K):
    """The layer's routing against the oracle's (each from its own fp32
    logits).  Returns the mask of tokens routed identically."""
    idx_gpu = np.asarray(idx_gpu)
    T, E = L64.shape
    same = np.all(idx_gpu == idx_ref, axis=1)
    dec = decided_tokens(L64, scale, K)
    bad = ~same & dec
    assert not bad.any(), f"{int(bad.sum())} tokens with decided rankings routed differently"
    band = 2 * LOGIT_TOL * scale
    for t in np.nonzero(~same)[0]:
        g = idx_gpu[t]
        assert len(set(g.tolist())) == K and g.min() >= 0 and g.max() < E, f"token {t}: invalid experts"
        lo, hi = L64[t] - band[t], L64[t] + band[t]
        assert np.all(hi[g[:-1]] >= lo[g[1:]]), f"token {t}: slots out of order beyond the bound"
        rest = np.setdiff1d(np.arange(E), g)
        if rest.size:
            assert hi[g].min() >= lo[rest].max(), f"token {t}: an unselected expert ranks above the bound"
    return same


def check_dispatch_valid(v, T, K, E):
    """Properties of the GPU's counts, offsets and dispatch order given its
    own top-K (used when some near-tied token was routed differently)."""
    idx = to_np(v["topk_idx"])
    counts, offsets = to_np(v["counts"]), to_np(v["offsets"])
    row_of, src_tok = to_np(v["row_of"]), to_np(v["src_tok"])
    assert np.array_equal(counts, np.bincount(idx.ravel(), minlength=E))
    assert offsets[0] == 0 and np.array_equal(np.diff(offsets), counts)
    assert np.array_equal(np.sort(row_of.ravel()), np.arange(T * K))
    tok = np.repeat(np.arange(T), K)
    assert np.array_equal(src_tok[row_of.ravel()], tok)
    ex = idx.ravel()
    r = row_of.ravel()
    assert np.all((offsets[ex] <= r) & (r < offsets[ex + 1]))
    for e in range(E):
        assert np.all(np.diff(src_tok[offsets[e]:offsets[e + 1]]) > 0)


def weight_tol(scale, idx):
    """|dw| bound through the layer: fp32 softmax error plus half the spread
    of the two sides' selected logits (each within LOGIT_TOL x scale of fp64)."""
    sel = np.take_along_axis(scale, np.asarray(idx), 1)
    return W_TOL + 2 * LOGIT_TOL * sel.max(axis=1)


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


def stratified_rows(offsets, seed=0, block=128):
    """Rows in the oracle's grouped numbering: one random row of every
    block-row slice of every non-empty group (slices counted from the
    group's first row, as the GEMM tiles are), plus each group's first and
    last row."""
    g = np.random.default_rng(seed)
    rows = []
    E = len(offsets) - 1
    for e in range(E):
        r0, r1 = int(offsets[e]), int(offsets[e + 1])
        if r1 == r0:
            continue
        rows += [r0, r1 - 1]
        for b0 in range(r0, r1, block):
            rows.append(int(g.integers(b0, min(b0 + block, r1))))
    return np.unique(np.array(rows, np.int64))


def check_stratified_rows(h, y_perm, row_of, xs, idx, offsets, src_tok, same, W1, W2):
    """h (and y_perm, unless None) of the stratified rows against the expert
    FFN evaluated from the definition on the oracle's routing (idx, offsets,
    src_tok), for rows of tokens routed identically on both sides (`same`).
    h, y_perm, row_of: the GPU's tensors; W1, W2: the layer's weights (any
    device).  Returns (rows checked, experts touched)."""
    rows_o = stratified_rows(offsets)
    tok = np.asarray(src_tok)[rows_o]
    keep = same[tok]
    rows_o, tok = rows_o[keep], tok[keep]
    e_of = np.searchsorted(offsets, rows_o, side="right") - 1
    k_of = np.argmax(idx[tok] == e_of[:, None], axis=1)
    assert np.all(idx[tok, k_of] == e_of)
    rows_g = to_np(row_of)[tok, k_of]
    sel = torch.from_numpy(rows_g).to(h.device)
    h_g = to_np(h[sel])
    yp_g = to_np(y_perm[sel]) if y_perm is not None else None
    h_ref = np.zeros(h_g.shape)
    yp_ref = np.zeros(yp_g.shape) if yp_g is not None else None
    for e in np.unique(e_of):
        m = e_of == e
        he, ye = oracle.expert_ffn(xs[tok[m]], to_np(W1[int(e)]), to_np(W2[int(e)]))
        h_ref[m] = he
        if yp_ref is not None:
            yp_ref[m] = ye
    check_rounded(h_g, h_ref, "h (stratified rows)")
    if yp_g is not None:
        check_output(yp_g, yp_ref, "y_perm (stratified rows)")
    return len(rows_o), len(np.unique(e_of))


def run_layer(x, w, K, fill_nan=True):
    """Runs the whole layer with moe.MoELayer on the tensors' device; the
    workspace is filled with 0xFF bytes first (NaN in bf16 and fp32, -1 in
    int32) so that any row a kernel fails to write shows up."""
    import dropless_moe_expert_gb300 as moe
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
    T, E = xs.shape[0], Wr.shape[1]
    ref = oracle.forward(xs, Wr, bias, W1, W2, K)
    _, scale, L64 = check_logits(to_np(v["logits"]), xs, Wr, bias)
    idx = to_np(v["topk_idx"])
    same = check_routing(idx, ref["idx"], L64, scale, K)
    dw = np.abs(to_np(v["topk_w"]) - ref["w"]).max(axis=1)
    assert np.all(dw[same] <= weight_tol(scale, idx)[same]), "topk_w"
    if same.all():
        assert np.array_equal(to_np(v["counts"]), ref["counts"]), "counts"
        assert np.array_equal(to_np(v["offsets"]), ref["offsets"]), "offsets"
        assert np.array_equal(to_np(v["row_of"]), ref["row_of"]), "row_of"
        assert np.array_equal(to_np(v["src_tok"]), ref["src_tok"]), "src_tok"
    else:
        check_dispatch_valid(v, T, K, E)
    src_tok = to_np(v["src_tok"])
    import dropless_moe_expert_gb300 as moe
    if not moe.forward_fuses_permute(T, xs.shape[1], E, K, W1.shape[1] // 2):
        # the layer wrote x_perm (else GEMM1 read the rows straight from x)
        xp = v["x_perm"].view(torch.int16).cpu().numpy()
        assert np.array_equal(xp, x.view(torch.int16).cpu().numpy()[src_tok]), "x_perm"
    # rows of the equally routed tokens, matched through each side's row_of
    rg = to_np(v["row_of"])[same].ravel()
    ro = ref["row_of"][same].ravel()
    check_rounded(to_np(v["h"])[rg], ref["h"][ro], "h")
    check_output(to_np(v["y_perm"])[rg], ref["y_perm"][ro], "y_perm")
    return check_output(to_np(y)[same], ref["y"][same], "y")


# ------------------------------------------------------------ MXFP8 scale atoms
def unpack_plain_atoms(buf, R, K):
    """Scale bytes [R, K/32] of a plain matrix from its 512-byte atoms (128
    rows x 4 scale columns each; row r's 4 bytes at (r % 32) * 16 +
    ((r % 128) // 32) * 4)."""
    ns = K // 128
    r = np.arange(R)
    out = np.zeros((R, K // 32), np.uint8)
    for ks in range(ns):
        base = ((r // 128) * ns + ks) * 512 + (r % 32) * 16 + ((r % 128) // 32) * 4
        for b in range(4):
            out[:, ks * 4 + b] = buf[base + b]
    return out


def unpack_group_atoms(buf, offsets, K, rows=None):
    """Scale bytes [len(rows), K/32] of rows grouped by expert (each group's
    row blocks start at its first row); all TK rows when rows is None."""
    ns = K // 128
    offsets = np.asarray(offsets, np.int64)
    counts = np.diff(offsets)
    rbp = np.concatenate([[0], np.cumsum((counts + 127) // 128)])[:-1]
    r = np.arange(int(offsets[-1])) if rows is None else np.asarray(rows, np.int64)
    e = np.searchsorted(offsets, r, side="right") - 1
    i = r - offsets[e]
    rb = rbp[e] + i // 128
    j = i % 128
    out = np.zeros((r.shape[0], K // 32), np.uint8)
    for ks in range(ns):
        base = (rb * ns + ks) * 512 + (j % 32) * 16 + (j // 32) * 4
        for b in range(4):
            out[:, ks * 4 + b] = buf[base + b]
    return out


def check_mx_rounded(hd_gpu, h_ref, hs_ref, what="h"):
    """A value computed in fp32 and stored as MXFP8 (hd_gpu, dequantised)
    against the oracle's fp64 value before its quantisation: within half an
    E4M3 ulp of its block (2^-4 relative in the normal range, 2^-10 of the
    block scale below it, the scale allowed one binade above the oracle's
    scale code hs_ref)."""
    hd_gpu = np.asarray(hd_gpu, np.float64)
    h_ref = np.asarray(h_ref, np.float64)
    assert np.all(np.isfinite(hd_gpu)), f"{what}: non-finite values"
    X = np.repeat(np.ldexp(1.0, np.asarray(hs_ref).astype(np.int64) - 127), 32, axis=-1)
    bound = 2.0 ** -4 * np.abs(h_ref) * (1 + 1e-4) + 2.0 ** -9 * X + 1e-6 * np.sqrt(np.mean(h_ref ** 2))
    excess = np.abs(hd_gpu - h_ref) - bound
    assert np.all(excess <= 0), f"{what}: {int((excess > 0).sum())} elements beyond the E4M3 rounding bound"
