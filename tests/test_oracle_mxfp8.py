"""Pins of the MXFP8 oracle (oracle/mxfp8.py), on CPU.

E4M3 decoding and rounding are checked against PyTorch's float8_e4m3fn
conversion (an independent library routine); the block scale rule, the
rounding error bounds and the representable-input identities against their
closed forms."""
import numpy as np
import pytest
import torch

import oracle
from oracle import mxfp8 as mx


def _torch_e4m3(v):
    return torch.from_numpy(np.asarray(v, np.float32)).to(torch.float8_e4m3fn).float().numpy().astype(np.float64)


def test_decode_matches_library_for_all_codes():
    codes = np.arange(256, dtype=np.uint8)
    ours = oracle.e4m3_decode(codes)
    lib = torch.from_numpy(codes).view(torch.float8_e4m3fn).float().numpy().astype(np.float64)
    nan = (codes & 0x7F) == 0x7F
    assert np.all(np.isnan(ours[nan])) and np.all(np.isnan(lib[nan]))
    assert np.array_equal(ours[~nan], lib[~nan])
    assert np.array_equal(np.signbit(ours[~nan]), np.signbit(lib[~nan]))
    assert ours[0x7E] == 448.0 and ours[0x08] == 2.0 ** -6 and ours[0x01] == 2.0 ** -9


def test_encode_decode_round_trip():
    codes = np.array([c for c in range(256) if (c & 0x7F) != 0x7F], np.uint8)
    assert np.array_equal(oracle.e4m3_encode(oracle.e4m3_decode(codes)), codes)


def test_rounding_matches_library():
    g = np.random.default_rng(0)
    v = np.concatenate([g.standard_normal(20000) * 10.0 ** g.uniform(-4, 2.4, 20000),
                        g.uniform(-448, 448, 5000)]).astype(np.float32)
    v = v[np.abs(v) <= 448]
    assert np.array_equal(oracle.e4m3_round(v), _torch_e4m3(v))


def test_rounding_ties_go_to_even_mantissa():
    # midpoints between neighbours: 1 + 1/16 lies between 1 (man 0) and 1.125 (man 1)
    assert oracle.e4m3_round(1.0 + 1 / 16) == 1.0
    assert oracle.e4m3_round(1.125 + 1 / 16) == 1.25          # between man 1 and man 2 -> 2
    assert oracle.e4m3_round(-(2.0 ** -9) / 2) == 0.0 and np.signbit(oracle.e4m3_round(-(2.0 ** -10)))
    assert oracle.e4m3_round(3 * 2.0 ** -10) == 2 * 2.0 ** -9  # subnormal tie: 1.5 ulp -> 2 ulp
    assert oracle.e4m3_round(464.0) == 448.0 and oracle.e4m3_round(1000.0) == 448.0


@pytest.mark.parametrize("k", [-20, -3, 0, 5, 30])
def test_scale_rule(k):
    e = oracle.mx_scale_exponent
    assert e(448.0 * 2.0 ** k) == k                         # the largest element lands on 448
    assert e(448.0 * 2.0 ** k * (1 + 2.0 ** -20)) == k + 1  # just above: next power of two
    assert e(2.0 ** k) == k - 8                             # m = 1 -> 256
    assert e(1.75 * 2.0 ** k) == k - 8                      # m = 1.75 -> 448, not saturated
    assert e(1.8 * 2.0 ** k) == k - 7                       # m > 1.75 -> below 256
    assert e(0.0) == -127


def test_quantize_bounds_and_no_saturation():
    g = np.random.default_rng(1)
    V = g.standard_normal((64, 256)) * 10.0 ** g.uniform(-3, 3, (64, 1))
    V[3, :32] = 0.0                                         # one all-zero block
    codes, sc, deq = oracle.mx_quantize(V)
    e = sc.astype(np.int64) - 127
    X = np.repeat(np.ldexp(1.0, e), 32, axis=-1)
    q = V / X
    # the block maximum is in (224, 448]: never saturated, never more than one binade low
    amax = np.abs(q).reshape(64, 8, 32).max(-1)
    nz = amax > 0
    assert np.all(amax[nz] <= 448) and np.all(amax[nz] > 224)
    # rounding error: half an E4M3 ulp (2^-4 relative) in the normal range,
    # half the subnormal spacing (2^-10 X) below it
    err = np.abs(deq - V)
    normal = np.abs(q) >= 2.0 ** -6
    assert np.all(err[normal] <= 2.0 ** -4 * np.abs(V[normal]))
    assert np.all(err[~normal] <= 2.0 ** -10 * X[~normal])
    assert np.all(codes[3, :32] == 0) and deq[3, :32].tolist() == [0.0] * 32 and sc[3, 0] == 0
    assert np.array_equal(oracle.mx_dequantize(codes, sc), deq)


def test_representable_inputs_are_fixed_points():
    g = np.random.default_rng(2)
    codes = g.integers(0, 256, (16, 128)).astype(np.uint8)
    codes[(codes & 0x7F) == 0x7F] = 0x40
    codes[:, ::32] = 0x7E                                   # each block holds a 448: amax pins the scale
    sc = g.integers(110, 140, (16, 4)).astype(np.uint8)
    V = oracle.mx_dequantize(codes, sc)
    c2, s2, d2 = oracle.mx_quantize(V)
    assert np.array_equal(c2, codes) and np.array_equal(s2, sc) and np.array_equal(d2, V)


def _tiny_case(representable):
    g = np.random.default_rng(3)
    T, d, E, K, f = 40, 64, 4, 2, 64

    def mxval(shape):
        c = g.integers(0, 256, shape).astype(np.uint8)
        c[(c & 0x7F) == 0x7F] = 0x38
        c[..., ::32] = 0x7E
        s = g.integers(118, 122, shape[:-1] + (shape[-1] // 32,)).astype(np.uint8)
        return oracle.mx_dequantize(c, s).astype(np.float32)

    if representable:
        x, W1, W2 = mxval((T, d)), mxval((E, 2 * f, d)), mxval((E, d, f))
    else:
        x = g.standard_normal((T, d)).astype(np.float32)
        W1 = (g.standard_normal((E, 2 * f, d)) / 8).astype(np.float32)
        W2 = (g.standard_normal((E, d, f)) / 8).astype(np.float32)
    Wr = (g.standard_normal((d, E)) / 8).astype(np.float32)
    bias = g.standard_normal(E).astype(np.float32)
    return x, Wr, bias, W1, W2, K


def test_forward_on_representable_inputs_matches_the_bf16_oracle_before_h():
    x, Wr, bias, W1, W2, K = _tiny_case(True)
    ref = oracle.forward(x, Wr, bias, W1, W2, K)
    out = oracle.forward_mxfp8(x, Wr, bias, W1, W2, K)
    for k in ("idx", "counts", "offsets", "row_of", "src_tok"):
        assert np.array_equal(out[k], ref[k])
    assert np.array_equal(out["x_perm"], ref["x_perm"])     # quantising x changed nothing
    assert np.allclose(out["h"], ref["h"], rtol=1e-12, atol=1e-12)
    # h itself is then quantised: the MXFP8 y is the bf16 y with h replaced by its quantised value
    _, _, hd = oracle.mx_quantize(ref["h"])
    y_perm = np.zeros_like(ref["y_perm"])
    for e in range(W1.shape[0]):
        r0, r1 = ref["offsets"][e], ref["offsets"][e + 1]
        y_perm[r0:r1] = hd[r0:r1] @ np.asarray(W2[e], np.float64).T
    assert np.allclose(out["y"], oracle.combine(y_perm, ref["row_of"], ref["w"]), rtol=1e-12, atol=1e-12)


def test_forward_error_against_the_bf16_oracle_is_the_quantisation_error():
    x, Wr, bias, W1, W2, K = _tiny_case(False)
    ref = oracle.forward(x, Wr, bias, W1, W2, K)["y"]
    y = oracle.forward_mxfp8(x, Wr, bias, W1, W2, K)["y"]
    rel = np.linalg.norm(y - ref) / np.linalg.norm(ref)
    assert 1e-3 < rel < 0.1       # E4M3 keeps 3 mantissa bits: a few percent, never zero


def test_quantize_in_row_chunks_equals_one_pass():
    # 70000 rows of 32: three chunks, the last one partial, and a 3-D shape
    g = np.random.default_rng(4)
    V = g.standard_normal((2, 35000, 32)) * np.exp(2 * g.standard_normal((2, 35000, 1)))
    codes, scales, deq = oracle.mx_quantize(V)
    c1, s1, d1 = mx._mx_quantize_rows(V.reshape(-1, 32))
    assert codes.shape == V.shape and scales.shape == (2, 35000, 1)
    assert np.array_equal(codes.reshape(-1, 32), c1)
    assert np.array_equal(scales.reshape(-1, 1), s1)
    assert np.array_equal(deq.reshape(-1, 32), d1)


@pytest.mark.parametrize("K", [1, 2, 4])
def test_per_token_evaluation_equals_the_whole_forward(K):
    x, Wr, bias, W1, W2, _ = _tiny_case(False)
    ref = oracle.forward_mxfp8(x, Wr, bias, W1, W2, K)
    _, _, W1d = oracle.mx_quantize(W1)
    _, _, W2d = oracle.mx_quantize(W2)
    toks = np.array([0, 3, x.shape[0] - 1])
    idx, w, slots, y = oracle.forward_mxfp8_tokens(x[toks], ref["logits"][toks], K, lambda e: (W1d[e], W2d[e]))
    assert np.array_equal(idx, ref["idx"][toks])
    assert np.array_equal(w, ref["w"][toks])
    for i, t in enumerate(toks):
        assert np.array_equal(slots[i][0]["xq"], ref["xq"][t])
        assert np.array_equal(slots[i][0]["xs"], ref["xs"][t])
        for k in range(K):
            r = ref["row_of"][t, k]
            assert np.allclose(slots[i][k]["h"], ref["h"][r], rtol=1e-12, atol=1e-12)
            assert np.array_equal(slots[i][k]["hq"], ref["hq"][r])
            assert np.array_equal(slots[i][k]["hs"], ref["hs"][r])
            assert np.allclose(slots[i][k]["y_perm"], ref["y_perm"][r], rtol=1e-12, atol=1e-12)
    assert np.allclose(y, ref["y"][toks], rtol=1e-12, atol=1e-12)
