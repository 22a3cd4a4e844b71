"""Pins for the CPU oracle: checks against things other than the oracle itself.

Each test ties one part of the oracle to a library routine, a closed form, an identity
the pages state, hand arithmetic, or an invariant, chosen so that a plausible slip (a
dropped bias, a wrong sign, a transposed operand, a shifted tap, a missing rounding of
the intermediate) fails at least one of them.
"""
import math
import os

import numpy as np
import pytest
import torch
import torch.nn.functional as F

from gemm_conv_chains_gb300 import workloads as wl

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def f16_bits(values):
    return np.asarray(values, dtype=np.float64).astype(np.float16).view(np.uint16)


def bf16_bits(values):
    t = torch.tensor(np.asarray(values, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


# ------------------------------------------------------------------------------------
# storage formats
# ------------------------------------------------------------------------------------

def test_decode_fp16_exhaustive_vs_numpy(oracle_mod):
    bits = np.arange(65536, dtype=np.uint16)
    ref = bits.view(np.float16).astype(np.float64)
    got = oracle_mod.decode("f16", bits)
    assert np.array_equal(np.isnan(ref), np.isnan(got))
    ok = ~np.isnan(ref)
    assert np.array_equal(ref[ok], got[ok])
    # signed zeros survive
    assert math.copysign(1.0, got[0x8000]) == -1.0


def test_decode_bf16_exhaustive_vs_fp32_upper_half(oracle_mod):
    # bf16 is, by definition, the upper 16 bits of an IEEE binary32
    bits = np.arange(65536, dtype=np.uint16)
    ref = (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    got = oracle_mod.decode("bf16", bits)
    assert np.array_equal(np.isnan(ref), np.isnan(got))
    ok = ~np.isnan(ref)
    assert np.array_equal(ref[ok], got[ok])


def _interesting_doubles(rng, n):
    mags = np.exp2(rng.uniform(-30, 18, n))
    vals = mags * rng.choice([-1.0, 1.0], n)
    return vals


def test_encode_fp16_vs_numpy_rne(oracle_mod):
    rng = np.random.default_rng(1)
    vals = _interesting_doubles(rng, 200000)
    # midpoints between neighbouring fp16 values: the ties-to-even cases
    b = rng.integers(0, 0x7BFF, 20000).astype(np.uint16)
    lo = b.view(np.float16).astype(np.float64)
    hi = (b + 1).view(np.float16).astype(np.float64)
    vals = np.concatenate([vals, (lo + hi) / 2, -(lo + hi) / 2,
                           [0.0, -0.0, 65504.0, 65519.99, 65520.0, 1e6, -1e6,
                            2.0 ** -24, 2.0 ** -25, 3 * 2.0 ** -26, 2.0 ** -14]])
    ref = vals.astype(np.float16).view(np.uint16)
    got = oracle_mod.encode("f16", vals)
    assert np.array_equal(ref, got)


def test_encode_bf16_vs_torch_on_fp32_exact_values(oracle_mod):
    # torch rounds float32 -> bf16 to nearest-even; on values that are exact float32,
    # that is a single rounding, so it must agree with the oracle's direct rounding.
    rng = np.random.default_rng(2)
    vals = _interesting_doubles(rng, 200000).astype(np.float32)
    # ties: halfway between bf16 neighbours (exact in float32)
    b = rng.integers(0, 0x7F7F, 20000).astype(np.uint32)
    ties = ((b << 16) | 0x8000).view(np.float32)
    vals = np.concatenate([vals, ties, -ties, np.float32([3.3895314e38, 3.40e38, 1e-40, 0.0])])
    ref = torch.from_numpy(vals).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = oracle_mod.encode("bf16", vals.astype(np.float64))
    assert np.array_equal(ref, got)


def test_encode_hand_ties_and_overflow(oracle_mod):
    # 1 + 2^-11 lies halfway between 1 and 1 + 2^-10: ties to the even neighbour, 1.0
    assert oracle_mod.encode("f16", np.array([1 + 2.0 ** -11]))[0] == 0x3C00
    # 1 + 3*2^-11 lies halfway between 1 + 2^-10 (odd) and 1 + 2^-9 (even)
    assert oracle_mod.encode("f16", np.array([1 + 3 * 2.0 ** -11]))[0] == 0x3C02
    # largest finite fp16 is 65504; 65520 is the midpoint to 2^16 and rounds up: inf
    assert oracle_mod.encode("f16", np.array([65519.0]))[0] == 0x7BFF
    assert oracle_mod.encode("f16", np.array([65520.0]))[0] == 0x7C00
    assert oracle_mod.encode("f16", np.array([-70000.0]))[0] == 0xFC00
    # smallest subnormal 2^-24; half of it ties to 0 (even)
    assert oracle_mod.encode("f16", np.array([2.0 ** -24]))[0] == 0x0001
    assert oracle_mod.encode("f16", np.array([2.0 ** -25]))[0] == 0x0000
    # bf16: 1 + 2^-8 ties to 1.0; 1 + 3*2^-8 ties up to 1 + 2^-6
    assert oracle_mod.encode("bf16", np.array([1 + 2.0 ** -8]))[0] == 0x3F80
    assert oracle_mod.encode("bf16", np.array([1 + 3 * 2.0 ** -8]))[0] == 0x3F82


# ------------------------------------------------------------------------------------
# activations (closed forms)
# ------------------------------------------------------------------------------------

@pytest.mark.parametrize("x,expected", [(-4.0, 0.0), (-3.0, 0.0), (-1.5, -0.375), (-1.0, -1.0 / 3.0),
                                        (0.0, 0.0), (1.0, 2.0 / 3.0), (3.0, 3.0), (10.0, 10.0)])
def test_hardswish_closed_form(oracle_mod, x, expected):
    assert oracle_mod.activation("hardswish", x) == pytest.approx(expected, abs=0, rel=1e-15)


def test_hardswish_fp16_rounding(oracle_mod):
    v = oracle_mod.activation("hardswish", 1.0)
    assert oracle_mod.encode("f16", np.array([v]))[0] == 0x3955   # 0.66650390625


@pytest.mark.parametrize("x,expected", [(-2.0, 0.0), (-0.0, 0.0), (0.0, 0.0), (0.5, 0.5), (7.0, 7.0)])
def test_relu_closed_form(oracle_mod, x, expected):
    assert oracle_mod.activation("relu", x) == expected


def test_none_activation_is_identity(oracle_mod):
    for x in (-5.5, 0.0, 3.25):
        assert oracle_mod.activation("none", x) == x


# ------------------------------------------------------------------------------------
# GEMM stage and b2b chain
# ------------------------------------------------------------------------------------

def test_hand_2x2_chain(oracle_mod):
    # A = [[1,2],[3,4]], W0 = I, b0 = [0,-5], ReLU:  h = relu([[1,-3],[3,-1]]) = [[1,0],[3,0]]
    # W1 = [[1,1],[0,1]], b1 = [0,0.5], none:        y = [[1,1.5],[3,3.5]]
    A = f16_bits([[1, 2], [3, 4]])
    W0 = f16_bits([[1, 0], [0, 1]])
    b0 = f16_bits([0, -5])
    W1 = f16_bits([[1, 1], [0, 1]])
    b1 = f16_bits([0, 0.5])
    h = oracle_mod.gemm_bias_act("f16", A, W0, b0, "relu")
    assert np.array_equal(oracle_mod.decode("f16", h), [[1, 0], [3, 0]])
    y = oracle_mod.b2b_gemm("f16", A, W0, b0, W1, b1, "relu", "none")
    assert np.array_equal(oracle_mod.decode("f16", y), [[1, 1.5], [3, 3.5]])


def test_bias_is_column_broadcast_and_optional(oracle_mod):
    A = f16_bits(np.zeros((3, 4)))
    W = f16_bits(np.ones((4, 5)))
    b = f16_bits([1, 2, 3, 4, 5])
    out = oracle_mod.decode("f16", oracle_mod.gemm_bias_act("f16", A, W, b, "none"))
    assert np.array_equal(out, np.tile([1, 2, 3, 4, 5], (3, 1)))
    out = oracle_mod.decode("f16", oracle_mod.gemm_bias_act("f16", A, W, None, "none"))
    assert np.array_equal(out, np.zeros((3, 5)))


@pytest.mark.parametrize("dt", ["f16", "bf16"])
def test_gemm_integer_exact_vs_numpy(oracle_mod, dt):
    # Integer operands: every product and partial sum is an exact integer, so the
    # result is independent of summation order and equals numpy's int64 matmul.
    rng = np.random.default_rng(3)
    M, K, N = 37, 19, 11                      # distinct sizes: a transposed operand fails
    A = rng.integers(-3, 4, (M, K))
    W = rng.integers(-3, 4, (K, N))
    b = rng.integers(-2, 3, (N,))
    enc = f16_bits if dt == "f16" else bf16_bits
    for act in ("none", "relu", "hardswish"):
        got = oracle_mod.gemm_bias_act(dt, enc(A), enc(W), enc(b), act)
        z = (A @ W + b).astype(np.float64)
        ref = np.array([oracle_mod.activation(act, v) for v in z.ravel()]).reshape(z.shape)
        assert np.array_equal(got, oracle_mod.encode(dt, ref))
    # spot-check a hand-indexed element against the definition's indices
    got = oracle_mod.decode(dt, oracle_mod.gemm_bias_act(dt, enc(A), enc(W), enc(b), "none"))
    m, n = 5, 7
    assert got[m, n] == sum(int(A[m, k]) * int(W[k, n]) for k in range(K)) + b[n]


def test_gemm_random_vs_numpy_float64(oracle_mod):
    rng = np.random.default_rng(4)
    M, K, N = 64, 48, 40
    A = f16_bits(rng.uniform(-1, 1, (M, K)))
    W = f16_bits(rng.normal(0, 1 / math.sqrt(K), (K, N)))
    b = f16_bits(rng.uniform(-0.1, 0.1, (N,)))
    Ad, Wd, bd = (oracle_mod.decode("f16", t) for t in (A, W, b))
    z = Ad @ Wd + bd
    ref = np.where(z > 0, z, 0.0)
    got = oracle_mod.decode("f16", oracle_mod.gemm_bias_act("f16", A, W, b, "relu"))
    # one fp16 rounding of a value that differs only by summation order
    assert np.max(np.abs(got - ref) / np.maximum(np.abs(ref), 2.0 ** -14)) <= 2.0 ** -10


def test_b2b_rounds_the_intermediate(oracle_mod):
    # z0 = [1 + 2^-12, 1]; stored in fp16 it is [1, 1]; y = h0 - h1.
    # With the intermediate rounded (as the fused kernel stores it): y = 0.
    # Without that rounding it would be 2^-12 (itself exact in fp16).
    A = f16_bits([[1.0]])
    W0 = f16_bits([[1.0, 1.0]])
    b0 = f16_bits([2.0 ** -12, 0.0])
    W1 = f16_bits([[1.0], [-1.0]])
    y = oracle_mod.b2b_gemm("f16", A, W0, b0, W1, None, "none", "none")
    assert oracle_mod.decode("f16", y)[0, 0] == 0.0


def test_b2b_equals_two_stages(oracle_mod):
    w = wl.GEMM_SMALL.with_m(300)
    t = wl.gemm_inputs(w, seed=5)
    bits = {k: wl.to_bits(v) for k, v in t.items()}
    h = oracle_mod.gemm_bias_act("f16", bits["A"], bits["W0"], bits["b0"], "relu")
    y2 = oracle_mod.gemm_bias_act("f16", h, bits["W1"], bits["b1"], "relu")
    y = oracle_mod.b2b_gemm("f16", bits["A"], bits["W0"], bits["b0"], bits["W1"], bits["b1"],
                            "relu", "relu")
    assert np.array_equal(y, y2)


def test_b2b_past_the_first_row_block(oracle_mod):
    # The oracle forms the intermediate 4096 rows at a time.  M = 4096 + 300 reaches a
    # second, partial block, checked three independent ways: numpy's int64 matmul with
    # numpy's own fp16 rounding (integer data: h = relu(A W0 + b0) <= 98 is exact in fp16,
    # y = relu(h W1 + b1) <= 7842 is rounded once, by numpy); the rows of the second block
    # run on their own (rows are independent, so a slip in the block offset shows); and two
    # separate stages.  Distinct K0, N0, N1 catch a transposed operand.
    rng = np.random.default_rng(11)
    M, K0, N0, N1 = 4096 + 300, 24, 40, 16
    A = rng.integers(-2, 3, (M, K0))
    W0 = rng.integers(-2, 3, (K0, N0))
    b0 = rng.integers(-2, 3, (N0,))
    W1 = rng.integers(-2, 3, (N0, N1))
    b1 = rng.integers(-2, 3, (N1,))
    h = np.maximum(A @ W0 + b0, 0)
    assert np.abs(h).max() <= 2048                        # exact in fp16
    ref = np.maximum(h @ W1 + b1, 0).astype(np.float64).astype(np.float16).view(np.uint16)
    y = oracle_mod.b2b_gemm("f16", f16_bits(A), f16_bits(W0), f16_bits(b0), f16_bits(W1),
                            f16_bits(b1), "relu", "relu")
    assert y.shape == (M, N1)
    assert np.array_equal(y, ref)
    tail = oracle_mod.b2b_gemm("f16", f16_bits(A[4096:]), f16_bits(W0), f16_bits(b0),
                               f16_bits(W1), f16_bits(b1), "relu", "relu")
    assert np.array_equal(y[4096:], tail)
    h16 = oracle_mod.gemm_bias_act("f16", f16_bits(A), f16_bits(W0), f16_bits(b0), "relu")
    y2 = oracle_mod.gemm_bias_act("f16", h16, f16_bits(W1), f16_bits(b1), "relu")
    assert np.array_equal(y, y2)


# ------------------------------------------------------------------------------------
# convolution
# ------------------------------------------------------------------------------------

def _torch_conv_nhwc(x, Wt, b, pad, stride=1):
    """float64 library convolution (cross-correlation) on NHWC data."""
    xt = torch.from_numpy(x).permute(0, 3, 1, 2)
    wt = torch.from_numpy(Wt).permute(0, 3, 1, 2)
    bt = torch.from_numpy(b) if b is not None else None
    return F.conv2d(xt, wt, bt, padding=pad, stride=stride).permute(0, 2, 3, 1).numpy()


def _im2col_conv_nhwc(x, Wt, b, pad):
    """The interview notes' Im2Col + GEMM formulation: unfold windows, then one matmul."""
    N, H, W, C = x.shape
    Co, R, S, _ = Wt.shape
    Ho, Wo = H + 2 * pad - R + 1, W + 2 * pad - S + 1
    xp = np.zeros((N, H + 2 * pad, W + 2 * pad, C))
    xp[:, pad:pad + H, pad:pad + W, :] = x
    cols = np.empty((N, Ho, Wo, R, S, C))
    for r in range(R):
        for s in range(S):
            cols[:, :, :, r, s, :] = xp[:, r:r + Ho, s:s + Wo, :]
    y = cols.reshape(N * Ho * Wo, R * S * C) @ Wt.reshape(Co, R * S * C).T
    if b is not None:
        y = y + b
    return y.reshape(N, Ho, Wo, Co)


@pytest.mark.parametrize("shape", [
    # N, H, W, C, Co, R, S, pad
    (2, 5, 7, 3, 4, 3, 3, 1),
    (1, 6, 4, 8, 5, 3, 3, 0),
    (1, 4, 5, 2, 3, 1, 3, 2),
    (3, 3, 3, 4, 2, 1, 1, 0),
])
@pytest.mark.parametrize("dt", ["f16", "bf16"])
def test_conv_integer_exact_vs_torch_and_im2col(oracle_mod, shape, dt):
    N, H, W, C, Co, R, S, pad = shape
    rng = np.random.default_rng(sum(shape))
    x = rng.integers(-3, 4, (N, H, W, C)).astype(np.float64)
    Wt = rng.integers(-3, 4, (Co, R, S, C)).astype(np.float64)
    b = rng.integers(-2, 3, (Co,)).astype(np.float64)
    enc = f16_bits if dt == "f16" else bf16_bits
    got = oracle_mod.decode(dt, oracle_mod.conv2d_nhwc(dt, enc(x), enc(Wt), enc(b), pad, "none"))
    ref_lib = _torch_conv_nhwc(x, Wt, b, pad)
    ref_i2c = _im2col_conv_nhwc(x, Wt, b, pad)
    assert got.shape == ref_lib.shape == (N, H + 2 * pad - R + 1, W + 2 * pad - S + 1, Co)
    assert np.array_equal(got, ref_lib)
    assert np.array_equal(got, ref_i2c)


def test_conv_random_vs_torch_float64(oracle_mod):
    rng = np.random.default_rng(7)
    x = oracle_mod.decode("f16", f16_bits(rng.uniform(-1, 1, (2, 9, 11, 16))))
    Wt = oracle_mod.decode("f16", f16_bits(rng.normal(0, 1 / 12, (8, 3, 3, 16))))
    b = oracle_mod.decode("f16", f16_bits(rng.uniform(-0.1, 0.1, (8,))))
    z = _torch_conv_nhwc(x, Wt, b, 1)
    ref = z * np.clip(z + 3, 0, 6) / 6
    got = oracle_mod.decode("f16", oracle_mod.conv2d_nhwc("f16", f16_bits(x), f16_bits(Wt),
                                                          f16_bits(b), 1, "hardswish"))
    assert np.max(np.abs(got - ref) / np.maximum(np.abs(ref), 2.0 ** -14)) <= 2.0 ** -10


def _read_tiles():
    tiles = {}
    with open(os.path.join(GOLDEN, "tile_shapes.txt")) as f:
        for line in f:
            line = line.split("#")[0].strip()
            if not line:
                continue
            name, src, _, dst = line.split()
            tiles[name] = (tuple(src.split(",")), tuple(dst.split(",")))
    return tiles


def test_conv_receptive_field_matches_page_tile(oracle_mod):
    # Welder: a 1x1xC conv output tile reads a 3x3xC input tile.  Perturb one input
    # pixel; exactly the outputs whose 3x3 window covers it must change.
    (ih, iw, _), (oh, ow, _) = _read_tiles()["conv3x3"]
    assert (int(ih), int(iw), int(oh), int(ow)) == (3, 3, 1, 1)
    rng = np.random.default_rng(8)
    x = rng.integers(-3, 4, (1, 7, 8, 4)).astype(np.float64)
    Wt = rng.integers(1, 4, (2, 3, 3, 4)).astype(np.float64)      # all positive taps
    base = oracle_mod.decode("f16", oracle_mod.conv2d_nhwc("f16", f16_bits(x), f16_bits(Wt), None, 1, "none"))
    x2 = x.copy()
    x2[0, 3, 5, :] += 1.0                                       # all channels up by one
    pert = oracle_mod.decode("f16", oracle_mod.conv2d_nhwc("f16", f16_bits(x2), f16_bits(Wt), None, 1, "none"))
    changed = np.any(pert != base, axis=-1)[0]
    expect = np.zeros_like(changed)
    expect[3 - 1:3 + 2, 5 - 1:5 + 2] = True
    assert np.array_equal(changed, expect)


def test_one_by_one_conv_chain_is_b2b_gemm(oracle_mod):
    # Interview notes: a 1x1 conv reduces to a GEMM.  Two chained 1x1 convs on
    # [N,H,W,C] equal the b2b GEMM over the [N*H*W, C] view, bit for bit.
    w = wl.ConvChain("t", "f16", 3, 5, 6, 16, 24, 1, 1, 0, 8, "relu", "hardswish")
    t = {k: wl.to_bits(v) for k, v in wl.conv_inputs(w, seed=9).items()}
    conv = oracle_mod.b2b_conv_nhwc("f16", t["x"], t["W0"], t["b0"], t["W1"], t["b1"], 0,
                                    "relu", "hardswish")
    A = t["x"].reshape(-1, w.C)
    W0 = np.ascontiguousarray(t["W0"].reshape(w.C0, w.C).T)
    W1 = np.ascontiguousarray(t["W1"].T)
    gemm = oracle_mod.b2b_gemm("f16", A, W0, t["b0"], W1, t["b1"], "relu", "hardswish")
    assert np.array_equal(conv.reshape(-1, w.C1), gemm)


def test_b2b_conv_equals_conv_then_pointwise(oracle_mod):
    w = wl.ConvChain("t", "f16", 2, 7, 5, 8, 16, 3, 3, 1, 24, "hardswish", "none")
    t = {k: wl.to_bits(v) for k, v in wl.conv_inputs(w, seed=10).items()}
    h = oracle_mod.conv2d_nhwc("f16", t["x"], t["W0"], t["b0"], 1, "hardswish")
    y2 = oracle_mod.conv2d_nhwc("f16", h, t["W1"].reshape(w.C1, 1, 1, w.C0), t["b1"], 0, "none")
    y = oracle_mod.b2b_conv_nhwc("f16", t["x"], t["W0"], t["b0"], t["W1"], t["b1"], 1,
                                 "hardswish", "none")
    assert np.array_equal(y, y2)


# ------------------------------------------------------------------------------------
# three-operator chain (BOLT notes, "Enabling deeper operator fusion")
# ------------------------------------------------------------------------------------

@pytest.mark.parametrize("dt", ["f16", "bf16"])
def test_gemm3_integer_exact_vs_numpy(oracle_mod, dt):
    # integer data in {-1, 0, 1}: every sum is an exact integer far below 2^24 and every
    # intermediate is exactly representable, so float64 numpy with the same roundings
    # (identity on these integers) gives the same values
    rng = np.random.default_rng(50)
    A = rng.integers(-1, 2, (37, 64)).astype(np.float64)
    W0 = rng.integers(-1, 2, (64, 48)).astype(np.float64)
    W1 = rng.integers(-1, 2, (48, 32)).astype(np.float64)
    W2 = rng.integers(-1, 2, (32, 24)).astype(np.float64)
    b0, b1, b2 = (rng.integers(-2, 3, (n,)).astype(np.float64) for n in (48, 32, 24))
    enc = f16_bits if dt == "f16" else bf16_bits
    got = oracle_mod.decode(dt, oracle_mod.b2b_gemm3(dt, enc(A), enc(W0), enc(b0), enc(W1),
                                                     enc(b1), enc(W2), enc(b2), "relu", "relu",
                                                     "none"))
    h0 = np.maximum(A @ W0 + b0, 0)
    h1 = np.maximum(h0 @ W1 + b1, 0)
    ref = h1 @ W2 + b2
    if dt == "bf16":      # bf16 keeps 8 significant bits: round the larger integers as it does
        ref = oracle_mod.decode("bf16", bf16_bits(ref))
    assert np.all(np.abs(ref) < 65504)
    assert np.array_equal(got, ref)


def test_gemm3_is_b2b_then_one_more_operator(oracle_mod):
    # the first two operators are the two-operator chain, the third one more GEMM + bias +
    # act on its stored output
    w = wl.GemmChain("t", "bf16", 70, 32, 40, 24, "hardswish", "relu")
    t = {k: wl.to_bits(v) for k, v in wl.gemm_inputs(w, seed=51).items()}
    rng = np.random.default_rng(52)
    W2 = bf16_bits(rng.normal(0, 0.2, (24, 16)))
    b2 = bf16_bits(rng.uniform(-0.1, 0.1, 16))
    two = oracle_mod.b2b_gemm("bf16", t["A"], t["W0"], t["b0"], t["W1"], t["b1"], "hardswish",
                              "relu")
    three = oracle_mod.b2b_gemm3("bf16", t["A"], t["W0"], t["b0"], t["W1"], t["b1"], W2, b2,
                                 "hardswish", "relu", "hardswish")
    assert three.shape == (70, 16)
    assert np.array_equal(three, oracle_mod.gemm_bias_act("bf16", two, W2, b2, "hardswish"))


# ------------------------------------------------------------------------------------
# strided conv (Welder notes, tile propagation: a strided conv reads a strided region)
# ------------------------------------------------------------------------------------

@pytest.mark.parametrize("shape", [
    # N, H, W, C, Co, R, S, pad, stride
    (2, 9, 8, 3, 4, 3, 3, 1, 2),
    (1, 7, 7, 8, 5, 3, 3, 1, 2),     # odd size: the last window ends at the padding
    (1, 10, 6, 2, 3, 1, 1, 0, 2),    # 1x1 stride 2 (a downsampling projection)
    (1, 11, 9, 4, 2, 5, 3, 2, 3),
])
@pytest.mark.parametrize("dt", ["f16", "bf16"])
def test_strided_conv_integer_exact_vs_torch(oracle_mod, shape, dt):
    N, H, W, C, Co, R, S, pad, st = shape
    rng = np.random.default_rng(sum(shape) + 100)
    x = rng.integers(-3, 4, (N, H, W, C)).astype(np.float64)
    Wt = rng.integers(-3, 4, (Co, R, S, C)).astype(np.float64)
    b = rng.integers(-2, 3, (Co,)).astype(np.float64)
    enc = f16_bits if dt == "f16" else bf16_bits
    got = oracle_mod.decode(dt, oracle_mod.conv2d_nhwc(dt, enc(x), enc(Wt), enc(b), pad, "none",
                                                       stride=st))
    ref = _torch_conv_nhwc(x, Wt, b, pad, stride=st)
    Ho, Wo = (H + 2 * pad - R) // st + 1, (W + 2 * pad - S) // st + 1
    assert got.shape == ref.shape == (N, Ho, Wo, Co)
    assert np.array_equal(got, ref)


def test_strided_conv_brute_force(oracle_mod):
    # every output element from its own window, by plain loops over the definition
    rng = np.random.default_rng(31)
    N, H, W, C, Co, R, S, pad, st = 1, 6, 7, 2, 2, 3, 2, 1, 2
    x = rng.integers(-3, 4, (N, H, W, C)).astype(np.float64)
    Wt = rng.integers(-3, 4, (Co, R, S, C)).astype(np.float64)
    got = oracle_mod.decode("f16", oracle_mod.conv2d_nhwc("f16", f16_bits(x), f16_bits(Wt), None,
                                                          pad, "none", stride=st))
    Ho, Wo = (H + 2 * pad - R) // st + 1, (W + 2 * pad - S) // st + 1
    for ho in range(Ho):
        for wo in range(Wo):
            for co in range(Co):
                acc = 0.0
                for r in range(R):
                    for s_ in range(S):
                        hi, wi = ho * st + r - pad, wo * st + s_ - pad
                        if 0 <= hi < H and 0 <= wi < W:
                            acc += float(np.dot(x[0, hi, wi], Wt[co, r, s_]))
                assert got[0, ho, wo, co] == acc, (ho, wo, co)


def test_strided_conv_is_the_stride_one_conv_subsampled(oracle_mod):
    # output (ho, wo) of a stride-2 conv is output (2 ho, 2 wo) of the stride-1 conv with
    # the same padding: the same window, the same sum in the same order, bit for bit
    w = wl.ConvChain("t", "bf16", 2, 9, 10, 8, 16, 3, 3, 1, 8, "hardswish", "none")
    t = {k: wl.to_bits(v) for k, v in wl.conv_inputs(w, seed=12).items()}
    one = oracle_mod.conv2d_nhwc("bf16", t["x"], t["W0"], t["b0"], 1, "hardswish")
    two = oracle_mod.conv2d_nhwc("bf16", t["x"], t["W0"], t["b0"], 1, "hardswish", stride=2)
    assert two.shape == (2, 5, 5, 16)
    assert np.array_equal(two, one[:, ::2, ::2, :])


def test_strided_b2b_conv_equals_conv_then_pointwise(oracle_mod):
    w = wl.ConvChain("t", "f16", 2, 9, 7, 8, 16, 3, 3, 1, 24, "relu", "none")
    t = {k: wl.to_bits(v) for k, v in wl.conv_inputs(w, seed=13).items()}
    h = oracle_mod.conv2d_nhwc("f16", t["x"], t["W0"], t["b0"], 1, "relu", stride=2)
    y2 = oracle_mod.conv2d_nhwc("f16", h, t["W1"].reshape(w.C1, 1, 1, w.C0), t["b1"], 0, "none")
    y = oracle_mod.b2b_conv_nhwc("f16", t["x"], t["W0"], t["b0"], t["W1"], t["b1"], 1, "relu",
                                 "none", stride=2)
    assert y.shape == (2, 5, 4, 24)
    assert np.array_equal(y, y2)


# ------------------------------------------------------------------------------------
# batch normalisation folded into weights and bias (interview notes, SimplifyInference)
# ------------------------------------------------------------------------------------

def test_fold_batchnorm_power_of_two_scale_is_exact(oracle_mod):
    # gamma / sqrt(var + eps) = 2 and 0.5: scaling by a power of two is exact, and
    # (b - mean) * s + beta is exact for these small integers
    rng = np.random.default_rng(40)
    W = rng.integers(-8, 9, (2, 3, 3, 4)).astype(np.float64)
    b = np.array([3.0, -2.0])
    gamma = np.array([4.0, 1.0], np.float32)
    var = np.array([3.0, 3.0], np.float32)         # sqrt(var + 1) = 2
    mean = np.array([1.0, -4.0], np.float32)
    beta = np.array([0.5, -1.0], np.float32)
    Wf, bf = oracle_mod.fold_batchnorm("f16", f16_bits(W), f16_bits(b), gamma, beta, mean, var,
                                       1.0)
    s = np.array([2.0, 0.5])
    assert np.array_equal(oracle_mod.decode("f16", Wf), W * s[:, None, None, None])
    assert np.array_equal(oracle_mod.decode("f16", bf), (b - mean) * s + beta)


def test_fold_batchnorm_equals_conv_then_batchnorm(oracle_mod):
    # conv with folded weights and bias == batch norm applied to the conv's fp64 output,
    # up to the rounding of the folded weights to fp16 (checked in float64 by torch)
    rng = np.random.default_rng(41)
    x = oracle_mod.decode("f16", f16_bits(rng.uniform(-1, 1, (1, 6, 5, 8))))
    W = oracle_mod.decode("f16", f16_bits(rng.normal(0, 0.3, (4, 3, 3, 8))))
    b = oracle_mod.decode("f16", f16_bits(rng.uniform(-0.1, 0.1, (4,))))
    gamma = rng.uniform(0.5, 2.0, 4).astype(np.float32)
    beta = rng.uniform(-0.5, 0.5, 4).astype(np.float32)
    mean = rng.uniform(-0.2, 0.2, 4).astype(np.float32)
    var = rng.uniform(0.5, 2.0, 4).astype(np.float32)
    eps = 1e-5
    Wf, bf = oracle_mod.fold_batchnorm("f16", f16_bits(W), f16_bits(b), gamma, beta, mean, var,
                                       eps)
    z = _torch_conv_nhwc(x, W, b, 1)
    bn = (z - mean) * (gamma / np.sqrt(var.astype(np.float64) + eps)) + beta
    folded = _torch_conv_nhwc(x, oracle_mod.decode("f16", Wf), oracle_mod.decode("f16", bf), 1)
    assert np.max(np.abs(folded - bn)) < 2e-2 * max(1.0, np.max(np.abs(bn)))
    # each folded weight is the nearest fp16 value of the exact product
    s = gamma.astype(np.float64) / np.sqrt(var.astype(np.float64) + eps)
    assert np.array_equal(Wf, f16_bits(W * s[:, None, None, None]))


def test_fold_batchnorm_layouts_agree(oracle_mod):
    # [Co][K] filters and [K][Co] row-major GEMM weights fold per output channel alike
    rng = np.random.default_rng(42)
    W = f16_bits(rng.normal(0, 1, (5, 12)))
    gamma, beta, mean, var = (rng.uniform(0.5, 1.5, 5).astype(np.float32) for _ in range(4))
    Wa, ba = oracle_mod.fold_batchnorm("f16", W, None, gamma, beta, mean, var, 1e-3)
    Wb, bb = oracle_mod.fold_batchnorm("f16", np.ascontiguousarray(W.T), None, gamma, beta, mean,
                                       var, 1e-3, out_inner=True)
    assert np.array_equal(Wa, Wb.T) and np.array_equal(ba, bb)
    assert np.array_equal(oracle_mod.decode("f16", ba), oracle_mod.decode(
        "f16", f16_bits(-mean.astype(np.float64) * gamma / np.sqrt(var.astype(np.float64) + 1e-3)
                        + beta)))


# ------------------------------------------------------------------------------------
# pooling chain
# ------------------------------------------------------------------------------------

@pytest.mark.parametrize("hw", [(4, 4), (6, 8), (7, 5), (5, 9)])
def test_maxpool_vs_torch(oracle_mod, hw):
    H, W = hw
    rng = np.random.default_rng(H * 31 + W)
    x = f16_bits(rng.uniform(-4, 4, (2, H, W, 8)))
    got = oracle_mod.decode("f16", oracle_mod.maxpool2x2_nhwc("f16", x))
    xt = torch.from_numpy(oracle_mod.decode("f16", x)).permute(0, 3, 1, 2)
    ref = F.max_pool2d(xt, 2, 2).permute(0, 2, 3, 1).numpy()       # floor mode
    assert got.shape == (2, H // 2, W // 2, 8)
    assert np.array_equal(got, ref)


def test_hand_4x4_pool(oracle_mod):
    x = np.array([[1, 5, 2, 0],
                  [3, 4, -1, 7],
                  [-2, -3, 6, 6],
                  [-4, -1, 0, -9]], dtype=np.float64).reshape(1, 4, 4, 1)
    got = oracle_mod.decode("f16", oracle_mod.maxpool2x2_nhwc("f16", f16_bits(x)))
    assert np.array_equal(got.reshape(2, 2), [[5, 7], [-1, 6]])


def test_pool_tile_from_page(oracle_mod):
    # Welder: MaxPool maps a 2x2xF tile to 1x1xF; Conv+ReLU+MaxPool has reuse tile
    # (2,2,F) and output (1,1,F): perturbing one conv output changes exactly one pooled
    # output, the one whose 2x2 window holds it.
    tiles = _read_tiles()
    assert tiles["maxpool2x2"] == (("2", "2", "F"), ("1", "1", "F"))
    assert tiles["conv_relu_maxpool.reuse"] == (("2", "2", "F"), ("1", "1", "F"))
    x = np.zeros((1, 6, 6, 2))
    base = oracle_mod.decode("f16", oracle_mod.maxpool2x2_nhwc("f16", f16_bits(x)))
    for (h, w) in [(0, 0), (3, 4), (5, 5), (2, 1)]:
        x2 = x.copy()
        x2[0, h, w, 1] = 1.0
        pert = oracle_mod.decode("f16", oracle_mod.maxpool2x2_nhwc("f16", f16_bits(x2)))
        diff = np.argwhere(pert != base)
        assert diff.tolist() == [[0, h // 2, w // 2, 1]]


def test_conv_relu_maxpool_pool_order_invariant(oracle_mod):
    # max commutes with the monotone maps "add b", ReLU and rounding, so
    # max_i rnd(relu(z_i + b)) == rnd(relu(max_i z_i + b)); the fused kernel uses the
    # right-hand side.  z is exact here (integer operands), computed by torch.
    rng = np.random.default_rng(11)
    N, H, W, C, Co = 2, 6, 8, 4, 3
    x = rng.integers(-3, 4, (N, H, W, C)).astype(np.float64)
    Wt = rng.integers(-3, 4, (Co, 3, 3, C)).astype(np.float64)
    b = np.array([0.5, -1.25, 3.0])
    got = oracle_mod.conv_relu_maxpool("f16", f16_bits(x), f16_bits(Wt), f16_bits(b))
    z = _torch_conv_nhwc(x, Wt, None, 1)
    zmax = z.reshape(N, H // 2, 2, W // 2, 2, Co).max(axis=(2, 4))
    ref = oracle_mod.encode("f16", np.maximum(zmax + b, 0.0))
    assert np.array_equal(got, ref)


def test_conv_relu_maxpool_odd_sizes_floor(oracle_mod):
    w = wl.ConvPool("t", "f16", 1, 7, 9, 8, 8)
    t = {k: wl.to_bits(v) for k, v in wl.pool_inputs(w, seed=12).items()}
    y = oracle_mod.conv_relu_maxpool("f16", t["x"], t["Wt"], t["b"])
    assert y.shape == (1, 3, 4, 8)
    c = oracle_mod.conv2d_nhwc("f16", t["x"], t["Wt"], t["b"], 1, "relu")
    assert np.array_equal(y, oracle_mod.maxpool2x2_nhwc("f16", c))


def test_alignment_rule_golden():
    vals = {}
    with open(os.path.join(GOLDEN, "alignment.txt")) as f:
        for line in f:
            line = line.split("#")[0].strip()
            if line:
                k, v = line.split()
                vals[k] = int(v)
    assert vals["elements"] * vals["element_bits"] == vals["vector_bits"] == 8 * vals["vector_bytes"]
