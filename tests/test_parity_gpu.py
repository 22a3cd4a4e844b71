"""GPU parity: every entry point of libb2b.so against the CPU oracle, element by element.

Shapes span several 128-row tiles with ragged tails, padded channel counts, odd spatial
sizes, both storage types and every epilogue.  Integer-valued cases must match exactly
(they pin layouts, swizzles, tap offsets, padding and pool windows bit for bit); random
cases must be within 2e-2 * max(1, |ref|).
"""
import numpy as np
import pytest
import torch

import oracle
from gemm_conv_chains_gb300 import ops
from gemm_conv_chains_gb300 import workloads as wl

from gpu_util import check_no_device_error, compare, run_b2b_gemm, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    ops.lib()
    ops.get_device_error()   # start from a clean error word


# ------------------------------------------------------------------------------------
# b2b GEMM
# ------------------------------------------------------------------------------------
GEMM_SHAPES = [
    # dtype, M, K0, N0, N1
    ("f16", 1, 64, 64, 64),
    ("f16", 300, 64, 64, 64),
    ("f16", 1000, 64, 64, 64),
    ("bf16", 513, 256, 256, 128),
    ("f16", 257, 72, 40, 24),
    ("bf16", 129, 8, 8, 8),
    ("f16", 640, 128, 128, 256),
    ("f16", 200, 320, 96, 200),
    ("bf16", 384, 64, 256, 256),
    # wide N0: the intermediate is kept in TMEM (checked by test_plan), D1 after P or,
    # for N1 > N0 / 2, past the end of D0
    ("f16", 300, 128, 256, 64),
    ("bf16", 257, 72, 200, 72),
    ("f16", 1000, 64, 224, 96),
    ("f16", 300, 128, 160, 128),
    ("bf16", 257, 72, 200, 120),
    ("f16", 640, 128, 144, 96),
    # 256 < N0 <= 512: GEMM0 in two passes over the halves of N0 (one tile per CTA here)
    ("bf16", 300, 128, 384, 64),
    ("f16", 257, 72, 264, 24),
    ("bf16", 1000, 256, 512, 128),
    ("bf16", 129, 64, 320, 96),
]


@pytest.mark.parametrize("shape", GEMM_SHAPES, ids=lambda s: "-".join(map(str, s)))
def test_b2b_gemm_integer_exact(shape):
    dt, M, K0, N0, N1 = shape
    for acts in (("relu", "none"), ("none", "relu")):
        w = wl.GemmChain("int", dt, M, K0, N0, N1, *acts)
        run_b2b_gemm(w, seed=M, integer=True)


@pytest.mark.parametrize("shape", GEMM_SHAPES, ids=lambda s: "-".join(map(str, s)))
def test_b2b_gemm_random(shape):
    dt, M, K0, N0, N1 = shape
    w = wl.GemmChain("rnd", dt, M, K0, N0, N1, "hardswish", "relu")
    run_b2b_gemm(w, seed=M + 1)


def test_b2b_gemm_without_bias():
    w = wl.GemmChain("nobias", "f16", 300, 64, 64, 64, "relu", "hardswish", bias=False)
    run_b2b_gemm(w, seed=3)


def test_b2b_gemm_small_workload_full():
    run_b2b_gemm(wl.GEMM_SMALL, seed=0)


def test_b2b_gemm_ffn_workload_sampled_rows():
    # Full-size FFN-like chain in the benchmark's launch configuration; the oracle checks
    # a sample of rows (rows are independent) including the first and last tiles.
    w = wl.GEMM_FFN
    rng = np.random.default_rng(0)
    rows = np.unique(np.concatenate([np.arange(128), np.arange(w.M - 128, w.M),
                                     rng.choice(w.M, 1024, replace=False)]))
    run_b2b_gemm(w, seed=0, rows=rows)


@pytest.mark.parametrize("M", wl.FFN_SWEEP_M)
def test_b2b_gemm_ffn_sweep_sampled_rows(M):
    # The FFN-like chain over the M sweep 4096 .. 262144 (32 .. 2048 tiles; at 262144 every
    # CTA runs 13 or 14 tiles), in the benchmark's launch configuration.  The oracle checks
    # every tile of CTA 0 (tiles 0, G, 2G, ... for a grid of G CTAs), the last tile and a
    # random sample of rows.
    w = wl.GEMM_FFN.with_m(M)
    tiles = (M + 127) // 128
    grid = min(tiles, ops.num_sms())
    rng = np.random.default_rng(M)
    cta0 = np.concatenate([np.arange(128 * t, min(128 * t + 128, M)) for t in range(0, tiles, grid)])
    rows = np.unique(np.concatenate([cta0, np.arange(M - 128, M), rng.choice(M, 512, replace=False)]))
    run_b2b_gemm(w, seed=M + 7, rows=rows)


@pytest.mark.parametrize("integer", [True, False])
def test_b2b_gemm_narrow_four_buffers_sampled_rows(integer):
    # 64 -> 64 -> 64 keeps four tiles in flight (each epilogue group one tile ahead); with
    # 5 x SMs + 1 tiles CTA 0 cycles through the four buffers 1.5 times, the last tile ragged.
    nsm = ops.num_sms()
    M = 128 * nsm * 5 + 77
    acts = ("relu", "none") if integer else ("hardswish", "relu")
    w = wl.GemmChain("quad", "f16", M, 64, 64, 64, *acts)
    rng = np.random.default_rng(7)
    cta0 = np.concatenate([np.arange(128 * t, min(128 * t + 128, M)) for t in range(0, 5 * nsm + 1, nsm)])
    rows = np.unique(np.concatenate([cta0, rng.choice(M, 512, replace=False)]))
    run_b2b_gemm(w, seed=13, integer=integer, rows=rows)


@pytest.mark.parametrize("streamed", [False, True])
@pytest.mark.parametrize("integer", [True, False])
def test_b2b_gemm_wide_streamed_pairs_sampled_rows(integer, streamed):
    # K0 = 256, single CTAs with P in TMEM: with `streamed` both weights stream (W0 with
    # every tile's A chunks); else W0 (128 KiB) stays resident and A and W1 stream through
    # the ring, the output leaving from registers.  Both layouts are pinned (the model
    # takes CTA pairs at this size).  3 x SMs + 1 tiles give CTA 0 two tile pairs, the
    # second with one ragged tile.
    nsm = ops.num_sms()
    M = 128 * nsm * 3 + 77
    dims = (M, 256, 256, 128)
    n = ops.debug_plan("b2b_gemm", dims, cand=0)["ncand"]
    want = dict(p_tmem=1, resident=0, cta_pair=0, w0_res=0 if streamed else 1)
    cand = next(c for c in range(n)
                if all(ops.debug_plan("b2b_gemm", dims, cand=c)[k] == v for k, v in want.items()))
    ops.set_choice("b2b_gemm", dims, cand=cand)
    try:
        acts = ("relu", "none") if integer else ("hardswish", "hardswish")   # exact: no fractions
        w = wl.GemmChain("spairs", "bf16", M, 256, 256, 128, *acts)
        rng = np.random.default_rng(6)
        cta0 = np.concatenate([np.arange(128 * t, min(128 * t + 128, M))
                               for t in range(0, 3 * nsm + 1, nsm)])
        rows = np.unique(np.concatenate([cta0, rng.choice(M, 512, replace=False)]))
        run_b2b_gemm(w, seed=12, integer=integer, rows=rows)
    finally:
        ops.autotune_reset()


@pytest.mark.parametrize("integer", [True, False])
def test_b2b_gemm_wide_many_pairs_sampled_rows(integer):
    # N0 = 256 keeps P in TMEM and processes tiles in pairs on single CTAs (pinned: the
    # model takes CTA pairs at this size); with 5 x SMs + 1 tiles, CTA 0 runs three pairs,
    # the last with one ragged tile.  Rows of every tile of CTA 0 plus a random sample.
    nsm = ops.num_sms()
    M = 128 * nsm * 5 + 77
    dims = (M, 64, 256, 128)
    n = ops.debug_plan("b2b_gemm", dims, cand=0)["ncand"]
    cand = next(c for c in range(n) if ops.debug_plan("b2b_gemm", dims, cand=c)["p_tmem"] == 1
                and ops.debug_plan("b2b_gemm", dims, cand=c)["cta_pair"] == 0)
    ops.set_choice("b2b_gemm", dims, cand=cand)
    try:
        acts = ("relu", "none") if integer else ("hardswish", "relu")   # exact: no fractions
        w = wl.GemmChain("pairs", "bf16", M, 64, 256, 128, *acts)
        rng = np.random.default_rng(5)
        cta0 = np.concatenate([np.arange(128 * t, min(128 * t + 128, M))
                               for t in range(0, 5 * nsm + 1, nsm)])
        rows = np.unique(np.concatenate([cta0, rng.choice(M, 512, replace=False)]))
        run_b2b_gemm(w, seed=11, integer=integer, rows=rows)
    finally:
        ops.autotune_reset()


# ------------------------------------------------------------------------------------
# single GEMM stage (unfused path)
# ------------------------------------------------------------------------------------
@pytest.mark.parametrize("shape", [("f16", 300, 64, 64), ("bf16", 513, 256, 256),
                                   ("f16", 130, 24, 40), ("f16", 1, 8, 8)],
                         ids=lambda s: "-".join(map(str, s)))
@pytest.mark.parametrize("integer", [True, False])
def test_gemm_bias_act(shape, integer):
    dt, M, K, N = shape
    w = wl.GemmChain("g", dt, M, K, N, 8, "relu" if integer else "hardswish", "none")
    t = wl.gemm_inputs(w, seed=M, integer=integer)
    out = ops.gemm_bias_act(to_dev(t["A"]), to_dev(t["W0"]), to_dev(t["b0"]), w.act0)
    torch.cuda.synchronize()
    check_no_device_error()
    ref = oracle.gemm_bias_act(dt, wl.to_bits(t["A"]), wl.to_bits(t["W0"]), wl.to_bits(t["b0"]),
                               w.act0)
    compare(dt, wl.to_bits(out.cpu()), ref, integer, "gemm_bias_act")


@pytest.mark.parametrize("dt,K0,N0,N1", [("bf16", 256, 512, 128), ("f16", 72, 264, 24),
                                         ("bf16", 128, 384, 64)])
def test_b2b_gemm_wide_n0_sampled_rows(dt, K0, N0, N1):
    # 256 < N0 <= 512 over 40000 rows (313 tiles): every CTA runs two or three tiles, which
    # alternate the half of N0 computed first; the rows sampled cover first tiles (lower
    # half first), CTA 4's second tile (upper half first) and third tiles.  N0 = 264 loads
    # W0 one 64-wide block at a time with a one-block upper half; 384 a four-block box
    # whose upper half is half out of bounds.
    w = wl.GemmChain(f"wide{N0}", dt, 40000, K0, N0, N1, "hardswish", "relu", a_dist="normal")
    run_b2b_gemm(w, seed=17, rows=np.r_[0:512, 20000:20128, 39744:40000])


# ------------------------------------------------------------------------------------
# three-operator chain (BOLT notes, "Enabling deeper operator fusion")
# ------------------------------------------------------------------------------------
GEMM3_SHAPES = [
    # dtype, M, K0, N0, N1, N2
    ("f16", 1, 64, 64, 64, 64),
    ("bf16", 1000, 64, 64, 64, 64),
    ("f16", 257, 72, 40, 24, 96),        # padded widths, ragged rows
    ("bf16", 129, 8, 8, 8, 8),
    ("f16", 40000, 128, 128, 64, 64),    # 313 tiles: pairs and an odd last tile per CTA
    ("bf16", 300, 128, 96, 64, 64),
]


def run_gemm3(shape, acts, integer, seed, rows=None):
    dt, M, K0, N0, N1, N2 = shape
    w = wl.GemmChain3("g3", dt, M, K0, N0, N1, N2, *acts)
    t = wl.gemm3_inputs(w, seed=seed, integer=integer)
    out = ops.b2b_gemm3(*(to_dev(t[k]) for k in ("A", "W0", "b0", "W1", "b1", "W2", "b2")), *acts)
    torch.cuda.synchronize()
    check_no_device_error()
    b = {k: wl.to_bits(v) for k, v in t.items()}
    sel = slice(None) if rows is None else rows
    ref = oracle.b2b_gemm3(dt, b["A"][sel], b["W0"], b["b0"], b["W1"], b["b1"], b["W2"], b["b2"],
                           *acts)
    return compare(dt, wl.to_bits(out.cpu())[sel], ref, integer, "b2b_gemm3")


@pytest.mark.parametrize("shape", GEMM3_SHAPES, ids=lambda s: "-".join(map(str, s)))
def test_b2b_gemm3_integer_exact(shape):
    rows = np.r_[0:600, 39400:40000] if shape[1] > 5000 else None
    run_gemm3(shape, ("relu", "relu", "none"), True, seed=shape[1] + 3, rows=rows)


@pytest.mark.parametrize("shape", GEMM3_SHAPES, ids=lambda s: "-".join(map(str, s)))
def test_b2b_gemm3_random(shape):
    rows = np.r_[0:600, 19000:19300, 39400:40000] if shape[1] > 5000 else None
    run_gemm3(shape, ("hardswish", "relu", "hardswish"), False, seed=shape[1] + 4, rows=rows)


def test_mlp3_workload_sampled_rows():
    w = wl.MLP3
    run_gemm3(("bf16", w.M, w.K0, w.N0, w.N1, w.N2), (w.act0, w.act1, w.act2), False, seed=0,
              rows=np.r_[0:256, 16000:16128, w.M - 256:w.M])


# ------------------------------------------------------------------------------------
# b2b conv
# ------------------------------------------------------------------------------------
CONV_SHAPES = [
    # dtype, N, H, W, C, C0, R, S, pad, C1
    ("f16", 2, 9, 9, 64, 64, 3, 3, 1, 128),
    ("f16", 1, 17, 20, 16, 24, 3, 3, 1, 8),
    ("bf16", 2, 8, 16, 64, 64, 3, 3, 1, 64),
    ("f16", 1, 11, 13, 128, 64, 3, 3, 0, 64),
    ("f16", 1, 10, 12, 32, 32, 5, 5, 2, 16),
    ("f16", 2, 7, 9, 64, 64, 1, 1, 0, 64),     # the 1x1 path (GEMM over pixels)
    ("f16", 1, 6, 6, 16, 16, 1, 3, 1, 16),     # non-square filter, wider output
    ("bf16", 1, 5, 5, 8, 8, 1, 1, 1, 8),       # 1x1 with padding: zero border rows
    ("bf16", 16, 30, 44, 64, 64, 3, 3, 1, 32),  # 192 ragged tiles: both MMA issuers busy
]


def run_conv(dt, N, H, W, C, C0, R, S, pad, C1, act0, act1, integer, seed, stride=1):
    w = wl.ConvChain("c", dt, N, H, W, C, C0, R, S, pad, C1, act0, act1, stride=stride)
    t = wl.conv_inputs(w, seed=seed, integer=integer)
    args = [to_dev(t[k]) for k in ("x", "W0", "b0", "W1", "b1")]
    if stride == 1:
        out = ops.b2b_conv_nhwc(*args, pad, act0, act1)
    else:
        out = ops.b2b_conv_nhwc_strided(*args, pad, stride, act0, act1)
    torch.cuda.synchronize()
    check_no_device_error()
    assert out.shape == (N, w.Ho, w.Wo, C1)
    b = {k: wl.to_bits(v) for k, v in t.items()}
    ref = oracle.b2b_conv_nhwc(dt, b["x"], b["W0"], b["b0"], b["W1"], b["b1"], pad, act0, act1,
                               stride=stride)
    return compare(dt, wl.to_bits(out.cpu()), ref, integer, "b2b_conv_nhwc")


@pytest.mark.parametrize("shape", CONV_SHAPES, ids=lambda s: "-".join(map(str, s)))
def test_b2b_conv_integer_exact(shape):
    run_conv(*shape, "relu", "none", True, seed=sum(shape[1:]))


@pytest.mark.parametrize("shape", CONV_SHAPES, ids=lambda s: "-".join(map(str, s)))
def test_b2b_conv_random(shape):
    run_conv(*shape, "hardswish", "none", False, seed=sum(shape[1:]) + 1)


@pytest.mark.parametrize("shape", [("f16", 2, 9, 9, 64, 64, 3, 3, 1), ("f16", 1, 7, 5, 16, 24, 3, 3, 1),
                                   ("f16", 2, 6, 6, 64, 64, 1, 1, 0)],
                         ids=lambda s: "-".join(map(str, s)))
@pytest.mark.parametrize("integer", [True, False])
def test_conv_bias_act(shape, integer):
    dt, N, H, W, C, Co, R, S, pad = shape
    w = wl.ConvChain("c", dt, N, H, W, C, Co, R, S, pad, 8, "relu", "none")
    t = wl.conv_inputs(w, seed=H * W, integer=integer)
    act = "relu" if integer else "hardswish"
    out = ops.conv_bias_act_nhwc(to_dev(t["x"]), to_dev(t["W0"]), to_dev(t["b0"]), pad, act)
    torch.cuda.synchronize()
    check_no_device_error()
    ref = oracle.conv2d_nhwc(dt, wl.to_bits(t["x"]), wl.to_bits(t["W0"]), wl.to_bits(t["b0"]),
                             pad, act)
    compare(dt, wl.to_bits(out.cpu()), ref, integer, "conv_bias_act_nhwc")


# strided first conv (Welder notes, tile propagation: a strided conv's input region)
STRIDED_SHAPES = [
    # dtype, N, H, W, C, C0, R, S, pad, C1, stride
    ("f16", 2, 9, 9, 64, 64, 3, 3, 1, 128, 2),       # resident filters, ragged 5 x 5 output
    ("bf16", 1, 17, 35, 16, 24, 3, 3, 1, 8, 2),      # narrow channels, two tile columns
    ("f16", 2, 28, 28, 64, 128, 1, 1, 0, 64, 2),     # strided 1x1 (a projection shortcut)
    ("f16", 1, 23, 19, 32, 32, 5, 5, 2, 16, 3),
    ("f16", 1, 30, 40, 64, 64, 3, 3, 1, 64, 4),
    ("f16", 2, 56, 56, 64, 128, 3, 3, 1, 128, 2),    # streamed filters (the workload's layers)
]


@pytest.mark.parametrize("shape", STRIDED_SHAPES, ids=lambda s: "-".join(map(str, s)))
def test_strided_conv_integer_exact(shape):
    run_conv(*shape[:10], "relu", "none", True, seed=sum(shape[1:]) + 5, stride=shape[10])


@pytest.mark.parametrize("shape", STRIDED_SHAPES, ids=lambda s: "-".join(map(str, s)))
def test_strided_conv_random(shape):
    run_conv(*shape[:10], "hardswish", "relu", False, seed=sum(shape[1:]) + 6, stride=shape[10])


@pytest.mark.parametrize("shape", [("f16", 2, 9, 9, 64, 64, 3, 3, 1, 2),
                                   ("bf16", 1, 14, 20, 16, 8, 1, 1, 0, 2),
                                   ("f16", 1, 13, 13, 32, 24, 3, 3, 1, 3)],
                         ids=lambda s: "-".join(map(str, s)))
@pytest.mark.parametrize("integer", [True, False])
def test_strided_conv_bias_act(shape, integer):
    dt, N, H, W, C, Co, R, S, pad, st = shape
    w = wl.ConvChain("c", dt, N, H, W, C, Co, R, S, pad, 8, "relu", "none", stride=st)
    t = wl.conv_inputs(w, seed=H * W + st, integer=integer)
    act = "relu" if integer else "hardswish"
    out = ops.conv_bias_act_nhwc_strided(to_dev(t["x"]), to_dev(t["W0"]), to_dev(t["b0"]), pad,
                                         st, act)
    torch.cuda.synchronize()
    check_no_device_error()
    ref = oracle.conv2d_nhwc(dt, wl.to_bits(t["x"]), wl.to_bits(t["W0"]), wl.to_bits(t["b0"]),
                             pad, act, stride=st)
    compare(dt, wl.to_bits(out.cpu()), ref, integer, "conv_bias_act_nhwc_strided")


def test_conv3x3s2_1x1_workload_sampled_images():
    w = wl.CONV3X3S2_1X1
    t = wl.conv_inputs(w, seed=0)
    out = ops.b2b_conv_nhwc_strided(*(to_dev(t[k]) for k in ("x", "W0", "b0", "W1", "b1")),
                                    w.pad, w.stride, w.act0, w.act1)
    torch.cuda.synchronize()
    check_no_device_error()
    b = {k: wl.to_bits(v) for k, v in t.items()}
    got = wl.to_bits(out.cpu())
    for n in (0, 17, w.N - 1):
        ref = oracle.b2b_conv_nhwc(w.dtype, b["x"][n:n + 1], b["W0"], b["b0"], b["W1"], b["b1"],
                                   w.pad, w.act0, w.act1, stride=w.stride)
        compare(w.dtype, got[n:n + 1], ref, False, f"conv3x3s2_1x1 image {n}")


def test_conv1x1_workload_sampled_images():
    w = wl.CONV1X1
    t = wl.conv_inputs(w, seed=0)
    out = ops.b2b_conv_nhwc(*(to_dev(t[k]) for k in ("x", "W0", "b0", "W1", "b1")), w.pad,
                            w.act0, w.act1)
    torch.cuda.synchronize()
    check_no_device_error()
    b = {k: wl.to_bits(v) for k, v in t.items()}
    got = wl.to_bits(out.cpu())
    for n in (0, 37, w.N - 1):
        ref = oracle.b2b_conv_nhwc(w.dtype, b["x"][n:n + 1], b["W0"], b["b0"], b["W1"], b["b1"],
                                   w.pad, w.act0, w.act1)
        compare(w.dtype, got[n:n + 1], ref, False, f"conv1x1 image {n}")


def test_conv3x3_1x1_workload_sampled_images():
    w = wl.CONV3X3_1X1
    t = wl.conv_inputs(w, seed=0)
    out = ops.b2b_conv_nhwc(*(to_dev(t[k]) for k in ("x", "W0", "b0", "W1", "b1")), w.pad,
                            w.act0, w.act1)
    torch.cuda.synchronize()
    check_no_device_error()
    b = {k: wl.to_bits(v) for k, v in t.items()}
    got = wl.to_bits(out.cpu())
    for n in (0, w.N - 1):
        ref = oracle.b2b_conv_nhwc(w.dtype, b["x"][n:n + 1], b["W0"], b["b0"], b["W1"], b["b1"],
                                   w.pad, w.act0, w.act1)
        compare(w.dtype, got[n:n + 1], ref, False, f"conv3x3_1x1 image {n}")


# ------------------------------------------------------------------------------------
# conv + ReLU + maxpool
# ------------------------------------------------------------------------------------
POOL_SHAPES = [
    # dtype, N, H, W, Cin, Cout
    ("f16", 2, 16, 16, 64, 64),
    ("f16", 1, 7, 9, 16, 8),
    ("bf16", 1, 20, 34, 32, 64),
    ("f16", 1, 2, 2, 8, 8),
    ("f16", 2, 18, 40, 64, 128),
]


def run_pool(dt, N, H, W, Cin, Cout, integer, seed):
    w = wl.ConvPool("p", dt, N, H, W, Cin, Cout)
    t = wl.pool_inputs(w, seed=seed, integer=integer)
    out = ops.conv_relu_maxpool(to_dev(t["x"]), to_dev(t["Wt"]), to_dev(t["b"]))
    torch.cuda.synchronize()
    check_no_device_error()
    ref = oracle.conv_relu_maxpool(dt, wl.to_bits(t["x"]), wl.to_bits(t["Wt"]), wl.to_bits(t["b"]))
    return compare(dt, wl.to_bits(out.cpu()), ref, integer, "conv_relu_maxpool")


@pytest.mark.parametrize("shape", POOL_SHAPES, ids=lambda s: "-".join(map(str, s)))
def test_conv_relu_maxpool_integer_exact(shape):
    run_pool(*shape, True, seed=sum(shape[1:]))


@pytest.mark.parametrize("shape", POOL_SHAPES, ids=lambda s: "-".join(map(str, s)))
def test_conv_relu_maxpool_random(shape):
    run_pool(*shape, False, seed=sum(shape[1:]) + 1)


POOL_PAIR_SHAPES = [
    # dtype, N, H, W, Cin, Cout over CTA pairs: an odd tile count (the last pair-tile's
    # second tile empty), ragged tiles, N0 = 16 / 48 / 128, partial channel blocks, pairs
    # with many pair-tiles (every MMA issuer busy); three issuers (Cout <= 64, one channel
    # block: nine or ten ring stages, ten split 4 + 3 + 3), two (Cout = 128: four
    # accumulators fill TMEM) and one (Cin = 128: six stages per tile)
    ("f16", 1, 16, 16, 64, 64), ("f16", 3, 18, 20, 16, 48), ("bf16", 2, 32, 48, 64, 128),
    ("f16", 1, 14, 30, 8, 16), ("bf16", 5, 36, 40, 64, 64), ("f16", 24, 56, 56, 64, 64),
    ("f16", 2, 17, 33, 128, 64),
]


@pytest.mark.parametrize("shape", POOL_PAIR_SHAPES, ids=lambda s: "-".join(map(str, s)))
@pytest.mark.parametrize("integer", [True, False])
def test_conv_relu_maxpool_cta_pair(shape, integer):
    # the pair layout (pinned) against the oracle and against the single-CTA layout: the
    # same products in the same order, but the pair adds the bias in fp32 after the sums
    # (the single-CTA kernel as a last MMA step), so the two agree bit for bit on integer
    # inputs (every sum exact) and within the tolerance otherwise
    dt, N, H, W, Cin, Cout = shape
    dims = (N, H, W, Cin, Cout)
    n = ops.debug_plan("conv_relu_maxpool", dims, cand=0)["ncand"]
    w = wl.ConvPool("p2", dt, N, H, W, Cin, Cout)
    t = wl.pool_inputs(w, seed=sum(dims) + integer, integer=integer)
    args = (to_dev(t["x"]), to_dev(t["Wt"]), to_dev(t["b"]))
    try:
        ops.set_choice("conv_relu_maxpool", dims, cand=0)
        assert ops.debug_plan("conv_relu_maxpool", dims)["cta_pair"] == 0
        single = ops.conv_relu_maxpool(*args)
        ops.set_choice("conv_relu_maxpool", dims, cand=n - 1)
        assert ops.debug_plan("conv_relu_maxpool", dims)["cta_pair"] == 1
        out = ops.conv_relu_maxpool(*args)
        torch.cuda.synchronize()
    finally:
        ops.autotune_reset()
    check_no_device_error()
    got = wl.to_bits(out.cpu())
    compare(dt, got, wl.to_bits(single.cpu()), integer, "conv_relu_maxpool pair vs single")
    b = {k: wl.to_bits(v) for k, v in t.items()}
    for i in sorted({0, N - 1}):
        ref = oracle.conv_relu_maxpool(dt, b["x"][i:i + 1], b["Wt"], b["b"])
        compare(dt, got[i:i + 1], ref, integer, f"conv_relu_maxpool pair image {i}")


def test_conv_pool_workload_sampled_images():
    w = wl.CONV_POOL
    t = wl.pool_inputs(w, seed=0)
    out = ops.conv_relu_maxpool(to_dev(t["x"]), to_dev(t["Wt"]), to_dev(t["b"]))
    torch.cuda.synchronize()
    check_no_device_error()
    got = wl.to_bits(out.cpu())
    b = {k: wl.to_bits(v) for k, v in t.items()}
    for n in (0, w.N - 1):
        ref = oracle.conv_relu_maxpool(w.dtype, b["x"][n:n + 1], b["Wt"], b["b"])
        compare(w.dtype, got[n:n + 1], ref, False, f"conv_pool image {n}")


@pytest.mark.parametrize("shape", [("f16", 2, 8, 8, 64), ("bf16", 1, 7, 9, 16), ("f16", 3, 2, 3, 8)])
def test_maxpool2x2(shape):
    dt, N, H, W, C = shape
    g = torch.Generator().manual_seed(H * W)
    x = (torch.rand((N, H, W, C), generator=g) * 8 - 4).to(wl.DTYPES[dt])
    out = ops.maxpool2x2_nhwc(x.cuda())
    torch.cuda.synchronize()
    ref = oracle.maxpool2x2_nhwc(dt, wl.to_bits(x))
    compare(dt, wl.to_bits(out.cpu()), ref, True, "maxpool2x2_nhwc")


# ------------------------------------------------------------------------------------
# unfused two-kernel path == fused chain (same tiles, same roundings)
# ------------------------------------------------------------------------------------
def test_unfused_gemm_chain_matches_fused_bitwise():
    w = wl.GemmChain("u", "bf16", 1000, 256, 256, 128, "hardswish", "hardswish", a_dist="normal")
    t = {k: to_dev(v) for k, v in wl.gemm_inputs(w, seed=4).items()}
    fused = ops.b2b_gemm(t["A"], t["W0"], t["b0"], t["W1"], t["b1"], w.act0, w.act1)
    h = ops.gemm_bias_act(t["A"], t["W0"], t["b0"], w.act0)
    unfused = ops.gemm_bias_act(h, t["W1"], t["b1"], w.act1)
    torch.cuda.synchronize()
    assert torch.equal(fused.view(torch.int16), unfused.view(torch.int16))


def test_unfused_conv_pool_matches_fused_bitwise():
    w = wl.ConvPool("u", "f16", 2, 16, 24, 64, 64)
    t = {k: to_dev(v) for k, v in wl.pool_inputs(w, seed=5).items()}
    fused = ops.conv_relu_maxpool(t["x"], t["Wt"], t["b"])
    c = ops.conv_bias_act_nhwc(t["x"], t["Wt"], t["b"], 1, "relu")
    unfused = ops.maxpool2x2_nhwc(c)
    torch.cuda.synchronize()
    assert torch.equal(fused.float(), unfused.float())


# ------------------------------------------------------------------------------------
# empty problems, failure detection
# ------------------------------------------------------------------------------------
def test_empty_problems_launch_nothing():
    A = torch.empty((0, 64), dtype=torch.float16, device="cuda")
    W = torch.zeros((64, 64), dtype=torch.float16, device="cuda")
    assert ops.b2b_gemm(A, W, None, W, None).shape == (0, 64)
    x = torch.empty((0, 8, 8, 64), dtype=torch.float16, device="cuda")
    Wt = torch.zeros((64, 3, 3, 64), dtype=torch.float16, device="cuda")
    assert ops.conv_relu_maxpool(x, Wt, None).shape == (0, 4, 4, 64)


def test_timeout_path_reports_and_context_survives():
    ops.get_device_error()
    ops.probe_timeout(20_000_000)            # 20 ms on a barrier nothing signals
    st, info = ops.get_device_error()
    assert st == 6 and info[0] == 6 and info[1] == 15, (st, info)
    assert ops.get_device_error()[0] == 0    # read-and-clear
    run_b2b_gemm(wl.GemmChain("after", "f16", 200, 64, 64, 64, "relu", "none"), integer=True)


# ------------------------------------------------------------------------------------
# the chain over CTA pairs (clusters of two CTAs sharing each 256-row MMA)
# ------------------------------------------------------------------------------------
def _pin_cta_pair(dims):
    n = ops.debug_plan("b2b_gemm", dims)["ncand"]
    ops.set_choice("b2b_gemm", dims, cand=n - 1)
    assert ops.debug_plan("b2b_gemm", dims)["cta_pair"] == 1


CTA_PAIR_SHAPES = [
    # dtype, M, K0, N0, N1
    ("bf16", 513, 256, 256, 128),     # three 256-row tiles, the last one's second CTA idle
    ("f16", 300, 64, 128, 128),
    ("bf16", 129, 8, 128, 128),       # one tile, ragged inside the first CTA
    ("f16", 1000, 448, 256, 128),     # seven K chunks of W0 (four ring stages)
    ("bf16", 700, 200, 128, 128),     # a partial last K chunk
]


@pytest.mark.parametrize("shape", CTA_PAIR_SHAPES, ids=lambda s: "-".join(map(str, s)))
@pytest.mark.parametrize("integer", [True, False])
def test_b2b_gemm_cta_pair(shape, integer):
    dt, M, K0, N0, N1 = shape
    _pin_cta_pair((M, K0, N0, N1))
    try:
        acts = ("relu", "none") if integer else ("hardswish", "relu")
        w = wl.GemmChain("cta2", dt, M, K0, N0, N1, *acts, a_dist="normal")
        run_b2b_gemm(w, seed=M + K0, integer=integer)
    finally:
        ops.autotune_reset()


@pytest.mark.parametrize("integer", [True, False])
def test_b2b_gemm_cta_pair_many_tiles_sampled_rows(integer):
    # 5 x SMs + 1 tiles of 128 rows: each pair runs five or six 256-row tiles (both TMEM
    # buffers reused), the last one ragged; rows of every tile of the first pair
    nsm = ops.num_sms()
    M = 128 * nsm * 5 + 77
    dims = (M, 256, 256, 128)
    _pin_cta_pair(dims)
    try:
        acts = ("relu", "none") if integer else ("hardswish", "hardswish")
        w = wl.GemmChain("cta2many", "bf16", M, 256, 256, 128, *acts, a_dist="normal")
        pairs = ops.debug_plan("b2b_gemm", dims)["tiles"]
        rng = np.random.default_rng(9)
        npairs_max = nsm // 2
        first = np.concatenate([np.arange(256 * t, min(256 * t + 256, M))
                                for t in range(0, pairs, npairs_max)])
        rows = np.unique(np.concatenate([first, np.arange(M - 256, M),
                                         rng.choice(M, 512, replace=False)]))
        run_b2b_gemm(w, seed=21, integer=integer, rows=rows)
    finally:
        ops.autotune_reset()
