"""Channel padding and memory guards on the GPU, through the C ABI.

Padding (BOLT notes, "Templated code generation", with the errata note: tensors padded
to 8 fp16 elements): channel counts that are not multiples of 8 are zero-padded with
ops.pad_channels; the padded problem's outputs must equal the oracle on the UNPADDED
problem in the real channels and be exactly 0 in the padded ones (zero inputs, weights
and biases give act(0) = 0 for every epilogue).

Guards: every output is written into the middle of a larger buffer whose slack is filled
with the byte 0x7E, checked unchanged after the call (no write outside the output);
every input sits in the middle of a buffer whose slack holds 0xFF bytes, a NaN in both
fp16 and bf16, so that a read outside an input would make an output non-finite, which
the comparison rejects.
"""
import numpy as np
import pytest
import torch

import oracle
from gemm_conv_chains_gb300 import ops
from gemm_conv_chains_gb300 import workloads as wl

from gpu_util import check_no_device_error, compare

pytestmark = pytest.mark.gpu

GUARD = 4096          # elements of slack on each side (8 KiB; keeps 16-byte alignment)
OUT_FILL = 0x7E
IN_FILL = 0xFF


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    ops.lib()
    ops.get_device_error()


def _guarded(shape, dtype, fill, src=None):
    """(buffer, view): `view` of `shape` in the middle of `buffer`, the slack set to `fill`."""
    n = int(np.prod(shape))
    buf = torch.empty(GUARD + n + GUARD, dtype=dtype, device="cuda")
    buf.view(torch.uint8).fill_(fill)
    view = buf[GUARD:GUARD + n].view(shape)
    if src is not None:
        view.copy_(src)
    assert view.data_ptr() % 16 == 0
    return buf, view


def _slack_intact(buf, n, fill, what):
    b = buf.view(torch.uint8).cpu().numpy()
    e = buf.element_size()
    lo, hi = b[:GUARD * e], b[(GUARD + n) * e:]
    assert np.all(lo == fill) and np.all(hi == fill), f"{what}: bytes outside the output changed"


def _inputs_guarded(tensors):
    """Copies each CPU tensor (None passes through) into the middle of a NaN-guarded buffer."""
    keep, views = [], []
    for t in tensors:
        if t is None:
            views.append(None)
            continue
        buf, v = _guarded(tuple(t.shape), t.dtype, IN_FILL, t.cuda())
        keep.append(buf)
        views.append(v)
    return keep, views


# ------------------------------------------------------------------------------------
# padded channels
# ------------------------------------------------------------------------------------
@pytest.mark.parametrize("dt", ["f16", "bf16"])
@pytest.mark.parametrize("integer", [True, False])
def test_b2b_gemm_padded_channels(dt, integer):
    # K0 3 -> 8, N0 20 -> 24, N1 60 -> 64 over 300 rows (three tiles, the last ragged)
    w = wl.GemmChain("pad", dt, 300, 3, 20, 60, "relu" if integer else "hardswish",
                     "none" if integer else "relu")
    t = wl.gemm_inputs(w, seed=21, integer=integer)
    pc = ops.pad_channels
    A = pc(t["A"], 1)
    W0 = pc(pc(t["W0"], 0), 1)
    b0 = pc(t["b0"], 0)
    W1 = pc(pc(t["W1"], 0), 1)
    b1 = pc(t["b1"], 0)
    assert A.shape == (300, 8) and W0.shape == (8, 24) and W1.shape == (24, 64)
    out = ops.b2b_gemm(*(x.cuda() for x in (A, W0, b0, W1, b1)), w.act0, w.act1)
    torch.cuda.synchronize()
    check_no_device_error()
    got = wl.to_bits(out.cpu())
    b = {k: wl.to_bits(v) for k, v in t.items()}
    ref = oracle.b2b_gemm(dt, b["A"], b["W0"], b["b0"], b["W1"], b["b1"], w.act0, w.act1)
    compare(dt, np.ascontiguousarray(got[:, :60]), ref, integer, "b2b_gemm padded")
    assert np.all(oracle.decode(dt, got[:, 60:]) == 0.0), "padded output channels not zero"


@pytest.mark.parametrize("integer", [True, False])
def test_b2b_conv_padded_channels(integer):
    # Cin 3 -> 8, C0 20 -> 24, C1 60 -> 64; 3x3 conv, odd spatial sizes
    w = wl.ConvChain("pad", "f16", 2, 11, 19, 3, 20, 3, 3, 1, 60,
                     "relu" if integer else "hardswish", "none")
    t = wl.conv_inputs(w, seed=22, integer=integer)
    pc = ops.pad_channels
    x = pc(t["x"], 3)
    W0 = pc(pc(t["W0"], 0), 3)
    b0 = pc(t["b0"], 0)
    W1 = pc(pc(t["W1"], 0), 1)
    b1 = pc(t["b1"], 0)
    assert x.shape[3] == 8 and W0.shape == (24, 3, 3, 8) and W1.shape == (64, 24)
    out = ops.b2b_conv_nhwc(*(v.cuda() for v in (x, W0, b0, W1, b1)), w.pad, w.act0, w.act1)
    torch.cuda.synchronize()
    check_no_device_error()
    got = wl.to_bits(out.cpu())
    b = {k: wl.to_bits(v) for k, v in t.items()}
    ref = oracle.b2b_conv_nhwc("f16", b["x"], b["W0"], b["b0"], b["W1"], b["b1"], w.pad, w.act0,
                               w.act1)
    compare("f16", np.ascontiguousarray(got[..., :60]), ref, integer, "b2b_conv_nhwc padded")
    assert np.all(oracle.decode("f16", got[..., 60:]) == 0.0), "padded output channels not zero"


@pytest.mark.parametrize("integer", [True, False])
def test_conv_relu_maxpool_padded_channels(integer):
    # Cin 3 -> 8, Cout 20 -> 24
    w = wl.ConvPool("pad", "f16", 2, 14, 22, 3, 20)
    t = wl.pool_inputs(w, seed=23, integer=integer)
    pc = ops.pad_channels
    x = pc(t["x"], 3)
    Wt = pc(pc(t["Wt"], 0), 3)
    bb = pc(t["b"], 0)
    out = ops.conv_relu_maxpool(x.cuda(), Wt.cuda(), bb.cuda())
    torch.cuda.synchronize()
    check_no_device_error()
    got = wl.to_bits(out.cpu())
    ref = oracle.conv_relu_maxpool("f16", wl.to_bits(t["x"]), wl.to_bits(t["Wt"]),
                                   wl.to_bits(t["b"]))
    compare("f16", np.ascontiguousarray(got[..., :20]), ref, integer, "conv_relu_maxpool padded")
    assert np.all(oracle.decode("f16", got[..., 20:]) == 0.0), "padded output channels not zero"


# ------------------------------------------------------------------------------------
# guard regions
# ------------------------------------------------------------------------------------
GUARD_GEMMS = [
    # dtype, M, K0, N0, N1: shared-memory P, P in TMEM with tile pairs, wide N0
    ("f16", 1000, 64, 64, 64),
    ("bf16", 128 * 152 * 2 + 77, 256, 256, 128),
    ("bf16", 300, 128, 384, 64),
    ("f16", 257, 72, 40, 24),
]


@pytest.mark.parametrize("shape", GUARD_GEMMS, ids=lambda s: "-".join(map(str, s)))
def test_b2b_gemm_guards(shape):
    _gemm_guarded(shape)


def _gemm_guarded(shape):
    dt, M, K0, N0, N1 = shape
    w = wl.GemmChain("guard", dt, M, K0, N0, N1, "hardswish", "relu", a_dist="normal")
    t = wl.gemm_inputs(w, seed=31)
    keep, (A, W0, b0, W1, b1) = _inputs_guarded([t[k] for k in ("A", "W0", "b0", "W1", "b1")])
    obuf, out = _guarded((M, N1), wl.DTYPES[dt], OUT_FILL)
    ops.b2b_gemm(A, W0, b0, W1, b1, w.act0, w.act1, out=out)
    torch.cuda.synchronize()
    check_no_device_error()
    _slack_intact(obuf, M * N1, OUT_FILL, "b2b_gemm")
    rows = np.unique(np.r_[0:128, M - 128:M, np.linspace(0, M - 1, 256).astype(int)])
    b = {k: wl.to_bits(v) for k, v in t.items()}
    ref = oracle.b2b_gemm(dt, b["A"][rows], b["W0"], b["b0"], b["W1"], b["b1"], w.act0, w.act1)
    compare(dt, wl.to_bits(out.cpu())[rows], ref, False, "b2b_gemm guarded")


@pytest.mark.parametrize("shape", [
    # dtype, M, K0, N0, N1 over CTA pairs: output staged per warp and stored with TMA (the
    # last tile's second CTA past M), and, with seven K chunks of W0, stored from registers
    ("bf16", 40000, 256, 256, 128), ("f16", 1000, 448, 256, 128), ("bf16", 700, 200, 128, 128)],
    ids=lambda s: "-".join(map(str, s)))
def test_b2b_gemm_cta_pair_guards(shape):
    dt, M, K0, N0, N1 = shape
    dims = (M, K0, N0, N1)
    n = ops.debug_plan("b2b_gemm", dims, cand=0)["ncand"]
    ops.set_choice("b2b_gemm", dims, cand=n - 1)
    try:
        assert ops.debug_plan("b2b_gemm", dims)["cta_pair"] == 1
        _gemm_guarded(shape)
    finally:
        ops.autotune_reset()


@pytest.mark.parametrize("shape", [("f16", 2, 9, 9, 64, 64, 3, 3, 1, 128),
                                   ("f16", 2, 7, 9, 64, 64, 1, 1, 0, 64),
                                   ("bf16", 1, 17, 20, 16, 24, 3, 3, 1, 8)],
                         ids=lambda s: "-".join(map(str, s)))
def test_b2b_conv_guards(shape):
    dt, N, H, W, C, C0, R, S, pad, C1 = shape
    w = wl.ConvChain("guard", dt, N, H, W, C, C0, R, S, pad, C1, "hardswish", "none")
    t = wl.conv_inputs(w, seed=32)
    keep, (x, W0, b0, W1, b1) = _inputs_guarded([t[k] for k in ("x", "W0", "b0", "W1", "b1")])
    oshape = (N, w.Ho, w.Wo, C1)
    obuf, out = _guarded(oshape, wl.DTYPES[dt], OUT_FILL)
    ops.b2b_conv_nhwc(x, W0, b0, W1, b1, pad, w.act0, w.act1, out=out)
    torch.cuda.synchronize()
    check_no_device_error()
    _slack_intact(obuf, int(np.prod(oshape)), OUT_FILL, "b2b_conv_nhwc")
    b = {k: wl.to_bits(v) for k, v in t.items()}
    ref = oracle.b2b_conv_nhwc(dt, b["x"], b["W0"], b["b0"], b["W1"], b["b1"], pad, w.act0, w.act1)
    compare(dt, wl.to_bits(out.cpu()), ref, False, "b2b_conv_nhwc guarded")


@pytest.mark.parametrize("shape", [("f16", 2, 16, 16, 64, 64), ("f16", 1, 7, 9, 16, 8),
                                   ("bf16", 1, 20, 34, 32, 64)],
                         ids=lambda s: "-".join(map(str, s)))
def test_conv_relu_maxpool_guards(shape):
    _pool_guarded(shape)


def _pool_guarded(shape):
    dt, N, H, W, Cin, Cout = shape
    w = wl.ConvPool("guard", dt, N, H, W, Cin, Cout)
    t = wl.pool_inputs(w, seed=33)
    keep, (x, Wt, bb) = _inputs_guarded([t[k] for k in ("x", "Wt", "b")])
    oshape = (N, H // 2, W // 2, Cout)
    obuf, out = _guarded(oshape, wl.DTYPES[dt], OUT_FILL)
    ops.conv_relu_maxpool(x, Wt, bb, out=out)
    torch.cuda.synchronize()
    check_no_device_error()
    _slack_intact(obuf, int(np.prod(oshape)), OUT_FILL, "conv_relu_maxpool")
    ref = oracle.conv_relu_maxpool(dt, wl.to_bits(t["x"]), wl.to_bits(t["Wt"]), wl.to_bits(t["b"]))
    compare(dt, wl.to_bits(out.cpu()), ref, False, "conv_relu_maxpool guarded")


@pytest.mark.parametrize("shape", [("f16", 1, 18, 20, 64, 64), ("bf16", 1, 20, 34, 32, 48)],
                         ids=lambda s: "-".join(map(str, s)))
def test_conv_relu_maxpool_cta_pair_guards(shape):
    # the pair layout: each CTA stores its own pooled tile (an odd tile count leaves the
    # last pair-tile's second tile empty: nothing stored past the output)
    dt, N, H, W, Cin, Cout = shape
    dims = (N, H, W, Cin, Cout)
    n = ops.debug_plan("conv_relu_maxpool", dims, cand=0)["ncand"]
    ops.set_choice("conv_relu_maxpool", dims, cand=n - 1)
    try:
        assert ops.debug_plan("conv_relu_maxpool", dims)["cta_pair"] == 1
        _pool_guarded(shape)
    finally:
        ops.autotune_reset()


def test_unfused_operators_guards():
    # the two-kernel path: GEMM stage, conv stage and the plain max-pool
    w = wl.GemmChain("g", "f16", 300, 64, 64, 8, "relu", "none")
    t = wl.gemm_inputs(w, seed=34)
    keep, (A, W0, b0) = _inputs_guarded([t["A"], t["W0"], t["b0"]])
    obuf, out = _guarded((300, 64), torch.float16, OUT_FILL)
    ops.gemm_bias_act(A, W0, b0, "relu", out=out)
    c = wl.ConvPool("p", "f16", 1, 9, 11, 16, 16)
    tp = wl.pool_inputs(c, seed=35)
    keep2, (x, Wt, bb) = _inputs_guarded([tp["x"], tp["Wt"], tp["b"]])
    cbuf, conv = _guarded((1, 9, 11, 16), torch.float16, OUT_FILL)
    ops.conv_bias_act_nhwc(x, Wt, bb, 1, "relu", out=conv)
    pbuf, pooled = _guarded((1, 4, 5, 16), torch.float16, OUT_FILL)
    ops.maxpool2x2_nhwc(conv, out=pooled)
    torch.cuda.synchronize()
    check_no_device_error()
    _slack_intact(obuf, 300 * 64, OUT_FILL, "gemm_bias_act")
    _slack_intact(cbuf, 9 * 11 * 16, OUT_FILL, "conv_bias_act_nhwc")
    _slack_intact(pbuf, 4 * 5 * 16, OUT_FILL, "maxpool2x2_nhwc")
    ref = oracle.gemm_bias_act("f16", wl.to_bits(t["A"]), wl.to_bits(t["W0"]), wl.to_bits(t["b0"]),
                               "relu")
    compare("f16", wl.to_bits(out.cpu()), ref, False, "gemm_bias_act guarded")
    ref = oracle.conv_relu_maxpool("f16", wl.to_bits(tp["x"]), wl.to_bits(tp["Wt"]),
                                   wl.to_bits(tp["b"]))
    compare("f16", wl.to_bits(pooled.cpu()), ref, False, "conv + maxpool guarded")
