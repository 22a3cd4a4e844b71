"""Batch normalisation folded into weights and bias on the GPU (b2b_fold_batchnorm) against
the oracle's fold, and a folded conv chain against the oracle chain on the same weights.

The kernel scales in fp32 and the oracle in double, each rounding once to the storage
type; a product that lands within an fp32 rounding of a tie may round the other way, so
the folded values must agree within one unit in the last place of the storage type, and
exactly when the scale is a power of two.
"""
import numpy as np
import pytest
import torch

import oracle
from gemm_conv_chains_gb300 import ops
from gemm_conv_chains_gb300 import workloads as wl

from gpu_util import check_no_device_error, compare

pytestmark = pytest.mark.gpu

DT = {"f16": torch.float16, "bf16": torch.bfloat16}


@pytest.fixture(autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    ops.lib()
    ops.get_device_error()


def _bn(Co, seed):
    g = torch.Generator().manual_seed(seed)
    gamma = torch.rand(Co, generator=g) * 1.5 + 0.5
    beta = torch.rand(Co, generator=g) - 0.5
    mean = (torch.rand(Co, generator=g) - 0.5) * 0.4
    var = torch.rand(Co, generator=g) * 1.5 + 0.5
    return gamma, beta, mean, var


def _ulp_close(dt, got, ref):
    g = oracle.decode(dt, got)
    r = oracle.decode(dt, ref)
    frac = 10 if dt == "f16" else 7
    ulp = np.exp2(np.floor(np.log2(np.maximum(np.abs(r), 2.0 ** -14))) - frac)
    assert np.all(np.abs(g - r) <= ulp), np.max(np.abs(g - r) / ulp)
    return float(np.mean(g == r))


@pytest.mark.parametrize("dt", ["f16", "bf16"])
@pytest.mark.parametrize("out_inner", [False, True])
def test_fold_matches_oracle(dt, out_inner):
    Co, K = 96, 3 * 3 * 40
    g = torch.Generator().manual_seed(7 + out_inner)
    W = (torch.randn((K, Co) if out_inner else (Co, 3, 3, 40), generator=g) * 0.2).to(DT[dt])
    b = (torch.rand(Co, generator=g) * 0.2 - 0.1).to(DT[dt])
    gamma, beta, mean, var = _bn(Co, 11)
    Wf, bf = ops.fold_batchnorm(W.cuda(), b.cuda(), *(v.cuda() for v in (gamma, beta, mean, var)),
                                eps=1e-5, out_inner=out_inner)
    torch.cuda.synchronize()
    check_no_device_error()
    rW, rb = oracle.fold_batchnorm(dt, wl.to_bits(W), wl.to_bits(b), gamma.numpy(), beta.numpy(),
                                   mean.numpy(), var.numpy(), 1e-5, out_inner=out_inner)
    assert _ulp_close(dt, wl.to_bits(Wf.cpu()), rW) > 0.99
    assert _ulp_close(dt, wl.to_bits(bf.cpu()), rb) > 0.9


def test_fold_power_of_two_scale_is_exact_and_in_place():
    Co, K = 16, 64
    W = torch.randn(Co, K, generator=torch.Generator().manual_seed(3)).to(torch.float16)
    b = torch.arange(Co, dtype=torch.float16)
    gamma = torch.full((Co,), 4.0)
    var = torch.full((Co,), 3.75)                  # sqrt(var + 0.25) = 2: s = 2
    mean = torch.linspace(-2, 2, Co)
    beta = torch.full((Co,), 0.5)
    Wd, bd = W.cuda(), b.cuda()
    ops.fold_batchnorm(Wd, bd, gamma.cuda(), beta.cuda(), mean.cuda(), var.cuda(), eps=0.25,
                       W_out=Wd, b_out=bd)          # in place
    torch.cuda.synchronize()
    assert torch.equal(Wd.cpu(), W * 2)
    assert torch.equal(bd.cpu(), ((b.float() - mean) * 2 + 0.5).to(torch.float16))


def test_folded_conv_chain():
    # the conv of a conv -> BN -> act block folded, then the fused chain on the folded
    # weights, against the oracle chain on the same folded weights
    w = wl.ConvChain("bn", "bf16", 2, 14, 14, 64, 64, 3, 3, 1, 128, "relu", "none")
    t = wl.conv_inputs(w, seed=21)
    gamma, beta, mean, var = _bn(w.C0, 22)
    dev = {k: v.cuda() for k, v in t.items()}
    W0f, b0f = ops.fold_batchnorm(dev["W0"], dev["b0"], gamma.cuda(), beta.cuda(), mean.cuda(),
                                  var.cuda())
    out = ops.b2b_conv_nhwc(dev["x"], W0f, b0f, dev["W1"], dev["b1"], 1, "relu", "none")
    torch.cuda.synchronize()
    check_no_device_error()
    bits = {k: wl.to_bits(v) for k, v in t.items()}
    ref = oracle.b2b_conv_nhwc("bf16", bits["x"], wl.to_bits(W0f.cpu()), wl.to_bits(b0f.cpu()),
                               bits["W1"], bits["b1"], 1, "relu", "none")
    compare("bf16", wl.to_bits(out.cpu()), ref, False, "folded conv chain")
