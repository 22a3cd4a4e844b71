"""Helpers shared by the GPU parity tests (not collected as tests).

Parity bar: integer-valued inputs (every product and partial sum an exact integer) must
match the oracle exactly; random inputs within |gpu - ref| <= 2e-2 * max(1, |ref|).
"""
import numpy as np
import torch

import oracle
from gemm_conv_chains_gb300 import ops
from gemm_conv_chains_gb300 import workloads as wl

RTOL = 2e-2


def to_dev(t):
    return None if t is None else t.cuda()


def check_no_device_error():
    st, info = ops.get_device_error()
    assert st == 0, f"device error word set: status {st}, info {info}"


def compare(dt, got_bits, ref_bits, exact, what=""):
    assert got_bits.shape == ref_bits.shape, (got_bits.shape, ref_bits.shape)
    g = oracle.decode(dt, got_bits)
    r = oracle.decode(dt, ref_bits)
    assert np.all(np.isfinite(g)), f"{what}: non-finite outputs"
    if exact:
        bad = g != r                      # by value: +0 == -0
        if bad.any():
            idx = np.argwhere(bad)
            raise AssertionError(f"{what}: {bad.sum()} of {bad.size} differ; first "
                                 f"{idx[:4].tolist()} got {g[bad][:4]} want {r[bad][:4]}")
        return 0.0
    err = np.abs(g - r)
    tol = RTOL * np.maximum(1.0, np.abs(r))
    bad = err > tol
    if bad.any():
        idx = np.argwhere(bad)
        raise AssertionError(f"{what}: {bad.sum()} of {bad.size} beyond tolerance; max err "
                             f"{err.max():.4g}; first {idx[:4].tolist()} got {g[bad][:4]} "
                             f"want {r[bad][:4]}")
    return float(err.max())


def run_b2b_gemm(w: wl.GemmChain, seed=0, integer=False, rows=None):
    """GPU b2b_gemm vs oracle; `rows` limits the oracle to a sample of rows."""
    t = wl.gemm_inputs(w, seed=seed, integer=integer)
    d = {k: to_dev(v) for k, v in t.items()}
    out = ops.b2b_gemm(d["A"], d["W0"], d["b0"], d["W1"], d["b1"], w.act0, w.act1)
    torch.cuda.synchronize()
    check_no_device_error()
    got = wl.to_bits(out.cpu())
    b = {k: wl.to_bits(v) for k, v in t.items()}
    A = b["A"] if rows is None else b["A"][rows]
    ref = oracle.b2b_gemm(w.dtype, A, b["W0"], b["b0"], b["W1"], b["b1"], w.act0, w.act1)
    return compare(w.dtype, got if rows is None else got[rows], ref, integer, w.name)
