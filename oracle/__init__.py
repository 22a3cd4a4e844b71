"""CPU oracle for the fused GEMM/conv chains -- TEST INFRASTRUCTURE ONLY.

Only the tests, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline leg may
import this package.  The product path (``gemm_conv_chains_gb300``) never imports it,
and this package imports nothing from the product path: the two share no code.

The arithmetic lives in ``oracle.c`` (plain C, single thread, double-precision sums,
one round-to-nearest-even into fp16/bf16 per stored tensor).  This module only builds
that file with gcc, loads it with ctypes and moves numpy arrays in and out.

Tensors cross this interface as numpy ``uint16`` arrays holding fp16/bf16 bit patterns,
so that the oracle and the GPU read identical bits.

Sources followed (page title, section):
  * BOLT notes -- "Persistent kernel (GEMM/Conv) fusion", "Threadblock residence",
    "Prerequisite: Epilogue fusion", "Graph Level" (Conv2D + BiasAdd + Hardswish);
  * Welder notes -- "Operator-tile and Tile-graph", "Tile-graph Scheduling" (Figure 5:
    Conv + ReLU + MaxPool, reuse tile (2,2,F) -> output (1,1,F));
  * AI Infra interview notes -- "Conv optimisation": im2col + GEMM, implicit GEMM,
    1x1 conv reduces to GEMM.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

F16 = 0
BF16 = 1
ACT_NONE = 0
ACT_RELU = 1
ACT_HARDSWISH = 2
ACTS = {"none": ACT_NONE, "relu": ACT_RELU, "hardswish": ACT_HARDSWISH}
DTYPES = {"f16": F16, "fp16": F16, "float16": F16, "bf16": BF16, "bfloat16": BF16}

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile oracle.c into liboracle.so next to it (gcc, no SIMD flags)."""
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-ffp-contract=off", "-fPIC", "-shared", "-std=c99",
           "-Wall", "-Wextra", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        build()
        lib = ctypes.CDLL(_LIB_PATH)
        u16p = ctypes.POINTER(ctypes.c_uint16)
        i64 = ctypes.c_int64
        ci = ctypes.c_int
        lib.oracle_decode.argtypes = [ci, ctypes.c_uint16]
        lib.oracle_decode.restype = ctypes.c_double
        lib.oracle_encode.argtypes = [ci, ctypes.c_double]
        lib.oracle_encode.restype = ctypes.c_uint16
        lib.oracle_decode_array.argtypes = [ci, i64, u16p, ctypes.POINTER(ctypes.c_double)]
        lib.oracle_decode_array.restype = None
        lib.oracle_encode_array.argtypes = [ci, i64, ctypes.POINTER(ctypes.c_double), u16p]
        lib.oracle_encode_array.restype = None
        lib.oracle_activation.argtypes = [ci, ctypes.c_double]
        lib.oracle_activation.restype = ctypes.c_double
        lib.oracle_gemm_bias_act.argtypes = [ci, i64, i64, i64, u16p, u16p, u16p, ci, u16p]
        lib.oracle_b2b_gemm.argtypes = [ci, i64, i64, i64, i64, u16p, u16p, u16p, ci,
                                        u16p, u16p, ci, u16p]
        lib.oracle_conv2d_nhwc.argtypes = [ci, i64, i64, i64, i64, u16p, i64, i64, i64, i64,
                                           u16p, u16p, ci, u16p]
        lib.oracle_maxpool2x2_nhwc.argtypes = [ci, i64, i64, i64, i64, u16p, u16p]
        lib.oracle_b2b_conv_nhwc.argtypes = [ci, i64, i64, i64, i64, u16p, u16p, i64, i64, i64,
                                             i64, u16p, ci, u16p, i64, u16p, ci, u16p]
        lib.oracle_conv_relu_maxpool.argtypes = [ci, i64, i64, i64, i64, u16p, u16p, u16p, i64,
                                                 u16p]
        lib.oracle_conv2d_nhwc_strided.argtypes = [ci, i64, i64, i64, i64, u16p, i64, i64, i64,
                                                   i64, i64, u16p, u16p, ci, u16p]
        lib.oracle_b2b_conv_nhwc_strided.argtypes = [ci, i64, i64, i64, i64, u16p, u16p, i64,
                                                     i64, i64, i64, i64, u16p, ci, u16p, i64,
                                                     u16p, ci, u16p]
        f32p = ctypes.POINTER(ctypes.c_float)
        lib.oracle_fold_batchnorm.argtypes = [ci, i64, i64, ci, u16p, u16p, f32p, f32p, f32p,
                                              f32p, ctypes.c_double, u16p, u16p]
        for name in ("oracle_gemm_bias_act", "oracle_b2b_gemm", "oracle_conv2d_nhwc",
                     "oracle_maxpool2x2_nhwc", "oracle_b2b_conv_nhwc",
                     "oracle_conv_relu_maxpool", "oracle_conv2d_nhwc_strided",
                     "oracle_b2b_conv_nhwc_strided", "oracle_fold_batchnorm"):
            getattr(lib, name).restype = ci
        _lib = lib
        return lib


# ------------------------------------------------------------------------------------
# helpers
# ------------------------------------------------------------------------------------

def _dt(dtype) -> int:
    if isinstance(dtype, int):
        return dtype
    return DTYPES[str(dtype).replace("torch.", "")]


def _act(act) -> int:
    if isinstance(act, int):
        return act
    return ACTS[act]


def _u16(a: np.ndarray | None, name: str):
    if a is None:
        return None, None
    a = np.ascontiguousarray(a)
    if a.dtype != np.uint16:
        raise TypeError(f"{name}: expected uint16 bit patterns, got {a.dtype}")
    return a, a.ctypes.data_as(ctypes.POINTER(ctypes.c_uint16))


def _check(rc: int, what: str):
    if rc != 0:
        raise RuntimeError(f"{what} failed with code {rc}")


def decode(dtype, bits: np.ndarray) -> np.ndarray:
    """Exact float64 values of fp16/bf16 bit patterns."""
    lib = _load()
    bits, p = _u16(bits, "bits")
    out = np.empty(bits.shape, dtype=np.float64)
    lib.oracle_decode_array(_dt(dtype), bits.size, p,
                            out.ctypes.data_as(ctypes.POINTER(ctypes.c_double)))
    return out


def encode(dtype, values: np.ndarray) -> np.ndarray:
    """Round float64 values to fp16/bf16 (nearest, ties to even), as uint16 bit patterns."""
    lib = _load()
    values = np.ascontiguousarray(values, dtype=np.float64)
    out = np.empty(values.shape, dtype=np.uint16)
    lib.oracle_encode_array(_dt(dtype), values.size,
                            values.ctypes.data_as(ctypes.POINTER(ctypes.c_double)),
                            out.ctypes.data_as(ctypes.POINTER(ctypes.c_uint16)))
    return out


def activation(act, x: float) -> float:
    return _load().oracle_activation(_act(act), float(x))


# ------------------------------------------------------------------------------------
# operators (each one call into oracle.c)
# ------------------------------------------------------------------------------------

def gemm_bias_act(dtype, A, W, b, act):
    """out = rnd(act(b + A @ W)); A [M,K], W [K,N] (row-major), b [N] or None."""
    lib = _load()
    A, pA = _u16(A, "A")
    W, pW = _u16(W, "W")
    b, pb = _u16(b, "b")
    M, K = A.shape
    K2, N = W.shape
    assert K == K2
    out = np.empty((M, N), dtype=np.uint16)
    _check(lib.oracle_gemm_bias_act(_dt(dtype), M, K, N, pA, pW, pb, _act(act),
                                    out.ctypes.data_as(ctypes.POINTER(ctypes.c_uint16))),
           "oracle_gemm_bias_act")
    return out


def b2b_gemm(dtype, A, W0, b0, W1, b1, act0, act1):
    """GEMM0 + bias + act0 -> intermediate (storage type) -> GEMM1 + bias + act1."""
    lib = _load()
    A, pA = _u16(A, "A")
    W0, pW0 = _u16(W0, "W0")
    W1, pW1 = _u16(W1, "W1")
    b0, pb0 = _u16(b0, "b0")
    b1, pb1 = _u16(b1, "b1")
    M, K0 = A.shape
    assert W0.shape[0] == K0
    N0 = W0.shape[1]
    assert W1.shape[0] == N0
    N1 = W1.shape[1]
    out = np.empty((M, N1), dtype=np.uint16)
    _check(lib.oracle_b2b_gemm(_dt(dtype), M, K0, N0, N1, pA, pW0, pb0, _act(act0),
                               pW1, pb1, _act(act1),
                               out.ctypes.data_as(ctypes.POINTER(ctypes.c_uint16))),
           "oracle_b2b_gemm")
    return out


def b2b_gemm3(dtype, A, W0, b0, W1, b1, W2, b2, act0, act1, act2):
    """A three-operator chain (BOLT notes, "Enabling deeper operator fusion": several GEMMs
    in one persistent kernel), written as its definition: three GEMM + bias + activation
    operators one after another, each intermediate stored in the storage type.
    A [M,K0], W0 [K0,N0], W1 [N0,N1], W2 [N1,N2] (row-major) -> out [M,N2]."""
    h0 = gemm_bias_act(dtype, A, W0, b0, act0)
    h1 = gemm_bias_act(dtype, h0, W1, b1, act1)
    return gemm_bias_act(dtype, h1, W2, b2, act2)


def conv_out_size(n, pad, k, stride=1):
    """Output length of a conv along one axis: floor((n + 2 pad - k) / stride) + 1."""
    return 0 if n + 2 * pad < k else (n + 2 * pad - k) // stride + 1


def conv2d_nhwc(dtype, x, Wt, b, pad, act, stride=1):
    """Direct convolution. x [N,H,W,C], Wt [Co,R,S,C] -> out [N,Ho,Wo,Co]."""
    lib = _load()
    x, px = _u16(x, "x")
    Wt, pW = _u16(Wt, "Wt")
    b, pb = _u16(b, "b")
    N, H, W, C = x.shape
    Co, R, S, C2 = Wt.shape
    assert C == C2
    Ho, Wo = conv_out_size(H, pad, R, stride), conv_out_size(W, pad, S, stride)
    out = np.empty((N, Ho, Wo, Co), dtype=np.uint16)
    _check(lib.oracle_conv2d_nhwc_strided(_dt(dtype), N, H, W, C, px, Co, R, S, pad, stride, pW,
                                          pb, _act(act),
                                          out.ctypes.data_as(ctypes.POINTER(ctypes.c_uint16))),
           "oracle_conv2d_nhwc_strided")
    return out


def maxpool2x2_nhwc(dtype, x):
    lib = _load()
    x, px = _u16(x, "x")
    N, H, W, C = x.shape
    out = np.empty((N, H // 2, W // 2, C), dtype=np.uint16)
    _check(lib.oracle_maxpool2x2_nhwc(_dt(dtype), N, H, W, C, px,
                                      out.ctypes.data_as(ctypes.POINTER(ctypes.c_uint16))),
           "oracle_maxpool2x2_nhwc")
    return out


def b2b_conv_nhwc(dtype, x, W0, b0, W1, b1, pad, act0, act1, stride=1):
    """conv RxS, stride `stride` (+bias, act0) -> intermediate -> 1x1 conv (+bias, act1).
    x [N,H,W,C], W0 [C0,R,S,C], W1 [C1,C0] -> out [N,Ho,Wo,C1]."""
    lib = _load()
    x, px = _u16(x, "x")
    W0, pW0 = _u16(W0, "W0")
    W1, pW1 = _u16(W1, "W1")
    b0, pb0 = _u16(b0, "b0")
    b1, pb1 = _u16(b1, "b1")
    N, H, W, C = x.shape
    C0, R, S, C2 = W0.shape
    assert C == C2
    C1, C0b = W1.shape
    assert C0b == C0
    Ho, Wo = conv_out_size(H, pad, R, stride), conv_out_size(W, pad, S, stride)
    out = np.empty((N, Ho, Wo, C1), dtype=np.uint16)
    _check(lib.oracle_b2b_conv_nhwc_strided(_dt(dtype), N, H, W, C, px, pW0, C0, R, S, pad,
                                            stride, pb0, _act(act0), pW1, C1, pb1, _act(act1),
                                            out.ctypes.data_as(ctypes.POINTER(ctypes.c_uint16))),
           "oracle_b2b_conv_nhwc_strided")
    return out


def fold_batchnorm(dtype, Wt, b, gamma, beta, mean, var, eps, out_inner=False):
    """Batch normalisation folded into the preceding operator's weights and bias
    (interview notes, SimplifyInference: BN -> scale + bias).  Wt [Co, ...] (conv filters,
    out_inner False) or [K, Co] (row-major GEMM weights, out_inner True); b [Co] or None;
    gamma, beta, mean, var float32 [Co].  Returns (W', b') in the storage type."""
    lib = _load()
    Wt, pW = _u16(Wt, "Wt")
    b, pb = _u16(b, "b")
    Co = Wt.shape[-1] if out_inner else Wt.shape[0]
    K = Wt.size // max(Co, 1)
    f32 = [np.ascontiguousarray(np.asarray(v, dtype=np.float32)) for v in (gamma, beta, mean, var)]
    assert all(v.shape == (Co,) for v in f32)
    fp = [v.ctypes.data_as(ctypes.POINTER(ctypes.c_float)) for v in f32]
    W_out = np.empty_like(Wt)
    b_out = np.empty((Co,), dtype=np.uint16)
    _check(lib.oracle_fold_batchnorm(_dt(dtype), Co, K, 1 if out_inner else 0, pW, pb, *fp,
                                     float(eps), W_out.ctypes.data_as(ctypes.POINTER(ctypes.c_uint16)),
                                     b_out.ctypes.data_as(ctypes.POINTER(ctypes.c_uint16))),
           "oracle_fold_batchnorm")
    return W_out, b_out


def conv_relu_maxpool(dtype, x, Wt, b):
    """conv3x3 pad 1 (+bias) -> ReLU -> intermediate -> max-pool 2x2/2 (floor)."""
    lib = _load()
    x, px = _u16(x, "x")
    Wt, pW = _u16(Wt, "Wt")
    b, pb = _u16(b, "b")
    N, H, W, C = x.shape
    Co, R, S, C2 = Wt.shape
    assert (R, S) == (3, 3) and C == C2
    out = np.empty((N, H // 2, W // 2, Co), dtype=np.uint16)
    _check(lib.oracle_conv_relu_maxpool(_dt(dtype), N, H, W, C, px, pW, pb, Co,
                                        out.ctypes.data_as(ctypes.POINTER(ctypes.c_uint16))),
           "oracle_conv_relu_maxpool")
    return out
