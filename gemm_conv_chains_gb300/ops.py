"""Python binding of libb2b.so (include/b2b.h): argument marshalling only.

Every function takes CUDA tensors, checks dtypes, shapes and contiguity (the C ABI sees
only pointers and sizes), allocates the output with torch when none is given, and calls
the entry point of the same name on the current torch stream.  All arithmetic runs in the
library's kernels; there is no other code path, and a missing or unloadable library
raises instead of falling back.
"""
from __future__ import annotations

import ctypes
import os
import threading
from typing import Optional

import torch

from . import build as _build

EPILOGUES = {"none": 0, "relu": 1, "hardswish": 2}
STATUS = {0: "B2B_OK", 1: "B2B_ERR_NULL", 2: "B2B_ERR_SHAPE", 3: "B2B_ERR_ALIGN",
          4: "B2B_ERR_UNSUPPORTED", 5: "B2B_ERR_CUDA", 6: "B2B_ERR_TIMEOUT"}

_lock = threading.Lock()
_lib = None


class B2BError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {STATUS.get(status, status)}")


def library_path() -> str:
    return _build.LIB_PATH


def lib() -> ctypes.CDLL:
    """Loads libb2b.so (building it first if it is absent or stale)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        path = _build.build()
        L = ctypes.CDLL(path)
        i32, i64, vp, u64 = ctypes.c_int32, ctypes.c_int64, ctypes.c_void_p, ctypes.c_uint64
        ci = ctypes.c_int
        L.b2b_gemm.argtypes = [ci, i64, i32, i32, i32, vp, vp, vp, ci, vp, vp, ci, vp, vp]
        L.b2b_conv_nhwc.argtypes = [ci, i32, i32, i32, i32, vp, vp, i32, i32, i32, i32, vp, ci,
                                    vp, i32, vp, ci, vp, vp]
        L.conv_relu_maxpool.argtypes = [ci, i32, i32, i32, i32, vp, vp, vp, i32, vp, vp]
        L.gemm_bias_act.argtypes = [ci, i64, i32, i32, vp, vp, vp, ci, vp, vp]
        L.conv_bias_act_nhwc.argtypes = [ci, i32, i32, i32, i32, vp, vp, i32, i32, i32, i32, vp,
                                         ci, vp, vp]
        L.maxpool2x2_nhwc.argtypes = [ci, i32, i32, i32, i32, vp, vp, vp]
        for name in ("b2b_gemm", "b2b_conv_nhwc", "conv_relu_maxpool", "gemm_bias_act",
                     "conv_bias_act_nhwc", "maxpool2x2_nhwc", "b2b_get_device_error",
                     "b2b_probe_timeout"):
            getattr(L, name).restype = ci
        L.b2b_status_str.argtypes = [ci]
        L.b2b_status_str.restype = ctypes.c_char_p
        L.b2b_version.argtypes = []
        L.b2b_version.restype = ctypes.c_char_p
        L.b2b_num_sms.argtypes = []
        L.b2b_num_sms.restype = i32
        L.b2b_set_wait_limit_ns.argtypes = [u64]
        L.b2b_set_wait_limit_ns.restype = None
        L.b2b_get_device_error.argtypes = [ctypes.POINTER(ctypes.c_uint32)]
        L.b2b_probe_timeout.argtypes = [u64, vp]
        L.b2b_set_trace.argtypes = [vp, ctypes.c_uint32, ctypes.c_uint32]
        L.b2b_set_trace.restype = ci
        p64 = ctypes.POINTER(i64)
        L.b2b_gemm3.argtypes = [ci, i64, i32, i32, i32, i32, vp, vp, vp, ci, vp, vp, ci, vp, vp,
                                ci, vp, vp]
        L.b2b_gemm3.restype = ci
        L.b2b_conv_nhwc_strided.argtypes = [ci, i32, i32, i32, i32, vp, vp, i32, i32, i32, i32,
                                            i32, vp, ci, vp, i32, vp, ci, vp, vp]
        L.b2b_conv_nhwc_strided.restype = ci
        L.conv_bias_act_nhwc_strided.argtypes = [ci, i32, i32, i32, i32, vp, vp, i32, i32, i32,
                                                 i32, i32, vp, ci, vp, vp]
        L.conv_bias_act_nhwc_strided.restype = ci
        L.b2b_fold_batchnorm.argtypes = [ci, i64, i64, i32, vp, vp, vp, vp, vp, vp,
                                         ctypes.c_float, vp, vp, vp]
        L.b2b_fold_batchnorm.restype = ci
        L.b2b_set_autotune.argtypes = [i32]
        L.b2b_set_autotune.restype = None
        L.b2b_autotune_reset.argtypes = []
        L.b2b_autotune_reset.restype = None
        L.b2b_set_choice.argtypes = [i32, p64, i32, i32, i32, i32]
        L.b2b_set_choice.restype = ci
        L.b2b_get_choice.argtypes = [i32, p64, i32, ctypes.POINTER(i32), i32]
        L.b2b_get_choice.restype = ci
        L.b2b_debug_plan.argtypes = [i32, p64, i32, ctypes.POINTER(ctypes.c_uint32), i32]
        L.b2b_debug_plan.restype = ci
        L.b2b_debug_plan_candidate.argtypes = [i32, p64, i32, i32, ctypes.POINTER(ctypes.c_uint32),
                                               i32]
        L.b2b_debug_plan_candidate.restype = ci
        L.b2b_set_candidates.argtypes = [i32, p64, i32, ctypes.POINTER(i32), i32]
        L.b2b_set_candidates.restype = ci
        L.b2b_get_tune_record.argtypes = [i32, p64, i32, ctypes.POINTER(i32), i32,
                                          ctypes.POINTER(i32)]
        L.b2b_get_tune_record.restype = ci
        _lib = L
        return L


# ------------------------------------------------------------------------------------
# marshalling helpers
# ------------------------------------------------------------------------------------

def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.float16:
        return 0
    if t.dtype == torch.bfloat16:
        return 1
    raise TypeError(f"expected float16 or bfloat16, got {t.dtype}")


def _epi(e) -> int:
    if isinstance(e, int):
        return e
    try:
        return EPILOGUES[e]
    except KeyError:
        raise ValueError(f"unknown epilogue {e!r}; expected one of {list(EPILOGUES)}") from None


def _check_tensor(t: torch.Tensor, name: str, dtype, shape) -> None:
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} has dtype {t.dtype}, expected {dtype}")
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {tuple(shape)}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _common_device(**tensors) -> torch.device:
    """The one device every given tensor (None skipped) lives on.  The library launches on
    the current device and encodes its tensor maps over the pointers it is given, so an
    operand on another device must be refused before anything is launched."""
    dev = None
    for name, t in tensors.items():
        if t is None:
            continue
        if dev is None:
            dev = t.device
        elif t.device != dev:
            raise ValueError(f"{name} is on {t.device}, the other operands on {dev}: "
                             "all operands and the output must be on one device")
    if dev is None:
        raise ValueError("no tensor operand given")
    return dev


def _stream(stream, device=None) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream(device)
    if isinstance(stream, torch.cuda.Stream):
        return ctypes.c_void_p(stream.cuda_stream)
    return ctypes.c_void_p(int(stream))


def _raise(status: int, what: str) -> None:
    if status != 0:
        raise B2BError(status, what)


# ------------------------------------------------------------------------------------
# fused chains
# ------------------------------------------------------------------------------------

def b2b_gemm(A, W0, b0, W1, b1, epi0="relu", epi1="relu", out=None, stream=None):
    """out[M,N1] = epi1(epi0(A[M,K0] @ W0[K0,N0] + b0) @ W1[N0,N1] + b1), one launch."""
    dt = A.dtype
    M, K0 = A.shape
    N0, N1 = W0.shape[1], W1.shape[1]
    _check_tensor(A, "A", dt, (M, K0))
    _check_tensor(W0, "W0", dt, (K0, N0))
    _check_tensor(W1, "W1", dt, (N0, N1))
    if b0 is not None:
        _check_tensor(b0, "b0", dt, (N0,))
    if b1 is not None:
        _check_tensor(b1, "b1", dt, (N1,))
    if out is None:
        out = torch.empty((M, N1), dtype=dt, device=A.device)
    _check_tensor(out, "out", dt, (M, N1))
    dev = _common_device(A=A, W0=W0, b0=b0, W1=W1, b1=b1, out=out)
    with torch.cuda.device(dev):
        _raise(lib().b2b_gemm(_dtype_code(A), M, K0, N0, N1, _ptr(A), _ptr(W0), _ptr(b0),
                              _epi(epi0), _ptr(W1), _ptr(b1), _epi(epi1), _ptr(out),
                              _stream(stream, dev)), "b2b_gemm")
    return out


def _conv_out(n, pad, k, stride):
    return 0 if n + 2 * pad < k else (n + 2 * pad - k) // stride + 1


def b2b_gemm3(A, W0, b0, W1, b1, W2, b2, epi0="relu", epi1="relu", epi2="relu", out=None,
              stream=None):
    """out = epi2(epi1(epi0(A @ W0 + b0) @ W1 + b1) @ W2 + b2) in one launch (b2b_gemm3).
    A [M,K0], W0 [K0,N0], W1 [N0,N1], W2 [N1,N2] -> out [M,N2]."""
    dt = A.dtype
    M, K0 = A.shape
    N0, N1, N2 = W0.shape[1], W1.shape[1], W2.shape[1]
    _check_tensor(A, "A", dt, (M, K0))
    _check_tensor(W0, "W0", dt, (K0, N0))
    _check_tensor(W1, "W1", dt, (N0, N1))
    _check_tensor(W2, "W2", dt, (N1, N2))
    for name, b, n in (("b0", b0, N0), ("b1", b1, N1), ("b2", b2, N2)):
        if b is not None:
            _check_tensor(b, name, dt, (n,))
    if out is None:
        out = torch.empty((M, N2), dtype=dt, device=A.device)
    _check_tensor(out, "out", dt, (M, N2))
    dev = _common_device(A=A, W0=W0, b0=b0, W1=W1, b1=b1, W2=W2, b2=b2, out=out)
    with torch.cuda.device(dev):
        _raise(lib().b2b_gemm3(_dtype_code(A), M, K0, N0, N1, N2, _ptr(A), _ptr(W0), _ptr(b0),
                               _epi(epi0), _ptr(W1), _ptr(b1), _epi(epi1), _ptr(W2), _ptr(b2),
                               _epi(epi2), _ptr(out), _stream(stream, dev)), "b2b_gemm3")
    return out


def b2b_conv_nhwc(x, W0, b0, W1, b1, pad=1, epi0="relu", epi1="relu", out=None, stream=None):
    """out = conv1x1(conv_RxS(x) + b0 -> epi0) + b1 -> epi1, NHWC, stride 1, one launch.
    x [N,H,W,C], W0 [C0,R,S,C], W1 [C1,C0] -> out [N,Ho,Wo,C1]."""
    return _b2b_conv(x, W0, b0, W1, b1, pad, 1, epi0, epi1, out, stream)


def b2b_conv_nhwc_strided(x, W0, b0, W1, b1, pad=1, stride=2, epi0="relu", epi1="relu",
                          out=None, stream=None):
    """b2b_conv_nhwc with the first conv at spatial stride `stride` (1..4):
    out [N, (H+2pad-R)//stride+1, (W+2pad-S)//stride+1, C1]."""
    return _b2b_conv(x, W0, b0, W1, b1, pad, stride, epi0, epi1, out, stream)


def _b2b_conv(x, W0, b0, W1, b1, pad, stride, epi0, epi1, out, stream):
    dt = x.dtype
    N, H, W, C = x.shape
    C0, R, S = W0.shape[0], W0.shape[1], W0.shape[2]
    C1 = W1.shape[0]
    _check_tensor(x, "x", dt, (N, H, W, C))
    _check_tensor(W0, "W0", dt, (C0, R, S, C))
    _check_tensor(W1, "W1", dt, (C1, C0))
    if b0 is not None:
        _check_tensor(b0, "b0", dt, (C0,))
    if b1 is not None:
        _check_tensor(b1, "b1", dt, (C1,))
    Ho, Wo = _conv_out(H, pad, R, stride), _conv_out(W, pad, S, stride)
    if out is None:
        out = torch.empty((N, Ho, Wo, C1), dtype=dt, device=x.device)
    _check_tensor(out, "out", dt, (N, Ho, Wo, C1))
    dev = _common_device(x=x, W0=W0, b0=b0, W1=W1, b1=b1, out=out)
    with torch.cuda.device(dev):
        if stride == 1:
            _raise(lib().b2b_conv_nhwc(_dtype_code(x), N, H, W, C, _ptr(x), _ptr(W0), C0, R, S,
                                       pad, _ptr(b0), _epi(epi0), _ptr(W1), C1, _ptr(b1),
                                       _epi(epi1), _ptr(out), _stream(stream, dev)),
                   "b2b_conv_nhwc")
        else:
            _raise(lib().b2b_conv_nhwc_strided(_dtype_code(x), N, H, W, C, _ptr(x), _ptr(W0), C0,
                                               R, S, pad, stride, _ptr(b0), _epi(epi0), _ptr(W1),
                                               C1, _ptr(b1), _epi(epi1), _ptr(out),
                                               _stream(stream, dev)), "b2b_conv_nhwc_strided")
    return out


def conv_relu_maxpool(x, Wt, b, out=None, stream=None):
    """out = maxpool2x2(relu(conv3x3_pad1(x, Wt) + b)), NHWC, one launch.
    x [N,H,W,Cin], Wt [Cout,3,3,Cin] -> out [N,H//2,W//2,Cout]."""
    dt = x.dtype
    N, H, W, Cin = x.shape
    Cout = Wt.shape[0]
    _check_tensor(x, "x", dt, (N, H, W, Cin))
    _check_tensor(Wt, "Wt", dt, (Cout, 3, 3, Cin))
    if b is not None:
        _check_tensor(b, "b", dt, (Cout,))
    if out is None:
        out = torch.empty((N, H // 2, W // 2, Cout), dtype=dt, device=x.device)
    _check_tensor(out, "out", dt, (N, H // 2, W // 2, Cout))
    dev = _common_device(x=x, Wt=Wt, b=b, out=out)
    with torch.cuda.device(dev):
        _raise(lib().conv_relu_maxpool(_dtype_code(x), N, H, W, Cin, _ptr(x), _ptr(Wt), _ptr(b),
                                       Cout, _ptr(out), _stream(stream, dev)), "conv_relu_maxpool")
    return out


# ------------------------------------------------------------------------------------
# single operators (the unfused two-kernel path)
# ------------------------------------------------------------------------------------

def gemm_bias_act(A, W, b, epi="relu", out=None, stream=None):
    """out[M,N] = epi(A[M,K] @ W[K,N] + b)."""
    dt = A.dtype
    M, K = A.shape
    N = W.shape[1]
    _check_tensor(A, "A", dt, (M, K))
    _check_tensor(W, "W", dt, (K, N))
    if b is not None:
        _check_tensor(b, "b", dt, (N,))
    if out is None:
        out = torch.empty((M, N), dtype=dt, device=A.device)
    _check_tensor(out, "out", dt, (M, N))
    dev = _common_device(A=A, W=W, b=b, out=out)
    with torch.cuda.device(dev):
        _raise(lib().gemm_bias_act(_dtype_code(A), M, K, N, _ptr(A), _ptr(W), _ptr(b), _epi(epi),
                                   _ptr(out), _stream(stream, dev)), "gemm_bias_act")
    return out


def conv_bias_act_nhwc(x, Wt, b, pad=1, epi="relu", out=None, stream=None):
    """out = epi(conv_RxS(x, Wt) + b); x [N,H,W,C], Wt [Co,R,S,C] -> [N,Ho,Wo,Co]."""
    return _conv_single(x, Wt, b, pad, 1, epi, out, stream)


def conv_bias_act_nhwc_strided(x, Wt, b, pad=1, stride=2, epi="relu", out=None, stream=None):
    """conv_bias_act_nhwc at spatial stride `stride` (1..4)."""
    return _conv_single(x, Wt, b, pad, stride, epi, out, stream)


def _conv_single(x, Wt, b, pad, stride, epi, out, stream):
    dt = x.dtype
    N, H, W, C = x.shape
    Co, R, S = Wt.shape[0], Wt.shape[1], Wt.shape[2]
    _check_tensor(x, "x", dt, (N, H, W, C))
    _check_tensor(Wt, "Wt", dt, (Co, R, S, C))
    if b is not None:
        _check_tensor(b, "b", dt, (Co,))
    Ho, Wo = _conv_out(H, pad, R, stride), _conv_out(W, pad, S, stride)
    if out is None:
        out = torch.empty((N, Ho, Wo, Co), dtype=dt, device=x.device)
    _check_tensor(out, "out", dt, (N, Ho, Wo, Co))
    dev = _common_device(x=x, Wt=Wt, b=b, out=out)
    with torch.cuda.device(dev):
        if stride == 1:
            _raise(lib().conv_bias_act_nhwc(_dtype_code(x), N, H, W, C, _ptr(x), _ptr(Wt), Co, R,
                                            S, pad, _ptr(b), _epi(epi), _ptr(out),
                                            _stream(stream, dev)), "conv_bias_act_nhwc")
        else:
            _raise(lib().conv_bias_act_nhwc_strided(_dtype_code(x), N, H, W, C, _ptr(x), _ptr(Wt),
                                                    Co, R, S, pad, stride, _ptr(b), _epi(epi),
                                                    _ptr(out), _stream(stream, dev)),
                   "conv_bias_act_nhwc_strided")
    return out


def fold_batchnorm(W, b, gamma, beta, mean, var, eps=1e-5, out_inner=False, W_out=None,
                   b_out=None, stream=None):
    """Batch norm folded into the preceding operator's weights and bias
    (b2b_fold_batchnorm): W [Co, ...] (conv filters, out_inner False) or [K, Co] (row-major
    GEMM weights, out_inner True), b [Co] or None, gamma/beta/mean/var float32 [Co].
    Returns (W', b') in W's dtype; W_out / b_out may be W / b."""
    dt = W.dtype
    Co = W.shape[-1] if out_inner else W.shape[0]
    K = W.numel() // max(Co, 1)
    _check_tensor(W, "W", dt, tuple(W.shape))
    if b is not None:
        _check_tensor(b, "b", dt, (Co,))
    for name, v in (("gamma", gamma), ("beta", beta), ("mean", mean), ("var", var)):
        _check_tensor(v, name, torch.float32, (Co,))
    W_out = torch.empty_like(W) if W_out is None else W_out
    b_out = torch.empty((Co,), dtype=dt, device=W.device) if b_out is None else b_out
    _check_tensor(W_out, "W_out", dt, tuple(W.shape))
    _check_tensor(b_out, "b_out", dt, (Co,))
    dev = _common_device(W=W, b=b, gamma=gamma, beta=beta, mean=mean, var=var, W_out=W_out,
                         b_out=b_out)
    with torch.cuda.device(dev):
        _raise(lib().b2b_fold_batchnorm(_dtype_code(W), Co, K, 1 if out_inner else 0, _ptr(W),
                                        _ptr(b), _ptr(gamma), _ptr(beta), _ptr(mean), _ptr(var),
                                        float(eps), _ptr(W_out), _ptr(b_out),
                                        _stream(stream, dev)), "b2b_fold_batchnorm")
    return W_out, b_out


def maxpool2x2_nhwc(x, out=None, stream=None):
    """out[N,H//2,W//2,C] = max over 2x2 windows (stride 2, floor mode) of x[N,H,W,C]."""
    dt = x.dtype
    N, H, W, C = x.shape
    _check_tensor(x, "x", dt, (N, H, W, C))
    if out is None:
        out = torch.empty((N, H // 2, W // 2, C), dtype=dt, device=x.device)
    _check_tensor(out, "out", dt, (N, H // 2, W // 2, C))
    dev = _common_device(x=x, out=out)
    with torch.cuda.device(dev):
        _raise(lib().maxpool2x2_nhwc(_dtype_code(x), N, H, W, C, _ptr(x), _ptr(out),
                                     _stream(stream, dev)), "maxpool2x2_nhwc")
    return out


# ------------------------------------------------------------------------------------
# diagnostics
# ------------------------------------------------------------------------------------

# Field names of b2b_debug_plan's output, in order (see include/b2b.h).
PLAN_FIELDS = ["smem", "stages", "stage_bytes", "resident", "alias", "off_ring", "ring", "off_w0",
               "off_w1", "w_res", "w0_chunk", "w1_chunk", "off_p0", "off_p1", "p", "off_out0",
               "off_out1", "out", "off_bias", "bias", "off_bar", "bar", "tmem_cols", "d0_col0",
               "d0_col1", "d1_col0", "d1_col1", "dual", "groups", "tiles", "kchunks0",
               "kchunks1", "N0p", "N1p", "mode", "p_tmem", "w1_group", "w1_per_stage", "halo",
               "a_stage_bytes", "nbuf", "off_p2", "off_p3", "d0_col2", "d0_col3", "d1_col2",
               "d1_col3", "cand", "ncand", "grid_choice", "pf_choice", "ring_extend", "off_w2",
               "off_p1_0", "off_p1_1", "d2_col0", "d2_col1", "p_split", "w0_res", "cta_pair",
               "two_issuers", "out_slots", "pt_col0", "pt_col1"]
_SIGNED_PLAN_FIELDS = ("grid_choice", "pf_choice")
PLAN_KINDS = {"b2b_gemm": 0, "gemm_bias_act": 1, "b2b_conv_nhwc": 2, "conv_bias_act_nhwc": 3,
              "conv_relu_maxpool": 4, "b2b_gemm3": 5}


def _dims(dims):
    return (ctypes.c_int64 * len(dims))(*[int(d) for d in dims])


def variant(dtype, *acts) -> list:
    """The trailing dims that name a call's variant for the plan and choice functions:
    the dtype code (torch.float16 / torch.bfloat16 or "f16" / "bf16"), then each epilogue
    kind.  Append it to the sizes (for the convs, after the stride)."""
    codes = {torch.float16: 0, torch.bfloat16: 1, "f16": 0, "bf16": 1}
    if dtype not in codes:
        raise TypeError(f"expected float16 or bfloat16, got {dtype!r}")
    return [codes[dtype]] + [_epi(a) for a in acts]


def debug_plan(kind: str, dims, cand: Optional[int] = None) -> dict:
    """The launch plan the entry point `kind` would use for `dims` (b2b_debug_plan; no CUDA
    call), or, with `cand`, the plan of that feasible layout candidate whatever is pinned
    (b2b_debug_plan_candidate).  Raises B2BError with the entry point's status if it would
    not launch."""
    arr = _dims(dims)
    out = (ctypes.c_uint32 * len(PLAN_FIELDS))()
    if cand is None:
        _raise(lib().b2b_debug_plan(PLAN_KINDS[kind], arr, len(dims), out, len(PLAN_FIELDS)),
               "b2b_debug_plan")
    else:
        _raise(lib().b2b_debug_plan_candidate(PLAN_KINDS[kind], arr, len(dims), int(cand), out,
                                              len(PLAN_FIELDS)), "b2b_debug_plan_candidate")
    plan = dict(zip(PLAN_FIELDS, [int(v) for v in out]))
    for k in _SIGNED_PLAN_FIELDS:
        plan[k] = ctypes.c_int32(plan[k]).value
    return plan


# ------------------------------------------------------------------------------------
# launch choices and the light-weight profiler (b2b_set_autotune and friends)
# ------------------------------------------------------------------------------------

def set_autotune(on: bool) -> None:
    """With the profiler on, the first call of an entry point for new sizes times every
    launch choice on the caller's stream and keeps the fastest (b2b_set_autotune)."""
    lib().b2b_set_autotune(1 if on else 0)


def autotune_reset() -> None:
    lib().b2b_autotune_reset()


def set_choice(kind: str, dims, cand: int = -1, grid: int = -1, prefetch_second: int = -1) -> None:
    """Pins the launch choice of entry point `kind` for `dims` (b2b_set_choice)."""
    arr = (ctypes.c_int64 * len(dims))(*[int(d) for d in dims])
    _raise(lib().b2b_set_choice(PLAN_KINDS[kind], arr, len(dims), int(cand), int(grid),
                                int(prefetch_second)), "b2b_set_choice")


def set_candidates(kind: str, dims, cands) -> None:
    """Hands the profiler a ranked list of layouts for `dims` (b2b_set_candidates): the
    first becomes the default, and the profiler times only these."""
    c = [int(x) for x in cands]
    arr = (ctypes.c_int32 * len(c))(*c)
    _raise(lib().b2b_set_candidates(PLAN_KINDS[kind], _dims(dims), len(dims), arr, len(c)),
           "b2b_set_candidates")


def tune_record(kind: str, dims) -> list:
    """Every launch choice the profiler timed for `dims`, the default first
    (b2b_get_tune_record): dicts of cand, grid (mode), ctas, prefetch_second, ns."""
    L, arr, n = lib(), _dims(dims), ctypes.c_int32(0)
    _raise(L.b2b_get_tune_record(PLAN_KINDS[kind], arr, len(dims), None, 0, ctypes.byref(n)),
           "b2b_get_tune_record")
    rows = n.value
    out = (ctypes.c_int32 * max(1, 5 * rows))()
    _raise(L.b2b_get_tune_record(PLAN_KINDS[kind], arr, len(dims), out, rows, ctypes.byref(n)),
           "b2b_get_tune_record")
    keys = ("cand", "grid", "ctas", "prefetch_second", "ns")
    return [dict(zip(keys, [int(v) for v in out[5 * i:5 * i + 5]])) for i in range(min(rows, n.value))]


def get_choice(kind: str, dims) -> dict:
    """The pinned or measured choice for `dims` (b2b_get_choice); source 0 = none."""
    arr = (ctypes.c_int64 * len(dims))(*[int(d) for d in dims])
    out = (ctypes.c_int32 * 7)()
    _raise(lib().b2b_get_choice(PLAN_KINDS[kind], arr, len(dims), out, 7), "b2b_get_choice")
    keys = ("source", "cand", "grid", "prefetch_second", "best_ns", "default_ns", "timed")
    return dict(zip(keys, [int(v) for v in out]))


def version() -> str:
    return lib().b2b_version().decode()


def status_str(status: int) -> str:
    return lib().b2b_status_str(status).decode()


def num_sms() -> int:
    return int(lib().b2b_num_sms())


def set_wait_limit_ns(ns: int) -> None:
    lib().b2b_set_wait_limit_ns(int(ns))


def get_device_error():
    """(status, info[4]); reads and clears the device error word (synchronises)."""
    info = (ctypes.c_uint32 * 4)()
    st = lib().b2b_get_device_error(info)
    return int(st), [int(v) for v in info]


def probe_timeout(limit_ns: int, stream=None) -> None:
    _raise(lib().b2b_probe_timeout(int(limit_ns), _stream(stream)), "b2b_probe_timeout")


TRACE_EVENTS = {1: "prod_acquire", 2: "prod_issued", 3: "mma_full", 4: "mma_g0_done",
                5: "mma_p_ready", 6: "mma_g1_done", 7: "mma_acc_free", 8: "epi_acc_ready",
                9: "epi_p_done", 10: "epi_d1_ready", 11: "epi_staging", 12: "epi_stored",
                13: "mma_wait", 14: "mma_issued",
                15: "prod_w1_issued", 16: "mma_w1_full",
                17: "kernel_entry", 18: "epi_drained", 19: "setup_done", 20: "dep_ready",
                21: "epi_p1_done", 22: "mma_g2_done", 23: "prod_start", 24: "mma_setup"}


def set_trace(buf, cta: int = 0) -> None:
    """Records the per-step timeline of CTA `cta` of later launches into `buf` (a zeroed,
    contiguous CUDA int64 tensor of 2 * capacity words); None turns it off.  Traced launches
    run a separate build of the kernels with the recording compiled in, a little slower
    than the plain build every other launch uses."""
    if buf is None:
        _raise(lib().b2b_set_trace(None, 0, 0), "b2b_set_trace")
        return
    if not (buf.is_cuda and buf.dtype == torch.int64 and buf.is_contiguous()):
        raise ValueError("trace buffer must be a contiguous CUDA int64 tensor")
    _raise(lib().b2b_set_trace(_ptr(buf), buf.numel() // 2, int(cta)), "b2b_set_trace")


def read_trace(buf):
    """Decodes a trace buffer into (nanoseconds since the first event, event, group, tile),
    sorted by time."""
    raw = buf.cpu().view(-1, 2).tolist()
    ev = [(c, w & ((1 << 63) - 1)) for c, w in raw if w != 0]
    if not ev:
        return []
    t0 = min(c for c, _ in ev)
    return sorted((c - t0, TRACE_EVENTS.get(w & 0xFF, str(w & 0xFF)), (w >> 8) & 0xFF,
                   (w >> 16) & 0xFFFF) for c, w in ev)


def pad_channels(t: torch.Tensor, dim: int, multiple: int = 8) -> torch.Tensor:
    """Zero-pads `dim` of t up to a multiple of `multiple` (BOLT's kernel padding to an
    8-element, 128-bit alignment).  Padded inputs, weights and biases give padded output
    channels that are exactly zero."""
    size = t.shape[dim]
    target = -(-size // multiple) * multiple
    if target == size:
        return t.contiguous()
    pad_shape = list(t.shape)
    pad_shape[dim] = target - size
    return torch.cat([t, t.new_zeros(pad_shape)], dim=dim).contiguous()
