"""The C-ABI boundary without a GPU: the library loads, exports every symbol the header
declares, and rejects bad arguments on the host with the documented status before it
touches CUDA."""
import ctypes
import os
import re

import pytest
import torch

from gemm_conv_chains_gb300 import ops

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "b2b.h")

OK, NULL, SHAPE, ALIGN, UNSUP, CUDA = 0, 1, 2, 3, 4, 5
F16, BF16 = 0, 1
FAKE = 0x10000          # a 16-byte aligned fake address: never dereferenced here
MIS = 0x10008           # 8-byte aligned only


def header_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:b2b_status|const char\*|int32_t|void)\s+(\w+)\s*\(",
                                 text, flags=re.M)))


@pytest.fixture(scope="module")
def L():
    return ops.lib()


def test_header_declares_the_entry_points():
    names = header_functions()
    for n in ("b2b_gemm", "b2b_conv_nhwc", "conv_relu_maxpool", "gemm_bias_act",
              "conv_bias_act_nhwc", "maxpool2x2_nhwc", "b2b_status_str", "b2b_get_device_error",
              "b2b_conv_nhwc_strided", "conv_bias_act_nhwc_strided", "b2b_set_autotune",
              "b2b_set_choice", "b2b_get_choice", "b2b_fold_batchnorm", "b2b_gemm3",
              "b2b_debug_plan_candidate", "b2b_set_candidates", "b2b_get_tune_record"):
        assert n in names


def test_library_exports_every_declared_symbol(L):
    for name in header_functions():
        assert hasattr(L, name), name


def test_status_strings(L):
    for s, tag in [(0, b"B2B_OK"), (1, b"B2B_ERR_NULL"), (2, b"B2B_ERR_SHAPE"),
                   (3, b"B2B_ERR_ALIGN"), (4, b"B2B_ERR_UNSUPPORTED"), (5, b"B2B_ERR_CUDA"),
                   (6, b"B2B_ERR_TIMEOUT")]:
        assert L.b2b_status_str(s).startswith(tag)
    assert L.b2b_version().decode().count(".") == 2


def gemm(L, dt=F16, M=256, K0=64, N0=64, N1=64, A=FAKE, W0=FAKE, b0=None, e0=1, W1=FAKE,
         b1=None, e1=1, D=FAKE):
    return L.b2b_gemm(dt, M, K0, N0, N1, A, W0, b0, e0, W1, b1, e1, D, None)


@pytest.mark.parametrize("kw,expect", [
    (dict(dt=2), UNSUP), (dict(e0=3), UNSUP), (dict(e1=-1), UNSUP),
    (dict(M=-1), SHAPE), (dict(K0=0), SHAPE), (dict(N1=-8), SHAPE),
    (dict(K0=12), ALIGN), (dict(N0=4), ALIGN), (dict(N1=30), ALIGN),
    (dict(N0=520), UNSUP), (dict(N0=264, N1=136), UNSUP), (dict(N1=512), UNSUP),
    (dict(A=None), NULL), (dict(W1=None), NULL), (dict(D=None), NULL),
    (dict(A=MIS), ALIGN), (dict(D=MIS), ALIGN), (dict(b0=FAKE + 1), ALIGN),
    (dict(M=0, A=None, D=None), OK),
    (dict(M=2 ** 31), UNSUP),
])
def test_b2b_gemm_argument_checks(L, kw, expect):
    assert gemm(L, **kw) == expect


def conv(L, dt=F16, N=2, H=8, W=8, C=64, x=FAKE, W0=FAKE, C0=64, R=3, S=3, pad=1, b0=None,
         e0=1, W1=FAKE, C1=64, b1=None, e1=0, y=FAKE):
    return L.b2b_conv_nhwc(dt, N, H, W, C, x, W0, C0, R, S, pad, b0, e0, W1, C1, b1, e1, y, None)


@pytest.mark.parametrize("kw,expect", [
    (dict(dt=5), UNSUP), (dict(N=-1), SHAPE), (dict(C=20), ALIGN), (dict(C0=300), ALIGN),
    (dict(C1=264), UNSUP), (dict(R=0), SHAPE), (dict(pad=-1), SHAPE), (dict(R=9), UNSUP),
    (dict(pad=4), UNSUP), (dict(H=1, pad=0), SHAPE),
    (dict(x=None), NULL), (dict(W1=MIS), ALIGN),
    (dict(N=0, x=None, y=None), OK), (dict(H=0, x=None), OK),
])
def test_b2b_conv_argument_checks(L, kw, expect):
    assert conv(L, **kw) == expect


@pytest.mark.parametrize("stride,kw,expect", [
    (0, {}, SHAPE), (-1, {}, SHAPE), (5, {}, UNSUP),
    (2, dict(H=1, pad=0), SHAPE),                       # H + 2 pad < R: no output
    (2, dict(C1=264), UNSUP), (3, dict(x=None), NULL), (2, dict(N=0, x=None, y=None), OK),
])
def test_strided_conv_argument_checks(L, stride, kw, expect):
    a = dict(dt=F16, N=2, H=9, W=9, C=64, x=FAKE, W0=FAKE, C0=64, R=3, S=3, pad=1, b0=None,
             e0=1, W1=FAKE, C1=64, b1=None, e1=1, y=FAKE)
    a.update(kw)
    assert L.b2b_conv_nhwc_strided(a["dt"], a["N"], a["H"], a["W"], a["C"], a["x"], a["W0"],
                                   a["C0"], a["R"], a["S"], a["pad"], stride, a["b0"], a["e0"],
                                   a["W1"], a["C1"], a["b1"], a["e1"], a["y"], None) == expect
    single = L.conv_bias_act_nhwc_strided(a["dt"], a["N"], a["H"], a["W"], a["C"], a["x"],
                                          a["W0"], a["C0"], a["R"], a["S"], a["pad"], stride,
                                          a["b0"], a["e0"], a["y"], None)
    if "C1" not in kw:
        assert single == expect


@pytest.mark.parametrize("args,expect", [
    ((F16, 2, 1, 8, 64, FAKE, FAKE, None, 64, FAKE), SHAPE),     # H < 2
    ((F16, 2, 8, 8, 60, FAKE, FAKE, None, 64, FAKE), ALIGN),
    ((F16, 2, 8, 8, 64, FAKE, FAKE, None, 320, FAKE), UNSUP),
    ((F16, 2, 8, 8, 64, None, FAKE, None, 64, FAKE), NULL),
    ((F16, 0, 8, 8, 64, None, None, None, 64, None), OK),
])
def test_conv_relu_maxpool_argument_checks(L, args, expect):
    assert L.conv_relu_maxpool(*args, None) == expect


def test_single_operator_argument_checks(L):
    assert L.gemm_bias_act(F16, 10, 12, 64, FAKE, FAKE, None, 1, FAKE, None) == ALIGN
    assert L.gemm_bias_act(F16, 0, 64, 64, None, None, None, 1, None, None) == OK
    assert L.conv_bias_act_nhwc(F16, 1, 4, 4, 64, FAKE, FAKE, 64, 3, 3, 5, None, 1, FAKE, None) == UNSUP
    assert L.maxpool2x2_nhwc(F16, 1, 4, 4, 12, FAKE, FAKE, None) == ALIGN
    assert L.maxpool2x2_nhwc(F16, 1, 1, 4, 16, FAKE, FAKE, None) == SHAPE


def gemm3(L, dt=F16, M=256, K0=64, N0=64, N1=64, N2=64, A=FAKE, W0=FAKE, b0=None, e0=1, W1=FAKE,
          b1=None, e1=1, W2=FAKE, b2=None, e2=0, D=FAKE):
    return L.b2b_gemm3(dt, M, K0, N0, N1, N2, A, W0, b0, e0, W1, b1, e1, W2, b2, e2, D, None)


@pytest.mark.parametrize("kw,expect", [
    (dict(e2=3), UNSUP), (dict(N2=0), SHAPE), (dict(N2=12), ALIGN), (dict(N2=264), UNSUP),
    (dict(N0=128, N1=128), UNSUP),            # two tiles of D0, D1, D2 exceed 512 columns
    (dict(W2=None), NULL), (dict(W2=MIS), ALIGN), (dict(b2=FAKE + 1), ALIGN),
    (dict(M=0, A=None, D=None), OK),
])
def test_b2b_gemm3_argument_checks(L, kw, expect):
    assert gemm3(L, **kw) == expect


def fold(L, dt=F16, Co=64, K=576, out_inner=0, W=FAKE, b=None, g=FAKE, be=FAKE, m=FAKE, v=FAKE,
         eps=1e-5, Wo=FAKE, bo=FAKE):
    return L.b2b_fold_batchnorm(dt, Co, K, out_inner, W, b, g, be, m, v, eps, Wo, bo, None)


@pytest.mark.parametrize("kw,expect", [
    (dict(dt=2), UNSUP), (dict(out_inner=2), UNSUP), (dict(Co=0), SHAPE), (dict(K=-1), SHAPE),
    (dict(eps=-1.0), SHAPE), (dict(eps=float("nan")), SHAPE), (dict(g=None), NULL),
    (dict(Wo=None), NULL), (dict(W=FAKE + 1), ALIGN), (dict(v=FAKE + 2), ALIGN),
    (dict(b=FAKE + 1), ALIGN),
])
def test_fold_batchnorm_argument_checks(L, kw, expect):
    assert fold(L, **kw) == expect


@pytest.mark.skipif(torch.cuda.is_available(), reason="would launch on fake pointers")
def test_valid_call_without_device_reports_cuda_error(L):
    assert gemm(L) == CUDA
    assert fold(L) == CUDA
    assert L.b2b_num_sms() == -1


def test_python_binding_rejects_cpu_tensors():
    A = torch.zeros(16, 64, dtype=torch.float16)
    W = torch.zeros(64, 64, dtype=torch.float16)
    with pytest.raises(ValueError):
        ops.b2b_gemm(A, W, None, W, None)
    with pytest.raises(TypeError):
        ops._dtype_code(A.float())
    with pytest.raises(ValueError):
        ops._epi("gelu")


def test_pad_channels_zero_fills():
    t = torch.arange(2 * 3 * 5, dtype=torch.float16).reshape(2, 3, 5)
    p = ops.pad_channels(t, dim=2)
    assert p.shape == (2, 3, 8)
    assert torch.equal(p[..., :5], t)
    assert torch.count_nonzero(p[..., 5:]) == 0
    assert ops.pad_channels(p, dim=2).shape == (2, 3, 8)


def test_operands_on_different_devices_are_refused_before_any_launch():
    # The library launches on the current device over the pointers it is given; the binding
    # must refuse operands spread over two devices.  CPU and meta tensors stand in for two
    # devices here (no GPU, and nothing is launched).
    from gemm_conv_chains_gb300 import ops
    a = torch.zeros(4)
    b = torch.zeros(4, device="meta")
    assert ops._common_device(A=a, W0=a, b0=None, out=a) == a.device
    with pytest.raises(ValueError, match="one device"):
        ops._common_device(A=a, W0=a, b0=None, out=b)
    with pytest.raises(ValueError):
        ops._common_device(A=None)
