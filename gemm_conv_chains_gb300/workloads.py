"""Seeded synthetic workloads shared by the tests, the benchmark and the smoke check.

This module only draws random numbers and names shapes; it holds none of the chain's
arithmetic, and it is the one piece of code that both the CUDA path's callers and the
CPU oracle's callers use.  Every tensor is drawn on the CPU from ``torch.Generator``
seeded per workload, in the fixed order input, W0, b0, W1, b1, then cast to the storage
dtype, so both sides read identical bits.

The five workloads stand in for the BERT / ResNet-50 operators that the BOLT notes
("Evaluation / Microbenchmarks") benchmark without printing shapes:

  gemm_small  fp16 b2b GEMM A[1024,64] . W0[64,64] (+b0, ReLU) . W1[64,64] (+b1, ReLU)
  gemm_ffn    bf16 b2b GEMM A[32768,256] . W0[256,256] (+b0, Hardswish) . W1[256,128]
              (+b1, Hardswish); the same shape is swept over M = 4096 .. 262144, and
              gemm_ffn_m262144 is its largest point
  conv1x1     fp16 two chained 1x1 convs on x[64,56,56,64], 64->64->64, ReLU/ReLU
  conv3x3_1x1 fp16 conv3x3 (pad 1) 64->64 + Hardswish, then conv1x1 64->128 + bias,
              on x[32,56,56,64]
  conv_pool   fp16 conv3x3 (pad 1) 64->64 + bias + ReLU + maxpool 2x2/2 on
              x[32,112,112,64] -> [32,56,56,64]

Distributions: inputs U[-1,1] (gemm_ffn: N(0,1)); weights N(0, std = 1/sqrt(K)) with K
the reduction length of the GEMM that reads them (K0; N0 for W1; 9*Cin for a 3x3
filter); biases U[-0.1, 0.1].
"""
from __future__ import annotations

import dataclasses
import math
from typing import Dict, Optional

import numpy as np
import torch

DTYPES = {"f16": torch.float16, "bf16": torch.bfloat16}


@dataclasses.dataclass(frozen=True)
class GemmChain:
    """b2b GEMM: out[M,N1] = act1(act0(A[M,K0] W0[K0,N0] + b0) W1[N0,N1] + b1)."""
    name: str
    dtype: str
    M: int
    K0: int
    N0: int
    N1: int
    act0: str
    act1: str
    a_dist: str = "uniform"        # "uniform" U[-1,1] or "normal" N(0,1)
    bias: bool = True

    @property
    def flops(self) -> int:
        return 2 * self.M * (self.K0 * self.N0 + self.N0 * self.N1)

    @property
    def floor_bytes(self) -> int:
        """A + W0 + b0 + W1 + b1 + out: the chain's irreducible HBM traffic."""
        e = 2
        b = (self.N0 + self.N1) * e if self.bias else 0
        return e * (self.M * self.K0 + self.K0 * self.N0 + self.N0 * self.N1
                    + self.M * self.N1) + b

    @property
    def unfused_bytes(self) -> int:
        """Floor plus the intermediate written by GEMM0 and read back by GEMM1."""
        return self.floor_bytes + 2 * 2 * self.M * self.N0

    def with_m(self, M: int) -> "GemmChain":
        return dataclasses.replace(self, M=M, name=f"{self.name}_m{M}")


@dataclasses.dataclass(frozen=True)
class GemmChain3:
    """Three-operator chain: out[M,N2] = act2(act1(act0(A W0 + b0) W1 + b1) W2 + b2)."""
    name: str
    dtype: str
    M: int
    K0: int
    N0: int
    N1: int
    N2: int
    act0: str
    act1: str
    act2: str

    @property
    def flops(self) -> int:
        return 2 * self.M * (self.K0 * self.N0 + self.N0 * self.N1 + self.N1 * self.N2)

    @property
    def floor_bytes(self) -> int:
        e = 2
        return e * (self.M * self.K0 + self.K0 * self.N0 + self.N0 * self.N1 + self.N1 * self.N2
                    + self.N0 + self.N1 + self.N2 + self.M * self.N2)

    @property
    def unfused_bytes(self) -> int:
        """Floor plus both intermediates written and read back."""
        return self.floor_bytes + 2 * 2 * self.M * (self.N0 + self.N1)


@dataclasses.dataclass(frozen=True)
class ConvChain:
    """conv RxS (pad, stride) + b0 + act0 -> conv1x1 + b1 + act1, NHWC."""
    name: str
    dtype: str
    N: int
    H: int
    W: int
    C: int
    C0: int
    R: int
    S: int
    pad: int
    C1: int
    act0: str
    act1: str
    stride: int = 1

    @property
    def Ho(self) -> int:
        return max(0, (self.H + 2 * self.pad - self.R) // self.stride + 1)

    @property
    def Wo(self) -> int:
        return max(0, (self.W + 2 * self.pad - self.S) // self.stride + 1)

    @property
    def M(self) -> int:
        return self.N * self.Ho * self.Wo

    @property
    def flops(self) -> int:
        return 2 * self.M * (self.R * self.S * self.C * self.C0 + self.C0 * self.C1)

    @property
    def floor_bytes(self) -> int:
        e = 2
        return e * (self.N * self.H * self.W * self.C + self.C0 * self.R * self.S * self.C
                    + self.C0 + self.C1 * self.C0 + self.C1 + self.M * self.C1)

    @property
    def unfused_bytes(self) -> int:
        return self.floor_bytes + 2 * 2 * self.M * self.C0


@dataclasses.dataclass(frozen=True)
class ConvPool:
    """conv3x3 (pad 1, stride 1) + bias + ReLU + maxpool 2x2 stride 2 (floor), NHWC."""
    name: str
    dtype: str
    N: int
    H: int
    W: int
    Cin: int
    Cout: int

    @property
    def flops(self) -> int:
        return 2 * self.N * self.H * self.W * 9 * self.Cin * self.Cout

    @property
    def floor_bytes(self) -> int:
        e = 2
        return e * (self.N * self.H * self.W * self.Cin + self.Cout * 9 * self.Cin + self.Cout
                    + self.N * (self.H // 2) * (self.W // 2) * self.Cout)

    @property
    def unfused_bytes(self) -> int:
        # conv output written, then read by the pool
        return self.floor_bytes + 2 * 2 * self.N * self.H * self.W * self.Cout


GEMM_SMALL = GemmChain("gemm_small", "f16", 1024, 64, 64, 64, "relu", "relu")
GEMM_FFN = GemmChain("gemm_ffn", "bf16", 32768, 256, 256, 128, "hardswish", "hardswish",
                     a_dist="normal")
CONV1X1 = ConvChain("conv1x1", "f16", 64, 56, 56, 64, 64, 1, 1, 0, 64, "relu", "relu")
CONV3X3_1X1 = ConvChain("conv3x3_1x1", "f16", 32, 56, 56, 64, 64, 3, 3, 1, 128,
                        "hardswish", "none")
CONV_POOL = ConvPool("conv_pool", "f16", 32, 112, 112, 64, 64)
# A downsampling stage: 3x3 stride 2 conv (56 -> 28, 64 -> 128 channels) + 1x1 (128 -> 128).
CONV3X3S2_1X1 = ConvChain("conv3x3s2_1x1", "f16", 32, 56, 56, 64, 128, 3, 3, 1, 128, "relu",
                          "none", stride=2)

# A wide chain: 256 -> 512 -> 128 over 32768 rows, bf16 (GEMM0 wider than one MMA).
GEMM_WIDE = GemmChain("gemm_wide", "bf16", 32768, 256, 512, 128, "hardswish", "hardswish",
                      a_dist="normal")
# A three-operator MLP head: 128 -> 128 -> 64 -> 64 over 32768 rows, bf16.
MLP3 = GemmChain3("mlp3", "bf16", 32768, 128, 128, 64, 64, "hardswish", "hardswish", "none")

FFN_SWEEP_M = [4096, 8192, 16384, 32768, 65536, 131072, 262144]
# The largest point of the FFN-like chain's M sweep: 2048 tiles, 13 or 14 per SM.
GEMM_FFN_LARGE = GEMM_FFN.with_m(FFN_SWEEP_M[-1])

WORKLOADS = {w.name: w for w in (GEMM_SMALL, GEMM_FFN, GEMM_FFN_LARGE, CONV1X1, CONV3X3_1X1,
                                 CONV_POOL, CONV3X3S2_1X1, MLP3, GEMM_WIDE)}


# ------------------------------------------------------------------------------------
# random draws
# ------------------------------------------------------------------------------------

def _gen(seed: int) -> torch.Generator:
    g = torch.Generator(device="cpu")
    g.manual_seed(seed)
    return g


def _uniform(g, shape, lo, hi):
    return torch.rand(shape, generator=g, dtype=torch.float32) * (hi - lo) + lo


def _normal(g, shape, std):
    return torch.randn(shape, generator=g, dtype=torch.float32) * std


def _ints(g, shape, lo, hi):
    """Integers uniformly in [lo, hi], exactly representable in fp16 and bf16."""
    return torch.randint(lo, hi + 1, shape, generator=g, dtype=torch.int64).to(torch.float32)


def gemm_inputs(w: GemmChain, seed: int = 0, integer: bool = False) -> Dict[str, torch.Tensor]:
    """A [M,K0], W0 [K0,N0], b0 [N0], W1 [N0,N1], b1 [N1] on the CPU, storage dtype."""
    g = _gen(seed)
    dt = DTYPES[w.dtype]
    if integer:
        A = _ints(g, (w.M, w.K0), -3, 3)
        W0 = _ints(g, (w.K0, w.N0), -3, 3)
        b0 = _ints(g, (w.N0,), -2, 2)
        W1 = _ints(g, (w.N0, w.N1), -3, 3)
        b1 = _ints(g, (w.N1,), -2, 2)
    else:
        A = _normal(g, (w.M, w.K0), 1.0) if w.a_dist == "normal" else _uniform(g, (w.M, w.K0), -1, 1)
        W0 = _normal(g, (w.K0, w.N0), 1.0 / math.sqrt(w.K0))
        b0 = _uniform(g, (w.N0,), -0.1, 0.1)
        W1 = _normal(g, (w.N0, w.N1), 1.0 / math.sqrt(w.N0))
        b1 = _uniform(g, (w.N1,), -0.1, 0.1)
    out = {"A": A, "W0": W0, "b0": b0, "W1": W1, "b1": b1}
    if not w.bias:
        out["b0"] = None
        out["b1"] = None
    return {k: (v.to(dt).contiguous() if v is not None else None) for k, v in out.items()}


def gemm3_inputs(w: GemmChain3, seed: int = 0, integer: bool = False) -> Dict[str, torch.Tensor]:
    """A [M,K0], W0 [K0,N0], b0, W1 [N0,N1], b1, W2 [N1,N2], b2 on the CPU, storage dtype.
    Integer data are in {-1, 0, 1} (biases too), so that three layers of sums stay exact
    and, for these sizes, finite in fp16."""
    g = _gen(seed)
    dt = DTYPES[w.dtype]
    dims = [(w.K0, w.N0), (w.N0, w.N1), (w.N1, w.N2)]
    if integer:
        A = _ints(g, (w.M, w.K0), -1, 1)
        ws = [(_ints(g, d, -1, 1), _ints(g, (d[1],), -1, 1)) for d in dims]
    else:
        A = _uniform(g, (w.M, w.K0), -1, 1)
        ws = [(_normal(g, d, 1.0 / math.sqrt(d[0])), _uniform(g, (d[1],), -0.1, 0.1)) for d in dims]
    out = {"A": A, "W0": ws[0][0], "b0": ws[0][1], "W1": ws[1][0], "b1": ws[1][1],
           "W2": ws[2][0], "b2": ws[2][1]}
    return {k: v.to(dt).contiguous() for k, v in out.items()}


def conv_inputs(w: ConvChain, seed: int = 0, integer: bool = False) -> Dict[str, torch.Tensor]:
    """x [N,H,W,C], W0 [C0,R,S,C], b0 [C0], W1 [C1,C0], b1 [C1] on the CPU."""
    g = _gen(seed)
    dt = DTYPES[w.dtype]
    if integer:
        x = _ints(g, (w.N, w.H, w.W, w.C), -3, 3)
        W0 = _ints(g, (w.C0, w.R, w.S, w.C), -3, 3)
        b0 = _ints(g, (w.C0,), -2, 2)
        W1 = _ints(g, (w.C1, w.C0), -3, 3)
        b1 = _ints(g, (w.C1,), -2, 2)
    else:
        x = _uniform(g, (w.N, w.H, w.W, w.C), -1, 1)
        W0 = _normal(g, (w.C0, w.R, w.S, w.C), 1.0 / math.sqrt(w.R * w.S * w.C))
        b0 = _uniform(g, (w.C0,), -0.1, 0.1)
        W1 = _normal(g, (w.C1, w.C0), 1.0 / math.sqrt(w.C0))
        b1 = _uniform(g, (w.C1,), -0.1, 0.1)
    return {k: v.to(dt).contiguous() for k, v in
            {"x": x, "W0": W0, "b0": b0, "W1": W1, "b1": b1}.items()}


def pool_inputs(w: ConvPool, seed: int = 0, integer: bool = False) -> Dict[str, torch.Tensor]:
    """x [N,H,W,Cin], Wt [Cout,3,3,Cin], b [Cout] on the CPU."""
    g = _gen(seed)
    dt = DTYPES[w.dtype]
    if integer:
        x = _ints(g, (w.N, w.H, w.W, w.Cin), -3, 3)
        Wt = _ints(g, (w.Cout, 3, 3, w.Cin), -3, 3)
        b = _ints(g, (w.Cout,), -2, 2)
    else:
        x = _uniform(g, (w.N, w.H, w.W, w.Cin), -1, 1)
        Wt = _normal(g, (w.Cout, 3, 3, w.Cin), 1.0 / math.sqrt(9 * w.Cin))
        b = _uniform(g, (w.Cout,), -0.1, 0.1)
    return {k: v.to(dt).contiguous() for k, v in {"x": x, "Wt": Wt, "b": b}.items()}


def to_bits(t: Optional[torch.Tensor]) -> Optional[np.ndarray]:
    """fp16/bf16 CPU tensor -> numpy uint16 array of the same bit patterns."""
    if t is None:
        return None
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def from_bits(a: np.ndarray, dtype: str) -> torch.Tensor:
    """numpy uint16 bit patterns -> CPU tensor of the storage dtype."""
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(DTYPES[dtype])
