"""Tile-graph model of the fused chains, on the host (no CUDA).

Welder notes, "Operator-tile and Tile-graph": once two operators are connected through a
reuse tile, every tile of the connected graph follows from the output tile (tile
propagation; for a convolution the input tile is the output tile plus the filter halo,
an upper bound on the region read), the memory traffic of a level is the sum of the
tiles it moves, and the footprint is what a best-fit allocation of the live buffers,
in topological order, needs.  Here the model is applied to the chain kernels of this
package: `propagate` gives the operand tiles of one output tile, `dram_traffic` the
unique bytes of a launch, `l2_to_smem_traffic` the bytes the kernel's TMA and global
loads move from L2 into the SMs for a given launch plan (`ops.debug_plan`; whole boxes,
out-of-bounds fill included), and
`smem_footprint` a best-fit allocation of buffers by lifetime.  Predictions are compared
with the ncu counters of the same launches in the profile summaries.

Welder notes, "Scheduling policy": the model also chooses.  `rank` enumerates the layouts
the planner finds feasible for a problem (`ops.debug_plan(..., cand=i)`), drops those over
the shared-memory / TMEM footprint, and orders the rest by their launch bounds; `choose`
hands the top k to the light-weight profiler (`ops.set_candidates`), which times only those
and keeps the fastest.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Dict, Iterable, List, Optional, Sequence, Tuple

from . import workloads as wl

ELEM = 2          # fp16 / bf16 bytes
TILE_M = 128      # rows of a 2-D tile = TMEM lanes
TILE_H, TILE_W = 8, 16   # output pixels of a conv tile


# ------------------------------------------------------------------------------------
# propagation
# ------------------------------------------------------------------------------------
@dataclasses.dataclass(frozen=True)
class TileGraph:
    """Operand tiles (element shapes) of one output tile of a fused chain."""
    kind: str
    tiles: Dict[str, Tuple[int, ...]]

    def bytes(self, name: str) -> int:
        return math.prod(self.tiles[name]) * ELEM


def propagate(w) -> TileGraph:
    """Every operand tile of the chain from its output tile.

    b2b GEMM: out (128, N1) <- P (128, N0), W1 (N0, N1) <- A (128, K0), W0 (K0, N0).
    Conv chain: out (8, 16, C1) <- P (8, 16, C0), W1 (C1, C0) <- x (7 st + R, 15 st + S, C)
    (the region an 8 x 16 output tile reads at stride st, an upper bound: every st-th pixel
    of it is used), W0 (C0, R, S, C).  Conv + pool: pooled (4, 8, F) <- conv out (8, 16, F) (the (2,2,F)
    reuse tile per pooled pixel) <- x (10, 18, C), W (F, 3, 3, C)."""
    if isinstance(w, wl.GemmChain):
        return TileGraph("gemm_chain", {"out": (TILE_M, w.N1), "P": (TILE_M, w.N0),
                                        "W1": (w.N0, w.N1), "A": (TILE_M, w.K0),
                                        "W0": (w.K0, w.N0)})
    if isinstance(w, wl.GemmChain3):
        return TileGraph("gemm_chain3", {"out": (TILE_M, w.N2), "P1": (TILE_M, w.N1),
                                         "W2": (w.N1, w.N2), "P0": (TILE_M, w.N0),
                                         "W1": (w.N0, w.N1), "A": (TILE_M, w.K0),
                                         "W0": (w.K0, w.N0)})
    if isinstance(w, wl.ConvChain):
        return TileGraph("conv_chain", {"out": (TILE_H, TILE_W, w.C1),
                                        "P": (TILE_H, TILE_W, w.C0), "W1": (w.C1, w.C0),
                                        "x": ((TILE_H - 1) * w.stride + w.R,
                                              (TILE_W - 1) * w.stride + w.S, w.C),
                                        "W0": (w.C0, w.R, w.S, w.C)})
    if isinstance(w, wl.ConvPool):
        return TileGraph("conv_pool", {"out": (TILE_H // 2, TILE_W // 2, w.Cout),
                                       "conv": (TILE_H, TILE_W, w.Cout),
                                       "x": (TILE_H + 2, TILE_W + 2, w.Cin),
                                       "W": (w.Cout, 3, 3, w.Cin)})
    raise TypeError(w)


# ------------------------------------------------------------------------------------
# traffic
# ------------------------------------------------------------------------------------
def dram_traffic(w, fused: bool = True) -> int:
    """Unique bytes of one launch: each tensor read or written once (the sum of the
    chain's input and output tensors).  Unfused, the intermediate is written by the first
    operator and read back by the second."""
    return w.floor_bytes if fused else w.unfused_bytes


def plan_of(w) -> dict:
    """The C planner's launch plan for a workload."""
    from . import ops
    return ops.debug_plan(*problem_of(w))


def tiles_per_cta(num_tiles: int, num_sms: int) -> List[int]:
    """Tiles of each CTA of the persistent grid (CTA b takes tiles b, b + grid, ...)."""
    grid = max(1, min(num_tiles, num_sms))
    return [len(range(b, num_tiles, grid)) for b in range(grid)]


def _overlap(lo: int, n: int, extent: int) -> int:
    """Length of [lo, lo + n) inside [0, extent): TMA fetches only in-bounds elements."""
    return max(0, min(lo + n, extent) - max(lo, 0))


def _strided_overlap(lo: int, n: int, step: int, extent: int) -> int:
    """How many of lo, lo + step, ..., lo + (n - 1) step lie in [0, extent)."""
    if step == 1:
        return _overlap(lo, n, extent)
    return sum(1 for i in range(n) if 0 <= lo + i * step < extent)


def _conv_tile_input_bytes(N, H, W, C, R, S, pad, halo: bool, stride: int = 1) -> int:
    """Input bytes inside the image that all tiles of an RxS conv (8 x 16 output tiles)
    read: one box of (8 + R - 1) x 16 pixels per column tap with halo loads, else one
    8 x 16 box per tap (pixels `stride` apart), each clipped to the image (the useful part
    of the boxes)."""
    Ho, Wo = (H + 2 * pad - R) // stride + 1, (W + 2 * pad - S) // stride + 1
    tiles_h, tiles_w = -(-Ho // TILE_H), -(-Wo // TILE_W)
    rows_per_box = TILE_H + R - 1 if halo else TILE_H
    row_offsets = [0] if halo else list(range(R))
    total = 0
    for th in range(tiles_h):
        for tw in range(tiles_w):
            for s in range(S):
                cols = _strided_overlap(tw * TILE_W * stride + s - pad, TILE_W, stride, W)
                for r in row_offsets:
                    rows = _strided_overlap(th * TILE_H * stride + r - pad, rows_per_box, stride, H)
                    total += rows * cols
    return N * total * C * ELEM


A_BOX = TILE_M * 64 * ELEM   # one 128-row x 64-element A box (16 KiB)


def l2_to_smem_traffic(w, plan: Optional[dict] = None, num_sms: int = 152) -> Dict[str, int]:
    """Bytes one fused launch moves from L2 into the SMs, by operand, for `plan`.

    Every TMA load moves its whole box: elements outside the tensor are filled with zeros
    in shared memory but cross the L2 -> SM crossbar all the same (ncu's
    l1tex__m_xbar2l1tex_read_bytes of the 3x3 conv chains on 56 x 56 and 64 x 64 images
    and of conv + pool equals the whole-box sum to the byte).  A: per tile, one box per
    K chunk (2-D; twice in wide chains, once per half of N0), or per column tap and channel block (halo boxes of (8 + R - 1) x 16
    pixels), or per tap and channel block (8 x 16 pixels).  Weights: once per CTA when
    resident; when streamed, W0 once per tile and W1 once per tile, or once per pair of
    tiles when the plan groups W1 (P in TMEM).  Biases: once per CTA (plain loads by the
    epilogue warps).  `A_in_bounds` (not in the total) is the part of A inside the
    tensor; A / A_in_bounds is the waste of ragged and halo tiles."""
    plan = plan or plan_of(w)
    if _pool_pair(plan):
        # conv + pool pairs: each CTA its own tile's halo boxes (an odd last pair-tile's
        # empty second tile included), its half of the filters once and the bias of every
        # channel once
        pairs = len(tiles_per_cta(-(-plan["tiles"] // 2), num_sms // 2))
        out = {"A": 2 * -(-plan["tiles"] // 2) * (plan["kchunks0"] // 3) * plan["a_stage_bytes"],
               "W0": 2 * pairs * plan["kchunks0"] * plan["w0_chunk"],
               "bias": 2 * pairs * plan["N0p"] * ELEM}
        out["total"] = sum(out.values())
        out["A_in_bounds"] = _conv_tile_input_bytes(w.N, w.H, w.W, w.Cin, 3, 3, 1, True)
        return out
    if plan.get("cta_pair"):
        return _cta_pair_traffic(w, plan, num_sms)
    per_cta = tiles_per_cta(plan["tiles"], num_sms)
    ctas = len(per_cta)
    tiles = plan["tiles"]
    out: Dict[str, int] = {}
    R = getattr(w, "R", 3 if isinstance(w, wl.ConvPool) else 1)
    a_tile = (plan["kchunks0"] // R * plan["a_stage_bytes"] if plan["halo"]
              else plan["kchunks0"] * A_BOX)
    w0 = plan["kchunks0"] * plan["w0_chunk"]
    if plan["p_split"]:
        # wide chains: GEMM0 in two passes over the halves of N0, each reading the A chunks
        # again with that half's W0 blocks (one box of four blocks, or one per block)
        a_tile *= 2
        n0blk = -(-plan["N0p"] // 64)
        hi = plan["w0_chunk"] if w.N0 % 64 == 0 else (n0blk - 4) * 8192
        w0 = plan["kchunks0"] * (plan["w0_chunk"] + hi)
    out["A"] = tiles * a_tile
    w1 = plan["kchunks1"] * plan["w1_chunk"]
    if isinstance(w, wl.GemmChain3):
        # W0, W1 by TMA boxes and W2 by the epilogue warps' loads (its bytes, unpadded),
        # once per CTA
        out["W0"], out["W1"] = ctas * w0, ctas * w1
        out["W2"] = ctas * w.N1 * w.N2 * ELEM
        out["bias"] = ctas * (w.N0 + w.N1 + w.N2) * ELEM
        out["total"] = sum(out.values())
        out["A_in_bounds"] = w.M * w.K0 * ELEM
        return out
    if plan["resident"]:
        out["W0"] = ctas * w0
        if w1:
            out["W1"] = ctas * w1
    elif plan.get("w0_res"):
        # W0 alone resident, W1 streamed (once per pair of tiles when grouped)
        out["W0"] = ctas * w0
        loads_w1 = sum(-(-n // 2) for n in per_cta) if plan["w1_group"] else tiles
        out["W1"] = loads_w1 * w1
    else:
        out["W0"] = tiles * w0
        if w1:
            loads_w1 = sum(-(-n // 2) for n in per_cta) if plan["w1_group"] else tiles
            out["W1"] = loads_w1 * w1
    if isinstance(w, wl.GemmChain):
        out["bias"] = ctas * (w.N0 + w.N1) * ELEM
        useful = w.M * w.K0 * ELEM
    elif isinstance(w, wl.ConvChain):
        out["bias"] = ctas * (w.C0 + w.C1) * ELEM
        useful = (w.N * w.H * w.W * w.C * ELEM if (w.R, w.S, w.pad, w.stride) == (1, 1, 0, 1) else
                  _conv_tile_input_bytes(w.N, w.H, w.W, w.C, w.R, w.S, w.pad, bool(plan["halo"]),
                                         w.stride))
    else:
        out["bias"] = ctas * w.Cout * ELEM
        useful = _conv_tile_input_bytes(w.N, w.H, w.W, w.Cin, 3, 3, 1, bool(plan["halo"]))
    out["total"] = sum(out.values())
    out["A_in_bounds"] = useful
    return out


def _cta_pair_traffic(w, plan: dict, num_sms: int) -> Dict[str, int]:
    """l2_to_smem_traffic of a plan over CTA pairs (b2b GEMM chains): 256-row tiles on up to
    num_sms / 2 pairs; each CTA loads its 128 rows of every A chunk, its halves of W0 and W1
    once, and its halves of the biases."""
    pairs = len(tiles_per_cta(plan["tiles"], num_sms // 2))
    ctas = 2 * pairs
    out: Dict[str, int] = {}
    out["A"] = plan["tiles"] * 2 * plan["kchunks0"] * A_BOX
    out["W0"] = ctas * plan["kchunks0"] * plan["w0_chunk"]
    out["W1"] = ctas * plan["kchunks1"] * plan["w1_chunk"]
    out["bias"] = ctas * (plan["N0p"] // 2 + plan["N1p"] // 2) * ELEM
    out["total"] = sum(out.values())
    out["A_in_bounds"] = w.M * w.K0 * ELEM
    return out


# ------------------------------------------------------------------------------------
# footprint
# ------------------------------------------------------------------------------------
@dataclasses.dataclass(frozen=True)
class Buffer:
    name: str
    size: int
    live: Tuple[int, int]        # [first step, last step] in topological order
    align: int = 1024


def best_fit(buffers: Sequence[Buffer]) -> Tuple[int, Dict[str, int]]:
    """Offsets of `buffers` such that two buffers live at a common step never overlap:
    buffers are placed largest first, each at the lowest aligned offset that fits beside
    the already placed buffers whose lifetimes intersect its own.  Returns (extent,
    offsets)."""
    placed: List[Tuple[Buffer, int]] = []
    offsets: Dict[str, int] = {}
    for b in sorted(buffers, key=lambda b: (-b.size, b.name)):
        busy = sorted((off, off + o.size) for o, off in placed
                      if not (o.live[1] < b.live[0] or b.live[1] < o.live[0]))
        off = 0
        for lo, hi in busy:
            if off + b.size <= lo:
                break
            off = max(off, -(-hi // b.align) * b.align)
        placed.append((b, off))
        offsets[b.name] = off
    extent = max((off + b.size for b, off in placed), default=0)
    return extent, offsets


def chain_buffers(plan: dict) -> List[Buffer]:
    """Shared-memory buffers of a launch plan, with lifetimes over the steps of one tile:
    0 load, 1 GEMM0, 2 epilogue 0 (writes P), 3 GEMM1 (reads P), 4 epilogue 1 (writes the
    output staging), 5 store.  The ring, resident weights, bias operands and barriers live
    throughout.  When the plan lets the output staging reuse the P buffers (`alias`: the
    epilogue waits for the previous store's reads before it writes P), a slot's P and its
    staging are used one after the other by the same tiles, so their lifetimes are
    disjoint; otherwise the tiles in flight (and the TMA store still reading a staging
    buffer while the next tile's P is written) keep every buffer live at every step."""
    whole = (0, 5)
    bufs = [Buffer("ring", plan["ring"], whole), Buffer("bias", plan["bias"], whole),
            Buffer("bar", plan["bar"], whole)]
    if _pool_pair(plan):
        # conv + pool pairs: half of the filters resident, one pooled staging tile per
        # epilogue warpgroup
        return bufs + [Buffer("weights", plan["w_res"], whole), Buffer("out0", plan["out"], whole),
                       Buffer("out1", plan["out"], whole)]
    if plan.get("cta_pair"):
        # CTA pairs: the halves of both weights resident, P in TMEM, and (when the ring keeps
        # five stages beside it) a 4 KiB output staging slot per epilogue warp
        extra = [Buffer("out", plan["out"], whole)] if plan["out"] else []
        return bufs + [Buffer("weights", plan["w_res"], whole)] + extra
    if plan["resident"] or plan.get("w0_res"):
        bufs.append(Buffer("weights", plan["w_res"], whole))
    if plan["mode"] == 3:
        # three-operator chain: two tiles in flight hold P0, P1 and the staging of both (with
        # `alias`, staging b shares P0[b]'s space: the P0 buffers are then that size)
        p1 = (plan["off_p1_1"] - plan["off_p1_0"])
        for b in range(2):
            bufs += [Buffer(f"P0{b}", plan["p"], whole), Buffer(f"P1{b}", p1, whole)]
            if not plan["alias"]:
                bufs.append(Buffer(f"out{b}", plan["out"], whole))
        return bufs
    chain = plan["mode"] == 0
    pbufs = plan["nbuf"] if (chain and not plan["p_tmem"]) else 0
    p_bytes = (plan["N0p"] + 63) // 64 * 128 * 128
    out_cols = plan["N1p"] if chain else plan["N0p"]
    per_chunk = 32 * 128 if plan["mode"] == 2 else 128 * 128   # pooled: 4 x 8 pixels per tile
    out_bytes = (out_cols + 63) // 64 * per_chunk
    # (W0 resident beside streamed W1: the output leaves from registers, no staging; the
    # conv chain's two-issuer layout: one 1 KiB slot per epilogue warp, `out` bytes in all)
    if plan.get("out_slots"):
        return bufs + [Buffer(f"P{i}", p_bytes, whole) for i in range(pbufs)] + \
            [Buffer("out", plan["out"], whole)]
    obufs = 0 if plan.get("w0_res") else (2 if plan["groups"] == 2 else 1)
    paired = bool(plan["alias"]) and pbufs == obufs
    for i in range(pbufs):
        bufs.append(Buffer(f"P{i}", p_bytes, (2, 3) if paired else whole))
    for i in range(obufs):
        bufs.append(Buffer(f"out{i}", out_bytes, (4, 5) if paired else whole))
    return bufs


def smem_footprint(plan: dict) -> int:
    """Best-fit shared-memory extent of a plan's buffers (without the 1 KiB the kernel
    adds to align its base)."""
    return best_fit(chain_buffers(plan))[0]


# ------------------------------------------------------------------------------------
# model vs. counters
# ------------------------------------------------------------------------------------
NCU_L2_TO_SM = "l1tex__m_xbar2l1tex_read_bytes.sum"
NCU_DRAM = ("dram__bytes_read.sum", "dram__bytes_write.sum")


def read_ncu_raw_csv(path: str) -> Dict[str, float]:
    """First launch of an `ncu -i <report> --page raw --csv` export, metric -> value in
    bytes where the unit is a byte multiple."""
    import csv
    scale = {"byte": 1, "Kbyte": 1e3, "Mbyte": 1e6, "Gbyte": 1e9}
    with open(path, newline="") as f:
        rows = list(csv.reader(f))
    hdr = next(i for i, r in enumerate(rows) if r and r[0] == "ID")
    names, units, vals = rows[hdr], rows[hdr + 1], rows[hdr + 2]
    out: Dict[str, float] = {}
    for n, u, v in zip(names, units, vals):
        try:
            x = float(v.replace(",", ""))
        except ValueError:
            continue
        out[n] = x * scale.get(u, 1)
    return out


# Per-SM TMA ingress from L2 measured on the GB300 for one SM loading alone (~89 B/clk);
# with every SM loading inside the FFN chain it was ~55 B/clk (48 KiB stages ~0.42 us
# apart), so the L2 bound below is optimistic.
L2_TO_SM_BYTES_PER_CLK = 89.0


def mma_factor(n: int, pair: bool = False) -> float:
    """How much longer than the bf16 peak allows a GEMM of MMA width N takes: an MMA of
    128 rows per SM needs N / 2 cycles at the peak, but short ones take a floor (measured,
    operands resident: M128 x N64 x K16 48 cycles, a pair's M256 x N64 x K16 43 cycles per
    SM's 128 rows; N >= 128 runs at the peak)."""
    return max(1.0, (43.0 if pair else 48.0) / max(1.0, n / 2))


def gemm_shapes(w) -> List[Tuple[float, int]]:
    """Each GEMM of the workload's fused launch: its FLOPs and its MMA width N (padded to
    16; GEMM0 of a wide chain runs in passes of at most 256)."""
    r16 = lambda n: -(-n // 16) * 16
    if isinstance(w, wl.GemmChain3):
        return [(2.0 * w.M * w.K0 * w.N0, r16(w.N0)), (2.0 * w.M * w.N0 * w.N1, r16(w.N1)),
                (2.0 * w.M * w.N1 * w.N2, r16(w.N2))]
    if isinstance(w, wl.GemmChain):
        out = [(2.0 * w.M * w.K0 * w.N0, r16(min(w.N0, 256)))]
        if w.N1:
            out.append((2.0 * w.M * w.N0 * w.N1, r16(w.N1)))
        return out
    if isinstance(w, wl.ConvChain):
        out = [(2.0 * w.M * w.R * w.S * w.C * w.C0, r16(w.C0))]
        if w.C1:
            out.append((2.0 * w.M * w.C0 * w.C1, r16(w.C1)))
        return out
    return [(float(w.flops), r16(w.Cout))]


def _mma_flops(w, pair: bool) -> float:
    """The workload's FLOPs weighted by mma_factor: its MMA time at the peak rate."""
    return sum(f * mma_factor(n, pair) for f, n in gemm_shapes(w))


def _pool_pair(plan: dict) -> bool:
    return bool(plan.get("cta_pair")) and plan["mode"] == 2


def launch_bounds(w, plan: Optional[dict] = None, hbm_gbs: float = 6791.4,
                  tensor_tflops: float = 1951.4, sm_mhz: float = 2070.0,
                  num_sms: int = 152) -> Dict[str, float]:
    """Lower bounds, in microseconds, on one fused launch from each resource it streams
    through.  HBM: the algorithmic bytes (inputs, weights, biases, output) over the copy
    bandwidth.  L2 -> SM: the busiest CTA's bytes (its tiles' A and streamed weights, W1
    once per pair of tiles when grouped, its resident weights and biases) over one SM's
    TMA ingress.  Tensor: the busiest CTA's share of the MMA FLOPs over one SM's share of
    the peak.  `floor` is the largest; `bound` names it."""
    plan = plan or plan_of(w)
    if _pool_pair(plan):
        # conv + pool pairs: per SM its own tile of each of its pair's pair-tiles (halo
        # boxes), its half of the filters, the bias of every channel, one tile's MMA FLOPs
        # per pair-tile
        n = max(tiles_per_cta(-(-plan["tiles"] // 2), num_sms // 2))
        R = getattr(w, "R", 3)
        cta_bytes = (plan["kchunks0"] // R * plan["a_stage_bytes"] * n
                     + plan["kchunks0"] * plan["w0_chunk"] + plan["N0p"] * ELEM)
        out = {"hbm_us": w.floor_bytes / (hbm_gbs * 1e3),
               "l2_us": cta_bytes / (L2_TO_SM_BYTES_PER_CLK * sm_mhz),
               "tensor_us": _mma_flops(w, True) / plan["tiles"] * n / (tensor_tflops * 1e6 / num_sms)}
        out["bound"] = max(out, key=out.get)[:-3]
        out["floor_us"] = max(out["hbm_us"], out["l2_us"], out["tensor_us"])
        return out
    if plan.get("cta_pair"):
        # pairs of SMs share each 256-row tile; per SM: 128 rows of each of its pair's tiles,
        # its weight halves, half of each tile's MMA FLOPs
        per_pair = tiles_per_cta(plan["tiles"], num_sms // 2)
        n = max(per_pair)
        t = l2_to_smem_traffic(w, plan, num_sms)
        ctas = 2 * len(per_pair)
        cta_bytes = (t["A"] / (2 * plan["tiles"]) * n + (t["W0"] + t["W1"] + t["bias"]) / ctas)
        out = {"hbm_us": w.floor_bytes / (hbm_gbs * 1e3),
               "l2_us": cta_bytes / (L2_TO_SM_BYTES_PER_CLK * sm_mhz),
               "tensor_us": _mma_flops(w, True) / (2 * plan["tiles"]) * n
               / (tensor_tflops * 1e6 / num_sms)}
        out["bound"] = max(out, key=out.get)[:-3]
        out["floor_us"] = max(out["hbm_us"], out["l2_us"], out["tensor_us"])
        return out
    per_cta = tiles_per_cta(plan["tiles"], num_sms)
    ctas, tiles, n = len(per_cta), plan["tiles"], max(per_cta)
    t = l2_to_smem_traffic(w, plan, num_sms)
    cta_bytes = t["A"] / tiles * n + t.get("bias", 0) / ctas + t.get("W2", 0) / ctas
    for k in ("W0", "W1"):
        if k not in t:
            continue
        if plan["resident"] or isinstance(w, wl.GemmChain3) or (k == "W0" and plan.get("w0_res")):
            cta_bytes += t[k] / ctas
        elif k == "W1" and plan["w1_group"]:
            loads = sum(-(-m // 2) for m in per_cta)
            cta_bytes += t[k] / loads * -(-n // 2)
        else:
            cta_bytes += t[k] / tiles * n
    out = {
        "hbm_us": w.floor_bytes / (hbm_gbs * 1e3),
        "l2_us": cta_bytes / (L2_TO_SM_BYTES_PER_CLK * sm_mhz),
        "tensor_us": _mma_flops(w, False) / tiles * n / (tensor_tflops * 1e6 / num_sms),
    }
    out["bound"] = max(out, key=out.get)[:-3]
    out["floor_us"] = max(out["hbm_us"], out["l2_us"], out["tensor_us"])
    return out


# ------------------------------------------------------------------------------------
# choosing: enumerate, check the footprint, rank, hand the top candidates to the profiler
# ------------------------------------------------------------------------------------
SMEM_LIMIT = 227 * 1024     # dynamic shared memory per CTA
TMEM_COLS = 512             # TMEM columns per SM
RANK_TOL = 0.02             # bounds closer than this (relative) count as equal
STEADY_TILES = 3            # tiles per CTA (or pair) from which the bounds rank layouts


@dataclasses.dataclass(frozen=True)
class GemmSingle(wl.GemmChain):
    """One GEMM + bias + activation (gemm_bias_act) in the chain's terms: N1 = 0, and the
    output is the M x N0 product."""

    @property
    def floor_bytes(self) -> int:
        return 2 * (self.M * self.K0 + self.K0 * self.N0 + self.N0 + self.M * self.N0)


@dataclasses.dataclass(frozen=True)
class ConvSingle(wl.ConvChain):
    """One conv + bias + activation (conv_bias_act_nhwc) in the chain's terms: C1 = 0, and
    the output is the M x C0 conv."""

    @property
    def floor_bytes(self) -> int:
        return 2 * (self.N * self.H * self.W * self.C + self.C0 * self.R * self.S * self.C
                    + self.C0 + self.M * self.C0)


def problem_of(w) -> Tuple[str, Tuple[int, ...]]:
    """The entry point and sizes (as the plan functions take them) of a workload."""
    if isinstance(w, GemmSingle):
        return "gemm_bias_act", (w.M, w.K0, w.N0)
    if isinstance(w, ConvSingle):
        return "conv_bias_act_nhwc", (w.N, w.H, w.W, w.C, w.C0, w.R, w.S, w.pad, w.stride)
    if isinstance(w, wl.GemmChain):
        return "b2b_gemm", (w.M, w.K0, w.N0, w.N1)
    if isinstance(w, wl.GemmChain3):
        return "b2b_gemm3", (w.M, w.K0, w.N0, w.N1, w.N2)
    if isinstance(w, wl.ConvChain):
        return "b2b_conv_nhwc", (w.N, w.H, w.W, w.C, w.C0, w.R, w.S, w.pad, w.C1, w.stride)
    return "conv_relu_maxpool", (w.N, w.H, w.W, w.Cin, w.Cout)


def workload_of(kind: str, dims) -> object:
    """The model's view of a problem given as an entry point and its sizes (the inverse of
    problem_of; dtype and epilogues do not enter the model)."""
    d = [int(x) for x in dims]
    if kind == "b2b_gemm":
        return wl.GemmChain("problem", "bf16", *d[:4], "none", "none")
    if kind == "gemm_bias_act":
        return GemmSingle("problem", "bf16", d[0], d[1], d[2], 0, "none", "none")
    if kind == "b2b_gemm3":
        return wl.GemmChain3("problem", "bf16", *d[:5], "none", "none", "none")
    if kind == "b2b_conv_nhwc":
        return wl.ConvChain("problem", "bf16", *d[:9], "none", "none",
                            stride=d[9] if len(d) > 9 else 1)
    if kind == "conv_bias_act_nhwc":
        return ConvSingle("problem", "bf16", *d[:8], 0, "none", "none",
                          stride=d[8] if len(d) > 8 else 1)
    if kind == "conv_relu_maxpool":
        return wl.ConvPool("problem", "bf16", *d[:5])
    raise ValueError(kind)


def fits(plan: dict) -> bool:
    """The footprint check of a candidate: its buffers' best-fit extent (plus the 1 KiB
    the kernel adds to align its base) within the shared memory of a CTA, and its
    accumulators within the SM's TMEM."""
    return smem_footprint(plan) + 1024 <= SMEM_LIMIT and plan["tmem_cols"] <= TMEM_COLS


@dataclasses.dataclass
class Candidate:
    cand: int                    # layout index, as b2b_debug_plan_candidate numbers it
    plan: dict
    bounds: Dict[str, float]     # launch_bounds of the plan
    tiles_per_unit: int          # tiles of the busiest CTA (or CTA pair)

    @property
    def demand(self) -> List[float]:
        """The three per-resource bounds, largest first."""
        return sorted((self.bounds["hbm_us"], self.bounds["l2_us"], self.bounds["tensor_us"]),
                      reverse=True)

    @property
    def shallow(self) -> bool:
        """Fewer than three ring stages: a load cannot be in flight beside the two stages
        the MMAs and the producer hold."""
        return self.plan["stages"] < 3


def orders(x: Candidate, y: Candidate) -> int:
    """-1 or 1 if the bounds order x before or after y, 0 if they do not: below the steady
    state (some CTA of either plan with fewer than STEADY_TILES tiles) the launch is mostly
    pipeline fill and drain, which the bounds do not see; in it, the lower demand wins,
    resource by resource from the binding one, bounds within RANK_TOL tying."""
    if min(x.tiles_per_unit, y.tiles_per_unit) < STEADY_TILES:
        return 0
    for a, b in zip(x.demand, y.demand):
        if abs(a - b) > RANK_TOL * max(a, b):
            return -1 if a < b else 1
    return 0


def compare(x: Candidate, y: Candidate) -> int:
    """The model's order: the bounds where they decide, else the planner's order of
    preference (more tiles in flight, resident weights, separate staging; rings of three
    or more stages before shallower ones)."""
    o = orders(x, y)
    if o:
        return o
    if x.shallow != y.shallow:
        return 1 if x.shallow else -1
    return (x.cand > y.cand) - (x.cand < y.cand)


def candidates(w, num_sms: int = 152) -> List[Candidate]:
    """Every layout the planner finds feasible for the workload, with its plan, bounds and
    tiles per CTA, in the planner's order; candidates over the footprint are dropped."""
    from . import ops
    kind, dims = problem_of(w)
    n = ops.debug_plan(kind, dims, cand=0)["ncand"]
    out = []
    for c in range(n):
        plan = ops.debug_plan(kind, dims, cand=c)
        if not fits(plan):
            continue
        units = num_sms // 2 if plan.get("cta_pair") else num_sms
        unit_tiles = -(-plan["tiles"] // 2) if _pool_pair(plan) else plan["tiles"]
        if plan["tiles"] == 0:
            b = {"hbm_us": 0.0, "l2_us": 0.0, "tensor_us": 0.0, "floor_us": 0.0, "bound": "hbm"}
            out.append(Candidate(c, plan, b, 0))
            continue
        out.append(Candidate(c, plan, launch_bounds(w, plan, num_sms=num_sms),
                             max(tiles_per_cta(unit_tiles, units))))
    return out


def rank(w, num_sms: int = 152) -> List[Candidate]:
    """The feasible layouts of a workload, best first (Welder notes, "Scheduling policy":
    candidates that pass the memory-footprint check are ordered by the cost model).  The
    order is built by repeatedly taking the best remaining candidate, scanning in the
    planner's order (`compare` may tie two candidates that a third separates)."""
    left = candidates(w, num_sms)
    out = []
    while left:
        best = 0
        for i in range(1, len(left)):
            if compare(left[i], left[best]) < 0:
                best = i
        out.append(left.pop(best))
    return out


def top(w, k: int = 3, num_sms: int = 152) -> List[Candidate]:
    """The model's best k layouts, and every later one the bounds do not order against the
    k-th (the model cannot tell those apart, so the profiler should)."""
    r = rank(w, num_sms)
    out = r[:k]
    for c in r[k:]:
        if orders(r[k - 1], c) != 0:
            break
        out.append(c)
    return out


def choose(w, k: int = 3, variant: Optional[Sequence[int]] = None) -> List[int]:
    """Hands the model's top layouts to the profiler (b2b_set_candidates): the first
    becomes the default of calls with these sizes (of one variant, if given:
    ops.variant(...)), and the profiler, when on, times only these.  The library ranks the
    same way by itself; this makes the choice explicit, or narrower with a smaller k.
    Returns the layout indices handed over."""
    from . import ops
    kind, dims = problem_of(w)
    cands = [c.cand for c in top(w, k)]
    ops.set_candidates(kind, list(dims) + list(variant or ()), cands)
    return cands


def bounds_report(measured_us: Optional[Dict[str, float]] = None) -> str:
    """Markdown table of launch_bounds for every workload, beside measured microseconds per
    launch where given (name -> us)."""
    measured_us = measured_us or {}
    lines = ["| workload | tiles per CTA or CTA pair (max) | HBM us | L2 -> SM us | tensor us "
             "| floor | measured us | floor / measured |", "|---|---|---|---|---|---|---|---|"]
    for name, w in wl.WORKLOADS.items():
        plan = plan_of(w)
        b = launch_bounds(w, plan)
        m = measured_us.get(name)
        got = "" if m is None else f"{m:.2f}"
        frac = "" if m is None else f"{b['floor_us'] / m:.2f}"
        lines.append(
            f"| {name} | {max(tiles_per_cta(plan['tiles'], 76 if plan.get('cta_pair') else 152))} "
            f"| {b['hbm_us']:.2f} "
            f"| {b['l2_us']:.2f} | {b['tensor_us']:.2f} | {b['floor_us']:.2f} ({b['bound']}) "
            f"| {got} | {frac} |")
    return "\n".join(lines)


def report(ncu: Optional[Dict[str, str]] = None) -> str:
    """Markdown table of the model for every workload, beside the counters of one
    captured launch per workload where an export is given (name -> csv path)."""
    ncu = ncu or {}
    lines = ["| workload | plan | DRAM unique MB | DRAM unfused MB | L2->SM model MB "
             "| A boxes / A in bounds | L2->SM ncu MB | model/ncu | smem model | smem planner |",
             "|---|---|---|---|---|---|---|---|---|---|"]
    for name, w in wl.WORKLOADS.items():
        plan = plan_of(w)
        t = l2_to_smem_traffic(w, plan)
        desc = ("CTA pairs, " if plan.get("cta_pair") else "") + \
            ("W0 resident" if plan.get("w0_res") else "resident" if plan["resident"] else "streamed") + \
            (", P in TMEM" if plan["p_tmem"] else f", {plan['nbuf']} P buffers") * (plan["mode"] == 0) + \
            (", halo" if plan["halo"] else "") + (", alias" if plan["alias"] else "")
        got = read_ncu_raw_csv(ncu[name]).get(NCU_L2_TO_SM) if name in ncu else None
        t_total = t["total"]
        lines.append(
            f"| {name} | {desc} | {dram_traffic(w) / 1e6:.2f} | {dram_traffic(w, False) / 1e6:.2f} "
            f"| {t['total'] / 1e6:.3f} | {t['A'] / t['A_in_bounds']:.3f} "
            f"| {'' if got is None else f'{got / 1e6:.3f}'} "
            f"| {'' if not got else f'{t_total / got:.3f}'} "
            f"| {smem_footprint(plan) + 1024} | {plan['smem']} |")
    return "\n".join(lines)


def main(argv: Optional[Sequence[str]] = None) -> None:
    import argparse
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("--ncu", nargs="*", default=[], metavar="WORKLOAD=CSV",
                    help="raw-page csv export of one captured chain launch per workload")
    ap.add_argument("--bounds", nargs="*", default=None, metavar="WORKLOAD=US",
                    help="print the per-resource launch bounds instead, beside measured "
                         "microseconds per launch")
    args = ap.parse_args(argv)
    if args.bounds is not None:
        print(bounds_report({k: float(v) for k, v in (a.split("=", 1) for a in args.bounds)}))
        return
    print(report(dict(a.split("=", 1) for a in args.ncu)))


if __name__ == "__main__":
    main()
