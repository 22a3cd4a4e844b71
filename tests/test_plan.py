"""Launch plans on the host (no GPU): every shared-memory region the kernel touches lies
inside the dynamic allocation, regions do not overlap, each is at least as large as the
kernel's accesses into it, and TMEM accumulators fit the allocation.

The sizes below are re-derived from what the kernel writes and reads, independently of
the planner: A chunks are 128 rows x 128 B; a weight chunk is 64 K-rows x 128 B per
64-wide N block (row-major weights) or N x 128 B (K-major filters); the P tile and the
output staging hold 16 KiB per 64 columns; a pooled staging tile 4 KiB per 64 columns;
the bias operands of the MMA 1 KiB plus 2 KiB per 64 columns of each GEMM.
"""
import ctypes
import itertools

import pytest

from gemm_conv_chains_gb300 import ops
from gemm_conv_chains_gb300 import workloads as wl

FIELDS = ["smem", "stages", "stage_bytes", "resident", "alias", "off_ring", "ring", "off_w0",
          "off_w1", "w_res", "w0_chunk", "w1_chunk", "off_p0", "off_p1", "p", "off_out0",
          "off_out1", "out", "off_bias", "bias", "off_bar", "bar", "tmem_cols", "d0_col0",
          "d0_col1", "d1_col0", "d1_col1", "dual", "groups", "tiles", "kchunks0", "kchunks1",
          "N0p", "N1p", "mode", "p_tmem", "w1_group", "w1_per_stage", "halo", "a_stage_bytes",
          "nbuf", "off_p2", "off_p3", "d0_col2", "d0_col3", "d1_col2", "d1_col3", "cand", "ncand",
          "grid_choice", "pf_choice", "ring_extend", "off_w2", "off_p1_0", "off_p1_1", "d2_col0",
          "d2_col1", "p_split", "w0_res", "cta_pair", "two_issuers", "out_slots", "pt_col0",
          "pt_col1"]
SMEM_LIMIT = 227 * 1024
KIND = {"b2b_gemm": 0, "gemm_bias_act": 1, "b2b_conv_nhwc": 2, "conv_bias_act_nhwc": 3,
        "conv_relu_maxpool": 4, "b2b_gemm3": 5}


def plan(kind, dims):
    arr = (ctypes.c_int64 * len(dims))(*dims)
    out = (ctypes.c_uint32 * len(FIELDS))()
    st = ops.lib().b2b_debug_plan(KIND[kind], arr, len(dims), out, len(FIELDS))
    return st, dict(zip(FIELDS, list(out)))


def rup(x, m):
    return -(-x // m) * m


def check(kind, dims, row_major_w):
    st, p = plan(kind, dims)
    R = {"b2b_conv_nhwc": dims[5] if len(dims) > 5 else 1, "conv_bias_act_nhwc": dims[5] if len(dims) > 5 else 1,
         "conv_relu_maxpool": 3}.get(kind, 1)
    if kind in ("b2b_conv_nhwc", "conv_bias_act_nhwc") and dims[5] == 1 and dims[6] == 1 and dims[7] == 0:
        R = 1   # a 1x1 pad-0 conv runs as a GEMM
    assert st == 0, (kind, dims, st)
    if p["cta_pair"] and kind == "conv_relu_maxpool":
        return check_pool_cta2(dims, p)
    if p["cta_pair"]:
        return check_cta2(kind, dims, p)
    mode = p["mode"]
    N0p, N1p = p["N0p"], p["N1p"]
    n0blk, n1blk = -(-N0p // 64), -(-N1p // 64)
    # what the kernel touches
    # (wide chains, 256 < N0: one half of N0, four 64-wide blocks, per chunk)
    w0_chunk = min(n0blk, 4 if mode == 0 and N0p > 256 else n0blk) * 8192 if row_major_w else N0p * 128
    w1_chunk = (n1blk * 8192 if row_major_w else N1p * 128) if mode == 0 else 0
    p_need = n0blk * 16384 if mode == 0 else 0
    out_need = {0: n1blk * 16384, 1: n0blk * 16384, 2: n0blk * 4096}[mode]
    assert p["w0_chunk"] == w0_chunk and p["w1_chunk"] == w1_chunk
    assert p["smem"] <= SMEM_LIMIT
    assert 2 <= p["stages"] <= 8
    assert p["ring"] == p["stages"] * p["stage_bytes"]
    w0_res = p["w0_res"] == 1
    assert p["stage_bytes"] >= p["a_stage_bytes"] + (0 if p["resident"] or w0_res else w0_chunk)
    if p["halo"]:
        # one box of (8 + R - 1) x 16 pixels x 64 channels per column tap feeds all row taps
        assert p["resident"] and p["a_stage_bytes"] == (8 + R - 1) * 16 * 128
    else:
        assert p["a_stage_bytes"] == 128 * 128
    if not p["resident"]:
        assert p["stage_bytes"] >= w1_chunk
    regions = [("ring", p["off_ring"], p["ring"]), ("bias", p["off_bias"], p["bias"]),
               ("bar", p["off_bar"], p["bar"])]
    if p["resident"]:
        assert not w0_res
        assert p["w_res"] >= p["kchunks0"] * w0_chunk + p["kchunks1"] * w1_chunk
        assert p["off_w1"] == p["off_w0"] + p["kchunks0"] * w0_chunk
        regions.append(("w", p["off_w0"], p["w_res"]))
    if w0_res:
        # W0 alone resident (one barrier per K chunk, at most 8), A and W1 through the ring,
        # tile pairs with P in TMEM, and no output staging (stores from registers)
        assert mode == 0 and row_major_w and p["p_tmem"] and p["dual"] and p["groups"] == 2
        assert p["kchunks0"] <= 8 and p["w_res"] >= p["kchunks0"] * w0_chunk
        assert p["stage_bytes"] >= max(128 * 128, w1_chunk) and not p["ring_extend"]
        regions.append(("w0", p["off_w0"], p["w_res"]))
    dual = p["dual"] == 1
    groups = p["groups"]
    assert groups in (1, 2) and (groups == 1 or dual)
    if mode == 2:
        assert groups == 2                       # the pool epilogue needs whole rows per warp
    p_tmem = p["p_tmem"] == 1
    wide = p["p_split"] > 0
    assert not p_tmem or (mode == 0 and not p["alias"] and (wide or (dual and groups == 2)))
    if wide:
        # 256 < N0 <= 512: one tile in flight, both warpgroups, P's halves packed in place at
        # 0 and 256, D1 between them
        assert p_tmem and not dual and groups == 1 and N0p > 256 and N1p <= 128
        assert p["p_split"] == 256 and p["tmem_cols"] == 512 and p["d0_col0"] == 0
        assert p["d1_col0"] == 128 and p["w1_group"] == 0 and not p["resident"]
        # GEMM0 by halves of N0: a ring stage holds an A chunk and four 64-wide W0 blocks;
        # D1 in the upper columns of the half computed first (the lower on even tiles)
        assert p["w0_chunk"] == 4 * 8192 and p["stage_bytes"] == 16384 + 4 * 8192
        assert p["d0_col1"] == 256 and p["d1_col1"] == 384
        # each tile's W1 packed as many chunks per ring stage as fit
        assert p["w1_per_stage"] == p["stage_bytes"] // w1_chunk
    elif not p["w1_group"]:
        assert p["w1_per_stage"] == 1
    if p["w1_group"]:
        # W1 packed w1_per_stage chunks per ring stage; all its stages in the ring at once
        assert p_tmem and not p["resident"]
        per = p["w1_per_stage"]
        assert per >= 1 and per * w1_chunk <= p["stage_bytes"]
        assert -(-p["kchunks1"] // per) <= p["stages"]
    nbuf = p["nbuf"]
    # (the pooled conv with two MMA issuers gives each issuer two accumulators)
    assert nbuf in (1, 2, 4) and (nbuf > 1) == dual
    assert mode == 0 or nbuf == 2 or (mode == 2 and p["two_issuers"] and nbuf == 4)
    assert nbuf != 4 or mode == 2 or (mode == 0 and not p_tmem and groups == 2 and not p["alias"])
    # P buffers used: tile i -> P[i mod nbuf]; none when P is in TMEM
    pbufs = 0 if p_tmem else (nbuf if mode == 0 else 0)
    obufs = 2 if groups == 2 else 1
    if mode == 0 and not p_tmem:
        need_p = max(p_need, out_need) if p["alias"] else p_need
        assert p["p"] >= need_p
        for b in range(pbufs):
            regions.append((f"p{b}", p[f"off_p{b}"], p["p"]))
    slots = p["out_slots"] == 1
    if slots:
        # the conv chain's two-issuer layout: halo boxes over resident filters, P in TMEM,
        # two sub-rings that each hold a whole tile's stages, and a 1 KiB output slot per
        # epilogue warp (32 rows x 16 columns)
        assert mode == 0 and p["two_issuers"] and p["halo"] and p["resident"] and p_tmem
        assert dual and groups == 2 and nbuf == 2 and N0p <= 64 and not p["alias"]
        assert p["stages"] // 2 >= p["kchunks0"] // R
        assert p["out"] == 8 * 1024 and p["off_out0"] == p["off_out1"]
        regions.append(("slots", p["off_out0"], p["out"]))
    if p["two_issuers"] and mode == 0:
        assert slots
    if p["alias"]:
        assert mode == 0
        # staging b (used by epilogue group b, which handles the tiles using P[b])
        for b in range(obufs):
            assert p[f"off_out{b}"] == p[f"off_p{b if dual else 0}"]
    elif slots:
        pass
    elif w0_res:
        assert p["out"] == 0
    else:
        assert p["out"] >= out_need
        for b in range(obufs):
            regions.append((f"out{b}", p[f"off_out{b}"], p["out"]))
    # bias operands: a 1 KiB ONES tile and a 2 KiB BIAS block per 64-wide N block of each GEMM
    assert p["bias"] >= 1024 + 2048 * (n0blk + (n1blk if mode == 0 else 0))
    assert p["bar"] >= 8 * 27 + 8                # 27 barriers, then the TMEM slot and flag
    usable = p["smem"] - 1024                    # the rest aligns the base to 1024
    if p["ring_extend"]:
        # extra ring stages run on into the output staging, never past it, and W1's stages
        # of a tile pair (after both tiles' GEMM0 chunks) stay out of them
        ext_end = p["off_ring"] + (p["stages"] + p["ring_extend"]) * p["stage_bytes"]
        assert p["p_tmem"] and not p["resident"] and p["w1_group"] and p["stages"] + p["ring_extend"] <= 8
        assert p["off_out0"] == p["off_ring"] + p["ring"]
        assert ext_end <= p["off_out0"] + (2 if groups == 2 else 1) * p["out"] <= p["off_bias"]
        total = p["stages"] + p["ring_extend"]
        per = p["w1_per_stage"]
        kst = p["kchunks0"] // (R if p["halo"] else 1)
        for j in range(-(-p["kchunks1"] // per)):
            assert (2 * kst + j) % total < p["stages"]
    for name, off, size in regions:
        assert off % 1024 == 0, name
        assert off + size <= usable, (name, off, size, usable)
    for (a, oa, sa), (b, ob, sb) in itertools.combinations(regions, 2):
        assert oa + sa <= ob or ob + sb <= oa, (a, b)
    # TMEM: every accumulator buffer in range, 32-column aligned, distinct buffers disjoint
    assert p["tmem_cols"] in (32, 64, 128, 256, 512)
    if wide:
        return p
    if p_tmem and slots:
        # two issuers: D0, P (packed) and D1 of each buffer in disjoint column ranges
        accs = []
        for b in range(2):
            accs += [(f"d0_{b}", p[f"d0_col{b}"], N0p), (f"p_{b}", p[f"pt_col{b}"], N0p // 2),
                     (f"d1_{b}", p[f"d1_col{b}"], N1p)]
        for name, col, n in accs:
            assert col % 32 == 0 and col + n <= p["tmem_cols"], (name, col, n)
        for (a, ca, na), (b, cb, nb) in itertools.combinations(accs, 2):
            assert ca + na <= cb or cb + nb <= ca, (a, b)
        return p
    if p_tmem:
        # buffer b: D0 [d0, d0 + N0p); P (packed) [d0, d0 + N0p/2); D1 [d1, d1 + N1p) after P
        spans = []
        for b in range(2):
            assert p[f"pt_col{b}"] == p[f"d0_col{b}"]
        for b in range(2):
            d0, d1 = p[f"d0_col{b}"], p[f"d1_col{b}"]
            assert d0 % 32 == 0 and d1 % 32 == 0
            assert d1 >= d0 + N0p // 2                  # D1 never overwrites P
            lo, hi = d0, max(d0 + N0p, d1 + N1p)
            assert hi <= p["tmem_cols"]
            spans.append((lo, hi))
        assert spans[0][1] <= spans[1][0] or spans[1][1] <= spans[0][0]
        return p
    accs = [(f"d0_{b}", p[f"d0_col{b}"], N0p) for b in range(nbuf)]
    if mode == 0:
        accs += [(f"d1_{b}", p[f"d1_col{b}"], N1p) for b in range(nbuf)]
    for name, col, n in accs:
        assert col % 32 == 0 and col + n <= p["tmem_cols"], (name, col, n)
    for (a, ca, na), (b, cb, nb) in itertools.combinations(accs, 2):
        assert ca + na <= cb or cb + nb <= ca, (a, b)
    assert N0p % 16 == 0 and 16 <= N0p <= 256 and N1p % 16 == 0 and N1p <= 256
    return p


def check_pool_cta2(dims, p):
    """A conv + pool plan over CTA pairs: per CTA a ring of halo boxes ((8 + 2) x 16 pixels x
    64 channels) of its own 8 x 16 tile, at least one tile's stages and one more; its half
    of the filters resident (N0p / 2 rows x 128 B per tap and channel block); one 4 KiB
    pooled staging tile per 64 channels for each epilogue warpgroup; the bias of every
    channel as 256 fp32 words; the barriers; MMA issuers in the leader as many as the ring
    holds tiles' stages (up to three; three only where their six accumulators fit TMEM),
    two accumulators in TMEM per issuer (four with fewer than three)."""
    N, H, W, C, C0 = dims[:5]
    N0p = p["N0p"]
    assert p["mode"] == 2 and N0p % 16 == 0 and N0p <= 128
    kc_tap = -(-C // 64)
    kst = 3 * kc_tap
    assert p["kchunks0"] == 9 * kc_tap and p["halo"] == 1 and p["resident"] == 1
    assert p["tiles"] == N * -(-H // 8) * -(-W // 16)
    assert p["stage_bytes"] == p["a_stage_bytes"] == 10 * 16 * 128
    assert p["ring"] == p["stages"] * p["stage_bytes"] and kst + 1 <= p["stages"] <= 10
    s0 = -(-N0p // 32) * 32
    issuers = min(3, p["stages"] // kst)
    if issuers == 3 and 6 * s0 > 512:
        issuers = 2
    assert p["two_issuers"] == issuers - 1
    assert p["w0_chunk"] == N0p // 2 * 128 and p["w_res"] >= p["kchunks0"] * p["w0_chunk"]
    nch = -(-N0p // 64)
    assert p["out"] == nch * 4096 and p["off_out1"] == p["off_out0"] + p["out"]
    assert p["bias"] >= 256 * 4
    nbuf = 6 if issuers == 3 else 4
    assert p["nbuf"] == nbuf and p["dual"] == 1 and p["groups"] == 2
    regions = [("ring", p["off_ring"], p["ring"]), ("w0", p["off_w0"], p["w_res"]),
               ("out", p["off_out0"], 2 * p["out"]), ("bias", p["off_bias"], p["bias"]),
               ("bar", p["off_bar"], p["bar"])]
    usable = p["smem"] - 1024
    for name, off, size in regions:
        assert off % 1024 == 0 and off + size <= usable, name
    for (a, oa, sa), (b, ob, sb) in itertools.combinations(regions, 2):
        assert oa + sa <= ob or ob + sb <= oa, (a, b)
    assert p["smem"] <= SMEM_LIMIT
    for b in range(4):
        assert p[f"d0_col{b}"] == b * s0
    assert nbuf * s0 <= p["tmem_cols"] <= 512
    return p


def check_cta2(kind, dims, p):
    """A plan over CTA pairs (clusters of two CTAs sharing each 256-row MMA): per CTA a ring
    of 16 KiB A chunks (128 rows x 64 K), its half of W0 and of W1 resident (64-wide blocks
    of 64 K-rows x 128 B), the ONES tile and a 2 KiB bias block per 64 columns of its halves,
    the barriers; P kept in TMEM over GEMM0's columns, two 256-row tiles in flight."""
    assert kind == "b2b_gemm" and p["mode"] == 0
    M, K0, N0, N1 = dims[:4]
    N0p, N1p = p["N0p"], p["N1p"]
    assert N0p % 128 == 0 and N1p % 128 == 0 and N0p <= 256 and N1p <= 256
    nb0, nb1 = N0p // 128, N1p // 128
    k0, k1 = -(-K0 // 64), -(-N0p // 64)
    assert p["kchunks0"] == k0 <= 8 and p["kchunks1"] == k1
    assert p["tiles"] == -(-M // 256)
    assert p["w0_chunk"] == nb0 * 8192 and p["w1_chunk"] == nb1 * 8192
    assert p["stage_bytes"] == p["a_stage_bytes"] == 128 * 128 and 3 <= p["stages"] <= 8
    assert p["ring"] == p["stages"] * p["stage_bytes"]
    assert p["resident"] and p["p_tmem"] and p["dual"] and p["groups"] == 2 and p["nbuf"] == 2
    assert not p["w0_res"] and not p["halo"] and p["p"] == 0
    # the output leaves through 4 KiB per epilogue warp (TMA stores) when the ring keeps
    # five stages beside it, else from registers
    assert p["out"] in (0, 8 * 4096)
    assert p["out"] == 0 or p["stages"] >= 5
    assert p["off_w1"] == p["off_w0"] + k0 * p["w0_chunk"]
    assert p["w_res"] == k0 * p["w0_chunk"] + k1 * p["w1_chunk"]
    assert p["bias"] >= 1024 + 2048 * (nb0 + nb1)
    assert p["bar"] >= 8 * 35 + 8                # 35 barriers, then the TMEM slot and flag
    assert p["smem"] <= SMEM_LIMIT
    usable = p["smem"] - 1024
    regions = [("ring", p["off_ring"], p["ring"]), ("w", p["off_w0"], p["w_res"]),
               ("bias", p["off_bias"], p["bias"]), ("bar", p["off_bar"], p["bar"])]
    if p["out"]:
        regions.append(("out", p["off_out0"], p["out"]))
    for name, off, size in regions:
        assert off % 1024 == 0 and off + size <= usable, (name, off, size, usable)
    for (a, oa, sa), (b, ob, sb) in itertools.combinations(regions, 2):
        assert oa + sa <= ob or ob + sb <= oa, (a, b)
    spans = []
    for b in range(2):
        d0, d1 = p[f"d0_col{b}"], p[f"d1_col{b}"]
        assert d0 % 32 == 0 and d1 % 32 == 0 and d1 >= d0 + N0p // 2
        spans.append((d0, max(d0 + N0p, d1 + N1p)))
        assert spans[-1][1] <= p["tmem_cols"] <= 512
    assert spans[0][1] <= spans[1][0] or spans[1][1] <= spans[0][0]
    return p


def test_ffn_offers_a_cta_pair_plan():
    # the FFN-like chain also runs over CTA pairs: each SM keeps half of W0 (64 KiB) and of
    # W1 (32 KiB) resident beside a five-stage ring of A chunks and 32 KiB of output staging
    dims = (32768, 256, 256, 128)
    n = ops.debug_plan("b2b_gemm", dims)["ncand"]
    ops.set_choice("b2b_gemm", dims, cand=n - 1)
    try:
        p = check("b2b_gemm", dims, True)
    finally:
        ops.autotune_reset()
    assert p["cta_pair"] == 1 and p["stages"] == 5 and p["out"] == 8 * 4096
    assert p["w_res"] == 96 * 1024
    assert p["tiles"] == 128
    # chains the pair kernel does not take offer no such plan
    for d in ((1000, 64, 64, 64), (1000, 64, 192, 128), (1000, 576, 256, 128)):
        m = ops.debug_plan("b2b_gemm", d)["ncand"]
        ops.set_choice("b2b_gemm", d, cand=m - 1)
        try:
            assert ops.debug_plan("b2b_gemm", d)["cta_pair"] == 0
        finally:
            ops.autotune_reset()


GEMM = [(1, 64, 64, 64), (640, 128, 128, 256), (200, 320, 96, 200), (384, 64, 256, 256),
        (32768, 256, 256, 128), (1024, 64, 64, 64), (129, 8, 8, 8), (257, 72, 40, 24),
        (100, 2048, 256, 256), (100, 8, 256, 8)]


@pytest.mark.parametrize("dims", GEMM)
def test_b2b_gemm_plans(dims):
    check("b2b_gemm", dims, True)


def test_b2b_gemm_plan_sweep():
    for n0 in range(8, 257, 24):
        for n1 in range(8, 257, 40):
            for k0 in (8, 64, 200, 512):
                check("b2b_gemm", (1000, k0, n0, n1), True)


def test_ffn_plan_keeps_p_in_tmem():
    dims = (32768, 256, 256, 128)
    p = check("b2b_gemm", dims, True)
    assert p["resident"] == 0      # 192 KiB of weights cannot stay beside the ring
    # 2 x (256 + 128) accumulator columns exceed 512, but D0 -> P + D1 in one 256-column
    # buffer per tile gives two tiles in flight with P in TMEM
    assert p["p_tmem"] == 1 and p["dual"] == 1
    # both weights stream: three 48 KiB stages (an A chunk and a W0 chunk each), W1 three
    # chunks to a stage, and a fourth stage over the two 32 KiB output staging buffers when
    # no CTA has a third tile (W1's stages of the pair, fills 8 and 9, land on stages 0, 1)
    assert p["w0_res"] == 0 and p["cta_pair"] == 0
    assert p["w1_group"] == 1 and p["w1_per_stage"] == 3
    assert p["stages"] == 3 and p["ring_extend"] == 1
    # the next layout keeps W0 (128 KiB) alone resident: five 16 KiB stages carry A and W1
    # chunks, W1 (4 chunks of 16 KiB) once per pair of tiles, no output staging
    ops.set_choice("b2b_gemm", dims, cand=p["cand"] + 1)
    try:
        q = check("b2b_gemm", dims, True)
    finally:
        ops.autotune_reset()
    assert q["w0_res"] == 1 and q["w_res"] == 4 * 32768 and q["out"] == 0
    assert q["stages"] == 5 and q["stage_bytes"] == 16384
    assert q["w1_group"] == 1 and q["w1_per_stage"] == 1


def test_large_chains_default_to_cta_pairs():
    # the tile-graph model takes CTA pairs (lower L2 -> SM bounds) once every CTA and every
    # pair runs three or more tiles -- past 152 x 256 rows on the 152 SMs (tiles then count
    # 256 rows); below, the planner's preference keeps single CTAs
    for M, pair in ((152 * 256, False), (152 * 256 + 1, True), (262144, True), (32768, False)):
        p = check("b2b_gemm", (M, 256, 256, 128), True)
        assert p["cta_pair"] == int(pair), M
        assert p["tiles"] == -(-M // (256 if pair else 128))
        assert p["cand"] == p["ncand"] - 1 if pair else p["cand"] < p["ncand"] - 1
    assert check("b2b_gemm", (262144, 64, 64, 64), True)["cta_pair"] == 0   # N0 not % 128


def test_small_chains_keep_four_tiles_in_flight():
    # 64 -> 64 -> 64: four (D0 + D1) buffers of 64 + 64 columns fill the 512 TMEM columns
    for dims in ((200704, 64, 64, 64), (1024, 64, 64, 64)):
        p = check("b2b_gemm", dims, True)
        assert p["nbuf"] == 4 and p["groups"] == 2 and p["resident"] == 1
    p = check("b2b_conv_nhwc", (32, 56, 56, 64, 64, 3, 3, 1, 128), False)
    assert p["dual"] == 1 and p["resident"] == 1


@pytest.mark.parametrize("dims", [(1000, 64, 64), (513, 256, 256), (130, 24, 40), (1, 8, 256)])
def test_gemm_bias_act_plans(dims):
    check("gemm_bias_act", dims, True)


CONV = [(2, 9, 9, 64, 64, 3, 3, 1, 128), (1, 17, 20, 16, 24, 3, 3, 1, 8),
        (1, 10, 12, 32, 32, 5, 5, 2, 16), (2, 7, 9, 64, 64, 1, 1, 0, 64),
        (32, 56, 56, 64, 64, 3, 3, 1, 128), (64, 56, 56, 64, 64, 1, 1, 0, 64),
        (1, 6, 6, 256, 256, 3, 3, 1, 256), (1, 6, 6, 16, 16, 1, 3, 1, 16)]


@pytest.mark.parametrize("dims", CONV)
def test_b2b_conv_plans(dims):
    check("b2b_conv_nhwc", dims, False)


@pytest.mark.parametrize("dims", [(2, 9, 9, 64, 64, 3, 3, 1), (1, 7, 5, 16, 24, 3, 3, 1),
                                  (2, 6, 6, 64, 64, 1, 1, 0), (1, 8, 8, 256, 256, 7, 7, 3)])
def test_conv_bias_act_plans(dims):
    check("conv_bias_act_nhwc", dims, False)


@pytest.mark.parametrize("dims", [(32, 112, 112, 64, 64), (1, 7, 9, 16, 8), (1, 2, 2, 8, 8),
                                  (2, 18, 40, 64, 128), (1, 16, 16, 256, 256)])
def test_conv_relu_maxpool_plans(dims):
    check("conv_relu_maxpool", dims, False)


def test_resident_3x3_convs_use_halo_boxes():
    for kind, dims in (("conv_relu_maxpool", (32, 112, 112, 64, 64)),
                       ("b2b_conv_nhwc", (32, 56, 56, 64, 64, 3, 3, 1, 128))):
        p = check(kind, dims, False)
        assert p["resident"] == 1 and p["halo"] == 1 and p["a_stage_bytes"] == 10 * 16 * 128


def test_workload_tile_counts():
    assert plan("b2b_gemm", (wl.GEMM_FFN.M, 256, 256, 128))[1]["tiles"] == 256
    assert plan("b2b_conv_nhwc", (32, 56, 56, 64, 64, 3, 3, 1, 128))[1]["tiles"] == 32 * 7 * 4
    assert plan("conv_relu_maxpool", (32, 112, 112, 64, 64))[1]["tiles"] == 32 * 14 * 7


def test_plan_rejects_like_the_entry_points():
    assert plan("b2b_gemm", (10, 12, 64, 64))[0] == 3        # K0 not a multiple of 8
    assert plan("b2b_gemm", (10, 64, 520, 64))[0] == 4       # N0 > 512
    assert plan("conv_relu_maxpool", (1, 1, 8, 8, 8))[0] == 2


def test_wide_chains_keep_p_in_tmem():
    for dims in ((300, 128, 256, 64), (257, 72, 200, 72), (1000, 64, 224, 96)):
        assert check("b2b_gemm", dims, True)["p_tmem"] == 1


def test_strided_conv_plans():
    # stride s: an 8 x 16 output tile's boxes take every s-th input pixel; no halo boxes
    # (the row taps are not whole box rows apart), tiles over the strided output
    for dims in ((32, 56, 56, 64, 128, 3, 3, 1, 256, 2), (2, 9, 9, 64, 64, 3, 3, 1, 128, 2),
                 (4, 28, 28, 64, 128, 1, 1, 0, 64, 2), (1, 17, 11, 16, 24, 5, 5, 2, 8, 3),
                 (1, 30, 33, 32, 16, 3, 3, 1, 16, 4)):
        p = check("b2b_conv_nhwc", dims, False)
        N, H, W = dims[:3]
        R, S, pad, st = dims[5], dims[6], dims[7], dims[9]
        Ho, Wo = (H + 2 * pad - R) // st + 1, (W + 2 * pad - S) // st + 1
        assert p["tiles"] == N * -(-Ho // 8) * -(-Wo // 16)
        assert p["halo"] == 0 and p["kchunks0"] == R * S * -(-dims[3] // 64)
        check("conv_bias_act_nhwc", dims[:8] + (st,), False)
    # an explicit stride 1 is the unstrided launch
    assert plan("b2b_conv_nhwc", (32, 56, 56, 64, 64, 3, 3, 1, 128, 1)) == \
        plan("b2b_conv_nhwc", (32, 56, 56, 64, 64, 3, 3, 1, 128))
    # a 1x1 pad-0 conv runs as a GEMM over the pixel rows at stride 1, as a strided
    # implicit GEMM at stride 2
    assert plan("b2b_conv_nhwc", (4, 28, 28, 64, 128, 1, 1, 0, 64))[1]["tiles"] == -(-4 * 28 * 28 // 128)
    assert plan("b2b_conv_nhwc", (4, 28, 28, 64, 128, 1, 1, 0, 64, 2))[1]["tiles"] == 4 * 2 * 1
    assert plan("b2b_conv_nhwc", (1, 9, 9, 64, 64, 3, 3, 1, 64, 5))[0] == 4     # stride > 4
    assert plan("b2b_conv_nhwc", (1, 9, 9, 64, 64, 3, 3, 1, 64, 0))[0] == 2


@pytest.mark.parametrize("dims", [(1000, 64, 64, 64, 64), (32768, 128, 128, 64, 64),
                                  (257, 72, 40, 24, 96), (129, 8, 8, 8, 8), (300, 128, 96, 64, 64)])
def test_gemm3_plans(dims):
    # three-operator chain: ring of A chunks, W0/W1/W2 resident, two P0, P1 and output
    # buffers, bias blocks of three GEMMs; two tiles of D0, D1, D2 in TMEM
    st, p = plan("b2b_gemm3", dims)
    assert st == 0, st
    M, K0, N0, N1, N2 = dims
    r16 = lambda n: -(-n // 16) * 16
    r32 = lambda n: -(-n // 32) * 32
    n0b, n1b, n2b = (-(-r16(n) // 64) for n in (N0, N1, N2))
    assert p["mode"] == 3 and p["resident"] == 1 and p["dual"] == 1 and p["groups"] == 2
    assert p["stages"] >= 2 and p["stage_bytes"] == 16384 and p["smem"] <= SMEM_LIMIT
    k0, k1, k2 = -(-K0 // 64), -(-r16(N0) // 64), -(-r16(N1) // 64)
    assert p["kchunks0"] == k0 and p["kchunks1"] == k1
    p0 = max(n0b, n2b) * 16384 if p["alias"] else n0b * 16384
    regions = [("ring", p["off_ring"], p["ring"]),
               ("w0", p["off_w0"], k0 * n0b * 8192), ("w1", p["off_w1"], k1 * n1b * 8192),
               ("w2", p["off_w2"], k2 * n2b * 8192),
               ("p0a", p["off_p0"], p0), ("p0b", p["off_p1"], p0),
               ("p1a", p["off_p1_0"], n1b * 16384), ("p1b", p["off_p1_1"], n1b * 16384),
               ("bias", p["off_bias"], 1024 + 2048 * (n0b + n1b + n2b)),
               ("bar", p["off_bar"], 8 * 43 + 8)]
    if p["alias"]:
        # output staging b shares P0[b]'s space, taken only where separate staging would
        # leave fewer than three ring stages
        assert p["off_out0"] == p["off_p0"] and p["off_out1"] == p["off_p1"] and p["out"] == 0
        assert p["stages"] >= 3
    else:
        regions += [("outa", p["off_out0"], n2b * 16384), ("outb", p["off_out1"], n2b * 16384)]
    for name, off, size in regions:
        assert off % 1024 == 0 and off + size <= p["smem"] - 1024, name
    for (a, oa, sa), (b, ob, sb) in itertools.combinations(regions, 2):
        assert oa + sa <= ob or ob + sb <= oa, (a, b)
    cols = [(p[f"d{i}_col{b}"], r32(n)) for i, n in enumerate((N0, N1, N2)) for b in range(2)]
    for c, n in cols:
        assert c % 32 == 0 and c + n <= p["tmem_cols"] <= 512
    for (ca, na), (cb, nb) in itertools.combinations(cols, 2):
        assert ca + na <= cb or cb + nb <= ca


def test_gemm3_mlp3_aliases_its_staging():
    # the three-operator workload (128 -> 128 -> 64 -> 64): separate staging leaves two
    # ring stages, sharing P0's space four
    st, p = plan("b2b_gemm3", (32768, 128, 128, 64, 64))
    assert st == 0 and p["alias"] == 1 and p["stages"] == 4


def test_gemm3_limits():
    assert plan("b2b_gemm3", (1000, 64, 128, 128, 64))[0] == 4   # 2 x (128 + 128 + 64) > 512
    assert plan("b2b_gemm3", (1000, 64, 64, 64, 12))[0] == 3     # N2 not a multiple of 8
    assert plan("b2b_gemm3", (1000, 8192, 128, 64, 64))[0] == 4  # W0 does not fit


@pytest.mark.parametrize("dims", [(32768, 256, 512, 128), (300, 128, 384, 64), (257, 72, 264, 24),
                                  (1, 64, 512, 128), (1000, 512, 320, 96)])
def test_wide_chains_split_gemm0(dims):
    # 256 < N0 <= 512 (N1 <= 128): GEMM0 in two passes over the halves of N0, P packed in
    # place in each half, both warpgroups on every tile
    p = check("b2b_gemm", dims, True)
    assert p["p_split"] == 256 and p["groups"] == 1 and p["nbuf"] == 1


def test_wide_chain_plan_sweep():
    # every width 256 < N0 <= 512 (multiples of 8) beside N1 up to 128: the two-pass plan,
    # its W0 half chunks within a ring stage, W1 packed, D1 inside TMEM on both parities
    for n0 in range(264, 513, 8):
        for n1 in (8, 64, 120, 128):
            for k0 in (8, 256, 1000):
                p = check("b2b_gemm", (4096, k0, n0, n1), True)
                assert p["p_split"] == 256 and p["tmem_cols"] == 512
                assert p["d1_col1"] + p["N1p"] <= 512 and p["d1_col0"] + p["N1p"] <= 256
                # the upper half's packed P (at 256) ends before D1 of odd tiles (at 384)
                assert 256 + (p["N0p"] - 256) // 2 <= p["d1_col1"]
                assert p["w1_per_stage"] * p["w1_chunk"] <= p["stage_bytes"]


def test_wide_chain_limits():
    assert plan("b2b_gemm", (1000, 64, 512, 136))[0] == 4     # N1 > 128 beside a wide N0
    assert plan("b2b_gemm", (1000, 64, 520, 64))[0] == 4      # N0 > 512
    assert plan("gemm_bias_act", (1000, 64, 264))[0] == 4     # single operators keep N <= 256


def test_two_issuers_only_for_the_n64_halo_convs():
    # the conv + pool kernel with N <= 64 whose ring holds two tiles' stages splits it
    # between two MMA issuers (three over CTA pairs when it holds three), and so does the conv chain with halo boxes and N0 <= 64 in
    # its own layout (P in TMEM, per-warp output slots, a six-stage ring); every other
    # kernel keeps one
    # (over CTA pairs, the model's pick for this pooled conv, the ring of nine stages holds
    # three tiles' stages: three issuers)
    pool = check("conv_relu_maxpool", (32, 112, 112, 64, 64), False)
    assert pool["cta_pair"] == 1 and pool["two_issuers"] == 2 and pool["stages"] == 9
    ops.set_choice("conv_relu_maxpool", (32, 112, 112, 64, 64), cand=0)
    try:
        pool = check("conv_relu_maxpool", (32, 112, 112, 64, 64), False)
        assert pool["cta_pair"] == 0 and pool["two_issuers"] == 1 and pool["stages"] // 2 >= 3
    finally:
        ops.autotune_reset()
    chain = check("b2b_conv_nhwc", (32, 56, 56, 64, 64, 3, 3, 1, 128), False)
    assert chain["two_issuers"] == 1 and chain["out_slots"] == 1 and chain["halo"] == 1
    assert chain["stages"] == 6 and chain["p_tmem"] == 1 and chain["out"] == 8 * 1024
    for kind, dims, rm in (("conv_bias_act_nhwc", (32, 56, 56, 64, 64, 3, 3, 1), False),
                           ("gemm_bias_act", (200704, 64, 64), True),
                           ("gemm_bias_act", (32768, 256, 256), True),
                           ("b2b_gemm", (1024, 64, 64, 64), True),
                           # a 1x1 chain (no halo boxes), a halo chain with N0 = 128
                           ("b2b_conv_nhwc", (64, 56, 56, 64, 64, 1, 1, 0, 64), False),
                           ("b2b_conv_nhwc", (8, 28, 28, 64, 128, 3, 3, 1, 64), False)):
        assert check(kind, dims, rm)["two_issuers"] == 0
    # the same pooled conv with streamed filters: nine stages per tile, one issuer; the
    # chain's other layouts keep one issuer
    ops.set_choice("conv_relu_maxpool", (32, 112, 112, 64, 64), cand=1)
    ops.set_choice("b2b_conv_nhwc", (32, 56, 56, 64, 64, 3, 3, 1, 128), cand=1)
    try:
        assert check("conv_relu_maxpool", (32, 112, 112, 64, 64), False)["two_issuers"] == 0
        other = check("b2b_conv_nhwc", (32, 56, 56, 64, 64, 3, 3, 1, 128), False)
        assert other["two_issuers"] == 0 and other["out_slots"] == 0
    finally:
        ops.autotune_reset()
