"""The host-side tile-graph model: propagation, traffic and footprint (CPU only).

Expected values are derived by hand from the tile shapes and the kernel's load schedule,
not from the model's own code: a 3x3 conv's interior tile reads a 10 x 18 input tile; the
FFN launch streams W0 once per tile and W1 once per tile pair on 152 CTAs; a best-fit
allocation lets buffers with disjoint lifetimes share an offset.
"""
import pytest

from gemm_conv_chains_gb300 import ops
from gemm_conv_chains_gb300 import tilegraph as tg
from gemm_conv_chains_gb300 import workloads as wl


def test_propagation_shapes():
    g = tg.propagate(wl.GEMM_FFN)
    assert g.tiles == {"out": (128, 128), "P": (128, 256), "W1": (256, 128),
                       "A": (128, 256), "W0": (256, 256)}
    c = tg.propagate(wl.CONV3X3_1X1)
    assert c.tiles["x"] == (10, 18, 64) and c.tiles["P"] == (8, 16, 64)
    assert c.tiles["out"] == (8, 16, 128)
    p = tg.propagate(wl.CONV_POOL)
    # the (2,2,F) reuse tile per pooled pixel: 4 x 8 pooled pixels need 8 x 16 conv pixels
    assert p.tiles["out"] == (4, 8, 64) and p.tiles["conv"] == (8, 16, 64)
    assert p.tiles["x"] == (10, 18, 64)
    assert p.bytes("x") == 10 * 18 * 64 * 2


def test_dram_traffic_is_the_sum_of_tensors():
    w = wl.GEMM_FFN
    assert tg.dram_traffic(w) == 2 * (32768 * 256 + 256 * 256 + 256 * 128 + 32768 * 128
                                      + 256 + 128)
    assert tg.dram_traffic(w, fused=False) - tg.dram_traffic(w) == 2 * 2 * 32768 * 256


def test_tiles_per_cta():
    n = tg.tiles_per_cta(256, 152)
    assert len(n) == 152 and sum(n) == 256 and n.count(2) == 104 and n.count(1) == 48
    assert tg.tiles_per_cta(7, 152) == [1] * 7


def test_ffn_l2_traffic_by_hand():
    # 256 tiles on 152 CTAs (104 with 2 tiles, 48 with 1): W0 streamed per tile, W1 once
    # per pair of tiles (P in TMEM), biases once per CTA.
    t = tg.l2_to_smem_traffic(wl.GEMM_FFN)
    assert t["A"] == 32768 * 256 * 2
    assert t["W0"] == 256 * 256 * 256 * 2
    assert t["W1"] == 152 * 256 * 128 * 2
    assert t["bias"] == 152 * (256 + 128) * 2
    assert t["total"] == 16_777_216 + 33_554_432 + 9_961_472 + 116_736   # 60.41 MB
    # with W0 resident (the next layout), W0 crosses once per CTA
    plan = dict(ops.debug_plan("b2b_gemm", (32768, 256, 256, 128)), w0_res=1)
    assert tg.l2_to_smem_traffic(wl.GEMM_FFN, plan)["W0"] == 152 * 256 * 256 * 2


def test_wide_chain_l2_traffic_by_hand():
    # N0 = 512: GEMM0 in two passes over the halves of N0, so every tile's A crosses twice;
    # W0 and W1 streamed per tile (one tile at a time), biases once per CTA.
    t = tg.l2_to_smem_traffic(wl.GEMM_WIDE)
    assert t["A"] == 2 * 32768 * 256 * 2
    assert t["W0"] == 256 * 256 * 512 * 2
    assert t["W1"] == 256 * 512 * 128 * 2
    assert t["bias"] == 152 * (512 + 128) * 2
    assert t["A_in_bounds"] * 2 == t["A"]
    assert t["total"] == 33_554_432 + 67_108_864 + 33_554_432 + 194_560   # 134.41 MB
    # a ragged upper half (N0 = 320) still moves a whole four-block box per K chunk
    w = wl.GemmChain("w320", "bf16", 1280, 128, 320, 64, "relu", "relu")
    assert tg.l2_to_smem_traffic(w)["W0"] == 10 * 2 * (2 * 4 * 64 * 64 * 2)
    # and with N0 not a multiple of 64 one box per block: 5 blocks per K chunk
    w = wl.GemmChain("w296", "bf16", 1280, 128, 296, 64, "relu", "relu")
    assert tg.l2_to_smem_traffic(w)["W0"] == 10 * 2 * (5 * 64 * 64 * 2)


def test_ffn_launch_bounds_by_hand():
    # 104 CTAs run two tiles: per busiest SM, A 2 x 64 KiB + W0 2 x 128 KiB + W1 64 KiB
    # (once per pair) + biases 768 B from L2; 2/256 of the MMA FLOPs on 1/152 of the peak
    b = tg.launch_bounds(wl.GEMM_FFN, hbm_gbs=6791.4, tensor_tflops=1951.4, sm_mhz=2070.0)
    assert abs(b["hbm_us"] - 25_363_200 / 6791.4e3) < 1e-9
    cta = 2 * 65536 + 2 * 131072 + 65536 + 768
    assert abs(b["l2_us"] - cta / (tg.L2_TO_SM_BYTES_PER_CLK * 2070.0)) < 1e-9
    flops = 2 * 32768 * (256 * 256 + 256 * 128)
    assert abs(b["tensor_us"] - flops * 2 / 256 / (1951.4e6 / 152)) < 1e-9
    assert b["bound"] == "tensor" and b["floor_us"] == b["tensor_us"]
    # a resident-weight chain charges its weights once per CTA
    b1 = tg.launch_bounds(wl.CONV1X1)
    assert b1["bound"] == "hbm"
    assert "| gemm_ffn | 2 |" in tg.bounds_report({"gemm_ffn": 9.3})


def test_conv_boxes_are_moved_whole():
    # conv3x3 -> 1x1 on 56 x 56 images: 32 x 7 x 4 tiles of 8 x 16 pixels (the fourth tile
    # column is half outside the image), 3 halo boxes of 10 x 16 pixels x 64 channels each;
    # resident filters once per CTA.  ncu's l1tex__m_xbar2l1tex_read_bytes.sum of one launch
    # reads 68,805,632: out-of-bounds fill crosses the crossbar like data.
    t = tg.l2_to_smem_traffic(wl.CONV3X3_1X1)
    assert t["A"] == 896 * 3 * 10 * 16 * 64 * 2
    assert t["W0"] == 152 * 9 * 64 * 64 * 2 and t["W1"] == 152 * 64 * 128 * 2
    assert t["bias"] == 152 * (64 + 128) * 2
    assert t["total"] == 68_805_632
    assert t["A"] > t["A_in_bounds"]
    # 112 x 112 images tile exactly; only the padding rows and columns are fill
    p = tg.l2_to_smem_traffic(wl.CONV_POOL)
    assert p["A"] == 32 * 14 * 7 * 3 * 10 * 16 * 64 * 2
    assert p["A_in_bounds"] < p["A"] < 1.07 * p["A_in_bounds"]


def test_conv_halo_boxes_read_less():
    # interior tiles of a 3x3 conv: halo loads move 3 boxes of 10 x 16 pixels, per-tap
    # loads 9 boxes of 8 x 16 pixels, per 64-channel block
    halo = tg._conv_tile_input_bytes(1, 64, 64, 64, 3, 3, 1, halo=True)
    taps = tg._conv_tile_input_bytes(1, 64, 64, 64, 3, 3, 1, halo=False)
    assert halo < taps
    interior_halo = 3 * 10 * 16 * 64 * 2
    interior_taps = 9 * 8 * 16 * 64 * 2
    assert interior_halo * 72 == interior_taps * 30
    # a 1-pixel image (pad 1): the pixel lies in the boxes of taps r, s in {0, 1} (4 per-tap
    # boxes) and in the halo boxes of column taps 0 and 1 (2 boxes); out-of-bounds fill is
    # not fetched
    assert tg._conv_tile_input_bytes(1, 1, 1, 8, 3, 3, 1, halo=False) == 4 * 8 * 2
    assert tg._conv_tile_input_bytes(1, 1, 1, 8, 3, 3, 1, halo=True) == 2 * 8 * 2


def test_best_fit_shares_offsets_by_lifetime():
    B = tg.Buffer
    ext, off = tg.best_fit([B("a", 4096, (0, 1)), B("b", 4096, (2, 3)), B("c", 1024, (0, 3))])
    assert off["a"] == off["b"] and ext == 5120       # a and b never live together
    ext, off = tg.best_fit([B("a", 4096, (0, 2)), B("b", 4096, (2, 3))])
    assert off["a"] != off["b"] and ext == 8192       # both live at step 2
    ext, off = tg.best_fit([B("a", 100, (0, 1)), B("b", 100, (0, 1))])
    assert sorted(off.values()) == [0, 1024] and ext == 1124   # 1 KiB alignment


@pytest.mark.parametrize("name", sorted(wl.WORKLOADS))
def test_footprint_matches_the_planner(name):
    # the C planner's layout is tight: the best-fit extent of the same buffers plus the
    # 1 KiB base alignment reproduces its dynamic shared memory size
    plan = tg.plan_of(wl.WORKLOADS[name])
    assert tg.smem_footprint(plan) + 1024 == plan["smem"]


def test_aliased_plan_needs_the_lifetime_analysis():
    # conv3x3 -> 1x1, halo layout with P in shared memory: the planner aliases each P
    # buffer with its group's output staging; without lifetimes the buffers would not fit
    # in 227 KiB
    plan = next(c.plan for c in tg.candidates(wl.CONV3X3_1X1)
                if c.plan["halo"] and not c.plan["p_tmem"] and c.plan["nbuf"] == 2)
    assert plan["alias"] == 1
    bufs = tg.chain_buffers(plan)
    no_reuse = sum(-(-b.size // 1024) * 1024 for b in bufs)
    assert no_reuse + 1024 > 227 * 1024 >= tg.smem_footprint(plan) + 1024


def test_read_ncu_raw_csv(tmp_path):
    # the raw page: a header row, a units row, then one row per launch
    p = tmp_path / "raw.csv"
    p.write_text('"ID","Kernel Name","l1tex__m_xbar2l1tex_read_bytes.sum","dram__bytes_read.sum",'
                 '"launch__grid_size"\n'
                 '"","","Mbyte","Kbyte",""\n'
                 '"0","chain_kernel","60.41","17,074.43","152"\n'
                 '"1","chain_kernel","1.00","2.00","152"\n')
    d = tg.read_ncu_raw_csv(str(p))
    assert d[tg.NCU_L2_TO_SM] == pytest.approx(60.41e6)
    assert d["dram__bytes_read.sum"] == pytest.approx(17_074_430)
    assert d["launch__grid_size"] == 152 and "Kernel Name" not in d
    table = tg.report({"gemm_ffn": str(p)})
    assert "| gemm_ffn |" in table and "60.410 | 1.000 | 60.410 | 1.000" in table


# ------------------------------------------------------------------------------------
# choosing: the model ranks the planner's layouts and its pick is the library's default
# ------------------------------------------------------------------------------------
MODEL_PROBLEMS = [
    ("b2b_gemm", (32768, 256, 256, 128)), ("b2b_gemm", (262144, 256, 256, 128)),
    ("b2b_gemm", (40000, 256, 256, 128)), ("b2b_gemm", (40000, 64, 256, 128)),
    ("b2b_gemm", (200000, 256, 256, 64)), ("b2b_gemm", (1024, 64, 64, 64)),
    ("b2b_gemm", (640, 128, 128, 256)), ("b2b_gemm", (300, 128, 256, 64)),
    ("b2b_gemm", (257, 72, 40, 24)), ("b2b_gemm", (32768, 256, 512, 128)),
    ("gemm_bias_act", (513, 256, 256)), ("gemm_bias_act", (300000, 64, 64)),
    ("b2b_conv_nhwc", (64, 56, 56, 64, 64, 1, 1, 0, 64)),
    ("b2b_conv_nhwc", (32, 56, 56, 64, 64, 3, 3, 1, 128)),
    ("b2b_conv_nhwc", (32, 56, 56, 64, 64, 3, 3, 1, 128, 2)),
    ("b2b_conv_nhwc", (1, 10, 12, 32, 32, 5, 5, 2, 16)),
    ("conv_bias_act_nhwc", (2, 9, 9, 64, 64, 3, 3, 1)),
    ("conv_bias_act_nhwc", (64, 28, 28, 128, 64, 3, 3, 1, 2)),
    ("conv_relu_maxpool", (32, 112, 112, 64, 64)), ("conv_relu_maxpool", (1, 7, 9, 16, 8)),
    ("b2b_gemm3", (40000, 128, 128, 64, 64)), ("b2b_gemm3", (262144, 64, 64, 64, 64)),
]


@pytest.fixture
def _no_choices():
    ops.autotune_reset()
    yield
    ops.autotune_reset()


def test_pair_and_streamed_bounds_by_hand():
    # FFN at 262144 rows.  CTA pairs: 1024 tiles of 256 rows on 76 pairs, the busiest with
    # 14; per SM its 128 rows of each tile's A (64 KiB per tile), its halves of W0 (64 KiB)
    # and W1 (32 KiB) once, its bias halves (128 + 64 elements).  Single CTAs, W0 streamed:
    # 2048 tiles on 152 CTAs, the busiest with 14: A and W0 (128 KiB) per tile, W1 (64 KiB)
    # once per pair of tiles, both biases.  One SM moves 89 B/clk at 2070 MHz.
    w = wl.GEMM_FFN_LARGE
    rate = 89.0 * 2070.0                       # bytes per microsecond
    by_cand = {c.cand: c for c in tg.candidates(w)}
    pair = by_cand[4]
    assert pair.plan["cta_pair"] == 1 and pair.tiles_per_unit == 14
    assert pair.bounds["l2_us"] == pytest.approx((14 * 65536 + 65536 + 32768 + 384) / rate)
    streamed = by_cand[0]
    assert streamed.plan["resident"] == 0 and streamed.plan["w0_res"] == 0
    assert streamed.tiles_per_unit == 14
    assert streamed.bounds["l2_us"] == pytest.approx(
        (14 * 65536 + 14 * 131072 + 7 * 65536 + 768) / rate)
    # HBM: 768 B per row (A in, output out) and the weights and biases once
    assert pair.bounds["hbm_us"] == pytest.approx((262144 * 768 + 197376) / 6791.4e3)


@pytest.mark.parametrize("kind,dims", MODEL_PROBLEMS, ids=lambda x: str(x))
def test_model_pick_is_the_library_default(kind, dims, _no_choices):
    """The library ranks layouts with its own copy of the model (C); both must pick the
    same layout, and every layout the planner offers must pass the model's footprint
    check."""
    w = tg.workload_of(kind, dims)
    ranked = tg.rank(w)
    n = ops.debug_plan(kind, dims, cand=0)["ncand"]
    assert sorted(c.cand for c in ranked) == list(range(n))       # none over the footprint
    assert ops.debug_plan(kind, dims)["cand"] == ranked[0].cand


def test_every_workload_defaults_to_the_model_pick(_no_choices):
    for name, w in wl.WORKLOADS.items():
        assert tg.plan_of(w)["cand"] == tg.rank(w)[0].cand, name


def test_pairs_only_in_the_steady_state(_no_choices):
    # two tiles per CTA (32768 rows): the bounds do not decide, the planner's preference
    # (single CTAs, P in TMEM, streamed weights) does; three or more (past 152 x 256 rows):
    # the pairs' lower L2 -> SM bound wins
    assert tg.rank(wl.GEMM_FFN)[0].plan["cta_pair"] == 0
    assert tg.rank(wl.GEMM_FFN.with_m(152 * 256 + 1))[0].plan["cta_pair"] == 1
    assert tg.rank(wl.GEMM_FFN_LARGE)[0].plan["cta_pair"] == 1


def test_top_extends_over_what_the_model_cannot_order(_no_choices):
    # one tile per CTA: no layout is ordered by the bounds, so the profiler gets them all
    small = tg.top(wl.GEMM_SMALL)
    assert [c.cand for c in small] == [c.cand for c in tg.rank(wl.GEMM_SMALL)]
    # steady state with distinct bounds: exactly the best three
    large = tg.top(wl.GEMM_FFN_LARGE)
    assert len(large) == 3 and large[0].plan["cta_pair"] == 1


def test_choose_hands_the_top_to_the_profiler(_no_choices):
    w = wl.GEMM_FFN_LARGE
    kind, dims = tg.problem_of(w)
    got = tg.choose(w, k=2)
    assert got == [c.cand for c in tg.rank(w)[:2]]
    c = ops.get_choice(kind, dims)
    assert (c["source"], c["cand"]) == (3, got[0])
    assert ops.debug_plan(kind, dims)["cand"] == got[0]
