"""Launch choices and the profiler's bookkeeping, on the host (no CUDA call).

Every feasible shared-memory / TMEM layout the planner offers for a problem must be a
valid plan (the same structural checks as the default plan), pinning a choice must be
reflected by b2b_debug_plan, and infeasible or out-of-range choices must be refused.
"""
import pytest

from gemm_conv_chains_gb300 import ops
from gemm_conv_chains_gb300 import tilegraph as tg
from test_plan import check

PROBLEMS = [
    ("b2b_gemm", (32768, 256, 256, 128)), ("b2b_gemm", (1024, 64, 64, 64)),
    ("b2b_gemm", (640, 128, 128, 256)), ("b2b_gemm", (300, 128, 256, 64)),
    ("b2b_gemm", (257, 72, 40, 24)), ("gemm_bias_act", (513, 256, 256)),
    ("b2b_conv_nhwc", (64, 56, 56, 64, 64, 1, 1, 0, 64)),
    ("b2b_conv_nhwc", (32, 56, 56, 64, 64, 3, 3, 1, 128)),
    ("b2b_conv_nhwc", (1, 10, 12, 32, 32, 5, 5, 2, 16)),
    ("conv_bias_act_nhwc", (2, 9, 9, 64, 64, 3, 3, 1)),
    ("conv_relu_maxpool", (32, 112, 112, 64, 64)), ("conv_relu_maxpool", (1, 7, 9, 16, 8)),
]


@pytest.fixture(autouse=True)
def _reset():
    ops.autotune_reset()
    yield
    ops.autotune_reset()


def _row_major(kind, dims):
    # b2b_gemm / gemm_bias_act take row-major [K][N] weights; 1x1 convs run as GEMMs with
    # K-major filters
    return kind in ("b2b_gemm", "gemm_bias_act")


@pytest.mark.parametrize("kind,dims", PROBLEMS, ids=lambda x: str(x))
def test_every_feasible_layout_is_a_valid_plan(kind, dims):
    default = ops.debug_plan(kind, dims)
    n = default["ncand"]
    assert 1 <= n <= 16 and 0 <= default["cand"] < n
    assert default["grid_choice"] == -1 and default["pf_choice"] == -1
    stages = []
    for cand in range(n):
        ops.set_choice(kind, dims, cand=cand)
        p = check(kind, dims, _row_major(kind, dims))
        assert p["cand"] == cand and p["ncand"] == n
        stages.append(p["stages"])
    # the default is the tile-graph model's pick
    assert default["cand"] == tg.rank(tg.workload_of(kind, dims))[0].cand
    assert all(s >= 2 for s in stages)


def test_infeasible_and_out_of_range_choices_are_refused():
    kind, dims = "b2b_gemm", (32768, 256, 256, 128)
    n = ops.debug_plan(kind, dims)["ncand"]
    with pytest.raises(ops.B2BError) as e:
        ops.set_choice(kind, dims, cand=n)
    assert e.value.status == 4          # B2B_ERR_UNSUPPORTED
    for bad in (dict(grid=3), dict(prefetch_second=2), dict(cand=-2), dict(grid=-3)):
        with pytest.raises(ops.B2BError) as e:
            ops.set_choice(kind, dims, **bad)
        assert e.value.status == 2      # B2B_ERR_SHAPE
    assert ops.get_choice(kind, dims)["source"] == 0


def test_pinned_choice_is_recorded_and_reset():
    kind, dims = "b2b_conv_nhwc", (64, 56, 56, 64, 64, 1, 1, 0, 64)
    assert ops.get_choice(kind, dims) == dict(source=0, cand=-1, grid=-1, prefetch_second=-1,
                                              best_ns=0, default_ns=0, timed=0)
    ops.set_choice(kind, dims, cand=1, grid=1, prefetch_second=0)
    c = ops.get_choice(kind, dims)
    assert (c["source"], c["cand"], c["grid"], c["prefetch_second"]) == (1, 1, 1, 0)
    p = ops.debug_plan(kind, dims)
    assert (p["cand"], p["grid_choice"], p["pf_choice"]) == (1, 1, 0)
    # another problem is unaffected
    assert ops.debug_plan(kind, (64, 56, 56, 64, 64, 1, 1, 0, 128))["grid_choice"] == -1
    ops.autotune_reset()
    assert ops.get_choice(kind, dims)["source"] == 0
    assert ops.debug_plan(kind, dims)["grid_choice"] == -1


def test_autotune_switch_needs_no_device():
    ops.set_autotune(True)
    ops.set_autotune(False)


def test_plan_of_a_forced_candidate_ignores_the_pinned_choice():
    kind, dims = "b2b_gemm", (32768, 256, 256, 128)
    n = ops.debug_plan(kind, dims)["ncand"]
    ops.set_choice(kind, dims, cand=n - 1)
    for cand in range(n):
        p = ops.debug_plan(kind, dims, cand=cand)
        assert p["cand"] == cand and p["grid_choice"] == -1
    with pytest.raises(ops.B2BError) as e:
        ops.debug_plan(kind, dims, cand=n)
    assert e.value.status == 4
    with pytest.raises(ops.B2BError) as e:
        ops.debug_plan(kind, dims, cand=-1)
    assert e.value.status == 2


def test_choices_are_filed_per_dtype_and_epilogue():
    """A choice pinned for one dtype / epilogue pair applies to that variant only; sizes
    alone pin it for every variant, and a variant's own entry takes precedence."""
    kind, dims = "b2b_gemm", (4096, 128, 128, 64)
    bf16_hs = list(dims) + ops.variant("bf16", "hardswish", "hardswish")
    f16_relu = list(dims) + ops.variant("f16", "relu", "relu")
    default = ops.debug_plan(kind, dims)["cand"]
    assert default != 1
    ops.set_choice(kind, bf16_hs, cand=1)
    assert ops.get_choice(kind, bf16_hs)["cand"] == 1
    assert ops.get_choice(kind, f16_relu)["source"] == 0
    assert ops.debug_plan(kind, bf16_hs)["cand"] == 1
    assert ops.debug_plan(kind, f16_relu)["cand"] == default
    # a query by sizes alone reads the most recent entry of any variant
    assert ops.get_choice(kind, dims)["cand"] == 1
    ops.set_choice(kind, f16_relu, cand=2)
    assert ops.get_choice(kind, dims)["cand"] == 2
    # sizes alone: a wildcard entry, which variants without their own entry fall back to
    ops.set_choice(kind, dims, cand=3)
    assert ops.get_choice(kind, dims)["cand"] == 3
    assert ops.get_choice(kind, bf16_hs)["cand"] == 1
    other = list(dims) + ops.variant("bf16", "relu", "none")
    # a variant with no entry of its own takes the wildcard's
    assert ops.get_choice(kind, other)["cand"] == ops.debug_plan(kind, other)["cand"] == 3


@pytest.mark.parametrize("kind,dims,nv", [
    ("b2b_gemm", (1024, 64, 64, 64), 3), ("gemm_bias_act", (513, 256, 256), 2),
    ("b2b_conv_nhwc", (2, 9, 9, 64, 64, 3, 3, 1, 64, 1), 3),
    ("conv_bias_act_nhwc", (2, 9, 9, 64, 64, 3, 3, 1, 1), 2),
    ("conv_relu_maxpool", (1, 7, 9, 16, 8), 1), ("b2b_gemm3", (1024, 64, 64, 64, 64), 4)])
def test_variant_dims_are_checked(kind, dims, nv):
    good = list(dims) + [1] + [2] * (nv - 1)
    ops.set_choice(kind, good, cand=0)
    assert ops.get_choice(kind, good)["source"] == 1
    for bad in (good[:-1] if nv > 1 else None, good + [0], good[:len(dims)] + [2] + good[len(dims) + 1:],
                good[:len(dims) + 1] + [3] * (nv - 1) if nv > 1 else None):
        if bad is None:
            continue
        with pytest.raises(ops.B2BError) as e:
            ops.debug_plan(kind, bad)
        assert e.value.status == 2, bad


def test_model_ranking_sets_the_default_and_is_recorded():
    kind, dims = "b2b_gemm", (32768, 256, 256, 128)
    n = ops.debug_plan(kind, dims)["ncand"]
    ops.set_candidates(kind, dims, [n - 1, 0])
    c = ops.get_choice(kind, dims)
    assert (c["source"], c["cand"], c["grid"]) == (3, n - 1, -1)
    assert ops.debug_plan(kind, dims)["cand"] == n - 1
    assert ops.tune_record(kind, dims) == []              # nothing measured yet
    for bad, status in (([], 2), ([0, 0], 2), ([-1], 2), ([n], 4)):
        with pytest.raises(ops.B2BError) as e:
            ops.set_candidates(kind, dims, bad)
        assert e.value.status == status
    # pinning replaces the ranking
    ops.set_choice(kind, dims, cand=0)
    assert ops.get_choice(kind, dims)["source"] == 1
