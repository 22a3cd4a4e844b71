"""Launch choices and the profiler's bookkeeping, on the host (no CUDA call).

Every feasible shared-memory / TMEM layout the planner offers for a problem must be a
valid plan (the same structural checks as the default plan), pinning a choice must be
reflected by b2b_debug_plan, and infeasible or out-of-range choices must be refused.
"""
import pytest

from gemm_conv_chains_gb300 import ops
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
    # the default is the first feasible layout with three or more ring stages, else the first
    first3 = next((i for i, s in enumerate(stages) if s >= 3), 0)
    assert default["cand"] == first3
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
