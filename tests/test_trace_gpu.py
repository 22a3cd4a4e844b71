"""The optional per-CTA event trace: it records every step of every tile of the chosen CTA,
in causal order (one global clock for all warps), and leaves the results unchanged."""
import pytest
import torch

from gemm_conv_chains_gb300 import ops
from gemm_conv_chains_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    yield
    ops.set_trace(None)


def test_trace_of_a_chain_is_complete_and_causal():
    w = wl.GemmChain("t", "f16", 128 * 400, 64, 64, 64, "relu", "relu")
    t = {k: v.cuda() for k, v in wl.gemm_inputs(w, seed=1).items()}
    ref = ops.b2b_gemm(t["A"], t["W0"], t["b0"], t["W1"], t["b1"], "relu", "relu")
    buf = torch.zeros(2 * 4096, dtype=torch.int64, device="cuda")
    ops.set_trace(buf, cta=3)
    out = ops.b2b_gemm(t["A"], t["W0"], t["b0"], t["W1"], t["b1"], "relu", "relu")
    ops.set_trace(None)
    torch.cuda.synchronize()
    assert torch.equal(out.view(torch.int16), ref.view(torch.int16))
    ev = ops.read_trace(buf)
    grid = min(ops.num_sms(), 400)
    ntiles = len(range(3, 400, grid))
    names = [e[1] for e in ev]
    for name in ("mma_g0_done", "mma_p_ready", "mma_g1_done", "epi_acc_ready", "epi_p_done",
                 "epi_d1_ready", "epi_stored"):
        assert names.count(name) == ntiles, (name, names.count(name), ntiles)
    when = {(e[1], e[3]): e[0] for e in ev}   # the last event of each kind per tile
    for it in range(ntiles):
        # An MMA issuer's stamp taken after it commits may come after the epilogue has seen
        # the MMAs complete, so each epilogue step is ordered after a stamp taken before the
        # MMAs it waits for were issued: the last GEMM0 chunk's arrival, P's publication.
        assert when[("mma_full", it)] <= when[("epi_acc_ready", it)]
        assert when[("mma_p_ready", it)] <= when[("mma_g1_done", it)]
        assert when[("mma_p_ready", it)] <= when[("epi_d1_ready", it)]
        assert when[("epi_d1_ready", it)] <= when[("epi_stored", it)]
    # the CTA's entry event comes first, then the end of its setup, then the end of the
    # wait for the previous grid; the first MMA follows both
    for name in ("kernel_entry", "setup_done", "dep_ready"):
        assert names.count(name) == 1, name
    assert all(when[("kernel_entry", 0)] <= e[0] for e in ev)
    assert when[("setup_done", 0)] <= when[("dep_ready", 0)] <= when[("mma_g0_done", 0)]
    # the producer starts after its own dependency wait and before its first load; the MMA
    # issuer sets up before its wait for the previous grid
    for name in ("prod_start", "mma_setup"):
        assert names.count(name) == 1, name
    assert when[("prod_start", 0)] <= when[("prod_acquire", 0)]
    assert when[("setup_done", 0)] <= when[("mma_setup", 0)] <= when[("dep_ready", 0)]


def test_trace_off_records_nothing():
    buf = torch.zeros(2 * 64, dtype=torch.int64, device="cuda")
    ops.set_trace(buf)
    ops.set_trace(None)
    w = wl.GemmChain("t", "bf16", 512, 64, 64, 64, "relu", "relu")
    t = {k: v.cuda() for k, v in wl.gemm_inputs(w, seed=2).items()}
    ops.b2b_gemm(t["A"], t["W0"], t["b0"], t["W1"], t["b1"])
    torch.cuda.synchronize()
    assert int(torch.count_nonzero(buf)) == 0
