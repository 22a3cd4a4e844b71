"""The bench's link between the ncu counters in profiles/traffic.json and the kernel source:
counters are reported only for the code they were taken on, and comments do not count."""
import json
import os
import shutil

import bench

SRC = ("chain_kernel.cuh", "chain_cta2_kernel.cuh", "ptx.cuh", "kernel_params.h", "kernel_units.cuh",
       "kernels_cta2_units.cuh", "api.cu")


def _copy_tree(tmp_path):
    csrc = tmp_path / "gemm_conv_chains_gb300" / "csrc"
    csrc.mkdir(parents=True)
    for name in SRC:
        shutil.copy(os.path.join(bench.ROOT, "gemm_conv_chains_gb300", "csrc", name), csrc / name)
    (tmp_path / "profiles").mkdir()
    shutil.copy(os.path.join(bench.ROOT, "profiles", "traffic.json"),
                tmp_path / "profiles" / "traffic.json")
    return csrc


def test_hash_ignores_comments_not_code(tmp_path, monkeypatch):
    csrc = _copy_tree(tmp_path)
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    h0 = bench.kernel_source_sha()
    p = csrc / "kernel_params.h"
    text = p.read_text()
    p.write_text("// a new comment line\n\n" + text.replace("#pragma once", "#pragma once  // x"))
    assert bench.kernel_source_sha() == h0
    p.write_text(text.replace("constexpr int kBlockM = 128;", "constexpr int kBlockM = 64;"))
    assert bench.kernel_source_sha() != h0


def test_traffic_only_for_the_captured_code(tmp_path, monkeypatch):
    csrc = _copy_tree(tmp_path)
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    rec = json.loads((tmp_path / "profiles" / "traffic.json").read_text())
    if rec["kernel_source_sha"] == bench.kernel_source_sha():
        assert bench.load_traffic("gemm_ffn") == rec["workloads"]["gemm_ffn"]["dram_bytes_per_launch"]
    p = csrc / "api.cu"
    p.write_text(p.read_text() + "\nstatic int b2b_unused_marker = 0;\n")
    assert bench.load_traffic("gemm_ffn") is None
