"""bench.py's host logic without a GPU: workload descriptions, algorithmic
bytes, the kernel source hash that keys the recorded DRAM traffic."""
import json
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
from tiled_tensor_core_persistent_gb300 import analysis, inputs  # noqa: E402


def test_case_bytes_single_and_grouped():
    c = inputs.make_case("b", 300, 200, 64, seed=1, dist="uniform", beta=0.5, c_dist="uniform", bias_std=0.1)
    # A, B, C and D in bf16, bias in bf16
    assert bench.case_bytes(c) == analysis.gemm_bytes(300, 200, 64, 2, 2, 2, 2)
    g = inputs.make_grouped_case("g", [(300, 200, 64), (10, 20, 30)], seed=2, dist="uniform")
    assert bench.case_bytes(g) == sum(bench.case_bytes(p) for p in g.problems)


def test_workload_config_describes_the_case():
    c = inputs.square_512()
    cfg = bench.workload_config(c, True)
    assert (cfg["M"], cfg["N"], cfg["K"]) == (512, 512, 512)
    assert "flush" in cfg["l2"]
    g = inputs.make_grouped_case("g", [(300, 64, 32), (20, 64, 32)], seed=3, dist="uniform", bias_std=0.1,
                                 act="gelu")
    gc = bench.workload_config(g, False)
    assert gc["problems"] == [[300, 64, 32], [20, 64, 32]] and gc["M"] == 320
    assert "grouped gemm, 2 problems" in gc["workload"] and "gelu" in gc["workload"]
    json.dumps(gc)   # serialisable into the bench line


def test_every_workload_has_a_factory_and_flush_flag():
    for name, (factory, flush) in bench.WORKLOADS.items():
        assert callable(factory) and isinstance(flush, bool), name
    assert bench.DEFAULT_WORKLOAD in bench.WORKLOADS


def test_kernel_source_hash_follows_the_code_not_the_comments(tmp_path):
    """A copy of csrc/ hashes like the package's; editing a comment, blank
    space or a test-only debug_* file keeps the hash, editing code (even inside
    a string literal that looks like a comment) changes it."""
    import shutil
    csrc = os.path.join(ROOT, "tiled_tensor_core_persistent_gb300", "csrc")
    d = tmp_path / "csrc"
    shutil.copytree(csrc, d)
    base = bench.source_hash(str(d))
    assert base == bench.kernel_source_hash()
    k = d / "gemm_kernel.cuh"
    text = k.read_text()
    k.write_text(text.replace("#pragma once", "#pragma once\n// a new comment\n/* and a block */\n\n", 1))
    assert bench.source_hash(str(d)) == base
    (d / "debug_extra.cu").write_text("int x;\n")
    assert bench.source_hash(str(d)) == base
    k.write_text(text.replace("#pragma once", "#pragma once\nstatic const char* kTag = \"// not a comment\";", 1))
    assert bench.source_hash(str(d)) != base
    k.write_text(text.replace("constexpr int kEpiChunk = 32;", "constexpr int kEpiChunk = 64;", 1))
    assert bench.source_hash(str(d)) != base


def test_recorded_traffic_only_for_the_current_source():
    with open(os.path.join(ROOT, "profiles", "traffic.json")) as f:
        rec = json.load(f)
    for name, entry in rec.items():
        got = bench.recorded_traffic(name)
        if entry.get("kernel_source_hash") == bench.kernel_source_hash():
            assert got == entry["dram_bytes_per_launch"]
        else:
            assert got is None
    assert bench.recorded_traffic("no_such_workload") is None
