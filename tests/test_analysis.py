"""Pins of the analytic models against the worked values printed on the pages."""
import json
import os

import pytest

from tiled_tensor_core_persistent_gb300 import analysis

with open(os.path.join(os.path.dirname(__file__), "golden", "page_values.json")) as f:
    PAGE = json.load(f)


def test_tile_intensity_widget():
    w = PAGE["tile_intensity_widget"]
    ai = analysis.boundary_intensity(w["M"], w["N"], w["K"], w["bytes_per_element"])
    assert round(ai, 2) == w["intensity_flop_per_byte"]
    assert 2 * w["M"] * w["N"] * w["K"] == w["flops"]
    fits = analysis.double_buffer_bytes(w["M"], w["N"], w["K"], w["bytes_per_element"]) <= w["smem_budget_kib"] * 1024
    assert fits == w["buffers_fit"]


def test_square_gemm_intensity_is_n_over_4():
    w = PAGE["square_gemm_intensity"]
    assert analysis.square_gemm_intensity_mixed(w["N"], w["in_bytes"], w["out_bytes"]) == w["intensity_flop_per_byte"]
    assert analysis.square_gemm_intensity_mixed(2048) == 2048 / 4


def test_ridge_and_square_tile():
    w = PAGE["a100_ridge"]
    ridge = analysis.ridge_point(w["peak_tflops"] * 1e12, w["bandwidth_tbs"] * 1e12)
    assert ridge == w["ridge_flop_per_byte"]
    # square tile intensity T / b must exceed the ridge: T > ridge * b
    assert ridge * w["bytes_per_element"] == w["min_square_tile"]
    T = w["min_square_tile"]
    assert analysis.boundary_intensity(T, T, 10 ** 9, w["bytes_per_element"]) == pytest.approx(T / 2, rel=1e-6)


def test_pipeline_widget():
    w = PAGE["pipeline_widget"]
    n, L, C = w["tiles"], w["load_us"], w["compute_us"]
    assert analysis.serial_time(n, L, C) == w["serial_us"]
    assert analysis.pipeline_time(n, L, C) == w["pipelined_us"]
    assert analysis.serial_time(n, L, C) / analysis.pipeline_time(n, L, C) == w["speedup"]
    # the slower stage sets the steady-state interval, whichever it is
    assert analysis.pipeline_time(n, C, L) == analysis.pipeline_time(n, L, C)


def test_roofline_is_min():
    assert analysis.roofline(100.0, 2.0, 10.0) == 20.0
    assert analysis.roofline(100.0, 20.0, 10.0) == 100.0


def test_swizzle_removes_column_bank_conflicts():
    w = PAGE["swizzle_bank_example"]
    rows, cols = w["rows"], w["cols"]
    for c in (0, 5, 31, 127):
        plain = {analysis.bank(r * cols + c) for r in range(rows)}
        swz = {analysis.bank(analysis.swizzle(r * cols + c, w["BBits"], w["MBase"], w["SShift"]))
               for r in range(rows)}
        assert rows // len(plain) == w["conflict_ways_unswizzled"]
        assert len(swz) == w["distinct_banks_swizzled"]


def test_swizzle_is_a_permutation_of_the_tile():
    w = PAGE["swizzle_bank_example"]
    n = w["rows"] * w["cols"]
    assert sorted(analysis.swizzle(o, w["BBits"], w["MBase"], w["SShift"]) for o in range(n)) == list(range(n))


def test_workload_intensities():
    # the metric workload (8192^3 bf16) and the two HBM-bound skinny shapes
    assert analysis.boundary_intensity(8192, 8192, 8192, 2) == pytest.approx(2730.67, rel=1e-5)
    assert analysis.boundary_intensity(16, 8192, 8192, 2) == pytest.approx(15.94, rel=1e-3)
    assert analysis.boundary_intensity(8192, 128, 8192, 2) == pytest.approx(124.1, rel=1e-3)
