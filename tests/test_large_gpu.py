"""Extreme sizes.  A GEMM whose output has more than 2^31 elements (49152 x
49152 fp32 D, 9.7 GB, 36,864 pair tiles per launch): every offset into D
past 2^31 elements must be formed in 64 bits, in the register-store epilogue
(ldd = N: 32-byte stores) and in the element-wise one (ldd = N + 1, whose
rows are not 16-byte multiples).  A K of 2^20 (split K) and a D of 2^20 - 3
rows.  Integer operands with fp32 D, so the sampled outputs (full rows
including the last ones, full columns and the four corner tiles) must equal
the oracle exactly; the guard rows around D (and the padding column) must
still hold the sentinel."""
import pytest
import torch

import tiled_tensor_core_persistent_gb300 as tcg
from tiled_tensor_core_persistent_gb300 import harness, inputs

from parity import check_rows_cols_corners, oracle_for

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    free, _ = torch.cuda.mem_get_info()
    if free < 24 << 30:
        pytest.skip("needs about 20 GB of free device memory")
    from tiled_tensor_core_persistent_gb300 import _build
    _build.build()
    tcg.debug_set()


@pytest.mark.parametrize("pad", [0, 1], ids=["register_stores", "elementwise"])
def test_output_beyond_2_31_elements(pad):
    M = N = 49152
    K = 64
    assert M * N > 2 ** 31
    case = inputs.make_case(f"big_d_pad{pad}", M, N, K, seed=700 + pad, dist="int4", d_dtype="f32", ldd=N + pad)
    dc = harness.DeviceCase(case, guard_rows=1)
    try:
        dc.run()
        torch.cuda.synchronize()
        assert tcg.device_status(dc.workspace) == 0, tcg.last_error()
        check_rows_cols_corners(dc.D_view[:, :N], oracle_for(case), M, N, 0.0, case.name, nrows=48, ncols=48,
                                corner=64, seed=pad, exact=True)
        s = dc.sentinel_stored
        assert bool((dc.D_full[0] == s).all()) and bool((dc.D_full[-1] == s).all()), "guard rows written"
        if pad:
            assert bool((dc.D_view[:, N] == s).all()), "padding column written"
    finally:
        del dc
        torch.cuda.empty_cache()


def test_long_k_split_exact():
    """K = 2^20 (split K, a long run of k-blocks per piece): integer operands
    keep every fp32 partial sum exact, so the sampled outputs equal the
    oracle's."""
    M, N, K = 200, 300, 1 << 20
    case = inputs.make_case("long_k", M, N, K, seed=710, dist="int4", d_dtype="f32")
    assert tcg.plan(M, N, K)["splits"] > 1
    dc = harness.DeviceCase(case, guard_rows=1)
    try:
        dc.run()
        torch.cuda.synchronize()
        assert tcg.device_status(dc.workspace) == 0, tcg.last_error()
        check_rows_cols_corners(dc.D_view[:, :N], oracle_for(case), M, N, 0.0, case.name, nrows=24, ncols=24,
                                corner=32, seed=7, exact=True)
        s = dc.sentinel_stored
        assert bool((dc.D_full[0] == s).all()) and bool((dc.D_full[-1] == s).all()), "guard rows written"
    finally:
        del dc
        torch.cuda.empty_cache()


def test_a_million_rows_exact():
    """M = 2^20 - 3 rows of a narrow D (4096 pair-tile rows, ragged last
    tile): exact on sampled rows including the last ones, on full columns and
    corners; guard rows untouched."""
    M, N, K = (1 << 20) - 3, 72, 40
    case = inputs.make_case("many_rows", M, N, K, seed=711, dist="int4", d_dtype="f32")
    dc = harness.DeviceCase(case, guard_rows=1)
    try:
        dc.run()
        torch.cuda.synchronize()
        assert tcg.device_status(dc.workspace) == 0, tcg.last_error()
        check_rows_cols_corners(dc.D_view[:, :N], oracle_for(case), M, N, 0.0, case.name, nrows=64, ncols=24,
                                corner=64, seed=8, exact=True)
        s = dc.sentinel_stored
        assert bool((dc.D_full[0] == s).all()) and bool((dc.D_full[-1] == s).all()), "guard rows written"
    finally:
        del dc
        torch.cuda.empty_cache()
