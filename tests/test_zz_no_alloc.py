"""tcg_gemm_noalloc: the GEMM for callers that cannot allocate device memory.

Such callers (a plugin handed only input/output pointers by an engine that
owns all device memory, a latency-critical loop where cudaMalloc/cudaFree are
not allowed) cannot supply the workspace tcg_gemm needs, so this entry point
takes its scratch from a fixed 32 MiB device array inside the library.  The
test calls it through the C ABI twice in a row and checks each result against
tcg_gemm with a caller-provided workspace.  The file is named to be collected
last and passes both alone and after the other tests.
"""
import numpy as np
import pytest
import torch

import tiled_tensor_core_persistent_gb300 as tcg
from tiled_tensor_core_persistent_gb300 import harness, inputs

from parity import TOL, assert_within

pytestmark = pytest.mark.gpu

WORKSPACE_ERROR = 5


@pytest.fixture(autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    from tiled_tensor_core_persistent_gb300 import _build
    _build.build()
    tcg.debug_set()
    yield
    tcg.debug_set()


def noalloc(case, dc, D):
    tcg.gemm_noalloc(case.M, case.N, case.K, case.alpha, dc.A, case.lda, case.opA, dc.B, case.ldb, case.opB,
                     case.beta, dc.C, case.ldc, case.c_dtype, D, case.ldd, case.d_dtype, bias=dc.bias,
                     bias_dtype=case.bias_dtype, act=case.act, ab_dtype=case.ab_dtype,
                     scale_a=case.scale_a, scale_b=case.scale_b)


@pytest.mark.parametrize("which", ["pair_tiles", "split_k"])
def test_noalloc_matches_workspace_entry_point_twice(which):
    if which == "pair_tiles":
        case = inputs.make_case("noalloc_pair", 1024, 1536, 640, seed=171, dist="uniform", beta=0.5,
                                c_dist="uniform", bias_std=0.1, act="gelu")
    else:
        tcg.debug_set(force_splits=4)  # split-K partials live in the scratch
        case = inputs.ragged(1, 1)     # 16 x 8192 x 8192
        assert tcg.plan(case.M, case.N, case.K)["splits"] == 4
    dc = harness.DeviceCase(case)
    dc.run()  # the existing entry point, caller-provided workspace
    torch.cuda.synchronize()
    assert tcg.device_status(dc.workspace) == 0
    ref = dc.result().numpy()
    for _ in range(2):
        D = torch.full_like(dc.D_view, float("nan"))
        noalloc(case, dc, D)
        torch.cuda.synchronize()
        got = D[:, :case.N].to(torch.float64).cpu().numpy()
        assert_within(got, ref, TOL[case.ab_dtype], f"noalloc {which}")


def test_noalloc_rejects_problems_beyond_the_scratch():
    case = inputs.make_case("noalloc_big", 16, 8192, 8192, seed=181, dist="uniform")
    tcg.debug_set(force_splits=16)  # 32 tiles x 16 splits of fp32 partials = 64 MiB
    dc = harness.DeviceCase(case)
    with pytest.raises(tcg.TcgError) as err:
        noalloc(case, dc, dc.D_view)
    assert err.value.code == WORKSPACE_ERROR
    assert "maximum" in tcg.last_error()
