"""tcg_gemm_noalloc: the GEMM for callers that cannot allocate device memory.

Such callers (a plugin handed only input/output pointers by an engine that
owns all device memory, a latency-critical loop where cudaMalloc/cudaFree are
not allowed) cannot supply the workspace tcg_gemm needs, so this entry point
takes its scratch from a fixed 32 MiB device array inside the library.  The
tests call it through the C ABI twice in a row.  It runs the same plan and
kernel as tcg_gemm, so each result must equal tcg_gemm's with a
caller-provided workspace bit for bit (split-K sums in a fixed order), and
integer-valued inputs with fp32 D must equal the oracle exactly.  The cases
cover pair tiles, split-K partials and arrival counters kept in the array,
and an operand with an odd leading dimension whose packed copy lives in the
array.  The file is named to be collected last and passes both alone and
after the other tests.
"""
import numpy as np
import pytest
import torch

import tiled_tensor_core_persistent_gb300 as tcg
from tiled_tensor_core_persistent_gb300 import harness, inputs

from parity import oracle_for

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


def make(which):
    if which == "pair_tiles":
        return inputs.make_case("noalloc_pair", 1024, 1536, 640, seed=171, dist="uniform", beta=0.5,
                                c_dist="uniform", bias_std=0.1, act="gelu")
    if which == "split_k":
        tcg.debug_set(force_splits=4)  # split-K partials and counters live in the scratch
        case = inputs.ragged(1, 1)     # 16 x 8192 x 8192
        assert tcg.plan(case.M, case.N, case.K)["splits"] == 4
        return case
    if which == "split_k_int_exact":
        tcg.debug_set(force_splits=3)
        return inputs.make_case("noalloc_int", 300, 520, 1100, seed=172, dist="int4", d_dtype="f32",
                                beta=0.5, c_dist="int4", c_dtype="f32", act="relu")
    if which == "packed_lda":
        # lda = K + 1 (odd): A is not TMA-addressable, so its packed copy goes into the scratch
        return inputs.make_case("noalloc_pack", 333, 290, 201, seed=173, dist="int4", d_dtype="f32", lda=202)
    raise ValueError(which)


@pytest.mark.parametrize("which", ["pair_tiles", "split_k", "split_k_int_exact", "packed_lda"])
def test_noalloc_matches_workspace_entry_point_twice(which):
    case = make(which)
    dc = harness.DeviceCase(case)
    if which == "packed_lda":
        assert tcg.workspace_size_for(case.M, case.N, case.K, "bf16", dc.A, case.lda, case.opA, dc.B, case.ldb,
                                      case.opB) > tcg.workspace_size(case.M, case.N, case.K)
    dc.run()  # the existing entry point, caller-provided workspace
    torch.cuda.synchronize()
    assert tcg.device_status(dc.workspace) == 0
    ref = dc.D_view[:, :case.N].clone()
    exact = case.d_dtype == "f32" and which != "pair_tiles"
    want = oracle_for(case).full() if exact else None
    if exact:
        assert np.array_equal(ref.to(torch.float64).cpu().numpy(), want)
    for _ in range(2):
        D = torch.full_like(dc.D_view, float("nan"))
        noalloc(case, dc, D)
        torch.cuda.synchronize()
        got = D[:, :case.N]
        assert torch.equal(got.view(torch.int16) if got.dtype == torch.bfloat16 else got.view(torch.int32),
                           ref.view(torch.int16) if ref.dtype == torch.bfloat16 else ref.view(torch.int32)), \
            f"noalloc {which}: not bit-identical to tcg_gemm"
        if exact:
            assert np.array_equal(got.to(torch.float64).cpu().numpy(), want)


def test_noalloc_rejects_problems_beyond_the_scratch():
    case = inputs.make_case("noalloc_big", 128, 8192, 8192, seed=181, dist="uniform")
    tcg.debug_set(force_splits=16)  # 32 tiles x 16 splits of 128 x 256 fp32 partials = 64 MiB
    dc = harness.DeviceCase(case)
    with pytest.raises(tcg.TcgError) as err:
        noalloc(case, dc, dc.D_view)
    assert err.value.code == WORKSPACE_ERROR
    assert "maximum" in tcg.last_error()
