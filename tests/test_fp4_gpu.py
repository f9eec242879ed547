"""GPU parity of the block-scaled four-bit formats against the oracle.

"CUTLASS" (stanleyjacob.dev), Part V: the latest tensor cores take
quantisation down to four-bit formats whose neighbouring elements share one
scale per small block.  NVFP4: FP4 E2M1 elements, one unsigned E4M3
scale per 16 consecutive K; MXFP4: one E8M0 scale per 32 (tcgen05
kind::mxf4nvf4 with 4 or 2 scales per MMA).  Element codes and scale codes
drawn from small sets make every product and partial sum exact in fp32, so
those results must equal the oracle bit for bit.
"""
import numpy as np
import pytest
import torch

from tiled_tensor_core_persistent_gb300 import harness, inputs
import tiled_tensor_core_persistent_gb300 as tcg

from parity import TOL, assert_within, check_rows_cols_corners, oracle_for

pytestmark = pytest.mark.gpu

NV_SCALES = [0x30, 0x34, 0x38, 0x3C, 0x40]   # 0.5, 0.75, 1, 1.5, 2 as unsigned E4M3
MX_SCALES = [126, 127, 128]                  # 0.5, 1, 2 as E8M0


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    from tiled_tensor_core_persistent_gb300 import _build
    _build.build()
    tcg.debug_set()
    yield
    tcg.debug_set()


def run(case, guard_rows=2):
    dc = harness.DeviceCase(case, guard_rows=guard_rows)
    dc.run()
    torch.cuda.synchronize()
    assert tcg.device_status(dc.workspace) == 0, tcg.last_error()
    return dc


def exact_case(M, N, K, fmt, seed):
    return inputs.make_fp4_case(f"{fmt}_{M}x{N}x{K}", M, N, K, seed=seed, fmt=fmt, dist="codes",
                                code_range=list(range(16)),
                                scale_codes=NV_SCALES if fmt == "nvfp4" else MX_SCALES, d_dtype="f32")


@pytest.mark.parametrize("shape", [(128, 128, 256), (128, 128, 64), (300, 200, 512), (257, 300, 1000),
                                   (1, 9, 32), (129, 129, 258), (640, 384, 4096)],
                         ids=lambda s: "x".join(map(str, s)))
@pytest.mark.parametrize("fmt", ["nvfp4", "mxfp4"])
def test_fp4_exact(shape, fmt):
    M, N, K = shape
    case = exact_case(M, N, K, fmt, seed=M + 5 * N + 7 * K)
    dc = run(case)
    got = dc.result().numpy()
    ref = oracle_for(case).full()
    assert np.array_equal(got, ref), f"max |diff| {np.abs(got - ref).max()}"
    assert dc.untouched_outside()


@pytest.mark.parametrize("fmt", ["nvfp4", "mxfp4"])
def test_fp4_quantised_normal_with_epilogue(fmt):
    case = inputs.make_fp4_case(f"{fmt}_q", 520, 390, 1024, seed=61, fmt=fmt, bias_std=0.1, act="gelu",
                                beta=0.5, alpha=0.5)
    dc = run(case)
    assert_within(dc.result().numpy(), oracle_for(case).full(), TOL[fmt], case.name)
    assert dc.untouched_outside()


def test_fp4_split_k():
    case = exact_case(64, 256, 8192, "nvfp4", seed=71)
    plan = tcg.plan(case.M, case.N, case.K, "nvfp4")
    assert plan["splits"] > 1 and plan["BN"] == 128
    assert np.array_equal(run(case).result().numpy(), oracle_for(case).full())


def test_fp4_layout_rules():
    case = exact_case(128, 128, 256, "nvfp4", seed=3)
    dc = harness.DeviceCase(case)
    args = (128, 128, 256, "nvfp4", dc.A, 256, "row", dc.B, 256, "col", 0, None, 0, "bf16", dc.D_view, 128, "f32")
    assert tcg.can_implement(*args) == 0
    assert tcg.can_implement(128, 128, 255, "nvfp4", dc.A, 256, "row", dc.B, 256, "col", 0, None, 0, "bf16",
                             dc.D_view, 128, "f32") == 2      # odd K
    assert tcg.can_implement(128, 128, 256, "nvfp4", dc.A, 272, "row", dc.B, 256, "col", 0, None, 0, "bf16",
                             dc.D_view, 128, "f32") == 2      # 136-byte rows: not a TMA pitch


def test_config_nvfp4_8192_bias_relu():
    """The 8192^3 NVFP4 workload: 256 full rows, 256 full columns and the four
    256 x 256 corner tiles against the oracle."""
    case = inputs.nvfp4_8192_relu()
    dc = run(case, guard_rows=0)
    check_rows_cols_corners(dc.D_view[:, :case.N], oracle_for(case), case.M, case.N, TOL["nvfp4"], case.name,
                            seed=19)


@pytest.mark.parametrize("fmt", ["nvfp4", "mxfp4"])
@pytest.mark.parametrize("width", [192, 256])
@pytest.mark.parametrize("shape", [(512, 512, 1024), (520, 700, 334), (256, 256, 64), (300, 1000, 128)],
                         ids=lambda s: "x".join(map(str, s)))
def test_fp4_pair_tiles_exact(shape, width, fmt):
    """Pair tiles with scale blocks by TMA: NVFP4 always 256 x 256 with one
    accumulator, MXFP4 256 x 256 (one accumulator) or 256 x 192 (two)."""
    M, N, K = shape
    if fmt == "nvfp4" and width == 192:
        pytest.skip("NVFP4 pair tiles are 256 wide")
    tcg.debug_set(force_cta2=4 if width == 192 else 3)
    try:
        case = exact_case(M, N, K, fmt, seed=M + 3 * N + K)
        plan = tcg.plan(M, N, K, fmt)
        assert plan["cluster"] == 2 and plan["BN"] == width
        dc = run(case)
        assert np.array_equal(dc.result().numpy(), oracle_for(case).full())
        assert dc.untouched_outside()
    finally:
        tcg.debug_set()
