"""GPU parity of block-scaled FP8 operands (MXE4M3 / MXE5M2) against the oracle.

"CUTLASS" (stanleyjacob.dev), Part V, data types: narrow formats in which a
few neighbouring elements share one scale, an operand handled together with
its scales.  Here: E4M3 / E5M2 elements with one E8M0 scale per
32 consecutive K of each A row and B column (the OCP Microscaling layout),
computed with the tensor cores' block-scaled MMA (tcgen05 kind::mxf8f6f4).
Integer elements with scales 2^-1..2^1 make every partial sum exact in fp32,
so those results must match the oracle bit for bit.
"""
import numpy as np
import pytest
import torch

from tiled_tensor_core_persistent_gb300 import harness, inputs
import tiled_tensor_core_persistent_gb300 as tcg

from parity import TOL, assert_within, check_rows_cols_corners, oracle_for

pytestmark = pytest.mark.gpu


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


def exact_case(M, N, K, fmt="e4m3", seed=1, **kw):
    return inputs.make_case(f"mx_int_{M}x{N}x{K}", M, N, K, seed=seed, dist="int4", ab_dtype=fmt,
                            d_dtype="f32", block_scaled=True, mx_scale_codes=(126, 128), **kw)


@pytest.mark.parametrize("shape", [(128, 128, 128), (128, 128, 32), (300, 200, 256), (257, 300, 1000),
                                   (1, 9, 7), (129, 129, 129), (640, 384, 4096)],
                         ids=lambda s: "x".join(map(str, s)))
@pytest.mark.parametrize("fmt", ["e4m3", "e5m2"])
def test_mx_integer_exact(shape, fmt):
    M, N, K = shape
    case = exact_case(M, N, K, fmt, seed=M + 2 * N + 3 * K)
    dc = run(case)
    got = dc.result().numpy()
    ref = oracle_for(case).full()
    assert np.array_equal(got, ref), f"max |diff| {np.abs(got - ref).max()}"
    assert dc.untouched_outside()


def test_mx_unit_scales_equal_plain_fp8():
    """All scale codes 127 (x1): the block-scaled GEMM equals the per-tensor one."""
    M, N, K = 256, 256, 512
    case = exact_case(M, N, K, seed=9)
    case.sfa[:] = 127
    case.sfb[:] = 127
    mx = run(case).result().numpy()
    plain = inputs.make_case("plain", M, N, K, seed=9, dist="int4", ab_dtype="e4m3", d_dtype="f32")
    plain.A, plain.B = case.A, case.B
    assert np.array_equal(mx, run(plain).result().numpy())


def test_mx_each_block_scale_reaches_its_block():
    """Scale codes that differ per (row, block) and per (column, block) over a
    wide range; D f32 against the oracle within fp32 accumulation error."""
    M, N, K = 384, 256, 1024
    case = inputs.make_case("mx_wide", M, N, K, seed=21, dist="int4", ab_dtype="e4m3", d_dtype="f32",
                            block_scaled=True, mx_scale_codes=(117, 137))
    dc = run(case)
    assert_within(dc.result().numpy(), oracle_for(case).full(), 1e-5, "wide scales")


@pytest.mark.parametrize("fmt", ["e4m3", "e5m2"])
def test_mx_quantised_normal_with_epilogue(fmt):
    """N(0,1) data quantised per OCP MX, bias + GELU + beta*C, bf16 D."""
    case = inputs.make_case(f"mx_q_{fmt}", 520, 390, 1000, seed=33, dist="normal", ab_dtype=fmt,
                            block_scaled=True, bias_std=0.1, act="gelu", beta=0.5, c_dist="uniform",
                            alpha=0.25)
    dc = run(case)
    assert_within(dc.result().numpy(), oracle_for(case).full(), TOL[fmt], case.name)
    assert dc.untouched_outside()


def test_mx_split_k_skinny():
    """Few output tiles: the planner splits K; partial sums of block-scaled products."""
    case = inputs.make_case("mx_skinny", 64, 256, 8192, seed=41, dist="int4", ab_dtype="e4m3",
                            d_dtype="f32", block_scaled=True, mx_scale_codes=(126, 128))
    plan = tcg.plan(case.M, case.N, case.K, "mxe4m3")
    assert plan["splits"] > 1 and plan["BN"] == 128 and plan["cluster"] == 1
    dc = run(case)
    assert np.array_equal(dc.result().numpy(), oracle_for(case).full())


def test_mx_requires_scales_and_fast_layout():
    case = exact_case(128, 128, 128)
    dc = harness.DeviceCase(case)
    with pytest.raises(tcg.TcgError) as e:
        tcg.gemm(128, 128, 128, 1.0, dc.A, case.lda, "row", dc.B, case.ldb, "col", 0.0, None, 0, "bf16",
                 dc.D_view, case.ldd, "f32", ab_dtype="mxe4m3", workspace=dc.workspace,
                 workspace_bytes=dc.ws_bytes)
    assert e.value.code == 1
    assert tcg.can_implement(128, 128, 128, "mxe4m3", dc.A, 128, "col", dc.B, 128, "col", 0, None, 0, "bf16",
                             dc.D_view, 128, "f32") == 2


def test_config_mxfp8_8192_bias_relu():
    """The 8192^3 MXFP8 workload (N(0,1) quantised per OCP MX, bias, ReLU, bf16 D):
    256 full rows, 256 full columns and the four 256 x 256 corner tiles
    against the oracle."""
    case = inputs.mxfp8_8192_relu()
    dc = run(case, guard_rows=0)
    check_rows_cols_corners(dc.D_view[:, :case.N], oracle_for(case), case.M, case.N, TOL["e4m3"], case.name,
                            seed=18)


@pytest.mark.parametrize("fmt", ["e4m3", "e5m2"])
@pytest.mark.parametrize("width", [192, 256])
@pytest.mark.parametrize("shape", [(512, 512, 1024), (520, 700, 333), (256, 256, 32), (300, 1000, 96)],
                         ids=lambda s: "x".join(map(str, s)))
def test_mx_pair_tiles_exact(shape, width, fmt):
    """256 x 192 and 256 x 256 tiles on CTA pairs (cta_group::2): each CTA copies
    its A rows' scales and the B scale blocks its tile's columns overlap into its
    own TMEM.  A 192-wide tile that starts half-way into a 128-column scale
    block (odd tile columns) reads its B scales from the block's third column."""
    M, N, K = shape
    tcg.debug_set(force_cta2=4 if width == 192 else 3)
    try:
        case = exact_case(M, N, K, fmt, seed=M + N + K)
        plan = tcg.plan(M, N, K, "mx" + fmt)
        assert plan["cluster"] == 2 and plan["BN"] == width
        dc = run(case)
        assert np.array_equal(dc.result().numpy(), oracle_for(case).full())
        assert dc.untouched_outside()
    finally:
        tcg.debug_set()
