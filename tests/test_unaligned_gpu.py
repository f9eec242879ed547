"""GPU parity of the slow path for matrices the TMA cannot address.

"CUTLASS" (stanleyjacob.dev), Part II, on alignment: pointers and leading
dimensions are normally expected on 8- or 16-element boundaries, and a tensor
that is not is either taken by a slower path or rejected.  Here
A and B with an unaligned base or row pitch are packed into the workspace
first, and C, D and bias with one are read and written element-wise by the
epilogue.  Every result is compared with the oracle, which reads the same
storage with the same leading dimensions.
"""
import numpy as np
import pytest
import torch

from tiled_tensor_core_persistent_gb300 import harness, inputs
import tiled_tensor_core_persistent_gb300 as tcg

from parity import TOL, assert_within, oracle_for, sample_indices

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


def tight(M, N, K, opA, opB, pad=0):
    """Leading dimensions equal to the contiguous extent (+ pad elements)."""
    lda = (K if opA == "row" else M) + pad
    ldb = (N if opB == "row" else K) + pad
    return dict(lda=lda, ldb=ldb, ldd=N + pad)


def run(case, offsets=None, guard_rows=2):
    dc = harness.DeviceCase(case, guard_rows=guard_rows, offsets=offsets)
    dc.run()
    torch.cuda.synchronize()
    assert tcg.device_status(dc.workspace) == 0, tcg.last_error()
    return dc


@pytest.mark.parametrize("combo", inputs.LAYOUT_COMBOS, ids=lambda c: c[0] + c[1])
@pytest.mark.parametrize("shape", [(300, 200, 129), (129, 257, 1001), (1, 9, 7), (260, 136, 64)],
                         ids=lambda s: "x".join(map(str, s)))
def test_tight_leading_dimensions_integer_exact(shape, combo):
    M, N, K = shape
    ld = tight(M, N, K, *combo)
    case = inputs.make_case(f"tight{M}x{N}x{K}", M, N, K, seed=M + 3 * N + 7 * K, dist="int4",
                            opA=combo[0], opB=combo[1], d_dtype="f32", **ld)
    dc = run(case)
    assert tcg.workspace_size_for(M, N, K, "bf16", dc.A, case.lda, case.opA, dc.B, case.ldb, case.opB) >= \
        tcg.workspace_size(M, N, K)
    got = dc.result().numpy()
    ref = oracle_for(case).full()
    assert np.array_equal(got, ref), f"max |diff| {np.abs(got - ref).max()}"
    assert dc.untouched_outside()


@pytest.mark.parametrize("which", ["A", "B", "C", "D", "bias", "all"])
def test_unaligned_pointers(which):
    """Each buffer one element past a 16-byte boundary (ld aligned otherwise)."""
    offsets = {"A": 1, "B": 1, "C": 1, "D": 1, "bias": 1} if which == "all" else {which: 1}
    case = inputs.make_case("offs", 333, 290, 200, seed=17, dist="uniform", beta=0.5, c_dist="uniform",
                            bias_std=0.1, act="gelu", alpha=1.25)
    dc = run(case, offsets=offsets)
    assert_within(dc.result().numpy(), oracle_for(case).full(), TOL["bf16"], "offsets " + which)
    assert dc.untouched_outside()


@pytest.mark.parametrize("d_dtype", ["bf16", "f32"])
@pytest.mark.parametrize("c_dtype", ["bf16", "f32"])
def test_unaligned_c_and_d_pitch(c_dtype, d_dtype):
    M, N, K = 257, 301, 320
    case = inputs.make_case("cdpitch", M, N, K, seed=23, dist="uniform", beta=0.75, c_dist="uniform",
                            c_dtype=c_dtype, d_dtype=d_dtype, ldc=N + 1, ldd=N + 3, bias_std=0.1,
                            bias_dtype="f32", act="relu")
    dc = run(case, offsets={"C": 1, "D": 1, "bias": 1})
    assert_within(dc.result().numpy(), oracle_for(case).full(), TOL["bf16"], "C/D pitch")
    assert dc.untouched_outside()


def test_in_place_with_unaligned_pitch():
    """D == C with ldc = ldd not a multiple of 16 bytes: every C element is read before it is overwritten."""
    M, N, K = 256, 333, 192
    case = inputs.make_case("inplace_odd", M, N, K, seed=29, dist="uniform", beta=1.0, c_dist="uniform",
                            ldc=N, ldd=N)
    ref = oracle_for(case).full()
    dc = harness.DeviceCase(case)
    dc.D_view.copy_(dc.C)
    tcg.gemm(M, N, K, case.alpha, dc.A, case.lda, "row", dc.B, case.ldb, "col", 1.0, dc.D_view, case.ldd,
             "bf16", dc.D_view, case.ldd, "bf16", workspace=dc.workspace, workspace_bytes=dc.ws_bytes)
    torch.cuda.synchronize()
    assert_within(dc.result().numpy(), ref, TOL["bf16"], "inplace odd pitch")


@pytest.mark.parametrize("ab", ["e4m3", "e5m2", "f16"])
def test_other_operand_types_with_odd_ld(ab):
    M, N, K = 300, 200, 1537
    opB = "col"
    case = inputs.make_case(f"odd_{ab}", M, N, K, seed=37, dist="int4", ab_dtype=ab, d_dtype="f32",
                            lda=K, ldb=K, ldd=N)
    dc = run(case, offsets={"A": 1} if ab != "f16" else {"A": 1, "B": 3})
    got = dc.result().numpy()
    ref = oracle_for(case).full()
    assert np.array_equal(got, ref), f"max |diff| {np.abs(got - ref).max()}"


def test_workspace_too_small_for_the_packed_copy_is_refused():
    case = inputs.make_case("small_ws", 300, 200, 129, seed=41, dist="int4", d_dtype="f32", lda=129)
    dc = harness.DeviceCase(case)
    with pytest.raises(tcg.TcgError) as e:
        tcg.gemm(case.M, case.N, case.K, 1.0, dc.A, case.lda, "row", dc.B, case.ldb, "col", 0.0, None, 0, "bf16",
                 dc.D_view, case.ldd, "f32", workspace=dc.workspace,
                 workspace_bytes=tcg.workspace_size(case.M, case.N, case.K))
    assert e.value.code == 5


@pytest.mark.parametrize("combo_idx", range(4))
def test_config_ragged_tight(combo_idx):
    """The ragged 4095 x 3001 x 1537 workload with tight leading dimensions
    (lda, ldb, ldc, ldd = the contiguous extents, all odd): sampled full rows
    and columns against the oracle."""
    case = inputs.ragged_tight(combo_idx)
    M, N = case.M, case.N
    dc = run(case, guard_rows=0)
    D = dc.D_view[:, :N]
    prob = oracle_for(case)
    rows = sample_indices(M, 40, combo_idx)
    cols = sample_indices(N, 40, combo_idx + 1)
    got_rows = D[torch.from_numpy(rows).long().to(D.device)].to(torch.float64).cpu().numpy()
    assert_within(got_rows, prob.select(rows, np.arange(N, dtype=np.int32)), TOL["bf16"], case.name + " rows")
    got_cols = D[:, torch.from_numpy(cols).long().to(D.device)].to(torch.float64).cpu().numpy()
    assert_within(got_cols, prob.select(np.arange(M, dtype=np.int32), cols), TOL["bf16"], case.name + " cols")


@pytest.mark.parametrize("splits", [2, 4])
def test_split_k_with_unaligned_c_and_d(splits):
    """Split K with C and D rows off the 16-byte grid: the pieces' sums are
    finished by all four epilogue warps, C read element-wise, D stored without
    the TMA."""
    tcg.debug_set(force_splits=splits)
    try:
        case = inputs.make_case(f"split_odd{splits}", 200, 301, 1024, seed=140 + splits, dist="uniform",
                                beta=0.5, c_dist="uniform", ldc=301, ldd=303, bias_std=0.1, act="relu")
        dc = run(case, offsets={"C": 1})
        assert_within(dc.result().numpy(), oracle_for(case).full(), TOL["bf16"], case.name)
        assert dc.untouched_outside()
    finally:
        tcg.debug_set()


def test_split_k_few_rows_with_c():
    """16 rows: one live row group, its split sums spread over the four warps."""
    tcg.debug_set(force_splits=3)
    try:
        case = inputs.make_case("split_m16", 16, 520, 1536, seed=151, dist="int4", beta=1.0, c_dist="int4",
                                c_dtype="f32", d_dtype="f32")
        assert tcg.plan(case.M, case.N, case.K)["swap"] == 0
        dc = run(case)
        assert np.array_equal(dc.result().numpy(), oracle_for(case).full())
        assert dc.untouched_outside()
    finally:
        tcg.debug_set()
