"""GPU parity: the CUDA path (through the C ABI) against the CPU oracle.

Every output the oracle can compute whole in seconds on the host cores is
compared element by element: the small cases, the 512^3 and 4096^3
workloads and all twelve ragged / skinny workloads (three shapes, four A / B
layouts).  The 8192^3 workloads are compared on 256 full rows, 256 full
columns (edges, both sides of every tile boundary, random positions) and
the four 256 x 256 corner tiles, which the oracle computes one element at a
time.  Integer-valued inputs with fp32 D must match bit for bit.
"""
import os

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


def run(case, guard_rows=0):
    dc = harness.DeviceCase(case, guard_rows=guard_rows)
    dc.run()
    torch.cuda.synchronize()
    assert tcg.device_status(dc.workspace) == 0, tcg.last_error()
    return dc


def check_full(case, tol=None, exact=False, guard_rows=2):
    dc = run(case, guard_rows=guard_rows)
    got = dc.result().numpy()
    ref = oracle_for(case).full()
    if exact:
        assert np.array_equal(got, ref), f"max |diff| {np.abs(got - ref).max()}"
    else:
        assert_within(got, ref, tol if tol is not None else TOL[case.ab_dtype], case.name)
    if guard_rows:
        assert dc.untouched_outside(), "wrote outside D's M x N window"
    return dc


# ------------------------------------------------------------ exact checks

def test_single_tile_integer_exact():
    case = inputs.make_case("t128", 128, 256, 128, seed=31, dist="int4", d_dtype="f32")
    check_full(case, exact=True)


def test_gemm512_integer_bit_exact():
    check_full(inputs.square_512(integer=True), exact=True)


def test_gemm512_uniform():
    check_full(inputs.square_512(integer=False))


EDGE_SHAPES = [(1, 1, 1), (128, 256, 64), (127, 255, 63), (129, 257, 65), (128, 128, 8),
               (300, 200, 1), (64, 384, 100), (5, 300, 1000), (260, 16, 130)]


@pytest.mark.parametrize("shape", EDGE_SHAPES, ids=lambda s: "x".join(map(str, s)))
@pytest.mark.parametrize("combo", inputs.LAYOUT_COMBOS, ids=lambda c: c[0] + c[1])
def test_edge_shapes_integer_exact(shape, combo):
    M, N, K = shape
    case = inputs.make_case(f"edge{M}x{N}x{K}", M, N, K, seed=M * 7 + N * 3 + K, dist="int4",
                            opA=combo[0], opB=combo[1], d_dtype="f32")
    check_full(case, exact=True)


def test_persistent_many_tiles_integer_exact():
    """More tiles than SMs: every CTA loops, both TMEM accumulators are reused."""
    case = inputs.make_case("many", 2048, 2560, 256, seed=41, dist="int4", d_dtype="f32")
    check_full(case, exact=True)


# ---------------------------------------------------------- epilogue paths

@pytest.mark.parametrize("act", ["none", "relu", "gelu"])
@pytest.mark.parametrize("bias_dtype", ["bf16", "f32"])
def test_bias_activation(act, bias_dtype):
    case = inputs.make_case(f"bias_{act}", 300, 520, 384, seed=51, dist="uniform", bias_std=0.1,
                            bias_dtype=bias_dtype, act=act)
    check_full(case)


@pytest.mark.parametrize("c_dtype", ["bf16", "f32"])
@pytest.mark.parametrize("d_dtype", ["bf16", "f32"])
def test_beta_c(c_dtype, d_dtype):
    case = inputs.make_case("beta", 333, 290, 200, seed=61, dist="uniform", beta=0.5,
                            c_dist="uniform", c_dtype=c_dtype, d_dtype=d_dtype, alpha=1.5)
    check_full(case)


def test_beta_zero_never_reads_c():
    case = inputs.make_case("nanC", 200, 300, 128, seed=71, dist="uniform")
    dc = harness.DeviceCase(case, guard_rows=1)
    nan_c = torch.full((case.M, case.ldd), float("nan"), dtype=torch.bfloat16, device="cuda")
    tcg.gemm(case.M, case.N, case.K, 1.0, dc.A, case.lda, "row", dc.B, case.ldb, "col", 0.0, nan_c,
             case.ldd, "bf16", dc.D_view, case.ldd, case.d_dtype, workspace=dc.workspace,
             workspace_bytes=dc.ws_bytes)
    torch.cuda.synchronize()
    assert_within(dc.result().numpy(), oracle_for(case).full(), TOL["bf16"], "nanC")


def test_k_zero_is_epilogue_only():
    case = inputs.make_case("k0", 130, 70, 0, seed=81, dist="uniform", beta=2.0, c_dist="uniform",
                            bias_std=0.5, act="relu", d_dtype="f32")
    check_full(case, tol=1e-6)


def test_in_place_c_equals_d():
    case = inputs.make_case("inplace", 256, 512, 192, seed=91, dist="uniform", beta=1.0,
                            c_dist="uniform", c_dtype="f32", d_dtype="f32")
    ref = oracle_for(case).full()
    dc = harness.DeviceCase(case)
    dc.D_view.copy_(dc.C)
    tcg.gemm(case.M, case.N, case.K, case.alpha, dc.A, case.lda, "row", dc.B, case.ldb, "col", 1.0,
             dc.D_view, case.ldd, "f32", dc.D_view, case.ldd, "f32", workspace=dc.workspace,
             workspace_bytes=dc.ws_bytes)
    torch.cuda.synchronize()
    assert_within(dc.result().numpy(), ref, 1e-4, "inplace")


# -------------------------------------------------------------------- FP8

def test_fp8_integer_exact():
    case = inputs.make_case("f8int", 256, 384, 512, seed=101, dist="int4", ab_dtype="e4m3",
                            d_dtype="f32")
    assert case.scale_a == 1.0 and case.scale_b == 1.0
    check_full(case, exact=True)


def test_fp8_scaled_bias_relu_small():
    case = inputs.make_case("f8small", 384, 640, 1024, seed=111, dist="normal", ab_dtype="e4m3",
                            bias_std=0.1, act="relu")
    check_full(case)


# ------------------------------------------------- the full-size workloads

@pytest.mark.slow
def test_config_4096_beta1():
    """The whole 4096 x 4096 output against the oracle (about 15 s of oracle time)."""
    check_full(inputs.square_4096_beta(), guard_rows=1)


def check_large(case, seed=0):
    dc = run(case)
    return check_rows_cols_corners(dc.D_view[:, :case.N], oracle_for(case), case.M, case.N,
                                   TOL[case.ab_dtype], case.name, seed=seed)


@pytest.mark.slow
def test_config_8192_bias_gelu():
    check_large(inputs.square_8192_gelu(), seed=4)


@pytest.mark.slow
@pytest.mark.parametrize("shape_idx", range(3), ids=["4095x3001x1537", "16x8192x8192", "8192x128x8192"])
@pytest.mark.parametrize("combo_idx", range(4), ids=["rowrow", "rowcol", "colrow", "colcol"])
def test_config_ragged(shape_idx, combo_idx):
    """Every element of each ragged / skinny workload, with guard rows around D."""
    check_full(inputs.ragged(shape_idx, combo_idx), guard_rows=1)


@pytest.mark.slow
def test_config_fp8_8192_bias_relu():
    check_large(inputs.fp8_8192_relu(), seed=17)


# ----------------------------------------------------------------- split-K

@pytest.mark.parametrize("splits", [2, 3, 5])
def test_forced_split_k_integer_exact(splits):
    try:
        tcg.debug_set(force_splits=splits)
        case = inputs.make_case(f"split{splits}", 300, 520, 1100, seed=121 + splits, dist="int4",
                                d_dtype="f32", opA="col", opB="row")
        assert tcg.plan(case.M, case.N, case.K)["splits"] == splits
        check_full(case, exact=True)
    finally:
        tcg.debug_set()


def test_forced_split_k_epilogue_and_determinism():
    try:
        tcg.debug_set(force_splits=4)
        case = inputs.make_case("split_epi", 250, 300, 2048, seed=131, dist="uniform", beta=0.5,
                                c_dist="uniform", bias_std=0.1, act="gelu")
        dc = check_full(case)
        first = dc.D_view.clone()
        for _ in range(3):
            dc.run()
        torch.cuda.synchronize()
        assert torch.equal(first.view(torch.int16), dc.D_view.view(torch.int16)), "split-K not deterministic"
    finally:
        tcg.debug_set()


def test_skinny_shapes_fill_the_gpu():
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    for (M, N, K) in [(16, 8192, 8192), (8192, 128, 8192)]:
        assert tcg.plan(M, N, K)["grid"] * 2 >= sms // 2


# ------------------------------------------------ 2-CTA pair tiles (cta_group::2)

PAIR_SHAPES = [(256, 256, 64), (300, 520, 384), (513, 700, 129), (1024, 1536, 512), (130, 258, 70)]


@pytest.mark.parametrize("shape", PAIR_SHAPES, ids=lambda s: "x".join(map(str, s)))
@pytest.mark.parametrize("combo", inputs.LAYOUT_COMBOS, ids=lambda c: c[0] + c[1])
def test_pair_tiles_integer_exact(shape, combo):
    M, N, K = shape
    try:
        tcg.debug_set(force_cta2=1)
        assert tcg.plan(M, N, K)["cluster"] == 2
        case = inputs.make_case(f"pair{M}x{N}x{K}", M, N, K, seed=M + 5 * N + 11 * K, dist="int4",
                                opA=combo[0], opB=combo[1], d_dtype="f32")
        check_full(case, exact=True)
    finally:
        tcg.debug_set()


def test_pair_tiles_many_units_epilogue():
    try:
        tcg.debug_set(force_cta2=1)
        case = inputs.make_case("pair_epi", 2304, 2816, 640, seed=151, dist="uniform", beta=0.5,
                                c_dist="uniform", bias_std=0.1, act="gelu")
        check_full(case)
    finally:
        tcg.debug_set()


def test_pair_tiles_fp8():
    try:
        tcg.debug_set(force_cta2=1)
        case = inputs.make_case("pair_f8", 768, 1024, 1024, seed=161, dist="int4", ab_dtype="e4m3",
                                d_dtype="f32")
        check_full(case, exact=True)
    finally:
        tcg.debug_set()


def test_planner_picks_pairs_for_large_square():
    pl = tcg.plan(8192, 8192, 8192)
    # at least 384 elements of K (six 128-byte atoms) in flight per CTA
    assert pl["cluster"] == 2 and pl["grid"] % 2 == 0 and pl["stages"] * pl["BK"] >= 384


# ------------------------------------- Stream-K (TCG_SK, read when the library loads)

_STREAM_K_CHILD = r"""
import sys, numpy as np, torch
sys.path.insert(0, {tests!r})
import tiled_tensor_core_persistent_gb300 as tcg
from tiled_tensor_core_persistent_gb300 import harness, inputs
from parity import TOL, assert_within, oracle_for
tcg.lib()
M, N, K = 2048 + 17, 2560, 1024 + 40
tiles = -(-M // 256) * -(-N // 256)
pl = tcg.plan(M, N, K)
assert pl["units"] < tiles, ("no Stream-K units planned", pl)
case = inputs.make_case("sk", M, N, K, seed=191, dist="int4", d_dtype="f32", opA="col", opB="col")
dc = harness.DeviceCase(case, guard_rows=2)
dc.run(); torch.cuda.synchronize()
assert tcg.device_status(dc.workspace) == 0
first = dc.D_view.clone()
assert np.array_equal(dc.result().numpy(), oracle_for(case).full()), "not exact"
assert dc.untouched_outside()
dc.run(); torch.cuda.synchronize()
assert torch.equal(first, dc.D_view), "not deterministic"
case2 = inputs.make_case("sk_epi", 4096, 4096, 1024, seed=202, dist="uniform", beta=0.5, c_dist="uniform",
                         bias_std=0.1, act="gelu")
dc2 = harness.DeviceCase(case2)
dc2.run(); torch.cuda.synchronize()
assert tcg.device_status(dc2.workspace) == 0
assert_within(dc2.result().numpy(), oracle_for(case2).full(), TOL["bf16"], "stream-k epilogue")
print("stream-k ok", pl)
"""


@pytest.mark.parametrize("mode", [1, 2, 3])
def test_stream_k_modes_exact_deterministic_and_epilogue(mode):
    """Stream-K schedules (off by default): integer-exact and run-to-run
    identical on a ragged shape with column-major A and B, and the full
    epilogue within tolerance.  The mode is read when the library loads, so
    each runs in a child process with TCG_SK set."""
    import subprocess
    import sys
    here = os.path.dirname(os.path.abspath(__file__))
    r = subprocess.run([sys.executable, "-c", _STREAM_K_CHILD.format(tests=here)],
                       env=dict(os.environ, TCG_SK=str(mode)), capture_output=True, text=True, timeout=900,
                       cwd=os.path.dirname(here))
    assert r.returncode == 0, r.stdout[-2000:] + r.stderr[-4000:]
    assert "stream-k ok" in r.stdout


_OVERRIDE_CHILD = r"""
import sys, numpy as np, torch
sys.path.insert(0, {tests!r})
import tiled_tensor_core_persistent_gb300 as tcg
from tiled_tensor_core_persistent_gb300 import harness, inputs
from parity import oracle_for
tcg.lib()
for M, N, K, force in ((2048 + 17, 2560, 1024 + 40, 1), (700, 900, 500, 2), (1000, 128, 300, 0)):
    tcg.debug_set(force_cta2=force)
    case = inputs.make_case("ovr", M, N, K, seed=M + N + K, dist="int4", d_dtype="f32", beta=0.5, c_dist="int4",
                            act="relu")
    dc = harness.DeviceCase(case, guard_rows=2)
    dc.run(); torch.cuda.synchronize()
    assert tcg.device_status(dc.workspace) == 0
    assert np.array_equal(dc.result().numpy(), oracle_for(case).full()), (M, N, K, tcg.plan(M, N, K))
    assert dc.untouched_outside()
    tcg.debug_set()
print("overrides ok")
"""


@pytest.mark.parametrize("env", [{"TCG_KATOMS": "1"}, {"TCG_KATOMS": "2"}, {"TCG_STAGES": "2"},
                                 {"TCG_GROUP_M": "3"}, {"TCG_NARROW": "0"}],
                         ids=lambda e: ",".join(f"{k}={v}" for k, v in e.items()))
def test_planner_overrides_stay_exact(env):
    """The planner's tuning overrides (read when the library loads) select
    other pipeline shapes and rasters; every one must stay integer-exact in
    pair and one-CTA tiles.  Each runs in a child process."""
    import subprocess
    import sys
    here = os.path.dirname(os.path.abspath(__file__))
    r = subprocess.run([sys.executable, "-c", _OVERRIDE_CHILD.format(tests=here)], env=dict(os.environ, **env),
                       capture_output=True, text=True, timeout=900, cwd=os.path.dirname(here))
    assert r.returncode == 0, r.stdout[-2000:] + r.stderr[-4000:]
    assert "overrides ok" in r.stdout


def test_tail_split_epilogue_bf16():
    case = inputs.make_case("tail_epi", 2048, 2560 + 256, 1024, seed=201, dist="uniform", beta=0.5,
                            c_dist="uniform", bias_std=0.1, act="gelu")
    check_full(case)


# -------------------------------------- fp16 / e5m2 operands, channel scales

@pytest.mark.parametrize("combo", inputs.LAYOUT_COMBOS, ids=lambda c: c[0] + c[1])
@pytest.mark.parametrize("force_cta2", [1, 2], ids=["pair", "one_cta"])
def test_f16_integer_exact(combo, force_cta2):
    try:
        tcg.debug_set(force_cta2=force_cta2)
        case = inputs.make_case("f16int", 300, 520, 384, seed=211, dist="int4", ab_dtype="f16",
                                opA=combo[0], opB=combo[1], d_dtype="f32")
        check_full(case, exact=True)
    finally:
        tcg.debug_set()


def test_f16_bias_gelu():
    case = inputs.make_case("f16gelu", 640, 768, 512, seed=221, dist="normal_sqrtk", ab_dtype="f16",
                            bias_std=0.1, act="gelu", beta=0.5, c_dist="uniform")
    check_full(case)


@pytest.mark.parametrize("force_cta2", [1, 2], ids=["pair", "one_cta"])
def test_e5m2_integer_exact(force_cta2):
    try:
        tcg.debug_set(force_cta2=force_cta2)
        case = inputs.make_case("e5m2int", 512, 768, 640, seed=231, dist="int4", ab_dtype="e5m2",
                                d_dtype="f32")
        check_full(case, exact=True)
    finally:
        tcg.debug_set()


def test_e5m2_scaled_bias_relu():
    case = inputs.make_case("e5m2", 384, 640, 1024, seed=241, dist="normal", ab_dtype="e5m2",
                            bias_std=0.1, act="relu")
    check_full(case)


@pytest.mark.parametrize("ab", ["bf16", "e4m3"])
@pytest.mark.parametrize("force_cta2", [1, 2], ids=["pair", "one_cta"])
def test_channel_scales(ab, force_cta2):
    try:
        tcg.debug_set(force_cta2=force_cta2)
        case = inputs.make_case("chan", 520, 768, 512, seed=251, dist="uniform" if ab == "bf16" else "normal",
                                ab_dtype=ab, beta=0.5, c_dist="uniform", bias_std=0.1, act="gelu",
                                channel_scales=True)
        check_full(case)
    finally:
        tcg.debug_set()


def test_channel_scales_integer_exact():
    """Power-of-two channel scales keep integer inputs exact."""
    case = inputs.make_case("chanint", 256, 512, 256, seed=261, dist="int4", d_dtype="f32")
    case.row_scale = torch.tensor([2.0 ** (i % 3) for i in range(case.M)], dtype=torch.float32)
    case.col_scale = torch.tensor([0.5 ** (j % 2) for j in range(case.N)], dtype=torch.float32)
    check_full(case, exact=True)


# ----------------------------------------------- the kernel's GELU, pinned

def gelu_sweep_case():
    """A GEMM whose outputs are GELU over a dense grid of pre-activations.

    A is one-hot (A[i, i mod K] = 1), so row i of A @ B is row (i mod K) of
    B; the fp32 bias adds a fine offset per column.  The pre-activations
    B[i mod K, j] + bias[j] cover [-10, 10] in steps of about 3e-4; the last
    16 columns hold special values in the bias over a zero B column: +-0,
    +-tiny (including an fp32 subnormal), moderate and huge magnitudes."""
    M, N, K = 256, 1040, 64
    specials = [0.0, -0.0, 1e-30, -1e-30, 1e-40, -1e-40, 3.0, -3.0, 5.5, -5.5, 20.0, -20.0,
                1e4, -1e4, 3e38, -3e38]
    nd = N - len(specials)
    grid = torch.linspace(-10.0, 10.0, K * nd, dtype=torch.float32).view(K, nd)
    Bl = torch.zeros(K, N, dtype=torch.float32)
    Bl[:, :nd] = grid.to(torch.bfloat16).to(torch.float32)
    gen = torch.Generator().manual_seed(301)
    bias = torch.zeros(N, dtype=torch.float32)
    bias[:nd] = (torch.rand(nd, generator=gen) * 2.0 - 1.0) * 0.01
    bias[nd:] = torch.tensor(specials, dtype=torch.float32)
    Al = torch.zeros(M, K, dtype=torch.float32)
    Al[torch.arange(M), torch.arange(M) % K] = 1.0
    A, lda = inputs._store(Al, "row", "bf16")
    B, ldb = inputs._store(Bl, "col", "bf16")
    return inputs.GemmCase("gelu_sweep", M, N, K, "row", "col", "bf16", "f32", A, lda, B, ldb,
                           bias=bias, bias_dtype="f32", act="gelu", ldd=N)


@pytest.mark.parametrize("force_cta2", [2, 1], ids=["one_cta", "pair"])
def test_gelu_error_bound(force_cta2):
    """The epilogue's GELU (Abramowitz & Stegun 7.1.26 for erf, with the
    hardware's approximate reciprocal and 2^x) against the oracle's exact
    0.5 x (1 + erf(x / sqrt 2)) in double, with fp32 D.  Bound per element:
    |D - D_ref| <= 1e-6 * max(1, |x|).  From 7.1.26's |error in erf| <=
    1.5e-7, about 2.4e-7 more from the approximate 2^x (relative, on
    exp(-z^2) <= 1) and about 3e-7 from the approximate reciprocal and the fp32
    polynomial, the error in erf stays under 1e-6; GELU multiplies it by
    |x| / 2 and the pre-activation and result roundings add about 1.2e-7 |x|.
    A wrong sign in the odd extension or a wrong coefficient fails it by
    orders of magnitude."""
    try:
        tcg.debug_set(force_cta2=force_cta2)
        case = gelu_sweep_case()
        dc = run(case, guard_rows=1)
        got = dc.result().numpy()
        ref = oracle_for(case).full()
        x = oracle_for(inputs.GemmCase("pre", case.M, case.N, case.K, "row", "col", "bf16", "f32", case.A,
                                       case.lda, case.B, case.ldb, bias=case.bias, bias_dtype="f32",
                                       act="none", ldd=case.N)).full()
        assert np.isfinite(got).all()
        err = np.abs(got - ref)
        bound = 1e-6 * np.maximum(1.0, np.abs(x))
        worst = float((err / bound).max())
        assert worst <= 1.0, f"GELU error {worst:.3f} x the bound at x = {x.flat[int(np.argmax(err / bound))]!r}"
        assert dc.untouched_outside()
        # sanity of the sweep itself: both signs, the whole range, the specials
        assert x.min() <= -9.99 and x.max() >= 9.99 and (np.abs(x) < 1e-3).any()
        assert got[0, -1] == 0.0 and got[0, -2] == np.float32(3e38)
    finally:
        tcg.debug_set()


# --------------------- split-K pieces summed by the finishing CTA (both paths)

@pytest.mark.parametrize("combo", inputs.LAYOUT_COMBOS, ids=lambda c: c[0] + c[1])
def test_skinny_pair_split_k_integer_exact(combo):
    """A tall, narrow, long-K problem runs on 256 x 128 pair tiles with split
    K; the finishing CTA of each tile takes its own piece from TMEM and the
    others from global memory, in piece order.  Integer inputs: exact, and
    run-to-run identical."""
    M, N, K = 2000, 120, 3000
    pl = tcg.plan(M, N, K, "bf16", combo[0], combo[1])
    assert pl["cluster"] == 2 and pl["BN"] == 128 and pl["splits"] > 1, pl
    case = inputs.make_case("skinny_pair", M, N, K, seed=401, dist="int4", opA=combo[0], opB=combo[1],
                            d_dtype="f32", beta=0.5, c_dist="int4", c_dtype="f32", bias_std=1.0,
                            bias_dtype="f32", act="relu")
    case.bias = torch.round(case.bias)
    dc = check_full(case, exact=True)
    first = dc.D_view.clone()
    dc.run()
    torch.cuda.synchronize()
    assert torch.equal(first, dc.D_view)


def test_split_k_own_quadrant_fixup_integer_exact():
    """One-CTA split-K tiles whose four row groups all hold rows (M a multiple
    of 128 plus a ragged last tile): the finishing CTA adds its own piece
    from TMEM.  Exact on integer inputs, in every split count."""
    for splits in (2, 3, 4):
        try:
            tcg.debug_set(force_splits=splits)
            case = inputs.make_case(f"ownq{splits}", 300, 384, 2048, seed=410 + splits, dist="int4",
                                    d_dtype="f32")
            assert tcg.plan(case.M, case.N, case.K)["splits"] == splits
            check_full(case, exact=True)
        finally:
            tcg.debug_set()


# ------------- GEMMs with few rows: the transposed product D^T = B^T A^T
# (taken on request only: measured no faster than the plain plan, whose
# skinny problems are all bound by B's bytes; the test knob force_cta2 = 5
# asks for it)

SWAP_SHAPES = [(1, 256, 64), (7, 300, 200), (16, 1000, 1000), (31, 520, 4096), (32, 2048, 64), (33, 384, 777),
               (48, 8192, 1024), (64, 700, 2048)]


@pytest.fixture
def transposed():
    tcg.debug_set(force_cta2=5)
    yield
    tcg.debug_set()


@pytest.mark.parametrize("shape", SWAP_SHAPES, ids=lambda s: "x".join(map(str, s)))
@pytest.mark.parametrize("opB", ["col", "row"])
def test_few_rows_transposed_product_integer_exact(shape, opB, transposed):
    """At most 64 rows and a row-major A: the transposed product (the
    kernel's tiles run over D's columns; the epilogue writes each tile back
    into row-major D and reads C the same way, bias per column).  Integer
    inputs with fp32 D, beta * C, an integer bias and ReLU: exact, with guard
    rows around D."""
    M, N, K = shape
    pl = tcg.plan(M, N, K, "bf16", "row", opB)
    assert pl["swap"] == 1 and pl["BN"] == (32 if M <= 32 else 64), pl
    case = inputs.make_case(f"swap{M}x{N}x{K}", M, N, K, seed=M * 31 + N + K, dist="int4", opB=opB,
                            d_dtype="f32", beta=0.5, c_dist="int4", c_dtype="f32", bias_std=2.0,
                            bias_dtype="f32", act="relu")
    case.bias = torch.round(case.bias)
    check_full(case, exact=True)


def test_few_rows_transposed_product_bf16_epilogue_and_split_k(transposed):
    """The transposed product with long K (split into pieces summed in a fixed
    order), bf16 C and D, bias and GELU, within the bf16 tolerance and
    run-to-run identical."""
    case = inputs.make_case("swap_epi", 16, 3000, 6144, seed=421, dist="uniform", beta=0.5, c_dist="uniform",
                            bias_std=0.1, act="gelu")
    pl = tcg.plan(case.M, case.N, case.K)
    assert pl["swap"] == 1 and pl["splits"] > 1, pl
    dc = check_full(case)
    first = dc.D_view.clone()
    dc.run()
    torch.cuda.synchronize()
    assert torch.equal(first.view(torch.int16), dc.D_view.view(torch.int16))


def test_few_rows_transposed_product_fp8_and_scales_exact(transposed):
    """e4m3 operands and power-of-two row / column scales (swapped into the
    transposed frame by the host): exact on integer inputs."""
    case = inputs.make_case("swap_f8", 24, 640, 512, seed=431, dist="int4", ab_dtype="e4m3", d_dtype="f32")
    case.row_scale = torch.tensor([2.0 ** (i % 3) for i in range(case.M)], dtype=torch.float32)
    case.col_scale = torch.tensor([0.5 ** (j % 2) for j in range(case.N)], dtype=torch.float32)
    assert tcg.plan(case.M, case.N, case.K, "e4m3")["swap"] == 1
    check_full(case, exact=True)


def test_few_rows_default_and_column_major_a_keep_the_plain_plan():
    assert tcg.plan(16, 8192, 8192)["swap"] == 0
    tcg.debug_set(force_cta2=5)
    try:
        case = inputs.make_case("noswap", 16, 640, 512, seed=441, dist="int4", opA="col", d_dtype="f32")
        assert tcg.plan(case.M, case.N, case.K, "bf16", "col", "col")["swap"] == 0
        check_full(case, exact=True)
    finally:
        tcg.debug_set()
