"""GPU parity of the grouped GEMM against the oracle.

"CUTLASS" (stanleyjacob.dev), Part V (numeric-types deep dive): the experts
of a mixture-of-experts layer run as one grouped GEMM, one problem per
expert, the problems of different sizes; Part III: grouped GEMMs with
irregular shapes.  One tcg_gemm_grouped launch computes every problem; each must equal
the oracle's result for that problem alone (bit for bit on integer inputs
with fp32 D), and nothing outside any problem's D may be written.
"""
import numpy as np
import pytest
import torch

import oracle
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


# irregular shapes: ragged M / N / K, a one-row problem, an empty problem, a
# problem with K == 0 (epilogue only) and a few multi-tile ones
SHAPES = [(300, 200, 129), (1, 64, 40), (0, 128, 64), (513, 257, 300), (128, 256, 64), (77, 1000, 8),
          (256, 96, 0), (1024, 384, 200)]


def run(gcase, guard_rows=2):
    dc = harness.GroupedDeviceCase(gcase, guard_rows=guard_rows)
    dc.run()
    torch.cuda.synchronize()
    assert tcg.device_status(dc.workspace) == 0, tcg.last_error()
    return dc


def exact_case(shapes, seed, **kw):
    return inputs.make_grouped_case("grouped_int", shapes, seed=seed, dist="int4", d_dtype="f32", **kw)


@pytest.mark.parametrize("tiles", ["pair", "single"])
@pytest.mark.parametrize("with_c", [False, True])
def test_grouped_integer_exact(tiles, with_c):
    tcg.debug_set(force_cta2=1 if tiles == "pair" else 2)
    try:
        kw = dict(beta=0.5, c_dist="int4") if with_c else {}
        gcase = exact_case(SHAPES, seed=51 + with_c, act="relu", **kw)
        plan = tcg.grouped_plan([dict(M=p.M, N=p.N, K=p.K) for p in gcase.problems])
        assert plan["cluster"] == (2 if tiles == "pair" else 1)
        dc = run(gcase)
    finally:
        tcg.debug_set()
    for g, (p, part) in enumerate(zip(gcase.problems, dc.parts)):
        ref = oracle_for(p).full()
        got = part.result().numpy()
        assert np.array_equal(got, ref), f"problem {g} {p.M}x{p.N}x{p.K}: max |diff| {np.abs(got - ref).max()}"
        assert part.untouched_outside(), f"problem {g} wrote outside its D"


@pytest.mark.parametrize("tiles", ["auto", "pair"])
@pytest.mark.parametrize("combo", range(4))
def test_grouped_layouts_bf16(combo, tiles):
    opA, opB = inputs.LAYOUT_COMBOS[combo]
    gcase = inputs.make_grouped_case("grouped_layouts", [(200, 136, 72), (33, 264, 520), (640, 512, 96)],
                                     seed=60 + combo, dist="uniform", opA=opA, opB=opB, beta=0.5,
                                     c_dist="uniform", bias_std=0.1, act="gelu")
    tcg.debug_set(force_cta2=1 if tiles == "pair" else 0)
    try:
        dc = run(gcase)
    finally:
        tcg.debug_set()
    for p, part in zip(gcase.problems, dc.parts):
        assert_within(part.result().numpy(), oracle_for(p).full(), TOL["bf16"], p.name)
        assert part.untouched_outside()


@pytest.mark.parametrize("fmt", ["e4m3", "e5m2"])
def test_grouped_fp8_per_problem_scales(fmt):
    """FP8 experts, each quantised with its own per-tensor scales (folded into
    the problem's alpha)."""
    gcase = inputs.make_grouped_case("grouped_fp8", [(300, 512, 256), (64, 256, 1024), (700, 300, 128)],
                                     seed=70, dist="normal", ab_dtype=fmt, bias_std=0.1, act="relu")
    scales = {p.scale_a * p.scale_b for p in gcase.problems}
    assert len(scales) == len(gcase.problems)   # the problems really differ in scale
    dc = run(gcase)
    for p, part in zip(gcase.problems, dc.parts):
        assert_within(part.result().numpy(), oracle_for(p).full(), TOL[fmt], p.name)


def test_grouped_workspace_reuse_sees_new_problems():
    """Two different grouped calls in a row on one workspace: the second must
    use its own problems' tensor maps, not the first call's."""
    a = exact_case([(256, 256, 128), (100, 300, 64)], seed=80)
    b = exact_case([(130, 70, 96), (400, 512, 32), (5, 5, 5)], seed=81)
    da = harness.GroupedDeviceCase(a)
    db = harness.GroupedDeviceCase(b)
    ws_bytes = max(da.ws_bytes, db.ws_bytes)
    da.ws_bytes = db.ws_bytes = ws_bytes
    da.workspace = db.workspace = torch.zeros(ws_bytes, dtype=torch.uint8, device="cuda")
    for _ in range(2):
        da.run()
        db.run()
    torch.cuda.synchronize()
    assert tcg.device_status(da.workspace) == 0
    for gc, dc in ((a, da), (b, db)):
        for p, part in zip(gc.problems, dc.parts):
            assert np.array_equal(part.result().numpy(), oracle_for(p).full())


def test_grouped_errors_queue_nothing():
    gcase = exact_case([(128, 128, 64), (64, 64, 64)], seed=90)
    dc = harness.GroupedDeviceCase(gcase)
    probs = [dict(q) for q in dc.problems]
    # an operand the TMA cannot address (odd leading dimension) in the second problem
    probs[1]["lda"] = 65
    with pytest.raises(tcg.TcgError) as e:
        tcg.gemm_grouped(probs, "row", "col", 0.0, "bf16", "f32", workspace=dc.workspace,
                         workspace_bytes=dc.ws_bytes)
    assert e.value.code == 2
    # block-scaled operands are not taken
    with pytest.raises(tcg.TcgError) as e:
        tcg.gemm_grouped(dc.problems, "row", "col", 0.0, "bf16", "f32", ab_dtype="mxe4m3",
                         workspace=dc.workspace, workspace_bytes=dc.ws_bytes)
    assert e.value.code in (1, 2)
    # a workspace too small for the table
    with pytest.raises(tcg.TcgError) as e:
        tcg.gemm_grouped(dc.problems, "row", "col", 0.0, "bf16", "f32", workspace=dc.workspace,
                         workspace_bytes=256)
    assert e.value.code == 5
    torch.cuda.synchronize()
    for part in dc.parts:
        assert bool((part.D_full.float() == part.sentinel_stored).all()), "a failed call wrote D"


def test_config_grouped_moe_bf16():
    """The MoE workload: 16 experts, 32768 routed rows, 4096 x 4096 weights,
    bias, GELU, bf16 D: per expert, sampled full rows and columns against
    the oracle (every row of the smallest experts)."""
    gcase = inputs.grouped_moe()
    dc = run(gcase, guard_rows=0)
    for g, (p, part) in enumerate(zip(gcase.problems, dc.parts)):
        D = part.D_view[:, :p.N]
        prob = oracle_for(p)
        rows = sample_indices(p.M, 6, 100 + g)
        cols = sample_indices(p.N, 6, 200 + g)
        got_rows = D[torch.from_numpy(rows).long().to(D.device)].to(torch.float64).cpu().numpy()
        assert_within(got_rows, prob.select(rows, np.arange(p.N, dtype=np.int32)), TOL["bf16"], f"{p.name} rows")
        got_cols = D[:, torch.from_numpy(cols).long().to(D.device)].to(torch.float64).cpu().numpy()
        assert_within(got_cols, prob.select(np.arange(p.M, dtype=np.int32), cols), TOL["bf16"], f"{p.name} cols")


def test_grouped_many_small_problems():
    """200 problems of random small shapes (zeros included): the unit -> problem
    search over many problems, and tiles of neighbouring problems on one CTA."""
    rng = np.random.default_rng(95)
    shapes = [(int(rng.integers(0, 300)), int(rng.integers(1, 300)), int(rng.integers(0, 200)))
              for _ in range(200)]
    # a few empty ones on purpose, first and last included
    shapes[0] = (0, 64, 64)
    shapes[57] = (50, 0, 64)
    shapes[-1] = (0, 0, 0)
    for tiles in ("pair", "single"):
        tcg.debug_set(force_cta2=1 if tiles == "pair" else 2)
        try:
            gcase = exact_case(shapes, seed=96, act="relu", bias_std=None)
            dc = run(gcase, guard_rows=1)
        finally:
            tcg.debug_set()
        for g, (p, part) in enumerate(zip(gcase.problems, dc.parts)):
            if p.M == 0 or p.N == 0:
                assert part.untouched_outside(), f"empty problem {g} was written"
                continue
            assert np.array_equal(part.result().numpy(), oracle_for(p).full()), f"{tiles}: problem {g} {p.M}x{p.N}x{p.K}"
            assert part.untouched_outside(), f"{tiles}: problem {g} wrote outside its D"


def test_grouped_unaligned_c_d_and_bias_per_problem():
    """C, D and bias that the TMA cannot address are taken element-wise, per
    problem, next to problems whose C and D go through the TMA."""
    mk = lambda name, M, N, K, seed, **kw: inputs.make_case(name, M, N, K, seed=seed, dist="int4", d_dtype="f32",
                                                            beta=0.5, c_dist="int4", act="relu", **kw)
    probs = [mk("aligned", 300, 256, 128, 1),
             mk("odd_ldc", 130, 200, 64, 2, ldc=201),
             mk("odd_ldd", 257, 96, 72, 3, ldd=97),
             mk("both", 64, 40, 200, 4, ldc=41, ldd=43)]
    gcase = inputs.GroupedCase("grouped_unaligned", probs)
    for tiles in ("pair", "single"):
        tcg.debug_set(force_cta2=1 if tiles == "pair" else 2)
        try:
            dc = run(gcase, guard_rows=1)
        finally:
            tcg.debug_set()
        for p, part in zip(gcase.problems, dc.parts):
            assert np.array_equal(part.result().numpy(), oracle_for(p).full()), f"{tiles}: {p.name}"
            assert part.untouched_outside(), f"{tiles}: {p.name} wrote outside its D"
