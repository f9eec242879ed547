"""Seeded random problems through the planner's whole decision space, each
compared element by element with the oracle.

Shapes are drawn so that the plans cover every way the planner splits work
on the GPU it runs on: whole 256 x 256 pair tiles, a last wave run as
half-width units, the wave-fitting 224 / 192 / 160-wide pair tiles, one-CTA
tiles, split K (with the round-robin and the own-row-group sums), 256 x 128
pair tiles with split K (among them wide GEMMs with at most 32 rows), and
the K-serpentine order of odd waves.  Integer
operands in [-4, 4], integer C and bias, fp32 D: every result is exact, so
any element that differs from the oracle is a bug.  Layouts, operand types
(bf16, f16, e4m3, e5m2), beta and the activation are drawn with the shape.
"""
import numpy as np
import pytest
import torch

import tiled_tensor_core_persistent_gb300 as tcg
from tiled_tensor_core_persistent_gb300 import harness, inputs

from parity import oracle_for

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


def draw_cases(n, seed=2026):
    rng = np.random.default_rng(seed)
    kinds = ["pairs_many_waves", "pairs_one_wave_tail", "wide_tail", "one_cta_small", "split_long_k", "tall_narrow",
             "few_rows_long_k"]
    cases = []
    for i in range(n):
        kind = kinds[i % len(kinds)]
        if kind == "pairs_many_waves":
            M, N, K = int(rng.integers(2048, 3300)), int(rng.integers(2048, 3300)), int(rng.integers(64, 400))
        elif kind == "pairs_one_wave_tail":
            M, N, K = 2048 + int(rng.integers(-40, 40)), 2560 + int(rng.integers(-100, 300)), int(rng.integers(100, 600))
        elif kind == "wide_tail":
            M, N, K = 2048 + int(rng.integers(0, 200)), 4096 + int(rng.integers(-200, 200)), int(rng.integers(64, 300))
        elif kind == "one_cta_small":
            M, N, K = int(rng.integers(1, 700)), int(rng.integers(1, 900)), int(rng.integers(1, 700))
        elif kind == "split_long_k":
            M, N, K = int(rng.integers(1, 400)), int(rng.integers(8, 600)), int(rng.integers(1500, 5000))
        elif kind == "tall_narrow":
            M, N, K = int(rng.integers(2048, 2600)), int(rng.integers(8, 129)), int(rng.integers(1600, 4000))
        else:
            M, N, K = int(rng.integers(1, 33)), int(rng.integers(4900, 9000)), int(rng.integers(1100, 3000))
        ab = ["bf16", "bf16", "f16", "e4m3", "e5m2"][int(rng.integers(0, 5))]
        if ab in ("e4m3", "e5m2"):
            opA, opB = "row", "col"
        else:
            opA, opB = inputs.LAYOUT_COMBOS[int(rng.integers(0, 4))]
        if kind == "few_rows_long_k":
            opA = "row"
        beta = [0.0, 0.5, 1.0][int(rng.integers(0, 3))]
        act = ["none", "relu"][int(rng.integers(0, 2))]
        cases.append(dict(kind=kind, M=M, N=N, K=K, ab=ab, opA=opA, opB=opB, beta=beta, act=act, seed=5000 + i))
    return cases


CASES = draw_cases(35)


@pytest.mark.parametrize("c", CASES, ids=lambda c: f"{c['kind']}-{c['M']}x{c['N']}x{c['K']}-{c['ab']}-{c['opA']}{c['opB']}")
def test_random_problem_integer_exact(c):
    case = inputs.make_case(f"fuzz{c['seed']}", c["M"], c["N"], c["K"], seed=c["seed"], dist="int4", ab_dtype=c["ab"],
                            opA=c["opA"], opB=c["opB"], d_dtype="f32", beta=c["beta"], c_dist="int4",
                            c_dtype="f32", bias_std=2.0, bias_dtype="f32", act=c["act"])
    if case.bias is not None:
        case.bias = torch.round(case.bias)
    dc = harness.DeviceCase(case, guard_rows=1)
    dc.run()
    torch.cuda.synchronize()
    assert tcg.device_status(dc.workspace) == 0, tcg.last_error()
    got = dc.result().numpy()
    ref = oracle_for(case).full()
    bad = np.argwhere(got != ref)
    assert bad.size == 0, f"{len(bad)} elements differ, first at {tuple(bad[0])}: {got[tuple(bad[0])]} vs {ref[tuple(bad[0])]}"
    assert dc.untouched_outside()


def test_the_random_problems_cover_every_plan_feature():
    """The draw above reaches each of the planner's ways of splitting work."""
    seen = set()
    for c in CASES:
        pl = tcg.plan(c["M"], c["N"], c["K"], c["ab"], c["opA"], c["opB"])
        if pl["cluster"] == 2 and pl["BN"] == 256 and pl["splits"] == 1:
            tiles = -(-c["M"] // 256) * -(-c["N"] // 256)
            seen.add("half_tail" if pl["units"] > tiles else "whole_pairs")
        if pl["cluster"] == 2 and pl["BN"] in (160, 192, 224):
            seen.add("narrow_pairs")
        if pl["cluster"] == 2 and pl["BN"] == 128 and pl["splits"] > 1:
            seen.add("skinny_pairs")
        if pl["cluster"] == 1:
            seen.add("one_cta")
        if pl["cluster"] == 1 and pl["splits"] > 1:
            seen.add("split_k")
        if c["M"] <= 32 and pl["cluster"] == 1 and pl["splits"] > 1 and c["N"] >= 4096:
            seen.add("few_rows_split_k")
        if pl["units"] > pl["grid"] // pl["cluster"]:
            seen.add("several_waves")
    assert {"half_tail", "whole_pairs", "narrow_pairs", "skinny_pairs", "one_cta", "split_k",
            "several_waves", "few_rows_split_k"} <= seen, seen
