"""Helpers that compare the CUDA path with the oracle (tests only)."""
from __future__ import annotations

import numpy as np

import oracle
from tiled_tensor_core_persistent_gb300 import inputs

# Tolerances of the comparison |D - D_ref| <= tol * max(1, |D_ref|):
# 1e-2 for bf16 operands, 5e-2 for e4m3 operands with per-tensor scales.
TOL = {"bf16": 1e-2, "f16": 1e-2, "e4m3": 5e-2, "e5m2": 5e-2, "nvfp4": 5e-2, "mxfp4": 5e-2}

_AB = {"bf16": oracle.BF16, "f16": oracle.F16, "e4m3": oracle.E4M3, "e5m2": oracle.E5M2,
       "nvfp4": oracle.E2M1, "mxfp4": oracle.E2M1}
_VEC = {"bf16": oracle.BF16, "f32": oracle.F32}


def oracle_for(case: inputs.GemmCase) -> oracle.Problem:
    return oracle.Problem(
        case.M, case.N, case.K, inputs.raw_bits(case.A), case.lda,
        oracle.ROW if case.opA == "row" else oracle.COL,
        inputs.raw_bits(case.B), case.ldb, oracle.ROW if case.opB == "row" else oracle.COL,
        alpha=case.alpha, beta=case.beta, C=inputs.raw_bits(case.C), ldc=case.ldc,
        bias=inputs.raw_bits(case.bias), act=case.act, scale_a=case.scale_a, scale_b=case.scale_b,
        ab_dtype=_AB[case.ab_dtype], c_dtype=_VEC[case.c_dtype] if case.C is not None else None,
        bias_dtype=_VEC[case.bias_dtype] if case.bias is not None else None,
        row_scale=None if case.row_scale is None else case.row_scale.numpy(),
        col_scale=None if case.col_scale is None else case.col_scale.numpy(),
        sfa=case.sfa, sfb=case.sfb, block=case.sf_block,
        sf_format=oracle.SF_UE4M3 if case.sf_format == "ue4m3" else oracle.SF_E8M0)


def assert_within(got: np.ndarray, ref: np.ndarray, tol: float, what: str = "") -> float:
    """Element-wise |got - ref| <= tol * max(1, |ref|); returns the worst ratio."""
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape, (got.shape, ref.shape)
    assert not np.isnan(ref).any(), "oracle produced NaN"
    assert not np.isnan(got).any(), f"{what}: NaN in GPU result ({int(np.isnan(got).sum())} elements)"
    err = np.abs(got - ref)
    bound = tol * np.maximum(1.0, np.abs(ref))
    ratio = err / bound
    worst = float(ratio.max()) if ratio.size else 0.0
    if worst > 1.0:
        idx = np.unravel_index(int(np.argmax(ratio)), ratio.shape)
        bad = int((ratio > 1.0).sum())
        raise AssertionError(f"{what}: {bad}/{ratio.size} elements out of tolerance {tol}; worst at "
                             f"{idx}: got {got[idx]!r} ref {ref[idx]!r}")
    return worst


def sample_indices(extent: int, count: int, seed: int, tile: int = 128) -> np.ndarray:
    """Edges, tile boundaries and random positions in [0, extent)."""
    rng = np.random.default_rng(seed)
    picks = {0, 1, extent - 1, extent - 2}
    for b in range(tile, extent, tile * max(1, extent // (tile * 8))):
        picks.update({b - 1, b})
    picks.update(rng.integers(0, extent, size=count).tolist())
    return np.array(sorted(p for p in picks if 0 <= p < extent), dtype=np.int32)
