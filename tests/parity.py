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


def spread_indices(extent: int, count: int, seed: int, tile: int = 128) -> np.ndarray:
    """`count` distinct indices of [0, extent) (all of them when extent <= count):
    both edges, both sides of every tile boundary, the rest drawn at random."""
    if extent <= count:
        return np.arange(extent, dtype=np.int32)
    picks = {0, 1, extent - 2, extent - 1}
    for b in range(tile, extent, tile):
        picks.update({b - 1, b})
    rng = np.random.default_rng(seed)
    if len(picks) > count:
        # more boundaries than wanted: keep the edges and an even spread of the rest
        inner = sorted(picks - {0, 1, extent - 2, extent - 1})
        keep = np.linspace(0, len(inner) - 1, count - 4).round().astype(int)
        picks = {0, 1, extent - 2, extent - 1} | {inner[i] for i in keep}
    while len(picks) < count:
        picks.update(rng.integers(0, extent, size=count - len(picks)).tolist())
    return np.array(sorted(picks), dtype=np.int32)


def check_rows_cols_corners(D, prob, M, N, tol, what, nrows=256, ncols=256, corner=256, seed=0,
                            exact=False) -> float:
    """The sampled comparison for outputs too large to compute whole on the
    CPU: `nrows` full rows and `ncols` full columns of D (edges, both sides of
    every 128-row / 128-column tile boundary, random positions) and the four
    corner tiles of corner x corner elements, each element against the oracle.
    D is the device M x N view; returns the worst error ratio."""
    import torch
    rows = spread_indices(M, nrows, seed)
    cols = spread_indices(N, ncols, seed + 1)
    all_rows = np.arange(M, dtype=np.int32)
    all_cols = np.arange(N, dtype=np.int32)

    def fetch(r, c):
        rr = torch.from_numpy(r).long().to(D.device)
        cc = torch.from_numpy(c).long().to(D.device)
        return D.index_select(0, rr).index_select(1, cc).to(torch.float64).cpu().numpy()

    def compare(got, ref, label):
        if exact:
            assert np.array_equal(got, ref), f"{what} {label}: max |diff| {np.abs(got - ref).max()}"
            return 0.0
        return assert_within(got, ref, tol, f"{what} {label}")

    worst = compare(fetch(rows, all_cols), prob.select(rows, all_cols), "rows")
    worst = max(worst, compare(fetch(all_rows, cols), prob.select(all_rows, cols), "cols"))
    cm, cn = min(corner, M), min(corner, N)
    for r0 in sorted({0, M - cm}):
        for c0 in sorted({0, N - cn}):
            r = np.arange(r0, r0 + cm, dtype=np.int32)
            c = np.arange(c0, c0 + cn, dtype=np.int32)
            worst = max(worst, compare(fetch(r, c), prob.select(r, c), f"corner ({r0}, {c0})"))
    return worst
