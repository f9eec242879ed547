"""Pins for the CPU oracle (no GPU).

Each test ties the oracle to something other than its own formula: exact
rational brute force, library routines on the decoded values (numpy matmul,
torch's dtype conversions), closed forms (identity, permutation, rank-1),
textbook constants (the normal CDF behind exact GELU) and invariants (layout
transposition, per-tensor scale folding, the 2*M*N*K operation count).  A
dropped term, a wrong sign or index, or a transposed operand in the oracle
fails at least one of them.
"""
import json
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle
from tiled_tensor_core_persistent_gb300 import inputs

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def bf16_bits(x: np.ndarray) -> np.ndarray:
    return inputs.raw_bits(torch.from_numpy(np.asarray(x, dtype=np.float32)).to(torch.bfloat16))


def bf16_values(bits: np.ndarray) -> np.ndarray:
    """Decode through torch (an implementation independent of the oracle's)."""
    t = torch.from_numpy(bits.view(np.int16).copy()).view(torch.bfloat16)
    return t.to(torch.float64).numpy()


def store(logical: np.ndarray, layout: str) -> tuple:
    """Row-major or column-major storage of a logical matrix (ld = inner extent)."""
    if layout == "row":
        return np.ascontiguousarray(logical), logical.shape[1]
    return np.ascontiguousarray(logical.T), logical.shape[0]


def op(layout):
    return oracle.ROW if layout == "row" else oracle.COL


# ---------------------------------------------------------------- decoders

def test_bf16_decoder_exhaustive_against_torch():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ours = oracle.decode_bf16(bits)
    ref = bf16_values(bits)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(ours), nan)
    assert np.array_equal(ours[~nan], ref[~nan])
    # signed zeros keep their sign
    assert np.array_equal(np.signbit(ours[~nan]), np.signbit(ref[~nan]))


def test_e4m3_decoder_exhaustive_against_torch():
    bits = np.arange(256, dtype=np.uint16).astype(np.uint8)
    ours = oracle.decode_e4m3(bits)
    ref = torch.from_numpy(bits.copy()).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    nan = np.isnan(ref)
    assert nan.sum() == 2  # 0x7F and 0xFF only
    assert np.array_equal(np.isnan(ours), nan)
    assert np.array_equal(ours[~nan], ref[~nan])
    assert np.nanmax(ours) == 448.0 and np.nanmin(ours) == -448.0


# ------------------------------------------------------ brute force (exact)

@pytest.mark.parametrize("M,N,K", [(1, 1, 1), (2, 3, 1), (3, 2, 4), (4, 4, 4), (7, 5, 3), (5, 7, 6)])
@pytest.mark.parametrize("layouts", [("row", "col"), ("col", "row"), ("row", "row"), ("col", "col")])
def test_tiny_shapes_exact_rational(M, N, K, layouts):
    """Every element against exact rational arithmetic on torch-decoded values."""
    rng = np.random.default_rng(M * 100 + N * 10 + K)
    a_bits = bf16_bits(rng.uniform(-2, 2, (M, K)))
    b_bits = bf16_bits(rng.uniform(-2, 2, (K, N)))
    c_bits = bf16_bits(rng.uniform(-2, 2, (M, N)))
    bias_bits = bf16_bits(rng.uniform(-1, 1, (N,)))
    a, b = bf16_values(a_bits), bf16_values(b_bits)
    c, bias = bf16_values(c_bits), bf16_values(bias_bits)
    alpha, beta = 0.75, -1.25  # exactly representable
    As, lda = store(a_bits, layouts[0])
    Bs, ldb = store(b_bits, layouts[1])
    got = oracle.Problem(M, N, K, As, lda, op(layouts[0]), Bs, ldb, op(layouts[1]),
                         alpha=alpha, beta=beta, C=c_bits, ldc=N, bias=bias_bits).full(1)
    for i in range(M):
        for j in range(N):
            s = Fraction(0)
            for k in range(K):
                s += Fraction(a[i, k]) * Fraction(b[k, j])
            ref = Fraction(alpha) * s + Fraction(beta) * Fraction(c[i, j]) + Fraction(bias[j])
            # K <= 6 products of bf16 values: the fp64 sum is exact here
            assert got[i, j] == float(ref), (i, j)


# ------------------------------------------------- library routine (numpy)

@pytest.mark.parametrize("layouts", [("row", "col"), ("col", "row"), ("row", "row"), ("col", "col")])
def test_integer_inputs_equal_numpy_matmul(layouts):
    """Integer-valued bf16 inputs: every partial sum is exact, so the oracle
    equals numpy's float64 matmul bit for bit in any summation order."""
    M, N, K = 37, 29, 513
    rng = np.random.default_rng(7)
    a = rng.integers(-4, 5, (M, K)).astype(np.float32)
    b = rng.integers(-4, 5, (K, N)).astype(np.float32)
    As, lda = store(bf16_bits(a), layouts[0])
    Bs, ldb = store(bf16_bits(b), layouts[1])
    got = oracle.Problem(M, N, K, As, lda, op(layouts[0]), Bs, ldb, op(layouts[1])).full()
    assert np.array_equal(got, a.astype(np.float64) @ b.astype(np.float64))


def test_random_bf16_close_to_numpy_matmul():
    M, N, K = 64, 48, 300
    rng = np.random.default_rng(11)
    a_bits = bf16_bits(rng.standard_normal((M, K)))
    b_bits = bf16_bits(rng.standard_normal((K, N)))
    got = oracle.Problem(M, N, K, a_bits, K, oracle.ROW, np.ascontiguousarray(b_bits.T), K,
                         oracle.COL).full()
    ref = bf16_values(a_bits) @ bf16_values(b_bits)
    np.testing.assert_allclose(got, ref, rtol=1e-12, atol=1e-12)


def test_padded_leading_dimensions_ignore_padding():
    """ld larger than the extent: padding (NaN) is never read."""
    M, N, K = 9, 11, 13
    rng = np.random.default_rng(3)
    a = rng.integers(-3, 4, (M, K)).astype(np.float32)
    b = rng.integers(-3, 4, (K, N)).astype(np.float32)
    lda, ldb = 24, 16
    As = np.full((M, lda), np.nan, np.float32); As[:, :K] = a
    Bs = np.full((N, ldb), np.nan, np.float32); Bs[:, :K] = b.T
    got = oracle.Problem(M, N, K, bf16_bits(As), lda, oracle.ROW, bf16_bits(Bs), ldb,
                         oracle.COL).full()
    assert np.array_equal(got, a.astype(np.float64) @ b.astype(np.float64))


# ------------------------------------------------------------ closed forms

def test_identity_and_permutation():
    n, N = 16, 10
    rng = np.random.default_rng(5)
    b_bits = bf16_bits(rng.uniform(-8, 8, (n, N)))
    b = bf16_values(b_bits)
    eye = bf16_bits(np.eye(n))
    got = oracle.Problem(n, N, n, eye, n, oracle.ROW, b_bits, N, oracle.ROW).full()
    assert np.array_equal(got, b)
    perm = rng.permutation(n)
    P = np.zeros((n, n), np.float32)
    P[np.arange(n), perm] = 1.0
    got = oracle.Problem(n, N, n, bf16_bits(P), n, oracle.ROW, b_bits, N, oracle.ROW).full()
    assert np.array_equal(got, b[perm])


def test_rank_one_closed_form():
    """(u v^T)(w x^T) = (v . w) u x^T, with small integers so all is exact."""
    M, K, N = 12, 20, 9
    rng = np.random.default_rng(9)
    u = rng.integers(-3, 4, M).astype(np.float64)
    v = rng.integers(-3, 4, K).astype(np.float64)
    w = rng.integers(-3, 4, K).astype(np.float64)
    x = rng.integers(-3, 4, N).astype(np.float64)
    A = np.outer(u, v)
    B = np.outer(w, x)
    got = oracle.Problem(M, N, K, bf16_bits(A), K, oracle.ROW,
                         bf16_bits(np.ascontiguousarray(B.T)), K, oracle.COL).full()
    assert np.array_equal(got, float(v @ w) * np.outer(u, x))


def test_operation_count_is_2mnk():
    M, N, K = 5, 6, 7
    a = bf16_bits(np.ones((M, K)))
    b = bf16_bits(np.ones((N, K)))
    out, n_mul, n_add = oracle.Problem(M, N, K, a, K, oracle.ROW, b, K, oracle.COL).count_ops()
    assert n_mul + n_add == 2 * M * N * K
    assert n_mul == M * N * K
    assert np.all(out == K)


# ------------------------------------------------------------- epilogue

def _small_problem(act="none", alpha=1.0, beta=0.0, with_c=False, with_bias=False, c_nan=False):
    M, N, K = 8, 12, 16
    rng = np.random.default_rng(21)
    a_bits = bf16_bits(rng.uniform(-1, 1, (M, K)))
    b_bits = bf16_bits(rng.uniform(-1, 1, (N, K)))
    c = rng.uniform(-1, 1, (M, N))
    if c_nan:
        c[:] = np.nan
    c_bits = bf16_bits(c) if with_c else None
    bias_bits = bf16_bits(rng.uniform(-1, 1, N)) if with_bias else None
    p = oracle.Problem(M, N, K, a_bits, K, oracle.ROW, b_bits, K, oracle.COL, alpha=alpha,
                       beta=beta, C=c_bits, ldc=N, bias=bias_bits, act=act)
    ref_ab = bf16_values(a_bits) @ bf16_values(b_bits).T
    return p, ref_ab, (bf16_values(c_bits) if with_c else None), \
        (bf16_values(bias_bits) if with_bias else None)


def test_alpha_zero_leaves_beta_c_plus_bias():
    p, _, c, bias = _small_problem(alpha=0.0, beta=0.5, with_c=True, with_bias=True)
    assert np.array_equal(p.full(), 0.5 * c + bias[None, :])


def test_beta_zero_never_reads_c():
    p, ref_ab, _, _ = _small_problem(beta=0.0, with_c=True, c_nan=True)
    got = p.full()
    assert not np.isnan(got).any()
    np.testing.assert_allclose(got, ref_ab, rtol=1e-13, atol=1e-13)


def test_relu_kills_negatives_and_keeps_positives():
    p, ref_ab, _, bias = _small_problem(act="relu", with_bias=True)
    pre = ref_ab + bias[None, :]
    got = p.full()
    assert (pre < 0).any() and (pre > 0).any()
    assert np.all(got[pre < 0] == 0.0)
    np.testing.assert_allclose(got[pre > 0], pre[pre > 0], rtol=1e-13, atol=1e-13)


def test_gelu_textbook_values():
    with open(os.path.join(GOLDEN, "normal_cdf.json")) as f:
        pts = json.load(f)["points"]
    x = np.array([p[0] for p in pts])
    phi = np.array([p[1] for p in pts])
    # the table's values are rounded to 15 decimals: |Phi - table| <= 5e-16
    err = np.abs(oracle.act("gelu", x) - x * phi)
    assert (err <= np.abs(x) * 6e-16 + 1e-16).all(), err
    assert oracle.act("gelu", np.array([0.0]))[0] == 0.0
    big = oracle.act("gelu", np.array([12.0, -12.0]))
    assert big[0] == 12.0 and abs(big[1]) < 1e-30


def test_fused_activation_equals_separate_pass():
    """The 'GEMM then activation' comparison the CUTLASS page's Lab 4 asks for."""
    for act in ("relu", "gelu"):
        p_fused, _, _, _ = _small_problem(act=act, with_bias=True, beta=0.5, with_c=True)
        p_plain, _, _, _ = _small_problem(act="none", with_bias=True, beta=0.5, with_c=True)
        np.testing.assert_array_equal(p_fused.full(), oracle.act(act, p_plain.full()))


def test_scales_fold_into_alpha():
    M, N, K = 6, 5, 32
    rng = np.random.default_rng(4)
    q_a = torch.from_numpy(rng.uniform(-400, 400, (M, K)).astype(np.float32)).to(torch.float8_e4m3fn)
    q_b = torch.from_numpy(rng.uniform(-400, 400, (N, K)).astype(np.float32)).to(torch.float8_e4m3fn)
    a_bits, b_bits = inputs.raw_bits(q_a), inputs.raw_bits(q_b)
    base = oracle.Problem(M, N, K, a_bits, K, oracle.ROW, b_bits, K, oracle.COL).full()
    ref = q_a.to(torch.float64).numpy() @ q_b.to(torch.float64).numpy().T
    np.testing.assert_allclose(base, ref, rtol=1e-13)
    scaled = oracle.Problem(M, N, K, a_bits, K, oracle.ROW, b_bits, K, oracle.COL,
                            alpha=2.0, scale_a=0.25, scale_b=3.0).full()
    np.testing.assert_allclose(scaled, 1.5 * base, rtol=1e-15)


def test_select_matches_full():
    case = inputs.make_case("sel", 40, 33, 70, seed=99, opA="col", opB="row", beta=0.5,
                            bias_std=0.1, act="gelu")
    p = oracle.Problem(case.M, case.N, case.K, inputs.raw_bits(case.A), case.lda, oracle.COL,
                       inputs.raw_bits(case.B), case.ldb, oracle.ROW, alpha=case.alpha,
                       beta=case.beta, C=inputs.raw_bits(case.C), ldc=case.ldc,
                       bias=inputs.raw_bits(case.bias), act="gelu")
    full = p.full()
    rows, cols = np.array([0, 17, 39]), np.array([1, 32, 5])
    assert np.array_equal(p.select(rows, cols), full[np.ix_(rows, cols)])


def test_k_zero_is_epilogue_only():
    M, N = 4, 6
    rng = np.random.default_rng(8)
    c_bits = bf16_bits(rng.uniform(-1, 1, (M, N)))
    bias_bits = bf16_bits(rng.uniform(-1, 1, N))
    a = np.zeros((M, 8), np.uint16)
    b = np.zeros((N, 8), np.uint16)
    got = oracle.Problem(M, N, 0, a, 8, oracle.ROW, b, 8, oracle.COL, beta=2.0, C=c_bits,
                         ldc=N, bias=bias_bits, act="relu").full()
    ref = np.maximum(2.0 * bf16_values(c_bits) + bf16_values(bias_bits)[None, :], 0.0)
    assert np.array_equal(got, ref)


def test_input_generator_recipes():
    """The generators honour their recipes (values, padding, integer range)."""
    c = inputs.square_512(integer=True)
    vals = c.A.to(torch.float32)[:, :c.K]
    assert torch.all(vals == vals.round()) and vals.abs().max() <= 4
    r = inputs.make_case("pad", 5, 7, 9, seed=1, opA="row", opB="row")
    assert r.lda == 16 and r.ldb == 8
    assert torch.isnan(r.A.to(torch.float32)[:, 9:]).all()
    f = inputs.make_case("f8", 8, 8, 32, seed=2, dist="normal", ab_dtype="e4m3")
    assert f.A.dtype == torch.float8_e4m3fn
    assert float(f.A.to(torch.float32)[:, :32].abs().max()) == 448.0


# ------------------------------------------- fp16 / e5m2 and channel scales

def test_f16_decoder_exhaustive_against_torch():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ours = oracle.decode_f16(bits)
    ref = torch.from_numpy(bits.view(np.int16).copy()).view(torch.float16).to(torch.float64).numpy()
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(ours), nan)
    assert np.array_equal(ours[~nan], ref[~nan])
    assert np.array_equal(np.signbit(ours[~nan]), np.signbit(ref[~nan]))


def test_e5m2_decoder_exhaustive_against_torch():
    bits = np.arange(256, dtype=np.uint16).astype(np.uint8)
    ours = oracle.decode_e5m2(bits)
    ref = torch.from_numpy(bits.copy()).view(torch.float8_e5m2).to(torch.float64).numpy()
    nan = np.isnan(ref)
    assert nan.sum() == 6  # exponent 31 with a non-zero fraction, both signs
    assert np.array_equal(np.isnan(ours), nan)
    assert np.array_equal(ours[~nan], ref[~nan])
    assert np.nanmax(ours[np.isfinite(ours)]) == 57344.0


@pytest.mark.parametrize("M,N,K", [(3, 4, 5), (6, 2, 7)])
def test_f16_tiny_exact_rational(M, N, K):
    rng = np.random.default_rng(M + N + K)
    a = torch.from_numpy(rng.uniform(-3, 3, (M, K)).astype(np.float32)).to(torch.float16)
    b = torch.from_numpy(rng.uniform(-3, 3, (N, K)).astype(np.float32)).to(torch.float16)
    a_bits = a.view(torch.int16).numpy().view(np.uint16)
    b_bits = b.view(torch.int16).numpy().view(np.uint16)
    got = oracle.Problem(M, N, K, a_bits, K, oracle.ROW, b_bits, K, oracle.COL, ab_dtype=oracle.F16).full(1)
    av, bv = a.double().numpy(), b.double().numpy()
    for i in range(M):
        for j in range(N):
            ref = sum((Fraction(av[i, k]) * Fraction(bv[j, k]) for k in range(K)), Fraction(0))
            assert got[i, j] == float(ref)


def test_e5m2_matches_numpy_on_decoded_values():
    M, N, K = 9, 7, 64
    rng = np.random.default_rng(12)
    qa = torch.from_numpy(rng.uniform(-100, 100, (M, K)).astype(np.float32)).to(torch.float8_e5m2)
    qb = torch.from_numpy(rng.uniform(-100, 100, (N, K)).astype(np.float32)).to(torch.float8_e5m2)
    got = oracle.Problem(M, N, K, qa.view(torch.uint8).numpy(), K, oracle.ROW, qb.view(torch.uint8).numpy(), K,
                         oracle.COL, ab_dtype=oracle.E5M2, scale_a=0.5, scale_b=0.25).full()
    ref = 0.125 * (qa.double().numpy() @ qb.double().numpy().T)
    np.testing.assert_allclose(got, ref, rtol=1e-13)


def test_channel_scales_are_row_and_column_factors():
    """Per-row and per-column scales multiply element (i, j) by r_i * c_j (indices not swapped)."""
    M, N, K = 5, 8, 24
    rng = np.random.default_rng(13)
    a_bits = bf16_bits(rng.uniform(-1, 1, (M, K)))
    b_bits = bf16_bits(rng.uniform(-1, 1, (N, K)))
    r = np.arange(1, M + 1, dtype=np.float32) * 0.5
    c = np.arange(1, N + 1, dtype=np.float32) * 0.25 + 1.0
    base = oracle.Problem(M, N, K, a_bits, K, oracle.ROW, b_bits, K, oracle.COL).full()
    scaled = oracle.Problem(M, N, K, a_bits, K, oracle.ROW, b_bits, K, oracle.COL,
                            row_scale=r, col_scale=c).full()
    np.testing.assert_allclose(scaled, base * r[:, None] * c[None, :], rtol=1e-13)
    only_rows = oracle.Problem(M, N, K, a_bits, K, oracle.ROW, b_bits, K, oracle.COL, row_scale=r).full()
    np.testing.assert_allclose(only_rows, base * r[:, None], rtol=1e-13)


# ------------------------------------------------------ block-scaled operands

def test_e8m0_decoder_exhaustive_against_torch():
    bits = np.arange(256, dtype=np.uint16).astype(np.uint8)
    ours = oracle.decode_e8m0(bits)
    ref = torch.from_numpy(bits.copy()).view(torch.float8_e8m0fnu).to(torch.float64).numpy()
    nan = np.isnan(ref)
    assert nan.sum() == 1 and nan[255]
    assert np.array_equal(np.isnan(ours), nan)
    assert np.array_equal(ours[~nan], ref[~nan])
    assert ours[127] == 1.0 and ours[128] == 2.0 and ours[126] == 0.5


def _mx_case(M, N, K, seed, lo=124, hi=130, fmt="e4m3"):
    """Integer-valued fp8 elements in [-4, 4] with random E8M0 scale codes."""
    rng = np.random.default_rng(seed)
    tdt = torch.float8_e4m3fn if fmt == "e4m3" else torch.float8_e5m2
    a = torch.from_numpy(rng.integers(-4, 5, (M, K)).astype(np.float32)).to(tdt)
    b = torch.from_numpy(rng.integers(-4, 5, (N, K)).astype(np.float32)).to(tdt)
    kb = (K + 31) // 32
    sfa = rng.integers(lo, hi + 1, (M, kb)).astype(np.uint8)
    sfb = rng.integers(lo, hi + 1, (N, kb)).astype(np.uint8)
    return a, b, sfa, sfb


@pytest.mark.parametrize("M,N,K", [(1, 1, 1), (3, 4, 33), (5, 2, 70), (2, 6, 96)])
@pytest.mark.parametrize("fmt", ["e4m3", "e5m2"])
def test_block_scaled_tiny_exact_rational(M, N, K, fmt):
    """Every element against exact rational arithmetic: a(i,k) and b(k,j) are
    multiplied by 2^(code - 127) of their 32-wide block along k (torch decodes
    the E8M0 codes and the fp8 elements independently of the oracle)."""
    a, b, sfa, sfb = _mx_case(M, N, K, M * 31 + N * 7 + K, fmt=fmt)
    dt = oracle.E4M3 if fmt == "e4m3" else oracle.E5M2
    got = oracle.Problem(M, N, K, a.view(torch.uint8).numpy(), K, oracle.ROW, b.view(torch.uint8).numpy(), K,
                         oracle.COL, ab_dtype=dt, sfa=sfa, sfb=sfb, alpha=0.5).full(1)
    av, bv = a.double().numpy(), b.double().numpy()
    sa = torch.from_numpy(sfa.copy()).view(torch.float8_e8m0fnu).double().numpy()
    sb = torch.from_numpy(sfb.copy()).view(torch.float8_e8m0fnu).double().numpy()
    for i in range(M):
        for j in range(N):
            ref = sum((Fraction(sa[i, k // 32]) * Fraction(av[i, k]) * Fraction(sb[j, k // 32]) * Fraction(bv[j, k])
                       for k in range(K)), Fraction(0))
            assert got[i, j] == float(Fraction(1, 2) * ref), (i, j)


def test_unit_block_scales_reduce_to_plain_fp8():
    M, N, K = 6, 9, 100
    a, b, sfa, sfb = _mx_case(M, N, K, 3)
    sfa[:] = 127
    sfb[:] = 127
    args = (M, N, K, a.view(torch.uint8).numpy(), K, oracle.ROW, b.view(torch.uint8).numpy(), K, oracle.COL)
    plain = oracle.Problem(*args, ab_dtype=oracle.E4M3).full()
    scaled = oracle.Problem(*args, ab_dtype=oracle.E4M3, sfa=sfa, sfb=sfb).full()
    assert np.array_equal(plain, scaled)


def test_one_block_scale_changes_only_its_block():
    """Raising the scale of block kb of row i of A by one code (x2) adds exactly
    that block's contribution to row i of D and leaves the other rows alone;
    the same for a column block of B (no swapped or shifted block index)."""
    M, N, K = 4, 5, 96
    a, b, sfa, sfb = _mx_case(M, N, K, 5)
    args = (M, N, K, a.view(torch.uint8).numpy(), K, oracle.ROW, b.view(torch.uint8).numpy(), K, oracle.COL)
    base = oracle.Problem(*args, ab_dtype=oracle.E4M3, sfa=sfa, sfb=sfb).full()
    av, bv = a.double().numpy(), b.double().numpy()
    sa = 2.0 ** (sfa.astype(np.float64) - 127)
    sb = 2.0 ** (sfb.astype(np.float64) - 127)
    i0, j0, kb = 2, 3, 1
    ks = np.arange(kb * 32, (kb + 1) * 32)
    sfa2 = sfa.copy()
    sfa2[i0, kb] += 1
    d = oracle.Problem(*args, ab_dtype=oracle.E4M3, sfa=sfa2, sfb=sfb).full() - base
    contrib = np.array([(sa[i0, kb] * av[i0, ks] * sb[j, kb] * bv[j, ks]).sum() for j in range(N)])
    np.testing.assert_array_equal(d[i0], contrib)
    assert not np.delete(d, i0, axis=0).any()
    sfb2 = sfb.copy()
    sfb2[j0, kb] += 1
    d = oracle.Problem(*args, ab_dtype=oracle.E4M3, sfa=sfa, sfb=sfb2).full() - base
    contrib = np.array([(sa[i, kb] * av[i, ks] * sb[j0, kb] * bv[j0, ks]).sum() for i in range(M)])
    np.testing.assert_array_equal(d[:, j0], contrib)
    assert not np.delete(d, j0, axis=1).any()


def test_mx_quantiser_and_blocked_layout():
    """The input generator's OCP MX quantisation keeps every value within the
    element format's relative step of its source, and the blocked scale layout
    is a permutation that puts (row r, column c) where the library reads it."""
    x = torch.randn((7, 70), generator=torch.Generator().manual_seed(0))
    q, codes = inputs.mx_quantize(x, "e4m3")
    scale = torch.from_numpy(codes.astype(np.float32) - 127).exp2().repeat_interleave(32, dim=1)[:, :70]
    deq = q.to(torch.float32) * scale
    assert torch.all((deq - x).abs() <= 2.0 ** -3 * x.abs() + 2.0 ** -9 * scale)
    sf = np.arange(300 * 9, dtype=np.int64).reshape(300, 9) % 251
    blk = inputs.mx_blocked_layout(sf.astype(np.uint8))
    assert blk.size == 384 * 12
    for r in (0, 31, 32, 127, 128, 299):
        for c in (0, 3, 4, 8):
            off = ((r // 128) * 3 + c // 4) * 512 + (r % 32) * 16 + (r % 128) // 32 * 4 + c % 4
            assert blk[off] == sf[r, c] % 251


# ------------------------------------------------------------ FP4 operands

def test_e2m1_decoder_against_e4m3_reencoding():
    """Each E2M1 code re-encoded bit by bit as the E4M3 code of the same value
    (exponent rebased from bias 1 to bias 7, fraction shifted into place) and
    decoded by torch must equal the oracle's decode."""
    codes = np.arange(16, dtype=np.uint8)
    ours = oracle.decode_e2m1(codes)
    for c in codes:
        s, e, f = (c >> 3) & 1, (c >> 1) & 3, c & 1
        if e == 0 and f == 0:
            bits = s << 7
        elif e == 0:   # subnormal 0.5 = 2^-1: E4M3 exponent field -1 + 7 = 6, fraction 0
            bits = (s << 7) | (6 << 3)
        else:
            bits = (s << 7) | ((e - 1 + 7) << 3) | (f << 2)
        ref = torch.tensor([bits], dtype=torch.uint8).view(torch.float8_e4m3fn).double().item()
        assert ours[c] == ref, (c, ours[c], ref)
    assert sorted(set(np.abs(ours))) == [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]


def test_ue4m3_decoder_against_torch():
    bits = np.arange(128, dtype=np.uint8)
    ours = oracle.decode_ue4m3(bits)
    ref = torch.from_numpy(bits.copy()).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(ours), nan) and nan.sum() == 1
    assert np.array_equal(ours[~nan], ref[~nan])
    assert np.array_equal(oracle.decode_ue4m3(bits | 0x80)[~nan], ours[~nan])  # the sign bit is ignored


@pytest.mark.parametrize("fmt", ["nvfp4", "mxfp4"])
@pytest.mark.parametrize("M,N,K", [(1, 1, 2), (3, 4, 34), (5, 2, 96), (2, 3, 130)])
def test_fp4_block_scaled_tiny_exact_rational(fmt, M, N, K):
    """Packed FP4 elements (even element in the low nibble) with per-block
    scales against exact rational arithmetic, elements and scales decoded
    independently of the oracle (nibble unpacking here, torch for the scales)."""
    case = inputs.make_fp4_case("t", M, N, K, seed=M * 13 + N * 5 + K, fmt=fmt, dist="codes",
                                code_range=list(range(16)),
                                scale_codes=[0x30, 0x38, 0x40, 0x44] if fmt == "nvfp4" else [125, 127, 129])
    got = oracle.Problem(M, N, K, case.A.numpy(), case.lda, oracle.ROW, case.B.numpy(), case.ldb, oracle.COL,
                         ab_dtype=oracle.E2M1, sfa=case.sfa, sfb=case.sfb, block=case.sf_block,
                         sf_format=oracle.SF_UE4M3 if fmt == "nvfp4" else oracle.SF_E8M0).full(1)
    grid = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]

    def unpack(storage):
        b = storage.numpy()
        nib = np.stack([b & 0xF, b >> 4], axis=-1).reshape(b.shape[0], -1)[:, :K]
        return [[Fraction(grid[n & 7]) * (-1 if n & 8 else 1) for n in row] for row in nib]

    def scale(code):
        if fmt == "nvfp4":
            return Fraction(torch.tensor([code], dtype=torch.uint8).view(torch.float8_e4m3fn).double().item())
        return Fraction(2) ** (int(code) - 127)

    a, b = unpack(case.A), unpack(case.B)
    blk = case.sf_block
    for i in range(M):
        for j in range(N):
            ref = sum((scale(case.sfa[i, k // blk]) * a[i][k] * scale(case.sfb[j, k // blk]) * b[j][k]
                       for k in range(K)), Fraction(0))
            assert got[i, j] == float(ref), (i, j)


def test_fp4_quantiser_keeps_values_within_one_step():
    case = inputs.make_fp4_case("q", 4, 3, 64, seed=2, fmt="nvfp4")
    rng = np.random.default_rng(2)
    x = rng.standard_normal((4, 64))  # the same first draw the generator quantised for A
    b = case.A.numpy()
    nib = np.stack([b & 0xF, b >> 4], axis=-1).reshape(4, -1)[:, :64]
    vals = oracle.decode_e2m1(nib) * np.repeat(oracle.decode_ue4m3(case.sfa), 16, axis=1)
    scale = np.repeat(oracle.decode_ue4m3(case.sfa), 16, axis=1)
    # the largest E2M1 step is 2 (between 4 and 6): half a step of the scaled grid, plus the scale's rounding
    assert np.all(np.abs(vals - x) <= 1.0 * scale + 0.07 * np.abs(x))


# ---------------------------------------------------------------- grouped GEMM

def _rank_one_problem(M, N, K, rng, layouts=("row", "col")):
    """A = u v^T, B = w x^T with small integers: D = (v . w) u x^T exactly."""
    u = rng.integers(-3, 4, M).astype(np.float64)
    v = rng.integers(-3, 4, K).astype(np.float64)
    w = rng.integers(-3, 4, K).astype(np.float64)
    x = rng.integers(-3, 4, N).astype(np.float64)
    A, lda = store(np.outer(u, v), layouts[0])
    B, ldb = store(np.outer(w, x), layouts[1])
    prob = oracle.Problem(M, N, K, bf16_bits(A), lda, op(layouts[0]), bf16_bits(B), ldb, op(layouts[1]))
    return prob, float(v @ w) * np.outer(u, x)


def test_grouped_rank_one_closed_forms():
    """Every problem of a batch of different shapes gets its own closed form,
    so a problem index mixed up anywhere (operands, sizes, output) fails."""
    rng = np.random.default_rng(31)
    shapes = [(5, 7, 3), (1, 12, 9), (9, 1, 4), (6, 6, 1), (3, 8, 17)]
    layouts = [("row", "col"), ("col", "row"), ("row", "row"), ("col", "col"), ("row", "col")]
    probs, refs = zip(*(_rank_one_problem(M, N, K, rng, lay) for (M, N, K), lay in zip(shapes, layouts)))
    got = oracle.grouped(list(probs))
    assert len(got) == len(shapes)
    for g, (d, ref, (M, N, K)) in enumerate(zip(got, refs, shapes)):
        assert d.shape == (M, N), g
        assert np.array_equal(d, ref), g


def test_grouped_problems_are_independent():
    """Changing one problem's inputs changes that problem's output only."""
    rng = np.random.default_rng(32)
    p0, r0 = _rank_one_problem(4, 5, 6, rng)
    p1, r1 = _rank_one_problem(3, 2, 7, rng)
    p1b, r1b = _rank_one_problem(3, 2, 7, rng)
    assert not np.array_equal(r1, r1b)
    a = oracle.grouped([p0, p1])
    b = oracle.grouped([p0, p1b])
    assert np.array_equal(a[0], r0) and np.array_equal(b[0], r0)
    assert np.array_equal(a[1], r1) and np.array_equal(b[1], r1b)


def test_grouped_empty_and_k_zero_problems():
    """An M == 0 problem contributes an empty result; a K == 0 problem is
    act(beta * C + bias), like a single GEMM with K == 0."""
    rng = np.random.default_rng(33)
    empty = oracle.Problem(0, 4, 8, np.zeros((1, 8), np.uint16), 8, oracle.ROW,
                           np.zeros((4, 8), np.uint16), 8, oracle.COL)
    c_bits = bf16_bits(rng.uniform(-1, 1, (2, 3)))
    bias_bits = bf16_bits(rng.uniform(-1, 1, 3))
    k0 = oracle.Problem(2, 3, 0, np.zeros((2, 8), np.uint16), 8, oracle.ROW, np.zeros((3, 8), np.uint16), 8,
                        oracle.COL, beta=0.5, C=c_bits, ldc=3, bias=bias_bits, act="relu")
    p2, r2 = _rank_one_problem(2, 2, 2, rng)
    got = oracle.grouped([empty, k0, p2])
    assert got[0].shape == (0, 4)
    assert np.array_equal(got[1], np.maximum(0.5 * bf16_values(c_bits) + bf16_values(bias_bits)[None, :], 0.0))
    assert np.array_equal(got[2], r2)


def test_moe_routing_recipe():
    """The grouped workload's routing: every row goes to exactly one expert, the
    counts are irregular and reproducible from the seed."""
    counts = inputs.moe_token_counts(32768, 16, seed=41)
    assert len(counts) == 16 and sum(counts) == 32768 and min(counts) >= 0
    assert counts == inputs.moe_token_counts(32768, 16, seed=41)
    assert len(set(counts)) > 8 and any(c % 128 for c in counts)
    assert counts != inputs.moe_token_counts(32768, 16, seed=42)


def test_integer_problems_match_numpy_for_random_shapes_and_layouts():
    """Property over random small shapes, layouts and padded leading dimensions:
    with integer inputs the oracle equals numpy's float64 matmul exactly."""
    hypothesis = pytest.importorskip("hypothesis")
    st = hypothesis.strategies

    @hypothesis.settings(max_examples=60, deadline=None)
    @hypothesis.given(M=st.integers(1, 9), N=st.integers(1, 9), K=st.integers(1, 12),
                      la=st.sampled_from(["row", "col"]), lb=st.sampled_from(["row", "col"]),
                      pad=st.integers(0, 3), seed=st.integers(0, 2**31 - 1))
    def check(M, N, K, la, lb, pad, seed):
        rng = np.random.default_rng(seed)
        a = rng.integers(-4, 5, (M, K)).astype(np.float64)
        b = rng.integers(-4, 5, (K, N)).astype(np.float64)

        def padded(x, layout):
            st_, ld = store(x, layout)
            out = np.zeros((st_.shape[0], ld + pad), dtype=np.float64)
            out[:, :ld] = st_
            return bf16_bits(out), ld + pad

        A, lda = padded(a, la)
        B, ldb = padded(b, lb)
        got = oracle.Problem(M, N, K, A, lda, op(la), B, ldb, op(lb)).full()
        assert np.array_equal(got, a @ b)

    check()
