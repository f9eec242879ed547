"""Seeded synthetic inputs for the GEMM workloads.

This module holds no GEMM arithmetic: it only draws operands with the value
distributions, shapes, storage orders and padded leading dimensions of the
workloads, on the CPU with ``torch.Generator``.  Both the CUDA path (through
the binding) and the oracle (through raw bits) consume exactly what it returns.

Storage convention (same as the C ABI): the logical A is M x K and the logical
B is K x N.  ``"row"`` stores a matrix row-major with leading dimension ld
(element (r,c) at r*ld + c), ``"col"`` stores it column-major (element (r,c)
at c*ld + r).  C and D are always row-major M x N.  Leading dimensions are
padded up to a multiple of 16 bytes; the padding is filled with NaN (bf16) or
the e4m3 NaN pattern so that a kernel reading it would be caught.
"""
from __future__ import annotations

from dataclasses import dataclass, field
from typing import Optional

import numpy as np
import torch

_ELEM_BYTES = {"bf16": 2, "e4m3": 1, "f32": 4, "f16": 2, "e5m2": 1}
_TORCH = {"bf16": torch.bfloat16, "e4m3": torch.float8_e4m3fn, "f32": torch.float32, "f16": torch.float16,
          "e5m2": torch.float8_e5m2}
E4M3_MAX = 448.0
E5M2_MAX = 57344.0
FP8_MAX = {"e4m3": E4M3_MAX, "e5m2": E5M2_MAX}


def padded_ld(extent: int, dtype: str) -> int:
    """Smallest leading dimension >= extent whose byte size is a multiple of 16."""
    q = 16 // _ELEM_BYTES[dtype]
    return max(q, (extent + q - 1) // q * q)


def _store(logical: torch.Tensor, layout: str, dtype: str, ld: Optional[int] = None):
    """Place a logical (rows x cols) fp32 matrix into padded storage of `dtype`."""
    rows, cols = logical.shape
    inner = cols if layout == "row" else rows
    outer = rows if layout == "row" else cols
    ld = padded_ld(inner, dtype) if ld is None else ld
    buf = torch.full((max(outer, 1), ld), float("nan"), dtype=torch.float32)
    if layout == "row":
        buf[:rows, :cols] = logical
    else:
        buf[:cols, :rows] = logical.t()
    return buf.to(_TORCH[dtype]), ld


def raw_bits(t: Optional[torch.Tensor]) -> Optional[np.ndarray]:
    """The raw storage bits of a CPU tensor as numpy (uint16 / uint8 / float32)."""
    if t is None:
        return None
    if t.dtype in (torch.bfloat16, torch.float16):
        return t.contiguous().view(torch.int16).numpy().view(np.uint16)
    if t.dtype in (torch.float8_e4m3fn, torch.float8_e5m2):
        return t.contiguous().view(torch.uint8).numpy()
    if t.dtype == torch.float32:
        return t.contiguous().numpy()
    if t.dtype == torch.uint8:  # packed FP4 storage
        return t.contiguous().numpy()
    raise TypeError(t.dtype)


@dataclass
class GemmCase:
    name: str
    M: int
    N: int
    K: int
    opA: str
    opB: str
    ab_dtype: str
    d_dtype: str
    A: torch.Tensor          # storage (CPU)
    lda: int
    B: torch.Tensor          # storage (CPU)
    ldb: int
    alpha: float = 1.0
    beta: float = 0.0
    C: Optional[torch.Tensor] = None
    ldc: int = 0
    c_dtype: str = "bf16"
    bias: Optional[torch.Tensor] = None
    bias_dtype: str = "bf16"
    act: str = "none"
    scale_a: float = 1.0
    scale_b: float = 1.0
    row_scale: Optional[torch.Tensor] = None   # fp32 [M] dequantisation scale per row
    col_scale: Optional[torch.Tensor] = None   # fp32 [N] dequantisation scale per column
    sfa: Optional[np.ndarray] = None           # uint8 E8M0 [M][ceil(K/32)] block scales of A's rows
    sfb: Optional[np.ndarray] = None           # uint8 E8M0 [N][ceil(K/32)] block scales of B's columns
    sf_block: int = 32                          # elements per block scale (32 MX, 16 NVFP4)
    sf_format: str = "e8m0"                     # "e8m0" or "ue4m3" scale codes
    ldd: int = 0
    meta: dict = field(default_factory=dict)

    @property
    def flops(self) -> int:
        return 2 * self.M * self.N * self.K


def _draw(gen, shape, dist, K):
    if dist == "uniform":
        return torch.rand(shape, generator=gen, dtype=torch.float32) * 2.0 - 1.0
    if dist == "int4":
        return torch.randint(-4, 5, shape, generator=gen, dtype=torch.int32).to(torch.float32)
    if dist == "normal_sqrtk":
        return torch.randn(shape, generator=gen, dtype=torch.float32) / float(np.sqrt(max(K, 1)))
    if dist == "normal":
        return torch.randn(shape, generator=gen, dtype=torch.float32)
    raise ValueError(dist)


MX_BLOCK = 32
# largest power-of-two exponent of each element format (e4m3: 448 = 1.75 * 2^8)
_EMAX = {"e4m3": 8, "e5m2": 15}


def mx_quantize(x: torch.Tensor, fmt: str, scale_dist: Optional[tuple] = None, gen=None):
    """OCP Microscaling quantisation along the last axis in blocks of 32:
    shared exponent E = floor(log2(amax of the block)) - emax(fmt), scale code
    E + 127 (E8M0), elements fp8(clamp(x / 2^E)).  All-zero blocks get scale 1.
    scale_dist = (lo, hi): instead draw each scale code uniformly in [lo, hi]
    and quantise x / 2^E with it (for integer-valued tests).  Returns the
    element codes (same shape, fp8 dtype) and the uint8 scale codes
    [..., ceil(n / 32)]."""
    n = x.shape[-1]
    nb = (n + MX_BLOCK - 1) // MX_BLOCK
    pad = nb * MX_BLOCK - n
    xp = torch.nn.functional.pad(x, (0, pad)).reshape(*x.shape[:-1], nb, MX_BLOCK)
    if scale_dist is None:
        amax = xp.abs().amax(dim=-1)
        e = torch.where(amax > 0, torch.floor(torch.log2(torch.where(amax > 0, amax, torch.ones_like(amax)))),
                        torch.zeros_like(amax)) - _EMAX[fmt]
        e = torch.where(amax > 0, e, torch.zeros_like(e)).clamp(-127, 127)
    else:
        lo, hi = scale_dist
        e = torch.randint(lo, hi + 1, xp.shape[:-1], generator=gen, dtype=torch.int64).to(torch.float32) - 127
    q = (xp / torch.exp2(e)[..., None]).clamp(-FP8_MAX[fmt], FP8_MAX[fmt])
    q = q.reshape(*x.shape[:-1], nb * MX_BLOCK)[..., :n].to(_TORCH[fmt])
    codes = (e + 127).to(torch.uint8).numpy()
    return q, codes


def mx_blocked_layout(sf: np.ndarray, rows_pad: int = 128, kb_pad: int = 4, pad_code: int = 127) -> np.ndarray:
    """The scale-factor layout the library reads (a permutation, no arithmetic):
    rows padded to a multiple of 128 and scale columns to a multiple of 4;
    for each block of 128 rows x 4 scale columns, 512 consecutive bytes, the
    byte of (row r, column c) at (r % 32) * 16 + (r % 128) // 32 * 4 + c % 4;
    blocks ordered by row block, then column block.  Padding bytes are 127."""
    R, C = sf.shape
    Rp = (R + rows_pad - 1) // rows_pad * rows_pad
    Cp = (C + kb_pad - 1) // kb_pad * kb_pad
    full = np.full((Rp, Cp), pad_code, dtype=np.uint8)
    full[:R, :C] = sf
    # [rb][r32_hi(4)][r32_lo(32)][cb][c4] -> [rb][cb][r32_lo][r32_hi][c4]
    t = full.reshape(Rp // 128, 4, 32, Cp // 4, 4).transpose(0, 3, 2, 1, 4)
    return np.ascontiguousarray(t).reshape(-1)


# FP4 E2M1 (OCP Microscaling formats): the eight magnitudes of codes 0..7
E2M1_GRID = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])
UE4M3_ONE = 0x38  # 1.0 as an unsigned E4M3 scale


def e2m1_codes(v: np.ndarray) -> np.ndarray:
    """Round to the nearest E2M1 value (ties to the even code), saturating at 6."""
    mag = np.minimum(np.abs(v), 6.0)
    mids = (E2M1_GRID[1:] + E2M1_GRID[:-1]) / 2
    code = np.searchsorted(mids, mag, side="left")          # mag <= mid -> lower code
    tie = np.isin(mag, mids)
    code = np.where(tie & (code % 2 == 1), code + 1, code)  # exact tie -> even code
    code = np.where(tie & (code % 2 == 1), code - 1, code)
    return (code | np.where(v < 0, 8, 0)).astype(np.uint8)


def pack_fp4(codes: np.ndarray, ld: int) -> np.ndarray:
    """Rows of 4-bit codes -> bytes, two per byte (even element in the low
    nibble), rows ld elements long (ld even; padding nibbles 7 = 6.0)."""
    rows, k = codes.shape
    full = np.full((rows, ld), 7, dtype=np.uint8)
    full[:, :k] = codes
    return (full[:, 0::2] | (full[:, 1::2] << 4)).astype(np.uint8)


def _fp4_scales(blocks: np.ndarray, fmt: str, gen_codes):
    """Per-block scale codes and values for FP4 quantisation of `blocks`
    [..., nb, blk]: NVFP4 amax / 6 rounded to unsigned E4M3, MXFP4
    2^(floor(log2 amax) - 2) as E8M0."""
    amax = np.abs(blocks).max(axis=-1)
    if gen_codes is not None:
        return gen_codes(amax.shape)
    if fmt == "nvfp4":
        s = np.where(amax > 0, np.minimum(amax / 6.0, 448.0), 1.0).astype(np.float32)
        codes = torch.from_numpy(s).to(torch.float8_e4m3fn).view(torch.uint8).numpy() & 0x7F
        codes = np.where(codes == 0, UE4M3_ONE, codes).astype(np.uint8)
        return codes
    e = np.where(amax > 0, np.floor(np.log2(np.where(amax > 0, amax, 1.0))) - 2, 0).clip(-127, 127)
    return (e + 127).astype(np.uint8)


def make_fp4_case(name, M, N, K, *, seed, fmt="nvfp4", dist="normal", lda=None, ldb=None, d_dtype="bf16",
                  alpha=1.0, beta=0.0, c_dist="uniform", bias_std=None, act="none", code_range=None,
                  scale_codes=None) -> GemmCase:
    """A block-scaled FP4 problem: A row-major, B column-major (both K-major),
    E2M1 elements packed two per byte.  fmt "nvfp4": unsigned E4M3 scales per
    16 elements; "mxfp4": E8M0 scales per 32.  dist "normal": N(0,1) quantised
    per block; dist "codes": element codes uniform over code_range (a list of
    E2M1 codes) and scale codes uniform over scale_codes (a list), for exact
    tests.  Order of draws: A, B (elements then scales), C, bias."""
    rng = np.random.default_rng(int(seed))
    blk = 16 if fmt == "nvfp4" else 32
    nb = (K + blk - 1) // blk
    ld_a = lda if lda is not None else (K + 31) // 32 * 32
    ld_b = ldb if ldb is not None else (K + 31) // 32 * 32

    def operand(rows):
        if dist == "codes":
            codes = rng.choice(np.asarray(code_range, dtype=np.uint8), size=(rows, K))
            sc = rng.choice(np.asarray(scale_codes, dtype=np.uint8), size=(rows, nb))
            return codes, sc
        x = rng.standard_normal((rows, nb * blk))
        xb = x.reshape(rows, nb, blk)
        sc = _fp4_scales(xb, fmt, None)
        if fmt == "nvfp4":
            sval = torch.from_numpy(sc.copy()).view(torch.float8_e4m3fn).to(torch.float64).numpy()
        else:
            sval = np.exp2(sc.astype(np.float64) - 127)
        codes = e2m1_codes(xb / sval[..., None]).reshape(rows, nb * blk)[:, :K]
        return codes, sc

    ca, sfa = operand(M)
    cb, sfb = operand(N)
    A = torch.from_numpy(pack_fp4(ca, ld_a))
    B = torch.from_numpy(pack_fp4(cb, ld_b))
    gen = torch.Generator().manual_seed(int(seed) + 1)
    C = None
    ldc = 0
    if beta != 0.0:
        c = _draw(gen, (M, N), c_dist, K)
        C, ldc = _store(c, "row", "bf16")
    bias = None
    if bias_std is not None:
        bias = (torch.randn((N,), generator=gen, dtype=torch.float32) * bias_std).to(torch.bfloat16)
    return GemmCase(name=name, M=M, N=N, K=K, opA="row", opB="col", ab_dtype=fmt, d_dtype=d_dtype, A=A, lda=ld_a,
                    B=B, ldb=ld_b, alpha=alpha, beta=beta, C=C, ldc=ldc, bias=bias, act=act,
                    ldd=padded_ld(N, d_dtype), sfa=sfa, sfb=sfb, sf_block=blk,
                    sf_format="ue4m3" if fmt == "nvfp4" else "e8m0", meta={"seed": seed, "dist": dist})


def make_case(name, M, N, K, *, seed, dist="uniform", opA="row", opB="col",
              ab_dtype="bf16", d_dtype="bf16", alpha=1.0, beta=0.0, c_dist=None,
              c_dtype="bf16", bias_std=None, bias_dtype="bf16", act="none",
              lda=None, ldb=None, ldc=None, ldd=None, channel_scales=False,
              block_scaled=False, mx_scale_codes=None) -> GemmCase:
    """Draw one GEMM problem.  Order of draws: A, B, C, bias, channel scales
    (all from `seed`).  channel_scales: fp32 row and column scales U[0.5, 2].
    block_scaled (fp8 operands, A row-major, B column-major): OCP MX blocks of
    32 along K with E8M0 scales (mx_quantize); mx_scale_codes = (lo, hi) draws
    the scale codes instead (after A and B, before C)."""
    gen = torch.Generator().manual_seed(int(seed))
    a = _draw(gen, (M, K), dist, K)
    b = _draw(gen, (K, N), dist, K)
    scale_a = scale_b = 1.0
    sfa = sfb = None
    if block_scaled:
        if ab_dtype not in FP8_MAX or opA != "row" or opB != "col":
            raise ValueError("block-scaled cases are fp8 with A row-major and B column-major")
        qa, sfa = mx_quantize(a, ab_dtype, mx_scale_codes, gen)
        qb, sfb = mx_quantize(b.t().contiguous(), ab_dtype, mx_scale_codes, gen)
        a = qa.to(torch.float32)
        b = qb.to(torch.float32).t()
    elif ab_dtype in FP8_MAX and dist != "int4":
        # per-tensor scale amax/fmax, then the quantised codes (the harness does
        # this, not the library): q = fp8(clamp(x / scale, -fmax, fmax)), fmax =
        # 448 (e4m3) or 57344 (e5m2).  Integer draws in [-4, 4] are FP8 codes
        # already and keep scale 1.
        fmax = FP8_MAX[ab_dtype]
        amax_a = float(a.abs().max()) if a.numel() else 1.0
        amax_b = float(b.abs().max()) if b.numel() else 1.0
        scale_a = (amax_a / fmax) if amax_a > 0 else 1.0
        scale_b = (amax_b / fmax) if amax_b > 0 else 1.0
        a = (a / scale_a).clamp(-fmax, fmax)
        b = (b / scale_b).clamp(-fmax, fmax)
    A, lda = _store(a, opA, ab_dtype, lda)
    B, ldb = _store(b, opB, ab_dtype, ldb)
    C = None
    if beta != 0.0:
        c = _draw(gen, (M, N), c_dist or dist, K)
        C, ldc = _store(c, "row", c_dtype, ldc)
    else:
        ldc = 0
    bias = None
    if bias_std is not None:
        bias = (torch.randn((N,), generator=gen, dtype=torch.float32) * bias_std).to(_TORCH[bias_dtype])
    row_scale = col_scale = None
    if channel_scales:
        row_scale = torch.rand((M,), generator=gen, dtype=torch.float32) * 1.5 + 0.5
        col_scale = torch.rand((N,), generator=gen, dtype=torch.float32) * 1.5 + 0.5
    ldd = padded_ld(N, d_dtype) if ldd is None else ldd
    return GemmCase(name=name, M=M, N=N, K=K, opA=opA, opB=opB, ab_dtype=ab_dtype,
                    d_dtype=d_dtype, A=A, lda=lda, B=B, ldb=ldb, alpha=alpha, beta=beta,
                    C=C, ldc=ldc, c_dtype=c_dtype, bias=bias, bias_dtype=bias_dtype,
                    act=act, scale_a=scale_a, scale_b=scale_b, row_scale=row_scale,
                    col_scale=col_scale, ldd=ldd, sfa=sfa, sfb=sfb, meta={"seed": seed, "dist": dist})


# The workloads, with their sizes and value recipes.  Seeds are fixed per case.
def square_512(integer: bool = False) -> GemmCase:
    """512^3, A row / B col bf16, alpha=1 beta=0, fp32 D; U[-1,1] or integers in [-4,4]."""
    if integer:
        return make_case("gemm512_int", 512, 512, 512, seed=2, dist="int4", d_dtype="f32")
    return make_case("gemm512_uniform", 512, 512, 512, seed=1, dist="uniform", d_dtype="f32")


def square_4096_beta() -> GemmCase:
    """4096^3 bf16, A,B ~ N(0,1)/sqrt(K), C ~ N(0,1), alpha=beta=1, bf16 D."""
    return make_case("gemm4096_beta1", 4096, 4096, 4096, seed=3, dist="normal_sqrtk",
                     alpha=1.0, beta=1.0, c_dist="normal")


def square_8192_gelu() -> GemmCase:
    """8192^3 bf16, A,B ~ N(0,1)/sqrt(K), D = GELU(AB + bias), bias ~ N(0,0.1), bf16 D."""
    return make_case("gemm8192_bias_gelu", 8192, 8192, 8192, seed=4, dist="normal_sqrtk",
                     bias_std=0.1, act="gelu")


RAGGED_SHAPES = [(4095, 3001, 1537), (16, 8192, 8192), (8192, 128, 8192)]
LAYOUT_COMBOS = [("row", "row"), ("row", "col"), ("col", "row"), ("col", "col")]


def ragged(shape_idx: int, combo_idx: int) -> GemmCase:
    """Ragged/skinny bf16 shapes, U[-1,1], C U[-1,1], beta=0.5, each A/B layout combo."""
    M, N, K = RAGGED_SHAPES[shape_idx]
    opA, opB = LAYOUT_COMBOS[combo_idx]
    seed = 5 + 4 * shape_idx + combo_idx
    return make_case(f"ragged_{M}x{N}x{K}_{opA}{opB}", M, N, K, seed=seed, dist="uniform",
                     opA=opA, opB=opB, alpha=1.0, beta=0.5, c_dist="uniform")


def ragged_tight(combo_idx: int) -> GemmCase:
    """The 4095 x 3001 x 1537 ragged shape with tight leading dimensions (each
    ld equal to the contiguous extent, so none is a multiple of 16 bytes):
    U[-1,1], C U[-1,1], beta=0.5, ldc = ldd = N."""
    M, N, K = RAGGED_SHAPES[0]
    opA, opB = LAYOUT_COMBOS[combo_idx]
    lda = K if opA == "row" else M
    ldb = N if opB == "row" else K
    return make_case(f"ragged_tight_{M}x{N}x{K}_{opA}{opB}", M, N, K, seed=105 + combo_idx,
                     dist="uniform", opA=opA, opB=opB, alpha=1.0, beta=0.5, c_dist="uniform",
                     lda=lda, ldb=ldb, ldc=N, ldd=N)


def mxfp8_8192_relu(fmt: str = "e4m3") -> GemmCase:
    """8192^3 MXFP8 (N(0,1) quantised in blocks of 32 along K with E8M0 scales),
    bias N(0,0.1), ReLU, bf16 D."""
    return make_case(f"gemm8192_mx{fmt}_bias_relu", 8192, 8192, 8192, seed=18, dist="normal",
                     ab_dtype=fmt, bias_std=0.1, act="relu", block_scaled=True)


def nvfp4_8192_relu() -> GemmCase:
    """8192^3 NVFP4 (N(0,1) quantised to E2M1 in blocks of 16 with unsigned
    E4M3 scales), bias N(0,0.1), ReLU, bf16 D."""
    return make_fp4_case("gemm8192_nvfp4_bias_relu", 8192, 8192, 8192, seed=19, fmt="nvfp4", bias_std=0.1,
                         act="relu")


def fp8_8192_relu() -> GemmCase:
    """8192^3 e4m3 (N(0,1) quantised with amax/448 per tensor), bias N(0,0.1), ReLU, bf16 D."""
    return make_case("gemm8192_e4m3_bias_relu", 8192, 8192, 8192, seed=17, dist="normal",
                     ab_dtype="e4m3", bias_std=0.1, act="relu")


# ---------------------------------------------------------------- grouped GEMM

@dataclass
class GroupedCase:
    """A grouped GEMM: independent problems that share the operand type, the
    layouts, alpha, beta, the activation and the C / D / bias types; each has
    its own sizes, A, B, C, bias and D."""
    name: str
    problems: list

    @property
    def flops(self) -> int:
        return sum(p.flops for p in self.problems)


def make_grouped_case(name, shapes, *, seed, **kw) -> GroupedCase:
    """One make_case per (M, N, K) of `shapes`; problem g draws from seed * 1000 + g."""
    return GroupedCase(name, [make_case(f"{name}[{g}]", M, N, K, seed=seed * 1000 + g, **kw)
                              for g, (M, N, K) in enumerate(shapes)])


def moe_token_counts(tokens: int, experts: int, seed: int) -> list:
    """Rows routed to each expert: a seeded multinomial over Dirichlet(1) expert
    probabilities, so the counts are irregular (some small, none guaranteed
    to be a multiple of a tile)."""
    rng = np.random.default_rng(seed)
    return [int(c) for c in rng.multinomial(tokens, rng.dirichlet(np.ones(experts)))]


def grouped_moe(experts: int = 16, tokens: int = 32768, N: int = 4096, K: int = 4096,
                ab_dtype: str = "bf16") -> GroupedCase:
    """A mixture-of-experts layer as a grouped GEMM: `tokens` rows of activations
    routed over `experts` experts (moe_token_counts, seed 41), expert e an
    (M_e x K) @ (K x N) GEMM with its own weights; A, B ~ N(0,1)/sqrt(K) (bf16)
    or N(0,1) quantised per tensor (fp8), bias ~ N(0, 0.1), GELU, bf16 D,
    A row-major, B column-major."""
    counts = moe_token_counts(tokens, experts, seed=41)
    dist = "normal_sqrtk" if ab_dtype in ("bf16", "f16") else "normal"
    return make_grouped_case(f"grouped_moe{experts}_{tokens}x{N}x{K}_{ab_dtype}_bias_gelu",
                             [(m, N, K) for m in counts], seed=41, dist=dist, ab_dtype=ab_dtype,
                             bias_std=0.1, act="gelu")
