"""Analytic performance models used to size tiles and to report rooflines.

* Arithmetic intensity of a GEMM boundary, ``2MNK / (b (MK + KN + MN))``: each
  input loaded once, the output written once, and the old output never read
  ("CuTe DSL and CUDA Tile", section "A tile is a plan for reuse").
* The square fp16-in / fp32-out GEMM intensity ``2N^3 / (2*2N^2 + 4N^2) = N/4``
  ("A10 CuTe, CUTLASS & CuTile", section 5 Performance Analysis).
* Roofline ``min(peak, intensity * bandwidth)`` and ridge ``peak / bandwidth``
  ("CUTLASS", Part V, the arithmetic-intensity deep dive).
* Ideal two-engine pipeline time ``L + C + (n - 1) max(L, C)``
  ("CuTe DSL and CUDA Tile", section "Pipelining hides a wait only when another
  resource can work").
* The XOR swizzle ``offset ^ ((offset & mask) >> shift)`` that spreads a column
  of a row-major tile over distinct shared-memory banks ("A10 CuTe, CUTLASS &
  CuTile", section 3.4 Swizzling).
"""
from __future__ import annotations


def boundary_intensity(M: int, N: int, K: int, bytes_per_element: float) -> float:
    """FLOP per byte when A, B are read once and D is written once."""
    return 2.0 * M * N * K / (bytes_per_element * (M * K + K * N + M * N))


def gemm_bytes(M: int, N: int, K: int, ab_bytes: float, d_bytes: float, c_bytes: float = 0.0,
               bias_bytes: float = 0.0) -> float:
    """Algorithmic bytes of one GEMM launch with the actual element sizes."""
    return ab_bytes * (M * K + K * N) + d_bytes * M * N + c_bytes * M * N + bias_bytes * N


def square_gemm_intensity_mixed(N: int, in_bytes: int = 2, out_bytes: int = 4) -> float:
    """2N^3 FLOP over two N x N inputs of in_bytes and one N x N output of out_bytes."""
    return 2.0 * N ** 3 / (2 * N * N * in_bytes + N * N * out_bytes)


def double_buffer_bytes(Mt: int, Nt: int, Kt: int, bytes_per_element: int) -> int:
    """Shared memory for two stages of an Mt x Kt A tile and a Kt x Nt B tile."""
    return 2 * bytes_per_element * (Mt * Kt + Kt * Nt)


def roofline(peak_flops: float, intensity: float, bandwidth: float) -> float:
    return min(peak_flops, intensity * bandwidth)


def ridge_point(peak_flops: float, bandwidth: float) -> float:
    return peak_flops / bandwidth


def pipeline_time(n: int, load: float, compute: float) -> float:
    """n independent tiles with a single loader and a single arithmetic unit that overlap perfectly."""
    if n <= 0:
        return 0.0
    return load + compute + (n - 1) * max(load, compute)


def serial_time(n: int, load: float, compute: float) -> float:
    return n * (load + compute)


def swizzle(offset: int, bbits: int, mbase: int, sshift: int) -> int:
    """XOR the BBits-wide field at bit (MBase + SShift) into the field at MBase."""
    yyy_mask = ((1 << bbits) - 1) << (mbase + sshift)
    return offset ^ ((offset & yyy_mask) >> sshift)


def bank(offset_elems: int, element_bytes: int = 4, banks: int = 32, bank_bytes: int = 4) -> int:
    return (offset_elems * element_bytes // bank_bytes) % banks
