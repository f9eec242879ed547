"""CPU oracle for the GEMM path -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the cpu_baseline / reference
leg of ``bench.py`` may import this package.  The library never imports it and
shares no code with it.

The arithmetic lives in ``gemm_oracle.c`` (plain C, fp64, one output element at
a time, summed in increasing k); this module only compiles it with gcc and
marshals numpy arrays through ctypes.  What it computes is

    D_ref(i,j) = act(alpha*sA*sB * sum_k a(i,k) b(k,j) + beta*c(i,j) + bias(j))

the one-GEMM identity of the "CUTLASS" page (stanleyjacob.dev), Part I, with
the epilogue of its Part II (LinearCombination), Part IV Stage 5 (bias, GELU,
dequantisation scale) and Part VII Lab 4 (activation after alpha*AB + beta*C).
With block scale factors (Part V, block-scaled narrow formats) a(i,k) and
b(k,j) are first multiplied by the E8M0 scale of their block of `blk` k's.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gemm_oracle.c")
_OUT_DIR = os.path.join(_HERE, "_build")
_SO = os.path.join(_OUT_DIR, "libgemm_oracle.so")

ROW, COL = 0, 1
BF16, E4M3, F32, F16, E5M2, E2M1 = 0, 1, 2, 3, 4, 5
SF_E8M0, SF_UE4M3 = 0, 1
ACT = {"none": 0, "relu": 1, "gelu": 2}

_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile gemm_oracle.c with gcc (portable -O2, no -march, no fast-math)."""
    os.makedirs(_OUT_DIR, exist_ok=True)
    stale = (not os.path.exists(_SO)) or os.path.getmtime(_SO) < os.path.getmtime(_SRC)
    if force or stale:
        tmp = _SO + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fno-fast-math",
               "-ffp-contract=off", "-o", tmp, _SRC, "-lm", "-lpthread"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _SO)
    return _SO


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        lib = ctypes.CDLL(build())
        P = ctypes.c_void_p
        i32, i64, f64 = ctypes.c_int, ctypes.c_longlong, ctypes.c_double
        problem = [i32, i32, i32, f64, P, i64, i32, P, i64, i32, i32, f64,
                   P, i64, i32, P, i32, i32, f64, f64]
        lib.oracle_gemm_select.argtypes = problem + [P, i32, P, i32, P, i32]
        lib.oracle_gemm_select.restype = i64
        lib.oracle_gemm_full.argtypes = problem + [P, i32, i32, P, P]
        lib.oracle_gemm_full.restype = i64
        lib.oracle_decode_bf16_array.argtypes = [P, P, i64]
        lib.oracle_decode_e4m3_array.argtypes = [P, P, i64]
        lib.oracle_decode_f16_array.argtypes = [P, P, i64]
        lib.oracle_decode_e5m2_array.argtypes = [P, P, i64]
        lib.oracle_set_channel_scales.argtypes = [P, P]
        lib.oracle_set_channel_scales.restype = None
        lib.oracle_act_array.argtypes = [i32, P, P, i64]
        lib.oracle_decode_e8m0_array.argtypes = [P, P, i64]
        lib.oracle_set_block_scales.argtypes = [P, i64, P, i64, i32, i32]
        lib.oracle_decode_ue4m3_array.argtypes = [P, P, i64]
        lib.oracle_decode_e2m1_array.argtypes = [P, P, i64]
        lib.oracle_set_block_scales.restype = None
        _lib = lib
        return lib


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _storage(x, dtype=None):
    """Raw storage of an operand: uint16 (bf16 bits), uint8 (e4m3 bits) or float32;
    `dtype` (BF16 / E4M3 / F32 / F16 / E5M2) overrides the guess from the array type."""
    if x is None:
        return None, None
    x = np.ascontiguousarray(x)
    if dtype is not None:
        return x, int(dtype)
    if x.dtype == np.uint16:
        return x, BF16
    if x.dtype == np.uint8:
        return x, E4M3
    if x.dtype == np.float32:
        return x, F32
    raise TypeError(f"unsupported storage dtype {x.dtype}")


class Problem:
    """One GEMM problem over raw host storage.

    A is the logical M x K matrix, stored row-major (opA=ROW, element (i,k) at
    i*lda+k) or column-major (opA=COL, element (i,k) at k*lda+i); B is the
    logical K x N matrix with the same convention; C is row-major M x N.
    Storage arrays hold raw bits: uint16 = bf16, uint8 = e4m3, float32 = f32;
    ab_dtype=E2M1 reads packed FP4 (element e of the storage at byte e // 2,
    low nibble for even e; lda / ldb count elements).  Block scales: sfa[M][.],
    sfb[N][.], one per `block` consecutive k, E8M0 (sf_format=SF_E8M0) or
    unsigned E4M3 (SF_UE4M3) codes.
    """

    def __init__(self, M, N, K, A, lda, opA, B, ldb, opB, alpha=1.0, beta=0.0,
                 C=None, ldc=0, bias=None, act="none", scale_a=1.0, scale_b=1.0,
                 ab_dtype=None, c_dtype=None, bias_dtype=None, row_scale=None, col_scale=None,
                 sfa=None, sfb=None, block=32, sf_format=SF_E8M0):
        self.M, self.N, self.K = int(M), int(N), int(K)
        self.A, ab = _storage(A, ab_dtype)
        self.B, ab2 = _storage(B, ab_dtype)
        if ab is not None and ab2 is not None and ab != ab2:
            raise TypeError("A and B must share a storage type")
        self.ab_dtype = ab if ab is not None else BF16
        self.lda, self.ldb, self.opA, self.opB = int(lda), int(ldb), int(opA), int(opB)
        self.alpha, self.beta = float(alpha), float(beta)
        self.C, self.c_dtype = _storage(C, c_dtype)
        self.ldc = int(ldc)
        self.bias, self.bias_dtype = _storage(bias, bias_dtype)
        self.row_scale = None if row_scale is None else np.ascontiguousarray(row_scale, dtype=np.float32)
        self.col_scale = None if col_scale is None else np.ascontiguousarray(col_scale, dtype=np.float32)
        self.act = ACT[act] if isinstance(act, str) else int(act)
        # block scale factors: uint8 E8M0 codes, sfa[M][ceil(K/block)], sfb[N][ceil(K/block)]
        self.sfa = None if sfa is None else np.ascontiguousarray(sfa, dtype=np.uint8)
        self.sfb = None if sfb is None else np.ascontiguousarray(sfb, dtype=np.uint8)
        self.block = int(block)
        self.sf_format = int(sf_format)
        if (self.sfa is None) != (self.sfb is None):
            raise ValueError("block scales come in pairs (sfa and sfb)")
        self.scale_a, self.scale_b = float(scale_a), float(scale_b)

    def _args(self):
        return (self.M, self.N, self.K, self.alpha, _ptr(self.A), self.lda, self.opA,
                _ptr(self.B), self.ldb, self.opB, self.ab_dtype, self.beta,
                _ptr(self.C), self.ldc, self.c_dtype if self.c_dtype is not None else BF16,
                _ptr(self.bias), self.bias_dtype if self.bias_dtype is not None else BF16,
                self.act, self.scale_a, self.scale_b)

    def _scales(self):
        L = _load()
        L.oracle_set_channel_scales(_ptr(self.row_scale), _ptr(self.col_scale))
        if self.sfa is None:
            L.oracle_set_block_scales(None, 0, None, 0, 32, 0)
        else:
            L.oracle_set_block_scales(_ptr(self.sfa), self.sfa.shape[1], _ptr(self.sfb), self.sfb.shape[1],
                                      self.block, self.sf_format)

    def full(self, nthreads: int = 0) -> np.ndarray:
        out = np.empty((self.M, self.N), dtype=np.float64)
        self._scales()
        n = _load().oracle_gemm_full(*self._args(), _ptr(out), int(nthreads), 0, None, None)
        if n < 0:
            raise MemoryError("oracle allocation failed")
        return out

    def count_ops(self):
        """Run the full GEMM single-threaded with the per-operation counter on."""
        out = np.empty((self.M, self.N), dtype=np.float64)
        n_mul, n_add = ctypes.c_longlong(0), ctypes.c_longlong(0)
        self._scales()
        _load().oracle_gemm_full(*self._args(), _ptr(out), 1, 1,
                                 ctypes.byref(n_mul), ctypes.byref(n_add))
        return out, n_mul.value, n_add.value

    def select(self, rows, cols, nthreads: int = 0) -> np.ndarray:
        rows = np.ascontiguousarray(rows, dtype=np.int32)
        cols = np.ascontiguousarray(cols, dtype=np.int32)
        out = np.empty((rows.size, cols.size), dtype=np.float64)
        self._scales()
        n = _load().oracle_gemm_select(*self._args(), _ptr(rows), int(rows.size),
                                       _ptr(cols), int(cols.size), _ptr(out), int(nthreads))
        if n < 0:
            raise MemoryError("oracle allocation failed")
        return out


def grouped(problems) -> list:
    """A grouped GEMM: a batch of independent problems of different shapes,
    each computed by the one-GEMM identity above with its own operands,
    C, bias and output.  "CUTLASS" page, Part V (numeric-types deep dive):
    the experts of a mixture-of-experts layer run as one grouped GEMM, one
    problem per expert, the problems of different sizes; Part III: grouped
    GEMMs with irregular shapes.  Returns the full fp64 result of every
    problem, in order (an M == 0 or N == 0 problem gives an empty array)."""
    return [p.full() for p in problems]


def decode_bf16(bits: np.ndarray) -> np.ndarray:
    bits = np.ascontiguousarray(bits, dtype=np.uint16)
    out = np.empty(bits.shape, dtype=np.float64)
    _load().oracle_decode_bf16_array(_ptr(bits), _ptr(out), bits.size)
    return out


def decode_e4m3(bits: np.ndarray) -> np.ndarray:
    bits = np.ascontiguousarray(bits, dtype=np.uint8)
    out = np.empty(bits.shape, dtype=np.float64)
    _load().oracle_decode_e4m3_array(_ptr(bits), _ptr(out), bits.size)
    return out


def decode_f16(bits: np.ndarray) -> np.ndarray:
    bits = np.ascontiguousarray(bits, dtype=np.uint16)
    out = np.empty(bits.shape, dtype=np.float64)
    _load().oracle_decode_f16_array(_ptr(bits), _ptr(out), bits.size)
    return out


def decode_e5m2(bits: np.ndarray) -> np.ndarray:
    bits = np.ascontiguousarray(bits, dtype=np.uint8)
    out = np.empty(bits.shape, dtype=np.float64)
    _load().oracle_decode_e5m2_array(_ptr(bits), _ptr(out), bits.size)
    return out


def decode_e8m0(bits: np.ndarray) -> np.ndarray:
    bits = np.ascontiguousarray(bits, dtype=np.uint8)
    out = np.empty(bits.shape, dtype=np.float64)
    _load().oracle_decode_e8m0_array(_ptr(bits), _ptr(out), bits.size)
    return out


def decode_ue4m3(bits: np.ndarray) -> np.ndarray:
    bits = np.ascontiguousarray(bits, dtype=np.uint8)
    out = np.empty(bits.shape, dtype=np.float64)
    _load().oracle_decode_ue4m3_array(_ptr(bits), _ptr(out), bits.size)
    return out


def decode_e2m1(nibbles: np.ndarray) -> np.ndarray:
    nibbles = np.ascontiguousarray(nibbles, dtype=np.uint8)
    out = np.empty(nibbles.shape, dtype=np.float64)
    _load().oracle_decode_e2m1_array(_ptr(nibbles), _ptr(out), nibbles.size)
    return out


def act(name: str, x: np.ndarray) -> np.ndarray:
    x = np.ascontiguousarray(x, dtype=np.float64)
    out = np.empty_like(x)
    _load().oracle_act_array(ACT[name], _ptr(x), _ptr(out), x.size)
    return out
