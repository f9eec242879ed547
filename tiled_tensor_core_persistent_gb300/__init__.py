"""GB300 (sm_103a) tiled tensor-core persistent GEMM -- Python binding.

Argument marshalling only: every step of the GEMM runs in the CUDA library
``libtcgemm.so`` (include/tcgemm.h) built in-tree from ``csrc/``.  There is no
CPU path: if the library is missing, every call raises.

    D = act(alpha * scale_a * scale_b * (A @ B) + beta * C + bias)

"CUTLASS" (stanleyjacob.dev), Part I (the GEMM identity), Part II (epilogue
functors, alignment), Part IV Stage 1 (workspace -> can_implement -> run).

Pointers may be given as ints (device addresses) or as torch tensors (their
data_ptr() is used); streams as ints (cudaStream_t) or torch.cuda.Stream.
"""
from __future__ import annotations

import ctypes
import os
import threading

from . import _build

ROW, COL = 0, 1
BF16, E4M3, F32, F16, E5M2, MXE4M3, MXE5M2, NVFP4, MXFP4 = 0, 1, 2, 3, 4, 5, 6, 7, 8
ACT_NONE, ACT_RELU, ACT_GELU = 0, 1, 2

DTYPES = {"bf16": BF16, "e4m3": E4M3, "f32": F32, "f16": F16, "e5m2": E5M2, "mxe4m3": MXE4M3,
          "mxe5m2": MXE5M2, "nvfp4": NVFP4, "mxfp4": MXFP4}
LAYOUTS = {"row": ROW, "col": COL}
ACTS = {"none": ACT_NONE, "relu": ACT_RELU, "gelu": ACT_GELU}

STATUS = {0: "TCG_OK", 1: "TCG_ERR_INVALID_ARG", 2: "TCG_ERR_UNSUPPORTED", 3: "TCG_ERR_MISALIGNED",
          4: "TCG_ERR_ARCH", 5: "TCG_ERR_WORKSPACE", 6: "TCG_ERR_LAUNCH", 7: "TCG_ERR_TIMEOUT",
          8: "TCG_ERR_CHECK"}

EXPORTED = ["tcg_can_implement", "tcg_workspace_size", "tcg_workspace_size_for", "tcg_workspace_init", "tcg_gemm",
            "tcg_device_status", "tcg_last_error", "tcg_plan", "tcg_debug_set", "tcg_gemm_noalloc",
            "tcg_debug_schedule", "tcg_grouped_workspace_size", "tcg_gemm_grouped", "tcg_grouped_plan",
            "tcg_debug_tma_swizzle128", "tcg_arch_status"]


class TcgError(RuntimeError):
    def __init__(self, code: int, where: str, detail: str = ""):
        self.code = code
        super().__init__(f"{where}: {STATUS.get(code, code)}" + (f" ({detail})" if detail else ""))


class Epilogue(ctypes.Structure):
    _fields_ = [("bias", ctypes.c_void_p), ("bias_dtype", ctypes.c_int), ("act", ctypes.c_int)]


class Scales(ctypes.Structure):
    _fields_ = [("scale_a", ctypes.c_float), ("scale_b", ctypes.c_float),
                ("row_scale", ctypes.c_void_p), ("col_scale", ctypes.c_void_p),
                ("block_sfa", ctypes.c_void_p), ("block_sfb", ctypes.c_void_p)]


class Problem(ctypes.Structure):
    """tcg_problem: one problem of a grouped GEMM."""
    _fields_ = [("M", ctypes.c_int), ("N", ctypes.c_int), ("K", ctypes.c_int), ("alpha", ctypes.c_float),
                ("A", ctypes.c_void_p), ("lda", ctypes.c_int), ("B", ctypes.c_void_p), ("ldb", ctypes.c_int),
                ("C", ctypes.c_void_p), ("ldc", ctypes.c_int), ("D", ctypes.c_void_p), ("ldd", ctypes.c_int),
                ("bias", ctypes.c_void_p)]


_lock = threading.Lock()
_lib = None


def library_path() -> str:
    """libtcgemm.so, or libtcgemm_debug.so (device-side checks) when TCG_DEBUG=1."""
    return _build.so_path()


def lib() -> ctypes.CDLL:
    """Load libtcgemm.so (it must have been built, e.g. by __graft_entry__.build())."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        path = library_path()
        if not os.path.exists(path):
            raise RuntimeError(f"{path} is missing: build it with __graft_entry__.build() "
                               "(there is no CPU fallback)")
        L = ctypes.CDLL(path)
        i32, sz, P, f32 = ctypes.c_int, ctypes.c_size_t, ctypes.c_void_p, ctypes.c_float
        L.tcg_can_implement.argtypes = [i32, i32, i32, i32, P, i32, i32, P, i32, i32, i32, P, i32, i32,
                                        P, i32, i32, Epilogue]
        L.tcg_can_implement.restype = i32
        L.tcg_arch_status.argtypes = [i32, i32]
        L.tcg_arch_status.restype = i32
        L.tcg_workspace_size.argtypes = [i32, i32, i32, i32]
        L.tcg_workspace_size.restype = sz
        L.tcg_workspace_size_for.argtypes = [i32, i32, i32, i32, P, i32, i32, P, i32, i32]
        L.tcg_workspace_size_for.restype = sz
        L.tcg_workspace_init.argtypes = [P, sz, P]
        L.tcg_workspace_init.restype = i32
        L.tcg_gemm.argtypes = [i32, i32, i32, f32, P, i32, i32, P, i32, i32, f32, P, i32, i32, P, i32, i32,
                               Epilogue, i32, Scales, P, sz, P]
        L.tcg_gemm.restype = i32
        L.tcg_gemm_noalloc.argtypes = [i32, i32, i32, f32, P, i32, i32, P, i32, i32, f32, P, i32, i32, P, i32,
                                       i32, Epilogue, i32, Scales, P]
        L.tcg_gemm_noalloc.restype = i32
        L.tcg_device_status.argtypes = [P, P]
        L.tcg_device_status.restype = i32
        L.tcg_last_error.argtypes = []
        L.tcg_last_error.restype = ctypes.c_char_p
        L.tcg_plan.argtypes = [i32, i32, i32, i32, i32, i32, ctypes.POINTER(ctypes.c_int)]
        L.tcg_plan.restype = i32
        L.tcg_debug_set.argtypes = [i32, ctypes.c_longlong, i32, i32]
        L.tcg_debug_set.restype = None
        L.tcg_debug_schedule.argtypes = [i32, i32, i32, i32, i32, i32, ctypes.POINTER(ctypes.c_int), i32]
        L.tcg_debug_schedule.restype = i32
        L.tcg_grouped_workspace_size.argtypes = [i32]
        L.tcg_grouped_workspace_size.restype = sz
        L.tcg_gemm_grouped.argtypes = [i32, ctypes.POINTER(Problem), i32, i32, f32, i32, i32, Epilogue, i32, P, sz,
                                       P]
        L.tcg_gemm_grouped.restype = i32
        L.tcg_grouped_plan.argtypes = [i32, ctypes.POINTER(Problem), i32, ctypes.POINTER(ctypes.c_int)]
        L.tcg_grouped_plan.restype = i32
        L.tcg_debug_tma_swizzle128.argtypes = [P, i32, P, P, P]
        L.tcg_debug_tma_swizzle128.restype = i32
        _lib = L
        return L


def _addr(x):
    if x is None:
        return None
    if isinstance(x, int):
        return x
    if hasattr(x, "data_ptr"):
        return x.data_ptr()
    raise TypeError(f"cannot take a device address of {type(x)}")


def _stream(s):
    if s is None:
        return None
    if isinstance(s, int):
        return s
    if hasattr(s, "cuda_stream"):
        return s.cuda_stream
    raise TypeError(f"cannot take a stream handle of {type(s)}")


def _enum(v, table):
    return table[v] if isinstance(v, str) else int(v)


def last_error() -> str:
    return lib().tcg_last_error().decode()


def can_implement(M, N, K, ab_dtype, A, lda, opA, B, ldb, opB, has_c, C, ldc, c_dtype, D, ldd, d_dtype,
                  bias=None, bias_dtype="bf16", act="none") -> int:
    epi = Epilogue(_addr(bias), _enum(bias_dtype, DTYPES), _enum(act, ACTS))
    return lib().tcg_can_implement(M, N, K, _enum(ab_dtype, DTYPES), _addr(A), lda, _enum(opA, LAYOUTS),
                                   _addr(B), ldb, _enum(opB, LAYOUTS), int(bool(has_c)), _addr(C), ldc,
                                   _enum(c_dtype, DTYPES), _addr(D), ldd, _enum(d_dtype, DTYPES), epi)


def arch_status(major: int, minor: int) -> int:
    return lib().tcg_arch_status(int(major), int(minor))


def workspace_size(M, N, K, ab_dtype="bf16") -> int:
    return int(lib().tcg_workspace_size(M, N, K, _enum(ab_dtype, DTYPES)))


def workspace_size_for(M, N, K, ab_dtype, A, lda, opA, B, ldb, opB) -> int:
    """Workspace bytes including packed copies of A/B that the TMA cannot address."""
    return int(lib().tcg_workspace_size_for(M, N, K, _enum(ab_dtype, DTYPES), _addr(A), lda,
                                            _enum(opA, LAYOUTS), _addr(B), ldb, _enum(opB, LAYOUTS)))


def workspace_init(workspace, nbytes, stream=None) -> None:
    st = lib().tcg_workspace_init(_addr(workspace), nbytes, _stream(stream))
    if st != 0:
        raise TcgError(st, "tcg_workspace_init", last_error())


def gemm(M, N, K, alpha, A, lda, opA, B, ldb, opB, beta, C, ldc, c_dtype, D, ldd, d_dtype, *,
         bias=None, bias_dtype="bf16", act="none", ab_dtype="bf16", scale_a=1.0, scale_b=1.0,
         row_scale=None, col_scale=None, block_sfa=None, block_sfb=None, workspace=None, workspace_bytes=0,
         stream=None) -> None:
    """Queue D = act(alpha*scale_a*scale_b*(A@B) + beta*C + bias) on `stream` (see tcgemm.h)."""
    epi = Epilogue(_addr(bias), _enum(bias_dtype, DTYPES), _enum(act, ACTS))
    st = lib().tcg_gemm(M, N, K, alpha, _addr(A), lda, _enum(opA, LAYOUTS), _addr(B), ldb,
                        _enum(opB, LAYOUTS), beta, _addr(C), ldc, _enum(c_dtype, DTYPES), _addr(D), ldd,
                        _enum(d_dtype, DTYPES), epi, _enum(ab_dtype, DTYPES),
                        Scales(scale_a, scale_b, _addr(row_scale), _addr(col_scale), _addr(block_sfa),
                               _addr(block_sfb)),
                        _addr(workspace), int(workspace_bytes), _stream(stream))
    if st != 0:
        raise TcgError(st, "tcg_gemm", last_error())


def gemm_noalloc(M, N, K, alpha, A, lda, opA, B, ldb, opB, beta, C, ldc, c_dtype, D, ldd, d_dtype, *,
                 bias=None, bias_dtype="bf16", act="none", ab_dtype="bf16", scale_a=1.0, scale_b=1.0,
                 row_scale=None, col_scale=None, block_sfa=None, block_sfb=None, stream=None) -> None:
    """tcg_gemm_noalloc: the same GEMM with the library's built-in device scratch (see tcgemm.h)."""
    epi = Epilogue(_addr(bias), _enum(bias_dtype, DTYPES), _enum(act, ACTS))
    st = lib().tcg_gemm_noalloc(M, N, K, alpha, _addr(A), lda, _enum(opA, LAYOUTS), _addr(B), ldb,
                                _enum(opB, LAYOUTS), beta, _addr(C), ldc, _enum(c_dtype, DTYPES), _addr(D),
                                ldd, _enum(d_dtype, DTYPES), epi, _enum(ab_dtype, DTYPES),
                                Scales(scale_a, scale_b, _addr(row_scale), _addr(col_scale), _addr(block_sfa),
                               _addr(block_sfb)), _stream(stream))
    if st != 0:
        raise TcgError(st, "tcg_gemm_noalloc", last_error())


def device_status(workspace, stream=None) -> int:
    """Synchronise, return and clear the workspace status word (0 = OK, 7 = timeout)."""
    return int(lib().tcg_device_status(_addr(workspace), _stream(stream)))


def plan(M, N, K, ab_dtype="bf16", opA="row", opB="col") -> dict:
    out = (ctypes.c_int * 11)()
    st = lib().tcg_plan(M, N, K, _enum(ab_dtype, DTYPES), _enum(opA, LAYOUTS), _enum(opB, LAYOUTS), out)
    if st != 0:
        raise TcgError(st, "tcg_plan", last_error())
    keys = ["BM", "BN", "BK", "stages", "splits", "grid", "cluster", "units", "group_m", "smem", "swap"]
    return dict(zip(keys, list(out)))


def debug_schedule(M, N, K, ab_dtype="bf16", num_sms=152, sk_mode=-1) -> list:
    """TEST-ONLY: the units of work tcg_gemm would run (see tcg_debug_schedule):
    a list of (worker, tile, m_blk, n_blk, kb0, kb1, split, nsplit, slot, half)."""
    L = lib()
    n = L.tcg_debug_schedule(M, N, K, _enum(ab_dtype, DTYPES), num_sms, sk_mode, None, 0)
    if n < 0:
        raise TcgError(1, "tcg_debug_schedule")
    buf = (ctypes.c_int * (10 * max(n, 1)))()
    L.tcg_debug_schedule(M, N, K, _enum(ab_dtype, DTYPES), num_sms, sk_mode, buf, n)
    return [tuple(buf[10 * i:10 * i + 10]) for i in range(n)]


def debug_set(fault_inject=0, wait_timeout_ns=0, force_splits=0, force_cta2=0) -> None:
    """TEST-ONLY knobs (see tcg_debug_set in tcgemm.h)."""
    lib().tcg_debug_set(int(fault_inject), int(wait_timeout_ns), int(force_splits), int(force_cta2))


def _problems(problems):
    """A tcg_problem array from dicts with keys M, N, K, alpha (default 1), A, lda, B, ldb, C, ldc,
    D, ldd, bias."""
    arr = (Problem * max(len(problems), 1))()
    for i, q in enumerate(problems):
        arr[i] = Problem(int(q["M"]), int(q["N"]), int(q["K"]), float(q.get("alpha", 1.0)), _addr(q.get("A")),
                         int(q.get("lda", 0)),
                         _addr(q.get("B")), int(q.get("ldb", 0)), _addr(q.get("C")), int(q.get("ldc", 0)),
                         _addr(q.get("D")), int(q.get("ldd", 0)), _addr(q.get("bias")))
    return arr


def grouped_workspace_size(num_problems: int) -> int:
    return int(lib().tcg_grouped_workspace_size(int(num_problems)))


def gemm_grouped(problems, opA, opB, beta, c_dtype, d_dtype, *, bias_dtype="bf16", act="none",
                 ab_dtype="bf16", workspace=None, workspace_bytes=0, stream=None) -> None:
    """Queue every problem of a grouped GEMM in one launch (tcg_gemm_grouped in tcgemm.h).
    problems: dicts with M, N, K, alpha, A, lda, B, ldb, C, ldc, D, ldd and bias (None allowed)."""
    arr = _problems(problems)
    epi = Epilogue(None, _enum(bias_dtype, DTYPES), _enum(act, ACTS))
    st = lib().tcg_gemm_grouped(len(problems), arr, _enum(opA, LAYOUTS), _enum(opB, LAYOUTS), beta,
                                _enum(c_dtype, DTYPES), _enum(d_dtype, DTYPES), epi, _enum(ab_dtype, DTYPES),
                                _addr(workspace), int(workspace_bytes), _stream(stream))
    if st != 0:
        raise TcgError(st, "tcg_gemm_grouped", last_error())


def grouped_plan(problems, ab_dtype="bf16") -> dict:
    out = (ctypes.c_int * 10)()
    st = lib().tcg_grouped_plan(len(problems), _problems(problems), _enum(ab_dtype, DTYPES), out)
    if st != 0:
        raise TcgError(st, "tcg_grouped_plan", last_error())
    keys = ["BM", "BN", "BK", "stages", "splits", "grid", "cluster", "units", "group_m", "smem"]
    return dict(zip(keys, list(out)))


def debug_tma_swizzle128(src, rows, dst, status, stream=None) -> None:
    """TEST-ONLY: one TMA load with 128-byte swizzling and back (tcg_debug_tma_swizzle128)."""
    st = lib().tcg_debug_tma_swizzle128(_addr(src), int(rows), _addr(dst), _addr(status), _stream(stream))
    if st != 0:
        raise TcgError(st, "tcg_debug_tma_swizzle128", last_error())
