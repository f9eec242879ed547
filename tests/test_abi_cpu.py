"""The C-ABI library on a machine without a GPU: it loads, exports every
function include/tcgemm.h declares, and validates arguments (no launch)."""
import os
import re

import pytest

import tiled_tensor_core_persistent_gb300 as tcg
from tiled_tensor_core_persistent_gb300 import _build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    _build.build()
    return tcg.lib()


def declared_functions():
    with open(os.path.join(ROOT, "include", "tcgemm.h")) as f:
        text = f.read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(tcg_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_binding_surface():
    assert declared_functions() == sorted(tcg.EXPORTED)


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name


def declared_arities():
    """Parameter count of every function prototype in the header."""
    with open(os.path.join(ROOT, "include", "tcgemm.h")) as f:
        text = re.sub(r"/\*.*?\*/", "", f.read(), flags=re.S)
    out = {}
    for name, params in re.findall(r"\b(tcg_[a-z0-9_]+)\s*\(([^)]*)\)\s*;", text):
        params = params.strip()
        out[name] = 0 if params in ("", "void") else params.count(",") + 1
    return out


def test_binding_argument_lists_match_the_header(lib):
    """Every ctypes prototype of the binding takes as many arguments as the
    header's declaration (a stale argtypes list would pass a wrong stack)."""
    arities = declared_arities()
    assert set(arities) == set(declared_functions())
    for name, n in arities.items():
        argtypes = getattr(lib, name).argtypes
        assert argtypes is not None and len(argtypes) == n, (name, n, argtypes)


def test_exports_with_nm(lib):
    import subprocess
    out = subprocess.run(["nm", "-D", "--defined-only", tcg.library_path()], capture_output=True,
                         text=True).stdout
    for name in declared_functions():
        assert re.search(rf"\bT {name}$", out, flags=re.M), name


# Arguments of a valid 300 x 200 x 128 bf16 problem (fake, aligned addresses:
# can_implement never dereferences them).
A, B, C, D, BIAS = 0x10000, 0x20000, 0x30000, 0x40000, 0x50000


def ci(M=300, N=200, K=128, ab="bf16", A_=A, lda=128, opA="row", B_=B, ldb=128, opB="col", has_c=0,
       C_=C, ldc=200, c_dtype="bf16", D_=D, ldd=200, d_dtype="bf16", bias=None, bias_dtype="bf16",
       act="none"):
    return tcg.can_implement(M, N, K, ab, A_, lda, opA, B_, ldb, opB, has_c, C_, ldc, c_dtype, D_, ldd,
                             d_dtype, bias=bias, bias_dtype=bias_dtype, act=act)


def test_valid_problem_is_ok(lib):
    assert ci() == 0
    assert ci(opA="col", lda=304, opB="row", ldb=200) == 0
    assert ci(has_c=1, bias=BIAS, act="gelu") == 0
    assert ci(ab="e4m3", lda=128, ldb=128) == 0
    assert ci(ab="f16") == 0
    assert ci(ab="e5m2", lda=128, ldb=128) == 0
    assert ci(ab="f16", opA="col", lda=304, opB="row", ldb=200) == 0


def test_arch_rule_maps_only_sm103_to_ok(lib):
    """The architecture rule: compute capability 10.3 runs, everything else is
    TCG_ERR_ARCH (4), including the other Blackwell parts (10.0, 12.0) and
    Hopper (9.0)."""
    assert tcg.arch_status(10, 3) == 0
    for major, minor in [(10, 0), (10, 1), (10, 2), (10, 4), (11, 0), (12, 0), (12, 1), (9, 0), (8, 0),
                         (0, 0), (-1, 3), (103, 0)]:
        assert tcg.arch_status(major, minor) == 4, (major, minor)


def test_validation_without_a_device_checks_the_arguments_only(lib):
    """With no CUDA device in the process the architecture rule is skipped and
    a valid problem is OK (the argument rules still apply, see below)."""
    import torch
    if torch.cuda.is_available():
        pytest.skip("a CUDA device is present")
    assert ci() == 0
    assert ci(lda=100) == 1


def test_empty_problem_is_ok(lib):
    assert ci(M=0, D_=None) == 0
    assert ci(N=0, D_=None) == 0


def test_invalid_arguments(lib):
    INVALID = 1
    assert ci(M=-1) == INVALID
    assert ci(ab="f32") == INVALID
    assert ci(opA=5) == INVALID
    assert ci(D_=None) == INVALID
    assert ci(has_c=1, C_=None) == INVALID
    assert ci(A_=None) == INVALID
    assert ci(lda=64) == INVALID          # lda < K for row-major A
    assert ci(opA="col", lda=296) == INVALID  # lda < M for column-major A
    assert ci(ldd=192) == INVALID
    assert ci(act=9) == INVALID


def test_pointer_not_aligned_to_its_element_is_refused(lib):
    """The refusing branch of the CUTLASS page's alignment rule (Part II): a pointer
    that is not aligned to its element size cannot be served by any path."""
    MISALIGNED = 3
    assert ci(A_=A + 1) == MISALIGNED
    assert ci(B_=B + 1) == MISALIGNED
    assert ci(D_=D + 1) == MISALIGNED
    assert ci(D_=D + 2, d_dtype="f32") == MISALIGNED
    assert ci(bias=BIAS + 1) == MISALIGNED
    assert ci(bias=BIAS + 2, bias_dtype="f32") == MISALIGNED
    assert ci(has_c=1, C_=C + 1) == MISALIGNED
    assert ci(ab="e4m3", A_=A + 1, lda=128, ldb=128) == 0   # 1-byte elements: any address


def test_unaligned_leading_dimensions_take_the_slow_path(lib):
    """The other branch of the same rule: Lab 3's lda misaligned by one element is
    accepted; the operand is packed into the workspace, which grows by its size."""
    assert ci(lda=129) == 0
    assert ci(A_=A + 2) == 0
    assert ci(ldd=201) == 0
    assert ci(bias=BIAS + 4) == 0
    assert ci(has_c=1, ldc=201, c_dtype="bf16") == 0
    base = tcg.workspace_size(300, 200, 128)
    assert tcg.workspace_size_for(300, 200, 128, "bf16", A, 128, "row", B, 128, "col") == base
    # A row-major 300 x 128 with lda 129: the copy holds 300 rows of K = 128 elements
    pa = (300 * 128 * 2 + 255) // 256 * 256
    assert tcg.workspace_size_for(300, 200, 128, "bf16", A, 129, "row", B, 128, "col") == base + pa
    assert tcg.workspace_size_for(300, 200, 128, "bf16", A + 2, 128, "row", B, 128, "col") == base + pa
    # B column-major 128 x 200 stored as 200 rows of K = 128, ldb 131 -> 200 x 128
    pb = (200 * 128 * 2 + 255) // 256 * 256
    assert tcg.workspace_size_for(300, 200, 128, "bf16", A, 129, "row", B, 131, "col") == base + pa + pb
    # a ragged contiguous extent is padded to 16 bytes: K = 127 bf16 -> 128, e4m3 -> 128
    assert tcg.workspace_size_for(300, 200, 127, "bf16", A, 127, "row", B, 128, "col") == \
        tcg.workspace_size(300, 200, 127) + (300 * 128 * 2 + 255) // 256 * 256
    assert tcg.workspace_size_for(300, 200, 100, "e4m3", A, 101, "row", B, 112, "col") == \
        tcg.workspace_size(300, 200, 100, "e4m3") + (300 * 112 + 255) // 256 * 256


def test_unsupported_fp8_layouts(lib):
    assert ci(ab="e4m3", opA="col", lda=304) == 2
    assert ci(ab="e5m2", opB="row", ldb=208) == 2


def test_k_zero_needs_no_operands(lib):
    assert ci(K=0, A_=None, B_=None, lda=0, ldb=0) == 0


def test_workspace_size_without_device(lib):
    assert tcg.workspace_size(8192, 8192, 8192) >= 256
    assert tcg.workspace_size(-1, 4, 4) == 0


# ---------------------------------------------------------------- grouped GEMM

def grouped(lib, problems, ab="bf16", ws=0x60000, ws_bytes=1 << 20):
    arr = tcg._problems(problems)
    return lib.tcg_gemm_grouped(len(problems), arr, tcg.ROW, tcg.COL, 0.0, tcg.BF16, tcg.BF16,
                                tcg.Epilogue(None, tcg.BF16, tcg.ACT_NONE), tcg.DTYPES[ab], ws, ws_bytes, None)


def test_grouped_validation_without_device(lib):
    ok = dict(M=300, N=200, K=128, A=A, lda=128, B=B, ldb=128, D=D, ldd=200)
    assert lib.tcg_gemm_grouped(-1, None, 0, 1, 0.0, 0, 0, tcg.Epilogue(None, 0, 0), 0, None, 0, None) == 1
    assert grouped(lib, [ok, dict(ok, lda=100)]) == 1                 # lda < K in the second problem
    assert grouped(lib, [ok, dict(ok, lda=136, A=A + 2)]) == 2        # A not TMA-addressable: no slow path here
    assert grouped(lib, [ok, dict(ok, ldb=129)]) == 2
    assert grouped(lib, [ok], ab="mxe4m3") == 2                       # block-scaled types are not taken
    assert grouped(lib, [dict(ok, A=A + 1)]) == 3                     # not aligned to the element
    assert grouped(lib, [dict(ok, M=0), dict(ok, N=0)]) == 0          # nothing to compute
    assert grouped(lib, []) == 0
    # a valid request needs the device (none here)
    assert grouped(lib, [ok, dict(ok, M=1, K=0, A=None, B=None)]) in (4, 6)


def test_grouped_workspace_size(lib):
    sizes = [tcg.grouped_workspace_size(g) for g in (0, 1, 16, 1000)]
    assert all(s >= 256 and s % 256 == 0 for s in sizes)
    assert sizes == sorted(sizes) and sizes[-1] > sizes[1]
    assert tcg.grouped_workspace_size(-1) == 0


def test_header_compiles_as_c99_and_links(lib, tmp_path):
    """A plain C99 program includes tcgemm.h, links libtcgemm.so and runs the
    validation and sizing entry points (no GPU needed)."""
    import shutil
    import subprocess
    gcc = shutil.which("gcc")
    if gcc is None:
        pytest.skip("gcc not found")
    so = tcg.library_path()
    exe = tmp_path / "abi_check"
    src = os.path.join(ROOT, "tests", "c", "abi_check.c")
    r = subprocess.run([gcc, "-std=c99", "-Wall", "-Wextra", "-Werror", "-I", os.path.join(ROOT, "include"), src,
                        "-o", str(exe), so, f"-Wl,-rpath,{os.path.dirname(so)}"], capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    r = subprocess.run([str(exe)], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stdout + r.stderr
    assert "abi_check ok" in r.stdout


def test_debug_variant_builds_and_exports_the_same_symbols(lib):
    """libtcgemm_debug.so (the kernel's device-side checks compiled in) builds
    from the same sources and exports the same C ABI."""
    import subprocess
    path = _build.build(debug=True)
    assert path.endswith("libtcgemm_debug.so")

    def exported(p):
        out = subprocess.run(["nm", "-D", "--defined-only", p], capture_output=True, text=True).stdout
        return {m.group(1) for m in re.finditer(r"\bT (tcg_[a-z0-9_]+)$", out, flags=re.M)}

    assert exported(path) == exported(tcg.library_path()) == set(declared_functions())
