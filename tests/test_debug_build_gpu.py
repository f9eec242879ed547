"""The debug build of the library (libtcgemm_debug.so, compiled with
TCG_DEBUG_CHECKS, loaded when TCG_DEBUG=1): the kernel checks its pipeline
bookkeeping on the device (stage, accumulator, epilogue-buffer, TMEM-column,
partial-slot and counter indices, the decoded units, and after every
mbarrier wait that the next phase is still open).  Every tile shape and
schedule runs clean under it, integer inputs stay exact, and a check failed
on purpose through the test knob (no invalid access: the check's condition is
forced false) ends the kernel with TCG_ERR_CHECK and leaves the context
usable.  Each run is a child process, since the library is chosen when it
loads.
"""
import os
import subprocess
import sys

import numpy as np
import pytest
import torch

import tiled_tensor_core_persistent_gb300 as tcg
from tiled_tensor_core_persistent_gb300 import harness, inputs

from parity import oracle_for

pytestmark = pytest.mark.gpu

HERE = os.path.dirname(os.path.abspath(__file__))

_CHILD = r"""
import sys, numpy as np, torch
sys.path.insert(0, {tests!r})
import tiled_tensor_core_persistent_gb300 as tcg
from tiled_tensor_core_persistent_gb300 import _build, harness, inputs
from parity import oracle_for
_build.build(debug=True)
assert tcg.library_path().endswith("libtcgemm_debug.so"), tcg.library_path()
tcg.lib()

def exact(case, force_cta2=0, force_splits=0, guard=1):
    tcg.debug_set(force_cta2=force_cta2, force_splits=force_splits)
    try:
        dc = harness.DeviceCase(case, guard_rows=guard)
        dc.run(); torch.cuda.synchronize()
        st = tcg.device_status(dc.workspace)
        assert st == 0, (case.name, st, tcg.last_error())
        assert np.array_equal(dc.result().numpy(), oracle_for(case).full()), case.name
        assert dc.untouched_outside(), case.name
        return dc
    finally:
        tcg.debug_set()

def int_case(name, M, N, K, seed, **kw):
    kw.setdefault("d_dtype", "f32")
    return inputs.make_case(name, M, N, K, seed=seed, dist="int4", **kw)

# one-CTA tiles, ragged edges, every layout
for opA, opB in inputs.LAYOUT_COMBOS:
    exact(int_case("one", 300, 520, 384, 1, opA=opA, opB=opB), force_cta2=2)
    exact(int_case("pair", 513, 700, 129, 2, opA=opA, opB=opB), force_cta2=1)
# narrow pair widths, several tiles per CTA (both accumulators reused)
exact(int_case("many", 2048 + 17, 2560, 300, 3, beta=0.5, c_dist="int4", c_dtype="f32"))
# split K (one-CTA tiles: round-robin and own-row-group fixups), skinny pairs, the transposed product
exact(int_case("split3", 300, 520, 1100, 4, opA="col", opB="row"), force_splits=3)
exact(int_case("split_m16", 16, 520, 1536, 5, opA="col"), force_splits=3)
exact(int_case("skinny_pair", 2000, 120, 3000, 6))
exact(int_case("swap", 16, 1000, 4096, 7, beta=0.5, c_dist="int4", c_dtype="f32"), force_cta2=5)
# 8-bit and block-scaled operands
exact(int_case("f8", 768, 1024, 1024, 8, ab_dtype="e4m3"), force_cta2=1)
exact(inputs.make_case("mx", 512, 512, 1024, seed=9, dist="int4", ab_dtype="e4m3", d_dtype="f32",
                       block_scaled=True, mx_scale_codes=(126, 128)), force_cta2=3)
exact(inputs.make_fp4_case("nv", 520, 700, 334, seed=10, fmt="nvfp4", dist="codes", code_range=list(range(16)),
                           scale_codes=[0x30, 0x34, 0x38, 0x3C, 0x40], d_dtype="f32"), force_cta2=3)
# a grouped GEMM
g = inputs.make_grouped_case("grp", [(200, 136, 72), (33, 264, 520), (0, 64, 64), (300, 256, 130)], seed=11,
                             dist="int4", d_dtype="f32")
gdc = harness.GroupedDeviceCase(g, guard_rows=1)
gdc.run(); torch.cuda.synchronize()
assert tcg.device_status(gdc.workspace) == 0, tcg.last_error()
for p, part in zip(g.problems, gdc.parts):
    assert np.array_equal(part.result().numpy(), oracle_for(p).full())

# a check failed on purpose: TCG_ERR_CHECK with code 199, then the same context computes exactly
case = int_case("forced", 512, 512, 512, 12)
dc = harness.DeviceCase(case)
tcg.debug_set(fault_inject=2, wait_timeout_ns=200_000_000)
dc.run(); torch.cuda.synchronize()
st = tcg.device_status(dc.workspace)
msg = tcg.last_error()
tcg.debug_set()
assert st == 8 and "199" in msg, (st, msg)
exact(case)
print("debug build ok")
"""


def run_child(extra_env=None):
    env = dict(os.environ, TCG_DEBUG="1", **(extra_env or {}))
    r = subprocess.run([sys.executable, "-c", _CHILD.format(tests=HERE)], env=env, capture_output=True, text=True,
                       timeout=1500, cwd=os.path.dirname(HERE))
    assert r.returncode == 0, r.stdout[-3000:] + r.stderr[-5000:]
    assert "debug build ok" in r.stdout


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    from tiled_tensor_core_persistent_gb300 import _build
    _build.build()


def test_debug_build_runs_every_tile_shape_clean_and_reports_a_forced_check():
    run_child()


def test_debug_build_with_stream_k_schedules():
    """Every tile of the launch in the Stream-K run (mode 3), so pieces of
    tiles cross CTA boundaries and each CTA owns two partial slots."""
    run_child({"TCG_SK": "3"})


def test_release_build_ignores_the_forced_check_knob():
    if _build_is_debug():
        pytest.skip("the debug library is loaded")
    case = inputs.make_case("forced_release", 256, 512, 256, seed=13, dist="int4", d_dtype="f32")
    dc = harness.DeviceCase(case)
    tcg.debug_set(fault_inject=2)
    try:
        dc.run()
        torch.cuda.synchronize()
        assert tcg.device_status(dc.workspace) == 0
    finally:
        tcg.debug_set()
    assert np.array_equal(dc.result().numpy(), oracle_for(case).full())


def _build_is_debug():
    return tcg.library_path().endswith("libtcgemm_debug.so")
