"""Failure detection without a GPU fault.

The failure is planted on the host: a test-only knob makes CTA 0's producer
skip its first stage (no loads, no arrival).  The MMA issuer's bounded wait
then runs out after a short limit, the kernel records TCG_ERR_TIMEOUT in the
workspace status word, drains its own copies, frees TMEM and returns.  The
host reads the status, and the context stays usable for the next GEMM.
"""
import numpy as np
import pytest
import torch

import tiled_tensor_core_persistent_gb300 as tcg
from tiled_tensor_core_persistent_gb300 import harness, inputs

from parity import oracle_for

pytestmark = pytest.mark.gpu

TIMEOUT = 7


@pytest.fixture(autouse=True)
def _reset():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    from tiled_tensor_core_persistent_gb300 import _build
    _build.build()
    tcg.debug_set()
    yield
    tcg.debug_set()


def test_bounded_wait_reports_timeout_and_context_survives():
    case = inputs.make_case("fault", 512, 512, 512, seed=141, dist="int4", d_dtype="f32")
    dc = harness.DeviceCase(case)
    tcg.debug_set(fault_inject=1, wait_timeout_ns=200_000_000)
    dc.run()
    assert tcg.device_status(dc.workspace) == TIMEOUT
    assert "ran out" in tcg.last_error()
    # status is cleared by the read
    assert tcg.device_status(dc.workspace) == 0
    tcg.debug_set()
    dc.run()
    torch.cuda.synchronize()
    assert tcg.device_status(dc.workspace) == 0
    assert np.array_equal(dc.result().numpy(), oracle_for(case).full())
