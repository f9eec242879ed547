"""Concurrent use: several GEMMs in flight at once on different streams (each
with its own workspace), and host threads calling the library at the same time
(the descriptor cache and the planner's caches are shared, behind locks).  The
persistent kernels never wait on CTAs of another launch, so launches that share
the GPU only slow each other down."""
import threading

import numpy as np
import pytest
import torch

from tiled_tensor_core_persistent_gb300 import harness, inputs
import tiled_tensor_core_persistent_gb300 as tcg

from parity import oracle_for

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    from tiled_tensor_core_persistent_gb300 import _build
    _build.build()
    tcg.debug_set()


SHAPES = [(1000, 700, 300), (256, 2048, 512), (64, 1000, 2000), (900, 900, 96)]


def cases():
    return [inputs.make_case(f"conc{i}", M, N, K, seed=300 + i, dist="int4", d_dtype="f32", beta=0.5,
                             c_dist="int4", act="relu") for i, (M, N, K) in enumerate(SHAPES)]


def test_launches_in_flight_on_several_streams():
    cs = cases()
    streams = [torch.cuda.Stream() for _ in cs]
    dcs = [harness.DeviceCase(c, guard_rows=1, stream=s) for c, s in zip(cs, streams)]
    torch.cuda.synchronize()
    for _ in range(5):
        for dc, s in zip(dcs, streams):
            with torch.cuda.stream(s):
                dc.run(s)
    torch.cuda.synchronize()
    for c, dc in zip(cs, dcs):
        assert tcg.device_status(dc.workspace) == 0
        assert np.array_equal(dc.result().numpy(), oracle_for(c).full()), c.name
        assert dc.untouched_outside()


def test_host_threads_call_concurrently():
    cs = cases()
    dcs = [harness.DeviceCase(c, guard_rows=1, stream=torch.cuda.Stream()) for c in cs]
    torch.cuda.synchronize()
    errors = []

    def worker(dc):
        try:
            for _ in range(20):
                dc.run()
            dc.stream.synchronize()
        except Exception as e:   # reported below
            errors.append(e)

    threads = [threading.Thread(target=worker, args=(dc,)) for dc in dcs]
    for t in threads:
        t.start()
    for t in threads:
        t.join()
    assert not errors, errors
    torch.cuda.synchronize()
    for c, dc in zip(cs, dcs):
        assert tcg.device_status(dc.workspace) == 0
        assert np.array_equal(dc.result().numpy(), oracle_for(c).full()), c.name
