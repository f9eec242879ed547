"""tcg_gemm inside a CUDA graph: captured once, replayed many times.

Launch-bound problems (512^3 takes ~10 us) are where a caller replays a
captured graph instead of calling the library each time.  The first call on
a device (which sets kernel attributes and queries the device) is made before
the capture; the captured call then records only its kernel launches, and the
replays read the buffers' current contents.  Split K, whose per-tile arrival
counters are reset by the kernel itself, must give the same result on every
replay.
"""
import numpy as np
import pytest
import torch

from tiled_tensor_core_persistent_gb300 import harness, inputs
import tiled_tensor_core_persistent_gb300 as tcg

from parity import TOL, assert_within, oracle_for

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    from tiled_tensor_core_persistent_gb300 import _build
    _build.build()
    tcg.debug_set()
    yield
    tcg.debug_set()


def capture(dc):
    stream = torch.cuda.Stream()
    with torch.cuda.stream(stream):
        dc.run(stream)          # first call outside the capture
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        dc.run(torch.cuda.current_stream())
    torch.cuda.synchronize()
    return graph


def test_graph_replay_reads_current_inputs():
    case = inputs.make_case("graph", 512, 512, 512, seed=201, dist="uniform", bias_std=0.1, act="gelu",
                            beta=0.5, c_dist="uniform")
    dc = harness.DeviceCase(case)
    graph = capture(dc)
    dc.D_view.zero_()
    graph.replay()
    torch.cuda.synchronize()
    assert_within(dc.result().numpy(), oracle_for(case).full(), TOL["bf16"], "replay 1")
    # new inputs in the same buffers: the replay must see them
    case2 = inputs.make_case("graph2", 512, 512, 512, seed=202, dist="uniform", bias_std=0.1, act="gelu",
                             beta=0.5, c_dist="uniform")
    dc.A.copy_(case2.A)
    dc.B.copy_(case2.B)
    dc.C.copy_(case2.C)
    dc.bias.copy_(case2.bias)
    for _ in range(3):
        graph.replay()
    torch.cuda.synchronize()
    assert_within(dc.result().numpy(), oracle_for(case2).full(), TOL["bf16"], "replay 2")
    assert tcg.device_status(dc.workspace) == 0


def test_graph_replay_split_k_is_repeatable():
    tcg.debug_set(force_splits=4)
    try:
        case = inputs.make_case("graph_split", 200, 300, 2048, seed=203, dist="int4", d_dtype="f32")
        dc = harness.DeviceCase(case)
        graph = capture(dc)
        ref = oracle_for(case).full()
        for _ in range(5):
            dc.D_view.zero_()
            graph.replay()
            torch.cuda.synchronize()
            assert np.array_equal(dc.result().numpy(), ref)
        assert tcg.device_status(dc.workspace) == 0
    finally:
        tcg.debug_set()
