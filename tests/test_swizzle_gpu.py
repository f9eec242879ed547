"""The TMA's 128-byte swizzle against the host model.

The pages explain shared-memory swizzling with a worked bank-conflict example
("CUTLASS" page, Part V deep dive on shared memory; pinned on the CPU in
test_analysis.py), but not the TMA's 128-byte pattern the GEMM kernel's
shared-memory descriptors assume.  Here one TMA load of a tile with distinct
random 16-byte chunks lands in 1024-byte-aligned shared memory and is copied
back byte for byte: byte o of the tile must sit at the model's offset
swizzle(o) = o XOR (((o >> 7) & 7) << 4) (the three row bits of each 1024-byte
group XORed into the 16-byte chunk index; analysis.swizzle with BBits=3,
MBase=4, SShift=3).
"""
import numpy as np
import pytest
import torch

import tiled_tensor_core_persistent_gb300 as tcg
from tiled_tensor_core_persistent_gb300 import analysis

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    from tiled_tensor_core_persistent_gb300 import _build
    _build.build()


@pytest.mark.parametrize("rows", [8, 24, 64])
def test_tma_128b_swizzle_matches_model(rows):
    rng = np.random.default_rng(rows)
    src = rng.integers(0, 256, size=rows * 128, dtype=np.uint8)
    d_src = torch.from_numpy(src).cuda()
    d_dst = torch.zeros(rows * 128, dtype=torch.uint8, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    tcg.debug_tma_swizzle128(d_src, rows, d_dst, status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    got = d_dst.cpu().numpy()
    expected = np.empty_like(src)
    for o in range(rows * 128):
        expected[analysis.swizzle(o, 3, 4, 3)] = src[o]
    assert np.array_equal(got, expected)
    # the layout really is permuted (rows 1..7 of every 8 move their chunks)
    assert not np.array_equal(got, src)
    # first row of every 1024-byte group is unchanged
    for r in range(0, rows, 8):
        assert np.array_equal(got[r * 128:(r + 1) * 128], src[r * 128:(r + 1) * 128])


def test_bad_arguments_are_refused():
    d = torch.zeros(64 * 128 + 16, dtype=torch.uint8, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    with pytest.raises(tcg.TcgError) as e:
        tcg.debug_tma_swizzle128(d, 65, d, status)
    assert e.value.code == 1
    with pytest.raises(tcg.TcgError) as e:
        tcg.debug_tma_swizzle128(d[1:], 8, d, status)
    assert e.value.code == 3
