"""The README's Python example runs as written (and its result is checked
against the oracle on a sample of rows)."""
import os
import re

import numpy as np
import pytest
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

pytestmark = pytest.mark.gpu


def test_readme_example_runs():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    from tiled_tensor_core_persistent_gb300 import _build
    _build.build()
    with open(os.path.join(ROOT, "README.md")) as f:
        blocks = re.findall(r"```python\n(.*?)```", f.read(), flags=re.S)
    assert blocks, "no python example in README.md"
    scope = {}
    exec(compile(blocks[0], "README.md", "exec"), scope)
    import oracle
    from tiled_tensor_core_persistent_gb300 import inputs
    A, B, bias, D, M, N, K = (scope[k] for k in ("A", "B", "bias", "D", "M", "N", "K"))
    rows = np.array([0, 1, 777, M - 1], dtype=np.int32)
    prob = oracle.Problem(M, N, K, inputs.raw_bits(A.cpu()), K, oracle.ROW, inputs.raw_bits(B.cpu()), K, oracle.COL,
                          bias=inputs.raw_bits(bias.cpu()), act="gelu")
    ref = prob.select(rows, np.arange(N, dtype=np.int32))
    got = D[torch.from_numpy(rows).long().cuda()].to(torch.float64).cpu().numpy()
    assert np.all(np.abs(got - ref) <= 1e-2 * np.maximum(1.0, np.abs(ref)))
