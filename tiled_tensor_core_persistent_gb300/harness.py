"""Device plumbing for running a GemmCase through the C ABI.

torch provides device memory and streams only; the GEMM itself is the one
``tcg_gemm`` call.  Used by the tests, ``__graft_entry__.smoke()`` and
``bench.py``.
"""
from __future__ import annotations

import torch

from . import gemm, workspace_size, workspace_init
from .inputs import GemmCase

_TORCH_DTYPE = {"bf16": torch.bfloat16, "f32": torch.float32, "e4m3": torch.float8_e4m3fn}


class DeviceCase:
    """A GemmCase uploaded to the device, with D (optionally guarded) and a workspace.

    guard_rows > 0 allocates D with that many extra rows before and after the
    M x ldd block, filled with a sentinel, so tests can check nothing outside
    D's M x N window was written.
    """

    SENTINEL = 1234.5

    def __init__(self, case: GemmCase, device="cuda", guard_rows: int = 0, stream=None):
        self.case = case
        self.device = torch.device(device)
        self.stream = stream
        dev = self.device
        self.A = case.A.to(dev)
        self.B = case.B.to(dev)
        self.C = case.C.to(dev) if case.C is not None else None
        self.bias = case.bias.to(dev) if case.bias is not None else None
        self.row_scale = case.row_scale.to(dev) if case.row_scale is not None else None
        self.col_scale = case.col_scale.to(dev) if case.col_scale is not None else None
        ddt = _TORCH_DTYPE[case.d_dtype]
        self.guard_rows = guard_rows
        rows = max(case.M, 1) + 2 * guard_rows
        self.D_full = torch.full((rows, max(case.ldd, 1)), self.SENTINEL, dtype=ddt, device=dev)
        self.sentinel_stored = float(torch.tensor(self.SENTINEL, dtype=ddt).float())
        self.D_view = self.D_full[guard_rows:guard_rows + case.M]
        self.ws_bytes = max(workspace_size(case.M, case.N, case.K, case.ab_dtype), 256)
        self.workspace = torch.zeros(self.ws_bytes, dtype=torch.uint8, device=dev)

    def run(self, stream=None) -> None:
        c = self.case
        gemm(c.M, c.N, c.K, c.alpha, self.A, c.lda, c.opA, self.B, c.ldb, c.opB, c.beta, self.C,
             c.ldc, c.c_dtype, self.D_view, c.ldd, c.d_dtype, bias=self.bias,
             bias_dtype=c.bias_dtype, act=c.act, ab_dtype=c.ab_dtype, scale_a=c.scale_a,
             scale_b=c.scale_b, row_scale=self.row_scale, col_scale=self.col_scale,
             workspace=self.workspace, workspace_bytes=self.ws_bytes,
             stream=stream if stream is not None else self.stream)

    def result(self) -> torch.Tensor:
        """D's M x N window as float64 on the host."""
        return self.D_view[:, :self.case.N].to(torch.float64).cpu()

    def untouched_outside(self) -> bool:
        """True when every element outside the M x N window still holds the sentinel."""
        full = self.D_full.to(torch.float32).cpu()
        g, M, N = self.guard_rows, self.case.M, self.case.N
        mask = torch.ones_like(full, dtype=torch.bool)
        mask[g:g + M, :N] = False
        return bool((full[mask] == self.sentinel_stored).all())
