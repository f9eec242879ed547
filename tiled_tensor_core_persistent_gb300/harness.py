"""Device plumbing for running a GemmCase through the C ABI.

torch provides device memory and streams only; the GEMM itself is the one
``tcg_gemm`` call.  Used by the tests, ``__graft_entry__.smoke()`` and
``bench.py``.
"""
from __future__ import annotations

import torch

from . import gemm, gemm_grouped, grouped_workspace_size, workspace_size_for
from .inputs import GemmCase, GroupedCase

_TORCH_DTYPE = {"bf16": torch.bfloat16, "f32": torch.float32, "e4m3": torch.float8_e4m3fn}


class DeviceCase:
    """A GemmCase uploaded to the device, with D (optionally guarded) and a workspace.

    guard_rows > 0 allocates D with that many extra rows before and after the
    M x ldd block, filled with a sentinel, so tests can check nothing outside
    D's M x N window was written.
    """

    SENTINEL = 1234.5

    def __init__(self, case: GemmCase, device="cuda", guard_rows: int = 0, stream=None,
                 offsets: dict | None = None, with_workspace: bool = True):
        """offsets: element offsets {"A", "B", "C", "D", "bias"} of each buffer's
        start from a 256-byte aligned allocation (to exercise unaligned pointers)."""
        self.case = case
        self.device = torch.device(device)
        self.stream = stream
        dev = self.device
        off = offsets or {}
        self.A = _upload(case.A, dev, off.get("A", 0))
        self.B = _upload(case.B, dev, off.get("B", 0))
        self.C = _upload(case.C, dev, off.get("C", 0)) if case.C is not None else None
        self.bias = _upload(case.bias, dev, off.get("bias", 0)) if case.bias is not None else None
        # block-scaled operands: the library reads the E8M0 scales in its blocked layout
        fp4 = case.ab_dtype in ("nvfp4", "mxfp4")
        self.ab_dtype = case.ab_dtype if (case.sfa is None or fp4) else "mx" + case.ab_dtype
        self.sfa = self.sfb = None
        if case.sfa is not None:
            from .inputs import UE4M3_ONE, mx_blocked_layout
            pad = UE4M3_ONE if case.sf_format == "ue4m3" else 127
            self.sfa = torch.from_numpy(mx_blocked_layout(case.sfa, pad_code=pad)).to(dev)
            self.sfb = torch.from_numpy(mx_blocked_layout(case.sfb, pad_code=pad)).to(dev)
        self.row_scale = case.row_scale.to(dev) if case.row_scale is not None else None
        self.col_scale = case.col_scale.to(dev) if case.col_scale is not None else None
        ddt = _TORCH_DTYPE[case.d_dtype]
        self.guard_rows = guard_rows
        rows = max(case.M, 1) + 2 * guard_rows
        ld = max(case.ldd, 1)
        self.d_off = off.get("D", 0)
        self.D_flat = torch.full((self.d_off + rows * ld,), self.SENTINEL, dtype=ddt, device=dev)
        self.D_full = self.D_flat[self.d_off:].view(rows, ld)
        self.sentinel_stored = float(torch.tensor(self.SENTINEL, dtype=ddt).float())
        self.D_view = self.D_full[guard_rows:guard_rows + case.M]
        self.ws_bytes = 0
        self.workspace = None
        if with_workspace:
            self.ws_bytes = max(workspace_size_for(case.M, case.N, case.K, self.ab_dtype, self.A, case.lda,
                                                   case.opA, self.B, case.ldb, case.opB), 256)
            self.workspace = torch.zeros(self.ws_bytes, dtype=torch.uint8, device=dev)

    def run(self, stream=None) -> None:
        c = self.case
        gemm(c.M, c.N, c.K, c.alpha, self.A, c.lda, c.opA, self.B, c.ldb, c.opB, c.beta, self.C,
             c.ldc, c.c_dtype, self.D_view, c.ldd, c.d_dtype, bias=self.bias,
             bias_dtype=c.bias_dtype, act=c.act, ab_dtype=self.ab_dtype, scale_a=c.scale_a,
             scale_b=c.scale_b, row_scale=self.row_scale, col_scale=self.col_scale,
             block_sfa=self.sfa, block_sfb=self.sfb,
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
        head = self.D_flat[:self.d_off].to(torch.float32).cpu()
        return bool((full[mask] == self.sentinel_stored).all()) and bool((head == self.sentinel_stored).all())


class GroupedDeviceCase:
    """A GroupedCase uploaded to the device: each problem's buffers as in
    DeviceCase (without a workspace of its own), and one grouped workspace."""

    def __init__(self, case: GroupedCase, device="cuda", guard_rows: int = 0, stream=None):
        self.case = case
        self.stream = stream
        self.parts = [DeviceCase(p, device, guard_rows=guard_rows, with_workspace=False) for p in case.problems]
        self.ws_bytes = grouped_workspace_size(len(case.problems))
        self.workspace = torch.zeros(self.ws_bytes, dtype=torch.uint8, device=torch.device(device))
        first = case.problems[0]
        self.shared = dict(opA=first.opA, opB=first.opB, beta=first.beta, c_dtype=first.c_dtype,
                           d_dtype=first.d_dtype, bias_dtype=first.bias_dtype, act=first.act,
                           ab_dtype=first.ab_dtype)
        for p in case.problems:
            for k, v in self.shared.items():
                if getattr(p, k) != v:
                    raise ValueError(f"grouped problems must share {k}")
        self.problems = [dict(M=p.M, N=p.N, K=p.K, alpha=p.alpha * p.scale_a * p.scale_b, A=d.A, lda=p.lda,
                              B=d.B, ldb=p.ldb, C=d.C, ldc=p.ldc, D=d.D_view, ldd=p.ldd, bias=d.bias)
                         for p, d in zip(case.problems, self.parts)]

    def run(self, stream=None) -> None:
        sh = self.shared
        gemm_grouped(self.problems, sh["opA"], sh["opB"], sh["beta"], sh["c_dtype"], sh["d_dtype"],
                     bias_dtype=sh["bias_dtype"], act=sh["act"], ab_dtype=sh["ab_dtype"],
                     workspace=self.workspace, workspace_bytes=self.ws_bytes,
                     stream=stream if stream is not None else self.stream)


def _upload(t: torch.Tensor, dev, offset: int) -> torch.Tensor:
    """Copy t to the device starting `offset` elements into a fresh allocation."""
    if offset == 0:
        return t.to(dev)
    flat = torch.empty((offset + t.numel(),), dtype=t.dtype, device=dev)
    flat[offset:] = t.reshape(-1).to(dev)
    return flat[offset:].view(t.shape)
