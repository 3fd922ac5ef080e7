"""GPU-side helpers for the parity tests: copy a gen.Problem to the device, run the
library through its Python binding (which calls the C ABI), return bf16 bit patterns."""
from __future__ import annotations

import numpy as np
import torch

import block_scaled_fp8_persistent_gb300 as bsfp8


class DeviceProblem:
    def __init__(self, p, c_rows_extra: int = 0, sentinel: int = 0x7FC1, c_offset: int = 0):
        dev = torch.device("cuda", 0)
        self.p = p
        self.A = torch.from_numpy(np.ascontiguousarray(p.A)).to(dev)
        self.B = torch.from_numpy(np.ascontiguousarray(p.B)).to(dev)
        self.sa = torch.from_numpy(np.ascontiguousarray(p.a_scales)).to(dev)
        self.sb = torch.from_numpy(np.ascontiguousarray(p.b_scales)).to(dev)
        self.off = torch.from_numpy(np.ascontiguousarray(p.offsets)).to(dev)
        ids = getattr(p, "expert_ids", None)
        self.ids = None if ids is None else torch.from_numpy(np.ascontiguousarray(ids)).to(dev)
        # C with optional guard rows after M_total, filled with a sentinel bit pattern, and
        # optionally starting c_offset bf16 elements into its allocation (c_offset = 8 makes
        # C 16-byte but not 32-byte aligned)
        rows = p.M_total + c_rows_extra
        flat = torch.full((c_offset + rows * p.N,), sentinel, dtype=torch.int16, device=dev)
        self.C_full = flat[c_offset:].view(rows, p.N).view(torch.bfloat16)
        self.C = self.C_full[: p.M_total]
        self.sentinel = sentinel

    def run(self, stream=None):
        p = self.p
        fmts = (getattr(p, "a_fmt", "mxfp8"), getattr(p, "b_fmt", "mxfp8"))
        if p.mode == "mx" and fmts != ("mxfp8", "mxfp8"):
            bsfp8.bsmx_grouped_gemm(*fmts, self.A, self.B, self.sa, self.sb, self.off, self.C,
                                    p.M_total, p.N, p.K, p.E, p.num_experts,
                                    expert_ids=self.ids, stream=stream)
            return
        if self.ids is not None:
            fn = (bsfp8.bsfp8_grouped_gemm_ids if p.mode == "blockwise"
                  else bsfp8.bsmxfp8_grouped_gemm_ids)
            fn(self.A, self.B, self.sa, self.sb, self.off, self.ids, self.C, p.M_total, p.N, p.K,
               p.E, p.num_experts, stream=stream)
            return
        fn = bsfp8.bsfp8_grouped_gemm if p.mode == "blockwise" else bsfp8.bsmxfp8_grouped_gemm
        fn(self.A, self.B, self.sa, self.sb, self.off, self.C, p.M_total, p.N, p.K, p.E,
           stream=stream)

    def c_bits(self) -> np.ndarray:
        torch.cuda.synchronize()
        return self.C.view(torch.int16).cpu().numpy().view(np.uint16)

    def guard_bits(self) -> np.ndarray:
        torch.cuda.synchronize()
        return self.C_full[self.p.M_total:].view(torch.int16).cpu().numpy().view(np.uint16)


def run_problem(p, **kw) -> np.ndarray:
    d = DeviceProblem(p, **kw)
    d.run()
    bits = d.c_bits()
    assert bsfp8.bsfp8_get_device_error() == 0
    return bits
