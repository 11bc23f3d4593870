"""Shared helpers of the GPU parity tests: move a seeded workload to the GPU,
run one append + decode step through the C ABI, read results back."""

from __future__ import annotations

import numpy as np
import torch

import paged_kv_cache_202_gb300 as pa

BF16_TOL = 1.5e-2   # max abs error, bf16 output
F32_TOL = 2e-3      # max abs error, float32 output


def to_dev(a: np.ndarray, dtype: str, dev="cuda") -> torch.Tensor:
    if dtype == "bf16":
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).to(dev)
    return torch.from_numpy(np.ascontiguousarray(a)).to(dev)


def bits(t: torch.Tensor) -> np.ndarray:
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).cpu().numpy().view(np.uint16)
    return t.cpu().numpy().view(np.uint32)


class DeviceStep:
    """One workload resident on the GPU."""

    def __init__(self, wl, dev="cuda"):
        self.wl = wl
        self.q = to_dev(wl.q, wl.dtype, dev)
        self.k_pool = to_dev(wl.k_pool, wl.dtype, dev)
        self.v_pool = to_dev(wl.v_pool, wl.dtype, dev)
        self.k_new = to_dev(wl.k_new, wl.dtype, dev)
        self.v_new = to_dev(wl.v_new, wl.dtype, dev)
        self.tables = torch.from_numpy(wl.block_tables).to(dev)
        self.seq_lens = torch.from_numpy(wl.seq_lens).to(dev)
        self.cache_lens = torch.from_numpy(wl.cache_lens).to(dev)
        out_dtype = torch.float32 if wl.dtype == "f32" else torch.bfloat16
        self.out = torch.full((wl.B, wl.Hq, wl.D), float("nan"), dtype=out_dtype, device=dev)

    def append(self):
        pa.pa_append_kv(self.k_new, self.v_new, self.k_pool, self.v_pool, self.tables,
                        self.cache_lens)

    def decode(self, plan: pa.Plan, max_seq_len: int | None = None, out=None):
        out = self.out if out is None else out
        pa.pa_decode(self.q, self.k_pool, self.v_pool, self.tables, self.seq_lens, self.wl.scale,
                     out, max_seq_len or self.wl.max_seq_len, plan)
        return out


def out_f64(t: torch.Tensor) -> np.ndarray:
    return t.float().cpu().numpy().astype(np.float64)


def tol(wl) -> float:
    return F32_TOL if wl.dtype == "f32" else BF16_TOL
