"""Device buffers of one FSDP unit for N_d logical ranks held in one GPU.

PyTorch provides the memory; the layout is the library's.  Every per-rank
buffer starts on a 256-byte boundary (rows of a 2-D allocation whose row
stride is rounded up), as the C ABI requires 16-byte aligned pointers even
when the shard size S or the padded size P_pad is not a multiple of 8.

HBM layout of one unit (n = N_d):
  grads   bf16 (n, P_pad)  rank k's full flat gradient
  master  fp32 (n, S)      rank r's shard of the fp32 master weights
  m, v    fp32 (n, S)      rank r's Adam moments
  accum   fp32 (n, S)      optional micro-step accumulator
  params  bf16 (n_out, P_pad) all-gathered parameters
"""
from __future__ import annotations

from typing import List, Sequence

import torch

from .zero import ZeroLayout, zero_flat_layout, zero_param_layout, zero_shard_numel

ROW_ALIGN = 128   # elements: 256 B for bf16, 512 B for fp32


def _round_up(x: int, a: int) -> int:
    return -(-x // a) * a


def aligned_rows(n_rows: int, n_cols: int, dtype, device, fill=None) -> torch.Tensor:
    """(n_rows, n_cols) view into an allocation whose rows start 256-B aligned."""
    stride = _round_up(max(n_cols, 1), ROW_ALIGN)
    if fill is None:
        base = torch.empty((n_rows, stride), dtype=dtype, device=device)
    else:
        base = torch.full((n_rows, stride), fill, dtype=dtype, device=device)
    return base[:, :n_cols]


def rows(t: torch.Tensor) -> List[torch.Tensor]:
    return [t[i] for i in range(t.shape[0])]


class FlatUnit:
    """Buffers and layout of one FlatParameter over n_ranks logical ranks."""

    def __init__(self, numels: Sequence[int], n_ranks: int, n_out: int = 1, accum: bool = False,
                 device="cuda", with_grads: bool = True):
        self.numels = [int(x) for x in numels]
        self.offsets, self.layout = zero_flat_layout(self.numels, n_ranks)
        L: ZeroLayout = self.layout
        self.n_ranks = int(n_ranks)
        self.P = int(L.numel)
        self.P_pad = int(L.numel_padded)
        self.S = int(L.shard_numel)
        self.device = device
        self.grads = aligned_rows(n_ranks, self.P_pad, torch.bfloat16, device, 0) \
            if with_grads else None
        self.master = aligned_rows(n_ranks, self.S, torch.float32, device, 0)
        self.m = aligned_rows(n_ranks, self.S, torch.float32, device, 0)
        self.v = aligned_rows(n_ranks, self.S, torch.float32, device, 0)
        self.accum = aligned_rows(n_ranks, self.S, torch.float32, device, 0) if accum else None
        self.params = aligned_rows(n_out, self.P_pad, torch.bfloat16, device, 0)

    # pointer lists for the C ABI
    def grad_rows(self):
        return rows(self.grads)

    def state_rows(self):
        return rows(self.master), rows(self.m), rows(self.v)

    def accum_rows(self):
        return rows(self.accum) if self.accum is not None else None

    def param_rows(self):
        return rows(self.params)

    def set_master_flat(self, flat: torch.Tensor):
        """Copy a (P_pad,) fp32 flat master vector into the rank shards."""
        self.master.copy_(flat.reshape(self.n_ranks, self.S))

    def master_flat(self) -> torch.Tensor:
        return self.master.reshape(-1) if self.master.is_contiguous() else \
            self.master.contiguous().reshape(-1)

    def state_bytes(self) -> int:
        n = 3 + (1 if self.accum is not None else 0)
        return n * self.n_ranks * self.S * 4


class ParamUnit:
    """Buffers of one parameter under the per-parameter Shard(0) layout
    (FSDP2): no FlatParameter and no padding.  Rank k's gradient and the
    gathered parameter hold exactly numel elements; rank r's state holds its
    chunk of ceil(dim0 / N_d) rows (fewer, or none, at the end)."""

    def __init__(self, dim0: int, row: int, n_ranks: int, device="cuda"):
        self.layout = zero_param_layout(dim0, row, n_ranks)
        self.n_ranks = int(n_ranks)
        self.numel = int(dim0) * int(row)
        self.sizes = [zero_shard_numel(self.layout, r) for r in range(n_ranks)]
        self.grads = aligned_rows(n_ranks, self.numel, torch.bfloat16, device, 0)
        width = max(max(self.sizes), 1)
        self.master = aligned_rows(n_ranks, width, torch.float32, device, 0)
        self.m = aligned_rows(n_ranks, width, torch.float32, device, 0)
        self.v = aligned_rows(n_ranks, width, torch.float32, device, 0)
        self.accum = None
        self.params = aligned_rows(1, self.numel, torch.bfloat16, device, 0)

    def set_master_flat(self, flat: torch.Tensor):
        """Scatter a (numel,) fp32 vector into the rank shards."""
        off = 0
        for r, n in enumerate(self.sizes):
            self.master[r, :n].copy_(flat[off:off + n])
            off += n

    def unit_tuple(self):
        return (rows(self.grads), rows(self.master), rows(self.m), rows(self.v), None,
                rows(self.params), self.layout)
