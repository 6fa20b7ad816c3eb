"""Seeded synthetic workloads for the sharded mixed-precision step.

This module only describes shapes and draws seeded random inputs.  It holds
none of the method's arithmetic, so the CUDA path and the CPU oracle can both
be fed from it without sharing any computation.

Workloads (all synthetic; no dataset or checkpoint is involved):

* ``tiny``: 3 tensors 4096x1024, 1024, 1000 (P = 4,196,328), N_d = 4,
  grads N(0, 1e-2), 10 steps.
* ``gpt2-small``: 12 transformer blocks of d = 768 plus a root unit holding the
  50257x768 token embedding (tied with the output head, counted once), the
  1024x768 position embedding and the final LayerNorm: 13 FSDP units,
  124,439,808 parameters, N_d = 8, grads N(0, 1e-3), 10 steps.
* ``llama3-8b-layer``: one decoder layer (d = 4096, ffn = 14336, GQA with 32
  query and 8 key/value heads of width 128, two RMSNorm weights) as a single
  FlatParameter of 218,112,000 parameters, N_d = 64, grads N(0, 1e-3) with an
  independent 1 % of entries per rank scaled by 100, 5 steps.
* ``7.5b``: 7.5e9 parameters in 32 equal units of 234,375,000 (padded to
  234,375,040 for N_d = 64), grads N(0, 1e-3), optionally accumulated in fp32
  over 4 micro-steps.
* ``sweep``: flat sizes 4^k (k = 10..15) and 4^k + 13, N_d in {2, 8, 64},
  grads N(0, 1e-2).

Every workload draws fp32 master weights from N(0, 0.02) and starts with
m = v = 0.  Gradients are drawn in fp32 and rounded to bf16 by PyTorch; the
padded tail of every flat buffer is zero.
"""
from __future__ import annotations

import dataclasses
import hashlib
from typing import List, Sequence

import torch

BASE_SEED = 20261202

ADAMW_DEFAULTS = dict(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.01)


@dataclasses.dataclass(frozen=True)
class Unit:
    """One FSDP unit: its tensors' element counts in registration order, and
    optionally their shapes as (dim 0, elements per dim-0 row) -- what a
    per-parameter Shard(0) layout splits."""
    name: str
    numels: tuple
    shapes: tuple = ()

    @property
    def numel(self) -> int:
        return int(sum(self.numels))

    def rows(self):
        """(dim0, row_numel) of every tensor; a 1-D tensor is dim0 rows of 1."""
        if self.shapes:
            return list(self.shapes)
        return [(int(n), 1) for n in self.numels]


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    units: tuple
    n_ranks: int
    grad_std: float
    master_std: float = 0.02
    outlier_frac: float = 0.0
    outlier_scale: float = 100.0
    steps: int = 10
    n_micro: int = 1

    @property
    def numel(self) -> int:
        return sum(u.numel for u in self.units)


def _unit(name: str, shapes) -> Unit:
    return Unit(name, tuple(a * b for a, b in shapes), tuple(shapes))


def _gpt2_block(i: int, d: int = 768) -> Unit:
    # GPT-2's Conv1D weights are stored (in, out)
    return _unit(f"h.{i}", (
        (d, 1), (d, 1),                # ln_1 weight, bias
        (d, 3 * d), (3 * d, 1),        # attn.c_attn weight, bias
        (d, d), (d, 1),                # attn.c_proj weight, bias
        (d, 1), (d, 1),                # ln_2 weight, bias
        (d, 4 * d), (4 * d, 1),        # mlp.c_fc weight, bias
        (4 * d, d), (d, 1),            # mlp.c_proj weight, bias
    ))


def gpt2_small_units() -> List[Unit]:
    d = 768
    # wte (tied with the output head), wpe, ln_f weight and bias
    root = _unit("root", ((50257, d), (1024, d), (d, 1), (d, 1)))
    return [_gpt2_block(i, d) for i in range(12)] + [root]


def llama3_8b_layer_unit() -> Unit:
    d, ffn, kv = 4096, 14336, 8 * 128
    # nn.Linear weights are stored (out, in)
    return _unit("layer", (
        (d, d), (kv, d), (kv, d), (d, d),       # q, k, v, o projections
        (ffn, d), (ffn, d), (d, ffn),           # gate, up, down
        (d, 1), (d, 1),                         # input and post-attention RMSNorm
    ))


def tiny_unit() -> Unit:
    return Unit("tiny", (4096 * 1024, 1024, 1000))


def model_7p5b_units(n_units: int = 32) -> List[Unit]:
    per = 7_500_000_000 // n_units
    return [Unit(f"u{i}", (per,)) for i in range(n_units)]


def sweep_sizes() -> List[int]:
    out = []
    for k in range(10, 16):
        out += [4 ** k, 4 ** k + 13]
    return out


SWEEP_RANKS = (2, 8, 64)


def workload(name: str) -> Workload:
    if name == "tiny":
        return Workload("tiny", (tiny_unit(),), 4, 1e-2, steps=10)
    if name == "gpt2-small":
        return Workload("gpt2-small", tuple(gpt2_small_units()), 8, 1e-3, steps=10)
    if name == "llama3-8b-layer":
        return Workload("llama3-8b-layer", (llama3_8b_layer_unit(),), 64, 1e-3,
                        outlier_frac=0.01, outlier_scale=100.0, steps=5)
    if name == "7.5b":
        return Workload("7.5b", tuple(model_7p5b_units()), 64, 1e-3, steps=2)
    if name == "7.5b-accum":
        return Workload("7.5b-accum", tuple(model_7p5b_units()), 64, 1e-3, steps=2, n_micro=4)
    if name.startswith("sweep:"):
        # sweep:<P>:<N_d>
        _, p, n = name.split(":")
        return Workload(name, (Unit("flat", (int(p),)),), int(n), 1e-2, steps=3)
    raise KeyError(name)


def padded(numel: int, n_ranks: int) -> int:
    """Smallest multiple of n_ranks that holds numel (used to size buffers)."""
    return -(-numel // n_ranks) * n_ranks


def seed_for(*parts) -> int:
    """Deterministic 63-bit seed from any tuple of labels."""
    h = hashlib.sha256(repr((BASE_SEED,) + tuple(parts)).encode()).digest()
    return int.from_bytes(h[:8], "little") & ((1 << 63) - 1)


def _generator(device, seed: int) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def fill_grad_(buf: torch.Tensor, numel: int, std: float, seed: int, outlier_frac: float = 0.0,
               outlier_scale: float = 100.0, chunk: int = 1 << 28) -> torch.Tensor:
    """Fill a bf16 buffer: first ``numel`` entries N(0, std) (a fraction scaled
    by ``outlier_scale``), rounded to bf16 by PyTorch; the tail is zero.
    Drawn in chunks so that the fp32 temporaries stay small."""
    assert buf.dtype == torch.bfloat16 and buf.dim() == 1
    g = _generator(buf.device, seed)
    buf[numel:].zero_()
    for s in range(0, numel, chunk):
        e = min(numel, s + chunk)
        x = torch.randn(e - s, generator=g, device=buf.device, dtype=torch.float32)
        x.mul_(std)
        if outlier_frac > 0.0:
            mask = torch.rand(e - s, generator=g, device=buf.device) < outlier_frac
            x = torch.where(mask, x * outlier_scale, x)
        buf[s:e].copy_(x)
    return buf


def fill_normal_f32_(buf: torch.Tensor, std: float, seed: int, chunk: int = 1 << 28):
    assert buf.dtype == torch.float32 and buf.dim() == 1
    g = _generator(buf.device, seed)
    for s in range(0, buf.numel(), chunk):
        e = min(buf.numel(), s + chunk)
        buf[s:e].normal_(0.0, std, generator=g)
    return buf


def make_grads(numel: int, n_ranks: int, std: float, seed_parts: Sequence, device="cpu",
               outlier_frac: float = 0.0, outlier_scale: float = 100.0) -> torch.Tensor:
    """(n_ranks, P_pad) bf16: one full flat gradient buffer per logical rank."""
    P_pad = padded(numel, n_ranks)
    out = torch.empty((n_ranks, P_pad), dtype=torch.bfloat16, device=device)
    for k in range(n_ranks):
        fill_grad_(out[k], numel, std, seed_for(*seed_parts, "grad", k), outlier_frac,
                   outlier_scale)
    return out


def make_master_flat(numel: int, n_ranks: int, std: float, seed_parts: Sequence,
                     device="cpu") -> torch.Tensor:
    """(P_pad,) fp32 master weights of one flat parameter; the padded tail is 0."""
    P_pad = padded(numel, n_ranks)
    out = torch.zeros(P_pad, dtype=torch.float32, device=device)
    fill_normal_f32_(out[:numel], std, seed_for(*seed_parts, "master"))
    return out


def bf16_bits(t: torch.Tensor):
    """numpy uint16 view of a CPU bf16 tensor's bit patterns."""
    import numpy as np
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)
