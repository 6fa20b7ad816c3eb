"""Drive the CUDA path and the oracle on the same seeded inputs.

Inputs come from fsdp_sharded_mixed_flatten_gb300.synthetic (no method
arithmetic); the GPU side goes through the C ABI binding, the reference
side through the oracle.  Used by the GPU parity tests and by the smoke check.
"""
from __future__ import annotations

import numpy as np
import torch

from fsdp_sharded_mixed_flatten_gb300 import (zero_adamw_shard_step, zero_all_gather,
                                              zero_reduce_scatter, zero_step)
from fsdp_sharded_mixed_flatten_gb300 import synthetic
from fsdp_sharded_mixed_flatten_gb300.buffers import FlatUnit, aligned_rows, rows

HP = dict(synthetic.ADAMW_DEFAULTS)


def hp_at(step, **over):
    d = dict(HP, step=int(step))
    d.update(over)
    return d


def bits(t: torch.Tensor) -> np.ndarray:
    return synthetic.bf16_bits(t)


class Case:
    """One FlatParameter stepped on the GPU and in the oracle side by side."""

    def __init__(self, numels, n_ranks, *, n_out=1, n_micro=1, grad_std=1e-2, tag="case",
                 path="fused", outlier_frac=0.0, hp_over=None):
        self.numels = list(numels)
        self.n_ranks = n_ranks
        self.n_micro = n_micro
        self.grad_std = grad_std
        self.tag = tag
        self.path = path
        self.outlier_frac = outlier_frac
        self.hp_over = hp_over or {}
        self.unit = FlatUnit(self.numels, n_ranks, n_out=n_out, accum=n_micro > 1 or path != "fused")
        u = self.unit
        self.P, self.P_pad, self.S = u.P, u.P_pad, u.S
        master0 = synthetic.make_master_flat(self.P, n_ranks, 0.02, (tag,))
        u.set_master_flat(master0.cuda())
        self.o_master = master0.numpy().reshape(n_ranks, self.S).copy()
        self.o_m = np.zeros_like(self.o_master)
        self.o_v = np.zeros_like(self.o_master)
        self.o_acc = np.zeros_like(self.o_master) if n_micro > 1 else None
        self.o_params = None
        if path != "fused":
            self.param_shards = aligned_rows(n_ranks, self.S, torch.bfloat16, "cuda", 0)
        self.last_grads = None

    def grads_for(self, step, micro):
        return synthetic.make_grads(self.P, self.n_ranks, self.grad_std,
                                    (self.tag, step, micro), outlier_frac=self.outlier_frac)

    def step(self, oracle, t):
        u = self.unit
        hp = hp_at(t, **self.hp_over)
        for k in range(1, self.n_micro + 1):
            g = self.grads_for(t, k)
            self.last_grads = g
            u.grads.copy_(g.cuda())
            self._gpu_micro(k, hp)
            out = oracle.zero_step(bits(g), self.o_master, self.o_m, self.o_v,
                                   accum=self.o_acc, micro_step=k, n_micro=self.n_micro,
                                   lr=hp["lr"], beta1=hp["beta1"], beta2=hp["beta2"],
                                   eps=hp["eps"], weight_decay=hp["weight_decay"], step=t)
            if out is not None:
                self.o_params = out

    def _gpu_micro(self, k, hp):
        u = self.unit
        K = self.n_micro
        master, m, v = u.state_rows()
        if self.path == "fused":
            zero_step(u.grad_rows(), master, m, v, u.accum_rows() if K > 1 else None, k, K,
                      u.param_rows(), u.layout, hp)
            return
        # unfused: reduce-scatter (into the accumulator), AdamW on shards, all-gather
        zero_reduce_scatter(u.grad_rows(), u.accum_rows(), u.layout, 1 if k > 1 else 0)
        if k == K:
            zero_adamw_shard_step(master, m, v, u.accum_rows(), float(K), rows(self.param_shards),
                                  u.layout, hp)
            zero_all_gather(rows(self.param_shards), u.param_rows(), u.layout)

    def gpu_state(self):
        torch.cuda.synchronize()
        u = self.unit
        return (u.master.cpu().numpy(), u.m.cpu().numpy(), u.v.cpu().numpy(),
                bits(u.params.cpu()))

    def compare(self):
        import parity
        g_master, g_m, g_v, g_params = self.gpu_state()
        parity.check_state("master", g_master, self.o_master)
        parity.check_state("m", g_m, self.o_m)
        parity.check_state("v", g_v, self.o_v)
        flat_master = g_master.reshape(-1)
        for o in range(g_params.shape[0]):
            parity.check_bf16(g_params[o], self.o_params)
            parity.check_bf16_is_rounded_master(g_params[o], flat_master)
        assert np.all(g_params[:, self.P:] == 0), "padding of the parameters is not zero"
        assert np.all(g_master.reshape(-1)[self.P:] == 0) if self.P_pad > self.P else True


def sample_indices(unit: FlatUnit, n_random: int, seed: int) -> np.ndarray:
    """Flat indices of a unit the oracle follows in the full-size tests: random
    ones plus every shard boundary, the first and last element, every tensor
    boundary and the whole padded tail."""
    rng = np.random.default_rng(seed)
    S, P, P_pad = unit.S, unit.P, unit.P_pad
    idx = set(rng.integers(0, P, size=n_random).tolist())
    for r in range(unit.n_ranks):
        for d in (0, 1, 2, 7, 8, S - 2, S - 1):
            if 0 <= d < S:
                idx.add(r * S + d)
    for off, n in zip(unit.offsets, unit.numels):
        for e in (off - 1, off, off + n - 1):
            if 0 <= e < P_pad:
                idx.add(e)
    idx.update(range(P, P_pad))
    idx.update((0, P - 1))
    return np.array(sorted(idx), dtype=np.int64)


class Sample:
    """The oracle's copy of one unit's state at sampled flat indices (the step
    is element-wise, so these elements can be followed exactly)."""

    def __init__(self, unit: FlatUnit, idx: np.ndarray, master_flat: torch.Tensor, n_micro=1):
        self.unit = unit
        self.idx = idx
        self.idx_t = torch.from_numpy(idx).to(master_flat.device)
        self.r_t, self.i_t = self.idx_t // unit.S, self.idx_t % unit.S
        self.master = master_flat[self.idx_t].cpu().numpy().copy()
        self.m = np.zeros_like(self.master)
        self.v = np.zeros_like(self.master)
        self.acc = np.zeros_like(self.master) if n_micro > 1 else None
        self.params = None

    def grads_at(self) -> np.ndarray:
        """Every rank's gradient at the sampled indices, (n_ranks, n) bf16 bits."""
        return bits(self.unit.grads[:, self.idx_t].cpu())

    def gpu_state(self):
        u = self.unit
        return (u.master[self.r_t, self.i_t].cpu().numpy(), u.m[self.r_t, self.i_t].cpu().numpy(),
                u.v[self.r_t, self.i_t].cpu().numpy(), bits(u.params[0, self.idx_t].cpu()))

    def compare(self):
        import parity
        g_master, g_m, g_v, g_p = self.gpu_state()
        parity.check_state("master", g_master, self.master)
        parity.check_state("m", g_m, self.m)
        parity.check_state("v", g_v, self.v)
        parity.check_bf16(g_p, self.params)
        parity.check_bf16_is_rounded_master(g_p, g_master)
        pad = self.idx >= self.unit.P
        assert np.all(g_p[pad] == 0) and np.all(g_master[pad] == 0)
