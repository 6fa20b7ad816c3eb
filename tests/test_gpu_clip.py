"""Global gradient-norm clipping across every shard and unit (the clipped
multi-unit step) against the oracle, through the C ABI."""
import math

import numpy as np
import pytest
import torch

import parity
from gpu_harness import bits, hp_at

import fsdp_sharded_mixed_flatten_gb300 as zf
from fsdp_sharded_mixed_flatten_gb300 import synthetic
from fsdp_sharded_mixed_flatten_gb300.buffers import FlatUnit

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from fsdp_sharded_mixed_flatten_gb300 import build
    build.build()
    zf.load()


class ClipRun:
    """Several units stepped with clipping on the GPU and in the oracle."""

    def __init__(self, specs, tag, n_micro=1, grad_std=1e-2, n_out=1):
        self.units, self.o_units = [], []
        self.n_micro, self.grad_std, self.tag = n_micro, grad_std, tag
        for i, (numels, n_ranks) in enumerate(specs):
            u = FlatUnit(numels, n_ranks, n_out=n_out, accum=True)
            master0 = synthetic.make_master_flat(u.P, n_ranks, 0.02, (tag, i))
            u.set_master_flat(master0.cuda())
            self.units.append(u)
            ms = master0.numpy().reshape(n_ranks, u.S).copy()
            self.o_units.append(dict(master=ms, m=np.zeros_like(ms), v=np.zeros_like(ms),
                                     accum=np.zeros_like(ms)))
        nbytes = zf.zero_clip_workspace_bytes(self.tuples(), n_micro)
        assert nbytes > 0
        self.workspace = torch.empty(max(nbytes // 8, 1), dtype=torch.float64, device="cuda")
        self.ws_bytes = nbytes
        self.norm = torch.zeros(1, dtype=torch.float32, device="cuda")
        self.o_params = [None] * len(self.units)
        self.o_norms = []

    def tuples(self):
        return [(u.grad_rows(), *u.state_rows(), u.accum_rows(), u.param_rows(), u.layout)
                for u in self.units]

    def step(self, oracle, t, max_norm, poison=None):
        """poison: (unit, rank, element, value) written into that gradient."""
        hp = hp_at(t)
        for k in range(1, self.n_micro + 1):
            for i, (u, ou) in enumerate(zip(self.units, self.o_units)):
                g = synthetic.make_grads(u.P, u.n_ranks, self.grad_std, (self.tag, i, t, k))
                if poison is not None and poison[0] == i:
                    g[poison[1], poison[2]] = poison[3]
                u.grads.copy_(g.cuda())
                ou["grads"] = bits(g)
            zf.zero_step_units_clip(self.tuples(), k, self.n_micro, hp, max_norm, self.workspace,
                                    self.ws_bytes, self.norm)
            outs, norm, coef = oracle.clipped_units_step(
                self.o_units, max_norm=max_norm, micro_step=k, n_micro=self.n_micro,
                lr=hp["lr"], beta1=hp["beta1"], beta2=hp["beta2"], eps=hp["eps"],
                weight_decay=hp["weight_decay"], step=t)
            if outs is not None:
                self.o_params = outs
                self.o_norms.append((norm, coef))
                torch.cuda.synchronize()
                got = float(self.norm.item())
                if poison is None:
                    assert abs(got - norm) <= 1e-6 * norm, (got, norm)

    def compare(self):
        torch.cuda.synchronize()
        for u, ou, op in zip(self.units, self.o_units, self.o_params):
            parity.check_state("master", u.master.cpu().numpy(), ou["master"])
            parity.check_state("m", u.m.cpu().numpy(), ou["m"])
            parity.check_state("v", u.v.cpu().numpy(), ou["v"])
            for o in range(u.params.shape[0]):
                pb = bits(u.params[o].cpu())
                parity.check_bf16(pb, op)
                parity.check_bf16_is_rounded_master(pb, u.master.cpu().numpy().reshape(-1))


SPECS = [([4099, 17], 4), ([100003], 8), ([64 * 77 + 3], 64), ([77777], 65), ([5], 8)]


def test_clipped_step_against_oracle(oracle):
    run = ClipRun(SPECS, "clip")
    # the total norm is ~ 1e-2 / sqrt(N_d) * sqrt(P): clip hard, then softly, then not at all
    for t, max_norm in ((1, 1e-2), (2, 0.2), (3, 1e3)):
        run.step(oracle, t, max_norm)
    assert run.o_norms[0][1] < 1.0 and run.o_norms[2][1] == 1.0
    run.compare()


def test_clipped_step_accumulation(oracle):
    run = ClipRun(SPECS[:3], "clip-acc", n_micro=3)
    run.step(oracle, 1, 5e-3)
    run.step(oracle, 2, 5e-3)
    assert all(c < 1.0 for _, c in run.o_norms)
    run.compare()


def test_clipped_many_units_several_norm_launches(oracle):
    """More units than one launch holds: the partial sums of several norm
    launches are reduced together."""
    specs = [([3000 + 41 * i], 64) for i in range(32)] + [([2000 + i], 3) for i in range(40)]
    run = ClipRun(specs, "clip-many")
    for t in (1, 2):
        run.step(oracle, t, 0.05)
    run.compare()


def test_no_clipping_equals_unclipped_step():
    """With a threshold above the norm the coefficient is exactly 1 and the
    clipped step equals zero_step_units bit for bit."""
    a = ClipRun(SPECS, "noclip")
    b_units = []
    for i, (numels, n_ranks) in enumerate(SPECS):
        u = FlatUnit(numels, n_ranks, accum=True)
        u.set_master_flat(synthetic.make_master_flat(u.P, n_ranks, 0.02, ("noclip", i)).cuda())
        b_units.append(u)
    for t in (1, 2):
        for i, (ua, ub) in enumerate(zip(a.units, b_units)):
            g = synthetic.make_grads(ua.P, ua.n_ranks, 1e-2, ("nc", i, t)).cuda()
            ua.grads.copy_(g)
            ub.grads.copy_(g)
        zf.zero_step_units_clip(a.tuples(), 1, 1, hp_at(t), 1e9, a.workspace, a.ws_bytes)
        zf.zero_step_units([(u.grad_rows(), *u.state_rows(), None, u.param_rows(), u.layout)
                            for u in b_units], 1, 1, hp_at(t))
    torch.cuda.synchronize()
    for ua, ub in zip(a.units, b_units):
        for x, y in ((ua.master, ub.master), (ua.m, ub.m), (ua.v, ub.v)):
            assert torch.equal(x.contiguous().view(torch.int32), y.contiguous().view(torch.int32))
        assert torch.equal(ua.params.contiguous().view(torch.int16),
                           ub.params.contiguous().view(torch.int16))


def test_averaged_gradient_left_in_accum(oracle):
    run = ClipRun(SPECS[:2], "clip-g")
    run.step(oracle, 1, 1e-3)
    torch.cuda.synchronize()
    for u, ou in zip(run.units, run.o_units):
        ref = oracle.reduce_scatter(ou["grads"]).reshape(-1)
        absmean = np.abs(((ou["grads"].astype(np.uint32) << 16).view(np.float32))).mean(axis=0)
        parity.check_mean(u.accum.cpu().numpy().reshape(-1), ref, absmean)


def test_workspace_too_small_rejected():
    run = ClipRun(SPECS[:2], "clip-ws")
    with pytest.raises(zf.ZeroError) as ei:
        zf.zero_step_units_clip(run.tuples(), 1, 1, hp_at(1), 1.0, run.workspace, 8)
    assert ei.value.code == -3
    with pytest.raises(zf.ZeroError) as ei:
        zf.zero_step_units_clip(run.tuples(), 1, 1, hp_at(1), -1.0, run.workspace, run.ws_bytes)
    assert ei.value.code == -1
    assert zf.zero_device_status() == zf.zero.ZERO_DEVICE_OK


@pytest.mark.parametrize("bad", ["nan", "inf"])
def test_nonfinite_gradient_shows_in_the_norm(oracle, bad):
    """A NaN or infinite gradient element makes the reported norm non-finite,
    the caller's signal to skip the step.  (The compensated rank sum turns an
    infinite value into NaN: its error term is inf - inf.)  With a NaN norm
    the coefficient is NaN and poisons every gradient, as in the oracle and in
    torch's clip_grad_norm_."""
    run = ClipRun(SPECS[:2], "nonfinite-" + bad)
    run.step(oracle, 1, 1.0, poison=(1, 3, 17, float(bad)))
    got = float(run.norm.item())
    assert math.isnan(got), got
    o_norm = run.o_norms[0][0]
    assert math.isnan(o_norm) if bad == "nan" else math.isinf(o_norm)
    if bad == "nan":
        for u, ou in zip(run.units, run.o_units):
            for name in ("master", "m", "v"):
                assert np.isnan(getattr(u, name).cpu().numpy()).all()
                assert np.isnan(ou[name]).all()
    assert zf.zero_device_status() == zf.zero.ZERO_DEVICE_OK
