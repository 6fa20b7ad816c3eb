"""Full-size workloads in the launch configuration the benchmark times, with
sampled parity: the step is element-wise, so the oracle recomputes a chosen
set of flat elements exactly (every rank's gradient at those elements plus
the owning rank's state) and the GPU's results there must match within the
stated tolerances.  The sample always holds every shard boundary, the first
and last element, every tensor boundary and the whole padded tail.
"""
import gc

import numpy as np
import pytest
import torch

import parity
from gpu_harness import bits, hp_at

import fsdp_sharded_mixed_flatten_gb300 as zf
from fsdp_sharded_mixed_flatten_gb300 import synthetic
from fsdp_sharded_mixed_flatten_gb300.buffers import FlatUnit

pytestmark = [pytest.mark.gpu, pytest.mark.slow]


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from fsdp_sharded_mixed_flatten_gb300 import build
    build.build()
    zf.load()
    yield
    gc.collect()
    torch.cuda.empty_cache()


def sample_indices(unit: FlatUnit, n_random: int, seed: int) -> np.ndarray:
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


class SampledUnit:
    def __init__(self, numels, n_ranks, w, tag, n_micro, n_random=3000):
        self.unit = FlatUnit(numels, n_ranks, accum=n_micro > 1)
        self.w, self.tag, self.n_micro = w, tag, n_micro
        u = self.unit
        flat = synthetic.make_master_flat(u.P, n_ranks, w.master_std, (tag,), device="cuda")
        u.set_master_flat(flat)
        self.idx = sample_indices(u, n_random, synthetic.seed_for(tag) & 0xFFFF)
        self.idx_t = torch.from_numpy(self.idx).cuda()
        self.r_t, self.i_t = self.idx_t // u.S, self.idx_t % u.S
        self.o_master = flat[self.idx_t].cpu().numpy().copy()
        del flat
        self.o_m = np.zeros_like(self.o_master)
        self.o_v = np.zeros_like(self.o_master)
        self.o_acc = np.zeros_like(self.o_master) if n_micro > 1 else None
        self.o_params = None

    def step(self, oracle, t):
        u, w = self.unit, self.w
        hp = hp_at(t)
        for k in range(1, self.n_micro + 1):
            for r in range(u.n_ranks):
                synthetic.fill_grad_(u.grads[r], u.P, w.grad_std,
                                     synthetic.seed_for(self.tag, t, k, "grad", r),
                                     w.outlier_frac, w.outlier_scale)
            zf.zero_step(u.grad_rows(), *u.state_rows(), u.accum_rows(), k, self.n_micro,
                         u.param_rows(), u.layout, hp)
            g_at = bits(u.grads[:, self.idx_t].cpu())
            out = oracle.sampled_step(g_at, self.o_master, self.o_m, self.o_v,
                                      acc_at=self.o_acc, micro_step=k, n_micro=self.n_micro,
                                      lr=hp["lr"], beta1=hp["beta1"], beta2=hp["beta2"],
                                      eps=hp["eps"], weight_decay=hp["weight_decay"], step=t)
            if out is not None:
                self.o_params = out

    def compare(self):
        u = self.unit
        torch.cuda.synchronize()
        g_master = u.master[self.r_t, self.i_t].cpu().numpy()
        g_m = u.m[self.r_t, self.i_t].cpu().numpy()
        g_v = u.v[self.r_t, self.i_t].cpu().numpy()
        g_p = bits(u.params[0, self.idx_t].cpu())
        parity.check_state("master", g_master, self.o_master)
        parity.check_state("m", g_m, self.o_m)
        parity.check_state("v", g_v, self.o_v)
        parity.check_bf16(g_p, self.o_params)
        parity.check_bf16_is_rounded_master(g_p, g_master)
        pad = self.idx >= u.P
        assert np.all(g_p[pad] == 0) and np.all(g_master[pad] == 0)


def _run(oracle, w, units, steps, n_micro):
    for ui, unit in enumerate(units):
        s = SampledUnit(unit.numels, w.n_ranks, w, (w.name, unit.name), n_micro)
        for t in range(1, steps + 1):
            s.step(oracle, t)
        s.compare()
        del s
        gc.collect()
        torch.cuda.empty_cache()


def test_gpt2_small_13_units_10_steps(oracle):
    w = synthetic.workload("gpt2-small")
    _run(oracle, w, w.units, w.steps, 1)


def test_llama3_8b_layer_5_steps_outliers(oracle):
    w = synthetic.workload("llama3-8b-layer")
    _run(oracle, w, w.units, w.steps, 1)


def test_7p5b_unit_fp32_accumulation_4_micro_steps(oracle):
    """Full-size unit of the 7.5B model (P_pad = 234,375,040, N_d = 64, S = 3,662,110,
    S mod 8 = 6), fp32 accumulation over 4 micro-steps, 2 optimizer steps."""
    w = synthetic.workload("7.5b-accum")
    _run(oracle, w, w.units[:1], w.steps, 4)


def test_7p5b_unit_plain(oracle):
    w = synthetic.workload("7.5b")
    _run(oracle, w, w.units[-1:], w.steps, 1)


SWEEP = [(4 ** 10, 2), (4 ** 10 + 13, 64), (4 ** 12 + 13, 8), (4 ** 13, 64), (4 ** 14 + 13, 2),
         (4 ** 15 + 13, 64), (4 ** 15, 8)]


@pytest.mark.parametrize("P,n_ranks", SWEEP, ids=[f"P{p}_N{n}" for p, n in SWEEP])
def test_sweep_points(oracle, P, n_ranks):
    w = synthetic.workload(f"sweep:{P}:{n_ranks}")
    _run(oracle, w, w.units, 2, 1)


def test_beyond_2_pow_31_elements(oracle):
    """Flat indices above 2^31 (64-bit index arithmetic)."""
    w = synthetic.workload(f"sweep:{2 ** 31 + 13}:2")
    _run(oracle, w, w.units, 1, 1)
