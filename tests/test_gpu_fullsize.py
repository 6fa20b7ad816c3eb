"""Full-size workloads in the launch configuration the benchmark times, with
sampled parity: every unit of a model is stepped by one zero_step_units call
per micro-step (the library packs the units into launches exactly as in the
benchmark), and the oracle recomputes a chosen set of flat elements of every
unit exactly (the step is element-wise: every rank's gradient at those
elements plus the owning rank's state).  The GPU's results there must match
within the stated tolerances.  The sample always holds every shard boundary,
the first and last element, every tensor boundary and the whole padded tail.
"""
import gc

import numpy as np
import pytest
import torch

from gpu_harness import Sample, hp_at, sample_indices

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


class SampledModel:
    """Units of a workload on the GPU, the oracle following a sample of each.
    shared_grads: one gradient buffer read by every unit (the 7.5B model streams
    its gradients unit by unit through one buffer, as the benchmark does)."""

    def __init__(self, w, units, tag, n_micro, shared_grads=False, n_random=3000):
        self.w, self.tag, self.n_micro, self.shared = w, tag, n_micro, shared_grads
        self.units, self.samples = [], []
        first = None
        for unit in units:
            fu = FlatUnit(unit.numels, w.n_ranks, accum=n_micro > 1,
                          with_grads=not (shared_grads and first is not None))
            if shared_grads:
                if first is None:
                    first = fu.grads
                else:
                    fu.grads = first
            flat = synthetic.make_master_flat(fu.P, w.n_ranks, w.master_std, (tag, unit.name),
                                              device="cuda")
            fu.set_master_flat(flat)
            idx = sample_indices(fu, n_random, synthetic.seed_for(tag, unit.name) & 0xFFFF)
            self.samples.append(Sample(fu, idx, flat, n_micro))
            del flat
            self.units.append(fu)
        self.names = [u.name for u in units]
        self.prepared = zf.zero.prepare_units(
            [(fu.grad_rows(), *fu.state_rows(), fu.accum_rows(), fu.param_rows(), fu.layout)
             for fu in self.units])

    def fill(self, t, k):
        w = self.w
        for fu, name in zip(self.units, self.names):
            for r in range(fu.n_ranks):
                synthetic.fill_grad_(fu.grads[r], fu.P, w.grad_std,
                                     synthetic.seed_for(self.tag, name, t, k, "grad", r),
                                     w.outlier_frac, w.outlier_scale)
            if self.shared:
                return

    def step(self, oracle, t):
        hp = hp_at(t)
        for k in range(1, self.n_micro + 1):
            self.fill(t, k)
            zf.zero_step_units(self.prepared, k, self.n_micro, hp)
            for s in self.samples:
                out = oracle.sampled_step(s.grads_at(), s.master, s.m, s.v, acc_at=s.acc,
                                          micro_step=k, n_micro=self.n_micro, lr=hp["lr"],
                                          beta1=hp["beta1"], beta2=hp["beta2"], eps=hp["eps"],
                                          weight_decay=hp["weight_decay"], step=t)
                if out is not None:
                    s.params = out

    def compare(self):
        torch.cuda.synchronize()
        for s in self.samples:
            s.compare()
        assert zf.zero_device_status() == zf.zero.ZERO_DEVICE_OK


def _run(oracle, w, units, steps, n_micro, shared_grads=False, n_random=3000):
    m = SampledModel(w, units, (w.name, "fullsize"), n_micro, shared_grads, n_random)
    for t in range(1, steps + 1):
        m.step(oracle, t)
    m.compare()
    del m
    gc.collect()
    torch.cuda.empty_cache()


def test_gpt2_small_13_units_10_steps(oracle):
    """All 13 units in one zero_step_units call (one packed launch), 10 steps."""
    w = synthetic.workload("gpt2-small")
    _run(oracle, w, w.units, w.steps, 1)


def test_llama3_8b_layer_5_steps_outliers(oracle):
    w = synthetic.workload("llama3-8b-layer")
    _run(oracle, w, w.units, w.steps, 1)


def test_7p5b_model_32_units_streamed_grads(oracle):
    """The whole 7.5B model (32 units of P_pad = 234,375,040, N_d = 64,
    S = 3,662,110, S mod 8 = 6) reading one shared gradient buffer, stepped by
    one zero_step_units call per step (three packed launches), 2 steps: the
    benchmark's headline step."""
    w = synthetic.workload("7.5b")
    _run(oracle, w, w.units, w.steps, 1, shared_grads=True, n_random=1000)


def test_7p5b_model_fp32_accumulation_4_micro_steps(oracle):
    """The whole 7.5B model with fp32 accumulation over 4 micro-steps, as the
    benchmark runs it: 32 units sharing one gradient buffer, every micro-step
    one zero_step_units call (two packed reduce-scatter launches for the first
    three, four packed fused launches for the last), 2 optimizer steps."""
    w = synthetic.workload("7.5b-accum")
    _run(oracle, w, w.units, w.steps, 4, shared_grads=True, n_random=600)


SWEEP = [(4 ** 10, 2), (4 ** 10 + 13, 64), (4 ** 12 + 13, 8), (4 ** 13, 64), (4 ** 14 + 13, 2),
         (4 ** 15 + 13, 64), (4 ** 15, 8),
         # S = 65,822: every rank's shard ends in 286 elements, as the 7.5B
         # model's do, in a launch of 7 rounds
         (64 * 65822, 64)]


@pytest.mark.parametrize("P,n_ranks", SWEEP, ids=[f"P{p}_N{n}" for p, n in SWEEP])
def test_sweep_points(oracle, P, n_ranks):
    w = synthetic.workload(f"sweep:{P}:{n_ranks}")
    _run(oracle, w, w.units, 2, 1)


def test_beyond_2_pow_31_elements(oracle):
    """Flat indices above 2^31 (64-bit index arithmetic)."""
    w = synthetic.workload(f"sweep:{2 ** 31 + 13}:2")
    _run(oracle, w, w.units, 1, 1)
