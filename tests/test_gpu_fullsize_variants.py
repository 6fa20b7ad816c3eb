"""The benchmark's variant steps at the sizes it times them, with sampled parity
against the oracle (the step is element-wise, so a sample of flat elements can
be followed exactly; every sample holds the shard and tensor boundaries):

* GPT-2-small (13 units, N_d = 8) with global gradient-norm clipping at
  max_norm = 1.0 -- the oracle forms the whole model's averaged gradient and
  its norm, then follows the sampled elements through the clipped update
  ("Data parallelism and ZeRO memory sharding", section 6);
* the ZeRO-1 form of a K = 4 micro-batch step on the Llama-3-8B layer
  (N_d = 64): full fp32 accumulators, one reduce-scatter at the end ("Lesson 5:
  ZeRO and FSDP", section 3 on gradient accumulation);
* GPT-2-small as 148 and the Llama-3-8B layer as 9 FSDP2 per-parameter
  Shard(0) units, each model in one zero_step_units call ("Lesson 5: ZeRO and
  FSDP", section 7.2).
"""
import gc

import numpy as np
import pytest
import torch

import parity
from gpu_harness import Sample, bits, hp_at, sample_indices

import fsdp_sharded_mixed_flatten_gb300 as zf
from fsdp_sharded_mixed_flatten_gb300 import synthetic
from fsdp_sharded_mixed_flatten_gb300.buffers import FlatUnit, ParamUnit, aligned_rows, rows

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


def _release():
    gc.collect()
    torch.cuda.empty_cache()


def _fill(fu, w, *seed_parts):
    for r in range(fu.n_ranks):
        synthetic.fill_grad_(fu.grads[r], fu.P, w.grad_std,
                             synthetic.seed_for(*seed_parts, "grad", r),
                             w.outlier_frac, w.outlier_scale)


def test_gpt2_small_global_norm_clipping_full_size(oracle):
    """The clipped GPT-2-small step the benchmark times (13 units, N_d = 8,
    max_norm = 1.0, which clips: the averaged gradient's norm is about 3.9),
    2 steps.  The oracle reduces every rank's whole gradient of every unit to
    the averaged gradient in double, takes the norm over all of them, and
    follows the sampled elements through the scaled AdamW update."""
    w = synthetic.workload("gpt2-small")
    tag = ("clip-fullsize",)
    units, samples = [], []
    for unit in w.units:
        fu = FlatUnit(unit.numels, w.n_ranks, accum=True)
        flat = synthetic.make_master_flat(fu.P, w.n_ranks, w.master_std, tag + (unit.name,),
                                          device="cuda")
        fu.set_master_flat(flat)
        idx = sample_indices(fu, 2000, synthetic.seed_for(tag, unit.name) & 0xFFFF)
        samples.append(Sample(fu, idx, flat))
        units.append(fu)
        del flat
    tuples = [(fu.grad_rows(), *fu.state_rows(), fu.accum_rows(), fu.param_rows(), fu.layout)
              for fu in units]
    nbytes = zf.zero_clip_workspace_bytes(tuples, 1)
    workspace = torch.empty(nbytes // 8, dtype=torch.float64, device="cuda")
    norm_gpu = torch.zeros(1, dtype=torch.float32, device="cuda")
    max_norm = 1.0
    for t in (1, 2):
        hp = hp_at(t)
        for fu, unit in zip(units, w.units):
            _fill(fu, w, *tag, unit.name, t)
        zf.zero_step_units_clip(tuples, 1, 1, hp, max_norm, workspace, nbytes, norm_gpu)
        # the oracle: every unit's averaged gradient in full, the global norm
        total, g_at, absmean_at = 0.0, [], []
        for fu, s in zip(units, samples):
            gb = bits(fu.grads.cpu())
            mean = oracle.reduce_scatter(gb)
            total += oracle.sum_squares(mean)
            g_at.append(mean[s.idx // fu.S, s.idx % fu.S].copy())
            x = (gb[:, s.idx].astype(np.uint32) << 16).view(np.float32)
            absmean_at.append(np.abs(x).mean(axis=0))
            del gb, mean
        coef = oracle.clip_coefficient(total, max_norm)
        norm = float(np.sqrt(total))
        torch.cuda.synchronize()
        got = float(norm_gpu.item())
        assert abs(got - norm) <= 1e-6 * norm, (got, norm)
        assert coef < 1.0, coef
        for fu, s, g, am in zip(units, samples, g_at, absmean_at):
            # the unscaled averaged gradient stays in the accumulator
            parity.check_mean(fu.accum[s.r_t, s.i_t].cpu().numpy(), g, am, what="mean")
            oracle.scale(g, coef)
            oracle.adamw(s.master, s.m, s.v, g, lr=hp["lr"], beta1=hp["beta1"],
                         beta2=hp["beta2"], eps=hp["eps"], weight_decay=hp["weight_decay"],
                         step=t)
            s.params = oracle.round_to_bf16(s.master)
    torch.cuda.synchronize()
    for s in samples:
        s.compare()
    assert zf.zero_device_status() == zf.zero.ZERO_DEVICE_OK
    del units, samples, tuples, workspace
    _release()


def test_zero1_llama3_8b_layer_k4_full_size(oracle):
    """The ZeRO-1 step the benchmark times: the Llama-3-8B layer (P = 218,112,000,
    N_d = 64, 1 % outliers), each rank accumulating its full fp32 gradient over
    K = 4 micro-batches (a 55.8 GB accumulator set), one reduce-scatter with the
    update at the end; 2 optimizer steps.  The accumulators at the sampled
    elements must equal the oracle's bit for bit (one fp32 rounding per add on
    both sides)."""
    w = synthetic.workload("llama3-8b-layer")
    K, N = 4, w.n_ranks
    tag = ("zero1-fullsize",)
    fu = FlatUnit(w.units[0].numels, N)
    flat = synthetic.make_master_flat(fu.P, N, w.master_std, tag, device="cuda")
    fu.set_master_flat(flat)
    s = Sample(fu, sample_indices(fu, 3000, synthetic.seed_for(tag) & 0xFFFF), flat)
    del flat
    acc = aligned_rows(N, fu.P_pad, torch.float32, "cuda", 5.0)   # junk: the first add resets
    acc_at = np.zeros((N, s.idx.size), np.float32)
    for t in (1, 2):
        hp = hp_at(t)
        for k in range(1, K + 1):
            _fill(fu, w, *tag, t, k)
            zf.zero1_accumulate(fu.grad_rows(), rows(acc), k == 1, fu.layout)
            oracle.zero1_accumulate(s.grads_at(), acc_at, first=(k == 1))
        torch.cuda.synchronize()
        got = acc[:, s.idx_t].cpu().numpy()
        assert np.array_equal(got.view(np.uint32), acc_at.view(np.uint32))
        zf.zero1_step(rows(acc), K, *fu.state_rows(), fu.param_rows(), fu.layout, hp)
        s.params = oracle.sampled_zero1_step(acc_at, s.master, s.m, s.v, n_micro=K, lr=hp["lr"],
                                             beta1=hp["beta1"], beta2=hp["beta2"],
                                             eps=hp["eps"], weight_decay=hp["weight_decay"],
                                             step=t)
    torch.cuda.synchronize()
    s.compare()
    assert zf.zero_device_status() == zf.zero.ZERO_DEVICE_OK
    del fu, s, acc
    _release()


class ParamSample:
    """The oracle's copy of one per-parameter Shard(0) unit at sampled
    elements.  Which rank owns an element, and where in that rank's shard it
    sits, come from the oracle's own shard bounds."""

    def __init__(self, oracle, pu: ParamUnit, dim0, row, master_flat, n_random, seed):
        rng = np.random.default_rng(seed)
        n, N = pu.numel, pu.n_ranks
        bounds = [oracle.param_shard_bounds(dim0, row, N, r) for r in range(N)]
        idx = set(rng.integers(0, n, size=min(n, n_random)).tolist()) | {0, n - 1}
        for b, e in bounds:
            if e > b:
                idx.update((b, b + 1, e - 2, e - 1))
        idx = np.array(sorted(i for i in idx if 0 <= i < n), dtype=np.int64)
        owner = np.empty_like(idx)
        local = np.empty_like(idx)
        for r, (b, e) in enumerate(bounds):
            sel = (idx >= b) & (idx < e)
            owner[sel] = r
            local[sel] = idx[sel] - b
        self.pu, self.idx = pu, idx
        dev = master_flat.device
        self.idx_t = torch.from_numpy(idx).to(dev)
        self.r_t, self.i_t = torch.from_numpy(owner).to(dev), torch.from_numpy(local).to(dev)
        self.master = master_flat[self.idx_t].cpu().numpy().copy()
        self.m = np.zeros_like(self.master)
        self.v = np.zeros_like(self.master)
        self.params = None

    def step(self, oracle, hp, t):
        g_at = bits(self.pu.grads[:, self.idx_t].cpu())
        self.params = oracle.sampled_step(g_at, self.master, self.m, self.v, lr=hp["lr"],
                                          beta1=hp["beta1"], beta2=hp["beta2"], eps=hp["eps"],
                                          weight_decay=hp["weight_decay"], step=t)

    def compare(self):
        pu = self.pu
        g_master = pu.master[self.r_t, self.i_t].cpu().numpy()
        parity.check_state("master", g_master, self.master)
        parity.check_state("m", pu.m[self.r_t, self.i_t].cpu().numpy(), self.m)
        parity.check_state("v", pu.v[self.r_t, self.i_t].cpu().numpy(), self.v)
        g_p = bits(pu.params[0, self.idx_t].cpu())
        parity.check_bf16(g_p, self.params)
        parity.check_bf16_is_rounded_master(g_p, g_master)


@pytest.mark.parametrize("name,n_params", [("gpt2-small", 148), ("llama3-8b-layer", 9)])
def test_fsdp2_per_parameter_full_size(oracle, name, n_params):
    """Every parameter of the model its own Shard(0) unit (no FlatParameter, no
    padding), all stepped by one zero_step_units call, as the benchmark times
    it; 2 steps."""
    w = synthetic.workload(name)
    tag = ("fsdp2-fullsize", name)
    pus, samples = [], []
    for u in w.units:
        for i, (d0, row) in enumerate(u.rows()):
            pu = ParamUnit(d0, row, w.n_ranks)
            flat = synthetic.make_master_flat(pu.numel, 1, w.master_std, tag + (u.name, i),
                                              device="cuda")
            pu.set_master_flat(flat)
            n_random = 400 if pu.numel > 100000 else 40
            samples.append(ParamSample(oracle, pu, d0, row, flat, n_random,
                                       synthetic.seed_for(tag, u.name, i) & 0xFFFF))
            pus.append((pu, u.name, i))
            del flat
    assert len(pus) == n_params
    prepared = zf.zero.prepare_units([pu.unit_tuple() for pu, _, _ in pus])
    for t in (1, 2):
        hp = hp_at(t)
        for pu, uname, i in pus:
            for r in range(pu.n_ranks):
                synthetic.fill_grad_(pu.grads[r], pu.numel, w.grad_std,
                                     synthetic.seed_for(*tag, uname, i, t, "grad", r),
                                     w.outlier_frac, w.outlier_scale)
        zf.zero_step_units(prepared, 1, 1, hp)
        for s in samples:
            s.step(oracle, hp, t)
    torch.cuda.synchronize()
    for s in samples:
        s.compare()
    assert zf.zero_device_status() == zf.zero.ZERO_DEVICE_OK
    del pus, samples, prepared
    _release()
