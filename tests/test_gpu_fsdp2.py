"""FSDP2-style per-parameter Shard(0) units (no FlatParameter, no padding)
through zero_step_units, against the oracle and against the flat FSDP1 step."""
import numpy as np
import pytest
import torch

import parity
from gpu_harness import bits, hp_at

import fsdp_sharded_mixed_flatten_gb300 as zf
from fsdp_sharded_mixed_flatten_gb300 import synthetic
from fsdp_sharded_mixed_flatten_gb300.buffers import FlatUnit

pytestmark = pytest.mark.gpu

SENTINEL = 12288.0   # exact in bf16 and fp32
CANARY = 64          # elements after every buffer that must stay untouched


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from fsdp_sharded_mixed_flatten_gb300 import build
    build.build()
    zf.load()


class ParamUnit:
    """One parameter's per-rank buffers, each exactly as long as its data,
    followed by a canary region."""

    def __init__(self, dim0, row, n_ranks, master0):
        self.dim0, self.row, self.n = dim0, row, n_ranks
        self.layout = zf.zero_param_layout(dim0, row, n_ranks)
        self.numel = dim0 * row
        self.sizes = [zf.zero_shard_numel(self.layout, r) for r in range(n_ranks)]
        dev = "cuda"

        def buf(n, dtype, fill):
            return torch.full((n + CANARY,), fill, dtype=dtype, device=dev)

        self.g_bufs = [buf(self.numel, torch.bfloat16, SENTINEL) for _ in range(n_ranks)]
        self.p_buf = buf(self.numel, torch.bfloat16, SENTINEL)
        self.state = {k: [buf(sz, torch.float32, SENTINEL) for sz in self.sizes]
                      for k in ("master", "m", "v", "accum")}
        off = 0
        for r, sz in enumerate(self.sizes):
            self.state["master"][r][:sz].copy_(master0[off:off + sz])
            self.state["m"][r][:sz].zero_()
            self.state["v"][r][:sz].zero_()
            off += sz

    def tuple(self, accum=False):
        return (self.g_bufs, self.state["master"], self.state["m"], self.state["v"],
                self.state["accum"] if accum else None, [self.p_buf], self.layout)

    def canaries_intact(self):
        bufs = self.g_bufs + [self.p_buf] + [b for k in self.state for b in self.state[k]]
        return all(bool(torch.all(b[-CANARY:] == SENTINEL)) for b in bufs)


# At N_d = 8 the last two shapes have S = 4098 (S mod 4096 = 2: the fused step's tail group),
# with the last rank's tail empty (32779 rows) or one element long (32783 rows).
SHAPES = [(5, 3), (64, 7), (1, 11), (9, 1), (130, 2), (4096, 1), (33, 768), (1000, 13),
          (32779, 1), (32783, 1)]


@pytest.mark.parametrize("n_ranks", [3, 4, 8, 64])
def test_fsdp2_units_against_oracle_and_flat(oracle, n_ranks):
    rng_tag = ("fsdp2", n_ranks)
    units, o_params, masters0 = [], [], []
    for i, (d0, row) in enumerate(SHAPES):
        m0 = synthetic.make_master_flat(d0 * row, 1, 0.02, rng_tag + (i,))
        masters0.append(m0)
        pu = ParamUnit(d0, row, n_ranks, m0.cuda())
        units.append(pu)
        prm = dict(dim0=d0, row=row, master=[], m=[], v=[])
        off = 0
        for sz in pu.sizes:
            prm["master"].append(m0.numpy()[off:off + sz].copy())
            prm["m"].append(np.zeros(sz, np.float32))
            prm["v"].append(np.zeros(sz, np.float32))
            off += sz
        o_params.append(prm)
    # the flat FSDP1 unit over the same parameters in the same order
    flat = FlatUnit([d0 * row for d0, row in SHAPES], n_ranks)
    flat.set_master_flat(torch.cat(masters0 + [torch.zeros(flat.P_pad - flat.P)]).cuda())
    for t in (1, 2):
        flat_g = []
        for i, (pu, prm) in enumerate(zip(units, o_params)):
            gs = synthetic.make_grads(pu.numel, n_ranks, 1e-2, rng_tag + (i, t))[:, :pu.numel]
            gs = gs.contiguous()
            for k in range(n_ranks):
                pu.g_bufs[k][:pu.numel].copy_(gs[k].cuda())
            prm["grads"] = bits(gs)
            flat_g.append(gs)
        fg = torch.cat(flat_g, dim=1)
        flat.grads[:, :flat.P].copy_(fg.cuda())
        zf.zero_step_units([pu.tuple() for pu in units], 1, 1, hp_at(t))
        zf.zero_step(flat.grad_rows(), *flat.state_rows(), None, 1, 1, flat.param_rows(),
                     flat.layout, hp_at(t))
        hp = hp_at(t)
        o_out = oracle.param_sharded_step(o_params, lr=hp["lr"], beta1=hp["beta1"],
                                          beta2=hp["beta2"], eps=hp["eps"],
                                          weight_decay=hp["weight_decay"], step=t)
    torch.cuda.synchronize()
    flat_master = flat.master.cpu().numpy().reshape(-1)
    flat_params = bits(flat.params[0].cpu())
    off = 0
    for pu, prm, out in zip(units, o_params, o_out):
        assert pu.canaries_intact(), "a kernel touched memory past a parameter's data"
        g_master = np.concatenate([pu.state["master"][r][:sz].cpu().numpy()
                                   for r, sz in enumerate(pu.sizes)])
        o_master = np.concatenate(prm["master"])
        parity.check_state("master", g_master, o_master)
        g_m = np.concatenate([pu.state["m"][r][:sz].cpu().numpy() for r, sz in enumerate(pu.sizes)])
        parity.check_state("m", g_m, np.concatenate(prm["m"]))
        pb = bits(pu.p_buf[:pu.numel].cpu())
        parity.check_bf16(pb, out, min_exact=0.99)
        # the flat FSDP1 step computes every element identically
        assert np.array_equal(g_master.view(np.uint32),
                              flat_master[off:off + pu.numel].view(np.uint32))
        assert np.array_equal(pb, flat_params[off:off + pu.numel])
        off += pu.numel
    assert zf.zero_device_status() == zf.zero.ZERO_DEVICE_OK


def test_fsdp2_clipped_and_accumulated():
    """Per-parameter units through the clipped step with micro-step
    accumulation: bit-identical to the same clipped step over flat units
    holding the same elements (one flat unit per parameter)."""
    n_ranks, K = 8, 2
    shapes = [(33, 768), (7, 5), (4096, 1)]
    pus, fus = [], []
    for i, (d0, row) in enumerate(shapes):
        m0 = synthetic.make_master_flat(d0 * row, 1, 0.02, ("f2c", i))
        pus.append(ParamUnit(d0, row, n_ranks, m0.cuda()))
        fu = FlatUnit([d0 * row], n_ranks, accum=True)
        fu.set_master_flat(torch.cat([m0, torch.zeros(fu.P_pad - fu.P)]).cuda())
        fus.append(fu)
    p_tuples = [pu.tuple(accum=True) for pu in pus]
    f_tuples = [(fu.grad_rows(), *fu.state_rows(), fu.accum_rows(), fu.param_rows(), fu.layout)
                for fu in fus]
    ws_p = zf.zero_clip_workspace_bytes(p_tuples, K)
    ws_f = zf.zero_clip_workspace_bytes(f_tuples, K)
    wp = torch.empty(ws_p // 8, dtype=torch.float64, device="cuda")
    wf = torch.empty(ws_f // 8, dtype=torch.float64, device="cuda")
    for k in range(1, K + 1):
        for i, (pu, fu) in enumerate(zip(pus, fus)):
            gs = synthetic.make_grads(pu.numel, n_ranks, 1e-2, ("f2c", i, k))
            for r in range(n_ranks):
                pu.g_bufs[r][:pu.numel].copy_(gs[r, :pu.numel].cuda())
            fu.grads[:, :fu.P].copy_(gs.cuda()[:, :fu.P])
        zf.zero_step_units_clip(p_tuples, k, K, hp_at(1), 0.05, wp, ws_p)
        zf.zero_step_units_clip(f_tuples, k, K, hp_at(1), 0.05, wf, ws_f)
    torch.cuda.synchronize()
    for pu, fu in zip(pus, fus):
        assert pu.canaries_intact()
        g_master = torch.cat([pu.state["master"][r][:sz] for r, sz in enumerate(pu.sizes)])
        # same elements, different owners: compare by element
        fm = fu.master.contiguous().reshape(-1)[:pu.numel]
        # the flat unit shards differently but the norm covers the same elements
        assert torch.allclose(g_master, fm, rtol=1e-6, atol=1e-7)


def test_unpadded_layout_rejected_where_unsupported():
    pu = ParamUnit(9, 1, 4, torch.zeros(9, device="cuda"))
    with pytest.raises(zf.ZeroError) as ei:
        zf.zero_all_gather(pu.state["master"], [pu.p_buf], pu.layout)
    assert ei.value.code == -1


def _pair_units(tag):
    """The same flat and per-parameter units twice, with equal seeded state."""
    from fsdp_sharded_mixed_flatten_gb300.buffers import ParamUnit as PU
    out = []
    for _ in range(2):
        units = []
        for i, (d0, row) in enumerate([(33, 768), (5, 3), (4096, 1), (130, 2)]):
            w = PU(d0, row, 8)
            w.set_master_flat(synthetic.make_master_flat(w.numel, 1, 0.02, (tag, i)).cuda())
            units.append(w)
        for i, (numels, n) in enumerate([([300_001, 77], 8), ([65_536], 64)]):
            f = FlatUnit(numels, n)
            f.set_master_flat(synthetic.make_master_flat(f.P, n, 0.02, (tag, "flat", i)).cuda())
            units.append(f)
        out.append(units)
    return out


def _fill(units, tag, t):
    gs = []
    for i, u in enumerate(units):
        n_ranks = u.n_ranks
        numel = u.numel if hasattr(u, "sizes") else u.P
        g = synthetic.make_grads(numel, n_ranks, 1e-2, (tag, i, t))[:, :u.grads.shape[1]]
        u.grads.copy_(g.cuda())
        gs.append(g.contiguous())
    return gs


def _tuple(u):
    if hasattr(u, "unit_tuple"):
        return u.unit_tuple()
    return (u.grad_rows(), *u.state_rows(), None, u.param_rows(), u.layout)


def _assert_same_state(a, b):
    for x, y in zip(a, b):
        for s, t in ((x.master, y.master), (x.m, y.m), (x.v, y.v)):
            assert torch.equal(s.contiguous().view(torch.int32), t.contiguous().view(torch.int32))
        assert torch.equal(x.params.contiguous().view(torch.int16),
                           y.params.contiguous().view(torch.int16))


def test_flat_and_per_parameter_units_in_one_call():
    """FSDP1 flat units and FSDP2 per-parameter units stepped by one
    zero_step_units call give the bits of one call per unit."""
    a, b = _pair_units("mixed")
    for t in (1, 2):
        _fill(a, "mixed", t)
        _fill(b, "mixed", t)
        zf.zero_step_units([_tuple(u) for u in a], 1, 1, hp_at(t))
        for u in b:
            zf.zero_step_units([_tuple(u)], 1, 1, hp_at(t))
    torch.cuda.synchronize()
    _assert_same_state(a, b)
    assert zf.zero_device_status() == zf.zero.ZERO_DEVICE_OK


@pytest.mark.parametrize("flags", [0, zf.ZERO_HOST_SM_COPY], ids=["copy_engines", "sm_copy"])
def test_host_step_with_per_parameter_units(flags):
    """The host-buffer step moves exactly numel elements per per-parameter
    unit (no padding) and gives the device step's bits."""
    dev, host_side = _pair_units("host-pp")
    h2d, d2h = torch.cuda.Stream(), torch.cuda.Stream()
    comp = torch.cuda.current_stream()
    for t in (1, 2):
        gs = _fill(dev, "host-pp", t)
        for u in host_side:
            u.grads.zero_()
        hg = [[g[k].clone().pin_memory() for k in range(g.shape[0])] for g in gs]
        hp_out = [torch.full((u.params.shape[1] + 64,), SENTINEL,
                             dtype=torch.bfloat16).pin_memory() for u in host_side]
        zf.zero_step_units([_tuple(u) for u in dev], 1, 1, hp_at(t))
        zf.zero_step_units_host([_tuple(u) for u in host_side], (hg, hp_out), 1, 1, hp_at(t),
                                flags, h2d, comp, d2h)
        d2h.synchronize()
        torch.cuda.synchronize()
        for u, hpo in zip(host_side, hp_out):
            n = u.numel if hasattr(u, "sizes") else u.P_pad
            assert torch.equal(hpo[:n].view(torch.int16), u.params[0, :n].cpu().view(torch.int16))
            # nothing written past the parameter's (per-parameter) or padded (flat) length
            assert bool(torch.all(hpo[u.params.shape[1]:] == SENTINEL))
    _assert_same_state(dev, host_side)
    assert zf.zero_device_status() == zf.zero.ZERO_DEVICE_OK
