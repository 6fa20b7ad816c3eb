"""Independent steps issued at the same time on two CUDA streams give the same
bits as the same steps issued one after the other.  The library keeps no
scratch state that two calls could share: every buffer, including the clipped
step's workspace, belongs to the caller."""
import pytest
import torch

from gpu_harness import hp_at

import fsdp_sharded_mixed_flatten_gb300 as zf
from fsdp_sharded_mixed_flatten_gb300 import synthetic
from fsdp_sharded_mixed_flatten_gb300.buffers import FlatUnit

pytestmark = pytest.mark.gpu

# (tensor sizes, N_d) of the units of the two groups
GROUP_A = [([300_001, 77], 8), ([1 << 20, 4097], 4)]
GROUP_B = [([2_000_003], 64), ([65_536, 12], 2)]


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from fsdp_sharded_mixed_flatten_gb300 import build
    build.build()
    zf.load()


def _units(specs, tag):
    units = []
    for i, (numels, n_ranks) in enumerate(specs):
        u = FlatUnit(numels, n_ranks, accum=True)
        u.set_master_flat(synthetic.make_master_flat(u.P, n_ranks, 0.02, (tag, i)).cuda())
        units.append(u)
    return units


def _tuples(units):
    return [(u.grad_rows(), *u.state_rows(), u.accum_rows(), u.param_rows(), u.layout)
            for u in units]


def _bits(units):
    out = []
    for u in units:
        for t in (u.master, u.m, u.v, u.accum):
            out.append(t.contiguous().view(torch.int32).cpu())
        out.append(u.params.contiguous().view(torch.int16).cpu())
    return out


class Group:
    """One group's units and, for the clipped group, its own workspace."""

    def __init__(self, specs, tag, clip, n_micro):
        self.units, self.clip, self.n_micro, self.tag = _units(specs, tag), clip, n_micro, tag
        self.tuples = _tuples(self.units)
        if clip:
            self.ws_bytes = zf.zero_clip_workspace_bytes(self.tuples, n_micro)
            self.ws = torch.empty(self.ws_bytes // 8, dtype=torch.float64, device="cuda")

    def fill(self, t, k):
        for i, u in enumerate(self.units):
            g = synthetic.make_grads(u.P, u.n_ranks, 1e-2, (self.tag, i, t, k))
            u.grads.copy_(g.cuda())

    def launch(self, t, k, stream):
        if self.clip:
            zf.zero_step_units_clip(self.tuples, k, self.n_micro, hp_at(t), 0.5, self.ws,
                                    self.ws_bytes, stream=stream)
        else:
            zf.zero_step_units(self.tuples, k, self.n_micro, hp_at(t), stream=stream)


def test_concurrent_streams_match_sequential():
    seq = [Group(GROUP_A, "streams-a", True, 2), Group(GROUP_B, "streams-b", False, 1)]
    con = [Group(GROUP_A, "streams-a", True, 2), Group(GROUP_B, "streams-b", False, 1)]
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    cur = torch.cuda.current_stream()
    for t in (1, 2, 3):
        for k in (1, 2):
            for g in seq + con:
                if k <= g.n_micro:
                    g.fill(t, k)
            torch.cuda.synchronize()
            for g in seq:                       # one after the other
                if k <= g.n_micro:
                    g.launch(t, k, cur)
            torch.cuda.synchronize()
            s1.wait_stream(cur)
            s2.wait_stream(cur)
            for g, s in zip(con, (s1, s2)):     # both at once
                if k <= g.n_micro:
                    g.launch(t, k, s)
            torch.cuda.synchronize()
    for a, b in zip(seq, con):
        for x, y in zip(_bits(a.units), _bits(b.units)):
            assert torch.equal(x, y)
    assert zf.zero_device_status() == zf.zero.ZERO_DEVICE_OK
