"""The clipped multi-unit step without a caller workspace.

zero_step_units_clip needs a small device workspace between its two passes.
Callers that cannot allocate device memory -- a runtime that gives all device
memory to its own pool at start-up and allows no allocation on the side, or a
deployment with a device-memory budget fixed before the optimizer runs -- use
zero_step_units_clip_noalloc, which keeps the partial sums in a fixed scratch
array inside the library.  Here it is called through the C ABI and must give
what the workspace variant gives, on two calls in a row (the second call runs
with the first call's partial sums still in the shared array).

This file is named to be collected last, so that a run stopping at the first
failure has already run every other test.
"""
import pytest
import torch

from gpu_harness import hp_at

import fsdp_sharded_mixed_flatten_gb300 as zf
from fsdp_sharded_mixed_flatten_gb300 import synthetic
from fsdp_sharded_mixed_flatten_gb300.buffers import FlatUnit

pytestmark = pytest.mark.gpu

SPECS = [([4099, 17], 4), ([100003], 8), ([64 * 77 + 3], 64), ([77777], 65)]


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from fsdp_sharded_mixed_flatten_gb300 import build
    build.build()
    zf.load()


def _make_units(tag):
    units = []
    for i, (numels, n_ranks) in enumerate(SPECS):
        u = FlatUnit(numels, n_ranks, accum=True)
        u.set_master_flat(synthetic.make_master_flat(u.P, n_ranks, 0.02, (tag, i)).cuda())
        units.append(u)
    return units


def _tuples(units):
    return [(u.grad_rows(), *u.state_rows(), u.accum_rows(), u.param_rows(), u.layout)
            for u in units]


@pytest.mark.parametrize("n_micro", [1, 2])
def test_no_alloc_matches_workspace_variant(n_micro):
    a_units = _make_units("na")        # no-allocation entry point
    b_units = _make_units("na")        # the existing entry point with a workspace
    ws_bytes = zf.zero_clip_workspace_bytes(_tuples(b_units), n_micro)
    workspace = torch.empty(ws_bytes // 8, dtype=torch.float64, device="cuda")
    norm_a = torch.zeros(1, dtype=torch.float32, device="cuda")
    norm_b = torch.zeros(1, dtype=torch.float32, device="cuda")
    for t, max_norm in ((1, 0.05), (2, 0.01)):        # two calls in a row, clipping active
        for k in range(1, n_micro + 1):
            for i, (ua, ub) in enumerate(zip(a_units, b_units)):
                g = synthetic.make_grads(ua.P, ua.n_ranks, 1e-2, ("na", i, t, k)).cuda()
                ua.grads.copy_(g)
                ub.grads.copy_(g)
            zf.zero_step_units_clip_noalloc(_tuples(a_units), k, n_micro, hp_at(t), max_norm,
                                            norm_a)
            zf.zero_step_units_clip(_tuples(b_units), k, n_micro, hp_at(t), max_norm, workspace,
                                    ws_bytes, norm_b)
        torch.cuda.synchronize()
        # Both entry points run the same kernels with the same grids and reduce
        # the partial sums in the same fixed order: the results are the same bits.
        na, nb = float(norm_a.item()), float(norm_b.item())
        assert nb > max_norm and na == nb, (na, nb)
        for ua, ub in zip(a_units, b_units):
            for x, y in ((ua.master, ub.master), (ua.m, ub.m), (ua.v, ub.v),
                         (ua.accum, ub.accum)):
                assert torch.equal(x.contiguous().view(torch.int32),
                                   y.contiguous().view(torch.int32))
            assert torch.equal(ua.params.contiguous().view(torch.int16),
                               ub.params.contiguous().view(torch.int16))
    assert zf.zero_device_status() == zf.zero.ZERO_DEVICE_OK


def test_no_alloc_rejects_oversized_calls():
    u = FlatUnit([4099], 4, accum=True)
    one = (u.grad_rows(), *u.state_rows(), u.accum_rows(), u.param_rows(), u.layout)
    with pytest.raises(zf.ZeroError) as ei:
        zf.zero_step_units_clip_noalloc([one] * 257, 1, 1, hp_at(1), 1.0)
    assert ei.value.code == -3 and "256" in str(ei.value)


def test_no_alloc_rejects_units_needing_too_many_slots():
    """84 units of 512 ranks: 3 units per norm launch (1024 pointers each), 28
    launches of 152 CTAs, 4256 partial sums > ZERO_NOALLOC_CLIP_SLOTS.  The call
    is refused before anything is launched: the state stays as it was."""
    units = []
    for i in range(84):
        u = FlatUnit([512], 512, accum=True)
        u.set_master_flat(synthetic.make_master_flat(u.P, 512, 0.02, ("slots", i)).cuda())
        u.grads.fill_(1.0)
        units.append(u)
    tuples = _tuples(units)
    assert zf.zero_clip_workspace_bytes(tuples, 1) // 8 > zf.zero.ZERO_NOALLOC_CLIP_SLOTS
    before = [u.master.clone() for u in units]
    with pytest.raises(zf.ZeroError) as ei:
        zf.zero_step_units_clip_noalloc(tuples, 1, 1, hp_at(1), 1.0)
    assert ei.value.code == -3 and "slots" in str(ei.value)
    torch.cuda.synchronize()
    for u, b in zip(units, before):
        assert torch.equal(u.master, b)
        assert not u.m.any() and not u.v.any() and not u.params.any()
    # a workspace of the size it asks for takes the same call
    nbytes = zf.zero_clip_workspace_bytes(tuples, 1)
    ws = torch.empty(nbytes // 8, dtype=torch.float64, device="cuda")
    zf.zero_step_units_clip(tuples, 1, 1, hp_at(1), 1.0, ws, nbytes)
    torch.cuda.synchronize()
    assert zf.zero_device_status() == zf.zero.ZERO_DEVICE_OK
