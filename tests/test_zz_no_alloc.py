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
import numpy as np
import pytest
import torch

import parity
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
        na, nb = float(norm_a.item()), float(norm_b.item())
        assert nb > max_norm and abs(na - nb) <= 1e-6 * nb
        for ua, ub in zip(a_units, b_units):
            parity.check_state("master", ua.master.cpu().numpy(), ub.master.cpu().numpy())
            parity.check_state("m", ua.m.cpu().numpy(), ub.m.cpu().numpy())
            parity.check_state("v", ua.v.cpu().numpy(), ub.v.cpu().numpy())
            parity.check_bf16(synthetic.bf16_bits(ua.params[0].cpu()),
                              synthetic.bf16_bits(ub.params[0].cpu()))
    assert zf.zero_device_status() == zf.zero.ZERO_DEVICE_OK


def test_no_alloc_rejects_oversized_calls():
    u = FlatUnit([4099], 4, accum=True)
    one = (u.grad_rows(), *u.state_rows(), u.accum_rows(), u.param_rows(), u.layout)
    with pytest.raises(zf.ZeroError) as ei:
        zf.zero_step_units_clip_noalloc([one] * 257, 1, 1, hp_at(1), 1.0)
    assert ei.value.code == -3 and "256" in str(ei.value)
