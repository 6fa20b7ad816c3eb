"""zero_step_units_host: the step with gradients copied in from pinned host
memory and the gathered parameters copied back, against zero_step_units on
the same gradients already on the device (bit for bit)."""
import pytest
import torch

from gpu_harness import hp_at

import fsdp_sharded_mixed_flatten_gb300 as zf
from fsdp_sharded_mixed_flatten_gb300 import synthetic
from fsdp_sharded_mixed_flatten_gb300.buffers import FlatUnit, aligned_rows

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from fsdp_sharded_mixed_flatten_gb300 import build
    build.build()
    zf.load()


def make_pair(specs, tag, accum=False):
    """Two identical sets of units (same initial master weights)."""
    sets = []
    for _ in range(2):
        us = []
        for i, (numels, n) in enumerate(specs):
            u = FlatUnit(numels, n, accum=accum)
            u.set_master_flat(synthetic.make_master_flat(u.P, n, 0.02, (tag, i)).cuda())
            us.append(u)
        sets.append(us)
    return sets


def tuples(us):
    return [(u.grad_rows(), *u.state_rows(), u.accum_rows(), u.param_rows(), u.layout)
            for u in us]


def assert_same(a, b):
    for ua, ub in zip(a, b):
        for x, y in ((ua.master, ub.master), (ua.m, ub.m), (ua.v, ub.v)):
            assert torch.equal(x.contiguous().view(torch.int32), y.contiguous().view(torch.int32))
        assert torch.equal(ua.params.contiguous().view(torch.int16),
                           ub.params.contiguous().view(torch.int16))


SPECS = [([4096 * 300 + 5, 1000], 8), ([999999], 3), ([77], 64)]


@pytest.mark.parametrize("flags", [0, zf.ZERO_HOST_SM_COPY], ids=["copy_engines", "sm_copy"])
@pytest.mark.parametrize("layout", ["strided", "rows", "odd_offset"])
def test_host_step_equals_device_step(layout, flags):
    """Rows in one pinned block (the second unit's rows then sit off the
    16-byte grid), in separate pinned buffers, or all at a 2-byte offset:
    with ZERO_HOST_SM_COPY the aligned rows go through the SMs and the others
    through the copy engines, with the same result."""
    dev, host_side = make_pair(SPECS, "host-" + layout)
    h2d, d2h = torch.cuda.Stream(), torch.cuda.Stream()
    comp = torch.cuda.current_stream()
    for t in (1, 2, 3):
        hg, hp_out = [], []
        for i, u in enumerate(host_side):
            g = synthetic.make_grads(u.P, u.n_ranks, 1e-2, ("host", layout, i, t))
            if layout == "strided":      # one pinned block, rows evenly spaced
                blk = g.pin_memory()
                hg.append([blk[k] for k in range(u.n_ranks)])
                hp_out.append(torch.empty(u.P_pad, dtype=torch.bfloat16).pin_memory())
            elif layout == "rows":       # separate pinned rows (not evenly spaced)
                hg.append([g[k].clone().pin_memory() for k in range(u.n_ranks)])
                hp_out.append(torch.empty(u.P_pad, dtype=torch.bfloat16).pin_memory())
            else:                        # every row and output 2 bytes past the grid
                blk = torch.empty(u.n_ranks * u.P_pad + 1, dtype=torch.bfloat16).pin_memory()
                blk[1:].view(u.n_ranks, u.P_pad).copy_(g)
                hg.append([blk[1 + k * u.P_pad:1 + (k + 1) * u.P_pad] for k in range(u.n_ranks)])
                hp_out.append(torch.empty(u.P_pad + 1, dtype=torch.bfloat16).pin_memory()[1:])
            dev[i].grads.copy_(g.cuda())
        zf.zero_step_units(tuples(dev), 1, 1, hp_at(t))
        zf.zero_step_units_host(tuples(host_side), (hg, hp_out), 1, 1, hp_at(t), flags,
                                h2d, comp, d2h)
        d2h.synchronize()
        torch.cuda.synchronize()
        for u, hpo in zip(host_side, hp_out):
            assert torch.equal(hpo.view(torch.int16), u.params[0].cpu().view(torch.int16))
    assert_same(dev, host_side)
    assert zf.zero_device_status() == zf.zero.ZERO_DEVICE_OK


def test_host_step_double_buffered_with_free_flag():
    """Two device gradient sets used alternately, the caller ordering the
    copies after the step that last read the set (ZERO_HOST_GRADS_FREE), the
    rows moved by the SMs (ZERO_HOST_SM_COPY)."""
    dev, host_side = make_pair(SPECS, "host-dbl")
    spare = [aligned_rows(u.n_ranks, u.P_pad, torch.bfloat16, "cuda", 0) for u in host_side]
    sets = [[u.grads for u in host_side], spare]
    h2d, d2h = torch.cuda.Stream(), torch.cuda.Stream()
    comp = torch.cuda.current_stream()
    done = {}
    blocks = []
    for t in range(1, 6):
        hg, hp_out = [], []
        for i, u in enumerate(host_side):
            g = synthetic.make_grads(u.P, u.n_ranks, 1e-2, ("host-dbl", i, t))
            blk = g.pin_memory()
            blocks.append(blk)
            hg.append([blk[k] for k in range(u.n_ranks)])
            hp_out.append(torch.empty(u.P_pad, dtype=torch.bfloat16).pin_memory())
            dev[i].grads.copy_(g.cuda())
        zf.zero_step_units(tuples(dev), 1, 1, hp_at(t))
        cur = sets[t % 2]
        if t - 2 in done:
            h2d.wait_event(done[t - 2])      # the step that last read this set is done
        units = [([cur[i][k] for k in range(u.n_ranks)], *u.state_rows(), None,
                  u.param_rows(), u.layout) for i, u in enumerate(host_side)]
        zf.zero_step_units_host(units, (hg, hp_out), 1, 1, hp_at(t),
                                zf.ZERO_HOST_GRADS_FREE | zf.ZERO_HOST_SM_COPY, h2d, comp, d2h)
        done[t] = comp.record_event()
        d2h.synchronize()
        for u, hpo in zip(host_side, hp_out):
            assert torch.equal(hpo.view(torch.int16), u.params[0].cpu().view(torch.int16))
    torch.cuda.synchronize()
    assert_same(dev, host_side)


def test_host_step_accumulation_copies_params_at_the_last_micro_step():
    dev, host_side = make_pair(SPECS[:2], "host-acc", accum=True)
    h2d, d2h = torch.cuda.Stream(), torch.cuda.Stream()
    comp = torch.cuda.current_stream()
    K = 3
    hp_out = [torch.full((u.P_pad,), 7.0, dtype=torch.bfloat16).pin_memory() for u in host_side]
    for k in range(1, K + 1):
        hg = []
        for i, u in enumerate(host_side):
            g = synthetic.make_grads(u.P, u.n_ranks, 1e-2, ("host-acc", i, k))
            blk = g.pin_memory()
            hg.append([blk[r] for r in range(u.n_ranks)])
            dev[i].grads.copy_(g.cuda())
        zf.zero_step_units(tuples(dev), k, K, hp_at(1))
        zf.zero_step_units_host(tuples(host_side), (hg, hp_out), k, K, hp_at(1), 0,
                                h2d, comp, d2h)
        torch.cuda.synchronize()
        if k < K:     # no optimizer step yet: the host buffers are untouched
            assert all(bool(torch.all(h == 7.0)) for h in hp_out)
    for u, hpo in zip(host_side, hp_out):
        assert torch.equal(hpo.view(torch.int16), u.params[0].cpu().view(torch.int16))
    assert_same(dev, host_side)


def test_host_step_sm_copy_many_rows():
    """More rows than one transfer launch holds (320 rows, 256 a launch), in
    and out, through the SMs: the device step's bits."""
    specs = [([1000 + 17 * i], 64) for i in range(5)]
    dev, host_side = make_pair(specs, "host-many")
    h2d, d2h = torch.cuda.Stream(), torch.cuda.Stream()
    comp = torch.cuda.current_stream()
    for t in (1, 2):
        hg, hp_out = [], []
        for i, u in enumerate(host_side):
            g = synthetic.make_grads(u.P, u.n_ranks, 1e-2, ("host-many", i, t))
            hg.append([g[k].clone().pin_memory() for k in range(u.n_ranks)])
            hp_out.append(torch.empty(u.P_pad, dtype=torch.bfloat16).pin_memory())
            dev[i].grads.copy_(g.cuda())
        zf.zero_step_units(tuples(dev), 1, 1, hp_at(t))
        zf.zero_step_units_host(tuples(host_side), (hg, hp_out), 1, 1, hp_at(t),
                                zf.ZERO_HOST_SM_COPY, h2d, comp, d2h)
        d2h.synchronize()
        torch.cuda.synchronize()
        for u, hpo in zip(host_side, hp_out):
            assert torch.equal(hpo.view(torch.int16), u.params[0].cpu().view(torch.int16))
    assert_same(dev, host_side)
    assert zf.zero_device_status() == zf.zero.ZERO_DEVICE_OK
