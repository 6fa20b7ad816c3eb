"""Failure injected on the host (ZERO_INJECT_FAILURE): a step whose launch or
copy fails reports ZERO_ERR_CUDA, leaves the optimizer state as it was, and
a retry once the failure is gone gives the same bits as a run that never
failed.  Nothing faults or hangs the GPU: the failing call is never made."""
import pytest
import torch

from gpu_harness import hp_at

import fsdp_sharded_mixed_flatten_gb300 as zf
from fsdp_sharded_mixed_flatten_gb300 import HostTables, synthetic
from fsdp_sharded_mixed_flatten_gb300.buffers import FlatUnit

pytestmark = pytest.mark.gpu

SPECS = [([300_001, 77], 8), ([1 << 20, 4097], 4), ([2_000_003], 64)]


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from fsdp_sharded_mixed_flatten_gb300 import build
    build.build()
    zf.load()


def _units(tag):
    units = []
    for i, (numels, n_ranks) in enumerate(SPECS):
        u = FlatUnit(numels, n_ranks, accum=True)
        u.set_master_flat(synthetic.make_master_flat(u.P, n_ranks, 0.02, (tag, i)).cuda())
        g = synthetic.make_grads(u.P, n_ranks, 1e-2, (tag, i, "g"))
        u.grads.copy_(g.cuda())
        units.append(u)
    return units


def _tuples(units):
    return [(u.grad_rows(), *u.state_rows(), u.accum_rows(), u.param_rows(), u.layout)
            for u in units]


def _state(units):
    out = []
    for u in units:
        for t in (u.master, u.m, u.v):
            out.append(t.contiguous().view(torch.int32).clone())
        out.append(u.params.contiguous().view(torch.int16).clone())
    return out


def _same(a, b):
    return len(a) == len(b) and all(torch.equal(x, y) for x, y in zip(a, b))


@pytest.mark.parametrize("label", ["clip norm pass", "clip update pass"])
def test_clipped_step_failure_then_retry(monkeypatch, label):
    clean, failing = _units("inject-clip"), _units("inject-clip")
    ws_bytes = zf.zero_clip_workspace_bytes(_tuples(clean), 1)
    ws = [torch.empty(ws_bytes // 8, dtype=torch.float64, device="cuda") for _ in range(2)]
    zf.zero_step_units_clip(_tuples(clean), 1, 1, hp_at(1), 0.5, ws[0], ws_bytes)
    before = _state(failing)
    monkeypatch.setenv("ZERO_INJECT_FAILURE", label)
    with pytest.raises(zf.ZeroError) as ei:
        zf.zero_step_units_clip(_tuples(failing), 1, 1, hp_at(1), 0.5, ws[1], ws_bytes)
    assert ei.value.code == -4 and "injected failure" in str(ei.value)
    torch.cuda.synchronize()
    assert _same(_state(failing), before), "a failed step changed the optimizer state"
    monkeypatch.delenv("ZERO_INJECT_FAILURE")
    zf.zero_step_units_clip(_tuples(failing), 1, 1, hp_at(1), 0.5, ws[1], ws_bytes)
    torch.cuda.synchronize()
    assert _same(_state(failing), _state(clean))
    assert zf.zero_device_status() == zf.zero.ZERO_DEVICE_OK


@pytest.mark.parametrize("flags", [0, zf.ZERO_HOST_SM_COPY], ids=["copy_engines", "sm_copy"])
@pytest.mark.parametrize("label", ["gradient copy to the device", "staged launch: step",
                                   "parameter copy to the host"])
def test_host_step_failure_then_retry(monkeypatch, label, flags):
    clean, failing = _units("inject-host"), _units("inject-host")
    host_g = [u.grads.cpu().pin_memory() for u in clean]
    host_p = [[torch.zeros(u.P_pad, dtype=torch.bfloat16).pin_memory() for u in clean]
              for _ in range(2)]

    def run(units, params):
        tables = HostTables([[g[k] for k in range(g.shape[0])] for g in host_g], params)
        s = torch.cuda.current_stream()
        zf.zero_step_units_host(_tuples(units), tables, 1, 1, hp_at(1), flags, s, s, s)

    run(clean, host_p[0])
    torch.cuda.synchronize()
    for u in failing:                 # the copies must bring the gradients back
        u.grads.zero_()
    before = _state(failing)
    monkeypatch.setenv("ZERO_INJECT_FAILURE", label)
    with pytest.raises(zf.ZeroError) as ei:
        run(failing, host_p[1])
    assert ei.value.code == -4 and label in str(ei.value)
    torch.cuda.synchronize()
    if label != "parameter copy to the host":
        assert _same(_state(failing), before), "a failed step changed the optimizer state"
        monkeypatch.delenv("ZERO_INJECT_FAILURE")
        run(failing, host_p[1])
        torch.cuda.synchronize()
        assert _same(_state(failing), _state(clean))
        for a, b in zip(host_p[0], host_p[1]):
            assert torch.equal(a.view(torch.int16), b.view(torch.int16))
    else:
        # the step ran; only the copy back failed: state and device params are final
        assert _same(_state(failing), _state(clean))
    assert zf.zero_device_status() == zf.zero.ZERO_DEVICE_OK
