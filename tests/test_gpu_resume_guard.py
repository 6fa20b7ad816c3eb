"""Two properties of a stateless library, on the GPU:
- resuming from saved state is exact: 10 steps equal 5 steps, a save of
  master/m/v to a file, a reload into fresh buffers and 5 more steps, bit for
  bit (the caller owns every byte of state and the step count);
- nothing outside a buffer is touched: every per-rank buffer of a flat unit
  sits between sentinel-filled guard bands that must survive the steps."""
import numpy as np
import pytest
import torch

from gpu_harness import hp_at

import fsdp_sharded_mixed_flatten_gb300 as zf
from fsdp_sharded_mixed_flatten_gb300 import synthetic
from fsdp_sharded_mixed_flatten_gb300.buffers import FlatUnit, rows

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from fsdp_sharded_mixed_flatten_gb300 import build
    build.build()
    zf.load()


NUMELS, N_RANKS = [4096 * 50 + 7, 999, 13], 8


def _fresh(tag):
    u = FlatUnit(NUMELS, N_RANKS)
    u.set_master_flat(synthetic.make_master_flat(u.P, N_RANKS, 0.02, (tag,)).cuda())
    return u


def _step(u, t):
    g = synthetic.make_grads(u.P, N_RANKS, 1e-2, ("resume", t))
    u.grads[:, :u.P_pad].copy_(g.cuda())
    zf.zero_step(u.grad_rows(), *u.state_rows(), None, 1, 1, u.param_rows(), u.layout, hp_at(t))


def test_resume_from_saved_state_is_bit_exact(tmp_path):
    straight = _fresh("resume-init")
    for t in range(1, 11):
        _step(straight, t)
    first = _fresh("resume-init")
    for t in range(1, 6):
        _step(first, t)
    torch.cuda.synchronize()
    path = tmp_path / "state.pt"
    torch.save({k: getattr(first, k).cpu().clone() for k in ("master", "m", "v")}, path)
    del first
    torch.cuda.empty_cache()
    resumed = _fresh("another-init")                # different weights until the load
    saved = torch.load(path)
    for k in ("master", "m", "v"):
        getattr(resumed, k).copy_(saved[k].cuda())
    for t in range(6, 11):
        _step(resumed, t)
    torch.cuda.synchronize()
    for k in ("master", "m", "v"):
        a, b = getattr(straight, k).contiguous(), getattr(resumed, k).contiguous()
        assert torch.equal(a.view(torch.int32), b.view(torch.int32)), k
    assert torch.equal(straight.params.contiguous().view(torch.int16),
                       resumed.params.contiguous().view(torch.int16))


GUARD = 256          # elements of sentinel before and after every buffer
SENTINEL = 12288.0   # exact in bf16 and fp32


def _guarded(n_rows, n_cols, dtype):
    """Rows of n_cols elements, each inside its own allocation of
    GUARD + n_cols + GUARD sentinels (rows stay 16-byte aligned)."""
    bases = [torch.full((GUARD + n_cols + GUARD,), SENTINEL, dtype=dtype, device="cuda")
             for _ in range(n_rows)]
    return bases, [b[GUARD:GUARD + n_cols] for b in bases]


def _guards_intact(bases):
    return all(bool(torch.all(b[:GUARD] == SENTINEL)) and bool(torch.all(b[-GUARD:] == SENTINEL))
               for b in bases)


@pytest.mark.parametrize("numels,n_ranks,n_micro", [([1000003], 8, 1), ([999999], 3, 3),
                                                    ([64 * 4099 + 5], 64, 2), ([5], 8, 1),
                                                    ([2 * 8 * 5000], 2, 1)])
@pytest.mark.parametrize("kernel", ["staged", "direct"])
def test_no_write_outside_any_buffer(monkeypatch, kernel, numels, n_ranks, n_micro):
    if kernel == "direct":
        monkeypatch.setenv("ZERO_STEP_KERNEL", "direct")
    else:
        monkeypatch.delenv("ZERO_STEP_KERNEL", raising=False)
    off, L = zf.zero_flat_layout(numels, n_ranks)
    P, P_pad, S = L.numel, L.numel_padded, L.shard_numel
    gb, grads = _guarded(n_ranks, P_pad, torch.bfloat16)
    mb, master = _guarded(n_ranks, S, torch.float32)
    m_b, m = _guarded(n_ranks, S, torch.float32)
    vb, v = _guarded(n_ranks, S, torch.float32)
    ab, acc = _guarded(n_ranks, S, torch.float32)
    pb, params = _guarded(2, P_pad, torch.bfloat16)
    for x in master + m + v + acc:
        x.zero_()
    for t in (1, 2):
        for k in range(1, n_micro + 1):
            g = synthetic.make_grads(P, n_ranks, 1e-2, ("guard", t, k)).cuda()
            for r in range(n_ranks):
                grads[r].copy_(g[r])
            zf.zero_step(grads, master, m, v, acc if n_micro > 1 else None, k, n_micro, params,
                         L, hp_at(t))
    torch.cuda.synchronize()
    for bases in (gb, mb, m_b, vb, ab, pb):
        assert _guards_intact(bases)
    assert zf.zero_device_status() == zf.zero.ZERO_DEVICE_OK
