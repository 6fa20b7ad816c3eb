"""ZeRO-1 local accumulation (full fp32 accumulators, one reduce-scatter at the
last micro-step) against the oracle, through the C ABI."""
import numpy as np
import pytest
import torch

import parity
from gpu_harness import bits, hp_at

import fsdp_sharded_mixed_flatten_gb300 as zf
from fsdp_sharded_mixed_flatten_gb300 import synthetic
from fsdp_sharded_mixed_flatten_gb300.buffers import FlatUnit, aligned_rows, rows

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from fsdp_sharded_mixed_flatten_gb300 import build
    build.build()
    zf.load()


CASES = [
    # numels, n_ranks, n_micro   (S mod 4 != 0 exercises the fp32 realignment)
    ([4096 * 1024, 1024, 1000], 4, 3),
    ([1000003], 8, 1),
    ([999999], 3, 2),
    ([64 * 4099 + 5], 64, 4),
    ([77777], 65, 2),
    ([5], 8, 2),
]


@pytest.mark.parametrize("numels,n_ranks,n_micro", CASES)
def test_zero1_against_oracle(oracle, numels, n_ranks, n_micro):
    u = FlatUnit(numels, n_ranks)
    master0 = synthetic.make_master_flat(u.P, n_ranks, 0.02, ("z1", n_ranks))
    u.set_master_flat(master0.cuda())
    acc = aligned_rows(n_ranks, u.P_pad, torch.float32, "cuda", 3.0)   # junk: reset by first
    o_master = master0.numpy().reshape(n_ranks, u.S).copy()
    o_m, o_v = np.zeros_like(o_master), np.zeros_like(o_master)
    o_acc = np.zeros((n_ranks, u.P_pad), np.float32)
    for t in (1, 2):
        hp = hp_at(t)
        for k in range(1, n_micro + 1):
            g = synthetic.make_grads(u.P, n_ranks, 1e-2, ("z1", n_ranks, t, k))
            u.grads.copy_(g.cuda())
            zf.zero1_accumulate(u.grad_rows(), rows(acc), k == 1, u.layout)
            oracle.zero1_accumulate(bits(g), o_acc, first=(k == 1))
        torch.cuda.synchronize()
        # the accumulators are element-wise fp32 sums, one rounding per add on both sides
        assert np.array_equal(acc.cpu().numpy().view(np.uint32), o_acc.view(np.uint32))
        zf.zero1_step(rows(acc), n_micro, *u.state_rows(), u.param_rows(), u.layout, hp)
        o_params = oracle.zero1_step(o_acc, o_master, o_m, o_v, n_micro=n_micro, lr=hp["lr"],
                                     beta1=hp["beta1"], beta2=hp["beta2"], eps=hp["eps"],
                                     weight_decay=hp["weight_decay"], step=t)
    torch.cuda.synchronize()
    parity.check_state("master", u.master.cpu().numpy(), o_master)
    parity.check_state("m", u.m.cpu().numpy(), o_m)
    parity.check_state("v", u.v.cpu().numpy(), o_v)
    pb = bits(u.params[0].cpu())
    parity.check_bf16(pb, o_params)
    parity.check_bf16_is_rounded_master(pb, u.master.cpu().numpy().reshape(-1))
    assert zf.zero_device_status() == zf.zero.ZERO_DEVICE_OK


def test_zero1_equals_zero2_on_exact_inputs():
    """Gradients on a 2^-10 grid: every sum is exact, so the ZeRO-1 form
    (accumulate locally, reduce-scatter once) and the ZeRO-2 form
    (reduce-scatter every micro-step) give identical bits."""
    numels, n_ranks, K = [64 * 1000 + 7], 64, 4
    a = FlatUnit(numels, n_ranks)
    b = FlatUnit(numels, n_ranks, accum=True)
    m0 = synthetic.make_master_flat(a.P, n_ranks, 0.02, ("z1x",)).cuda()
    a.set_master_flat(m0)
    b.set_master_flat(m0)
    acc = aligned_rows(n_ranks, a.P_pad, torch.float32, "cuda", 0)
    gen = torch.Generator().manual_seed(5)
    for k in range(1, K + 1):
        q = torch.randint(-32, 32, (n_ranks, a.P_pad), generator=gen).float() / 1024.0
        q[:, a.P:] = 0
        g = q.to(torch.bfloat16).cuda()
        a.grads.copy_(g)
        b.grads.copy_(g)
        zf.zero1_accumulate(a.grad_rows(), rows(acc), k == 1, a.layout)
        zf.zero_step(b.grad_rows(), *b.state_rows(), b.accum_rows(), k, K, b.param_rows(),
                     b.layout, hp_at(1))
    zf.zero1_step(rows(acc), K, *a.state_rows(), a.param_rows(), a.layout, hp_at(1))
    torch.cuda.synchronize()
    for x, y in ((a.master, b.master), (a.m, b.m), (a.v, b.v)):
        assert torch.equal(x.contiguous().view(torch.int32), y.contiguous().view(torch.int32))
    assert torch.equal(a.params.contiguous().view(torch.int16),
                       b.params.contiguous().view(torch.int16))


@pytest.mark.parametrize("n_ranks", [1, 3, 8, 64])
def test_zero1_equals_plain_step_on_special_values(n_ranks):
    """With one micro-step the ZeRO-1 form sums the same values as the plain
    step (its fp32 accumulators are the exactly widened bf16 gradients) in the
    same rank order, so the two give identical bits: signed zeros,
    infinities, NaNs and subnormals included, in rank 0 (whose values start
    both sums without a two-sum) and in later ranks."""
    numels = [n_ranks * (2 * 4096 + 77) + 3]
    a = FlatUnit(numels, n_ranks)
    b = FlatUnit(numels, n_ranks)
    m0 = synthetic.make_master_flat(a.P, n_ranks, 0.02, ("z1s", n_ranks)).cuda()
    a.set_master_flat(m0)
    b.set_master_flat(m0)
    g = synthetic.make_grads(a.P, n_ranks, 1e-2, ("z1s", n_ranks))
    gi = g.view(torch.int16)
    rng = np.random.default_rng(n_ranks)
    specials = np.array([0x8000, 0x7F80, 0xFF80, 0x7FC0, 0x0001, 0x8001] * 16,
                        dtype=np.uint16).view(np.int16)
    for k in sorted({0, n_ranks - 1, n_ranks // 2}):
        pos = rng.choice(a.P, size=specials.size, replace=False)   # the padding stays zero
        gi[k, torch.from_numpy(pos)] = torch.from_numpy(specials)
    gi[:, :64] = torch.tensor(np.uint16(0x8000).view(np.int16))   # every rank -0
    g = g.cuda()
    a.grads.copy_(g)
    b.grads.copy_(g)
    acc = aligned_rows(n_ranks, a.P_pad, torch.float32, "cuda", 3.0)
    for t in (1, 2):
        zf.zero1_accumulate(a.grad_rows(), rows(acc), True, a.layout)
        zf.zero1_step(rows(acc), 1, *a.state_rows(), a.param_rows(), a.layout, hp_at(t))
        zf.zero_step(b.grad_rows(), *b.state_rows(), None, 1, 1, b.param_rows(), b.layout,
                     hp_at(t))
    torch.cuda.synchronize()
    for x, y in ((a.master, b.master), (a.m, b.m), (a.v, b.v)):
        assert torch.equal(x.contiguous().view(torch.int32), y.contiguous().view(torch.int32))
    assert torch.equal(a.params.contiguous().view(torch.int16),
                       b.params.contiguous().view(torch.int16))
    assert zf.zero_device_status() == zf.zero.ZERO_DEVICE_OK

