"""CUDA path against the oracle, element by element, through the C ABI.

Sizes here are ones the oracle finishes in seconds; they span many CTA tiles,
ragged shard ends, every realignment of the gradient slices (S mod 8), padded
tails, rank counts on both sides of the 64-pointer argument block, several
all-gather destinations and micro-step accumulation.
"""
import numpy as np
import pytest
import torch

import parity
from gpu_harness import Case, bits, hp_at

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


def test_tiny_config_ten_steps(oracle):
    """3 tensors 4096x1024, 1024, 1000; N_d = 4; 10 AdamW steps."""
    w = synthetic.workload("tiny")
    c = Case(w.units[0].numels, w.n_ranks, grad_std=w.grad_std, tag="tiny")
    assert c.S % 8 == 2       # rank slices start off the 16-byte grid
    for t in range(1, w.steps + 1):
        c.step(oracle, t)
    c.compare()


CASES = [
    # (name, numels, n_ranks, n_out, n_micro, steps)
    ("one_rank", [12345], 1, 1, 1, 3),
    ("fewer_elements_than_ranks", [5], 8, 1, 1, 3),
    ("odd_shard_every_realignment", [1000003], 8, 1, 1, 3),
    ("padded_end_not_multiple_of_8", [999999], 3, 1, 1, 3),
    ("many_tensors_some_empty", [0, 7, 4099, 0, 1, 65536, 3], 4, 1, 1, 2),
    ("ranks_64_small_shards", [64 * 37 + 5], 64, 1, 1, 3),
    ("ranks_65", [65 * 1000 + 7], 65, 1, 1, 2),
    ("ranks_512", [512 * 33 + 1], 512, 1, 1, 2),
    ("gather_to_every_rank", [10007], 4, 4, 1, 2),
    ("accumulate_4_micro_steps", [100003], 8, 1, 4, 2),
    ("accumulate_3_micro_steps", [40001], 5, 2, 3, 2),
    # every shard a multiple of 8 elements: the kernels' aligned forms
    ("aligned_two_ranks", [2 * 8 * 5000], 2, 1, 1, 3),
    ("aligned_one_rank_two_outputs", [8 * 1111, 8 * 7], 1, 2, 1, 2),
    ("aligned_eight_ranks_two_outputs", [8 * 8 * 3001], 8, 2, 1, 2),
    ("aligned_accumulate_3_micro_steps", [16 * 8 * 777], 16, 1, 3, 2),
    # shards ending in a tail of 13..509 elements at N_d > 8: one short tile
    # per rank spanning several stages (S = 4196: 100-element tails, the last
    # rank's ending past the buffer's last full 16 bytes; S = 8701: S mod 8 = 5;
    # S = 4109 with N_d = 9)
    ("ranks_64_tail_100_two_group_tiles", [64 * 4196 - 3], 64, 1, 1, 2),
    ("ranks_16_tail_509", [16 * 8701], 16, 1, 1, 2),
    ("ranks_9_tail_13", [9 * 4109 - 4], 9, 2, 1, 2),
]


@pytest.fixture(params=["staged", "direct", "unfused"])
def kernel(request, monkeypatch):
    """Run a test with the bulk-copy staged fused kernel (default), again with
    the direct-load kernels, and again through the unfused entry points
    (zero_reduce_scatter, zero_adamw_shard_step, zero_all_gather)."""
    if request.param == "direct":
        monkeypatch.setenv("ZERO_STEP_KERNEL", "direct")
    else:
        monkeypatch.delenv("ZERO_STEP_KERNEL", raising=False)
    yield request.param
    assert zf.zero_device_status() == zf.zero.ZERO_DEVICE_OK


@pytest.mark.parametrize("name,numels,n_ranks,n_out,n_micro,steps", CASES,
                         ids=[c[0] for c in CASES])
def test_small_cases(oracle, kernel, name, numels, n_ranks, n_out, n_micro, steps):
    c = Case(numels, n_ranks, n_out=n_out, n_micro=n_micro, tag=name,
             path="unfused" if kernel == "unfused" else "fused")
    for t in range(1, steps + 1):
        c.step(oracle, t)
    c.compare()


@pytest.mark.parametrize("numels,n_ranks,n_micro", [([4096 * 1024, 1024, 1000], 4, 1),
                                                    ([999999], 3, 1), ([64 * 4099 + 5], 64, 2),
                                                    ([77777], 65, 3), ([5], 8, 1),
                                                    ([2 * 8 * 70001], 2, 1),
                                                    ([8 * 8 * 1234], 8, 2),
                                                    ([64 * 4196 - 3], 64, 1),
                                                    ([16 * 8701], 16, 1)])
def test_staged_equals_direct_bitwise(monkeypatch, numels, n_ranks, n_micro):
    """The bulk-copy staged kernels and the direct-load kernels give identical bits."""
    units = {}
    master0 = synthetic.make_master_flat(sum(numels),
                                         n_ranks, 0.02, ("sd",)).cuda()
    for kern in ("staged", "direct"):
        if kern == "direct":
            monkeypatch.setenv("ZERO_STEP_KERNEL", "direct")
        else:
            monkeypatch.delenv("ZERO_STEP_KERNEL", raising=False)
        u = FlatUnit(numels, n_ranks, n_out=2, accum=True)
        u.set_master_flat(master0)
        for t in (1, 2):
            for k in range(1, n_micro + 1):
                g = synthetic.make_grads(u.P, n_ranks, 1e-2, ("sd", t, k)).cuda()
                u.grads.copy_(g)
                zf.zero_step(u.grad_rows(), *u.state_rows(),
                             u.accum_rows() if n_micro > 1 else None, k, n_micro,
                             u.param_rows(), u.layout, hp_at(t))
        # and a plain reduce-scatter of the last gradients
        rs = aligned_rows(n_ranks, u.S, torch.float32, "cuda", 0)
        zf.zero_reduce_scatter(u.grad_rows(), rows(rs), u.layout, 0)
        torch.cuda.synchronize()
        units[kern] = (u, rs)
    monkeypatch.delenv("ZERO_STEP_KERNEL", raising=False)
    (a, rsa), (b, rsb) = units["staged"], units["direct"]
    for x, y in ((a.master, b.master), (a.m, b.m), (a.v, b.v), (rsa, rsb)):
        assert torch.equal(x.contiguous().view(torch.int32), y.contiguous().view(torch.int32))
    assert torch.equal(a.params.contiguous().view(torch.int16),
                       b.params.contiguous().view(torch.int16))
    assert zf.zero_device_status() == zf.zero.ZERO_DEVICE_OK


def test_bounded_wait_reports_timeout():
    """A barrier wait that nothing satisfies runs out, is reported, and the
    context stays usable for the next step."""
    assert zf.zero_device_status() == zf.zero.ZERO_DEVICE_OK
    zf.zero_selftest_wait_timeout(20_000_000)          # 20 ms
    assert zf.zero_device_status(clear=True) == zf.zero.ZERO_DEVICE_TIMEOUT
    assert zf.zero_device_status() == zf.zero.ZERO_DEVICE_OK
    u = FlatUnit([4099], 4)
    u.grads.normal_()
    zf.zero_step(u.grad_rows(), *u.state_rows(), None, 1, 1, u.param_rows(), u.layout, hp_at(1))
    torch.cuda.synchronize()
    assert zf.zero_device_status() == zf.zero.ZERO_DEVICE_OK


def test_late_step_bias_corrections(oracle):
    c = Case([30011], 4, tag="late", hp_over=dict(weight_decay=0.1))
    c.step(oracle, 10_000)
    c.step(oracle, 10_001)
    c.compare()


def test_outliers_and_zero_gradients(oracle):
    c = Case([200003], 16, tag="outliers", outlier_frac=0.05, grad_std=1e-3)
    c.step(oracle, 1)
    c.unit.grads.zero_()
    # a step with all-zero gradients: the moments decay, theta decays
    hp = hp_at(2)
    zf.zero_step(c.unit.grad_rows(), *c.unit.state_rows(), None, 1, 1, c.unit.param_rows(),
                 c.unit.layout, hp)
    zeros = np.zeros((c.n_ranks, c.P_pad), dtype=np.uint16)
    c.o_params = oracle.zero_step(zeros, c.o_master, c.o_m, c.o_v, lr=hp["lr"],
                                  beta1=hp["beta1"], beta2=hp["beta2"], eps=hp["eps"],
                                  weight_decay=hp["weight_decay"], step=2)
    c.compare()


@pytest.mark.parametrize("numels,n_ranks", [([4096 * 1024, 1024, 1000], 4), ([1000003], 8),
                                            ([64 * 1001 + 3], 64), ([77777], 65)])
def test_reduce_scatter_mean(oracle, numels, n_ranks):
    """The averaged gradient shard itself against the exact mean."""
    u = FlatUnit(numels, n_ranks, accum=True)
    g = synthetic.make_grads(u.P, n_ranks, 1e-2, ("rs", n_ranks), outlier_frac=0.01)
    # heavy cancellation in a few columns: rank n-1 cancels rank 0
    if n_ranks > 1:
        g[-1, :64] = -g[0, :64]
    u.grads.copy_(g.cuda())
    zf.zero_reduce_scatter(u.grad_rows(), u.accum_rows(), u.layout, 0)
    got = u.accum.cpu().numpy().reshape(-1)
    gb = bits(g)
    ref = oracle.reduce_scatter(gb).reshape(-1)
    absmean = np.abs(g.float().numpy()).mean(axis=0)
    parity.check_mean(got, ref, absmean)
    exact = np.count_nonzero(got.view(np.uint32) == ref.view(np.uint32)) / got.size
    assert exact > 0.999, f"only {exact:.5f} of the means are correctly rounded"


@pytest.mark.parametrize("numels,n_ranks,n_micro", [([4096 * 1024, 1024, 1000], 4, 1),
                                                    ([1000003], 8, 1), ([64 * 999 + 1], 64, 2),
                                                    ([3001], 65, 3)])
def test_fused_equals_unfused_bitwise(numels, n_ranks, n_micro):
    """zero_step is bit-identical to reduce-scatter + AdamW + all-gather."""
    units = [FlatUnit(numels, n_ranks, n_out=2, accum=True) for _ in range(2)]
    master0 = synthetic.make_master_flat(units[0].P, n_ranks, 0.02, ("fu",)).cuda()
    for u in units:
        u.set_master_flat(master0)
    pshards = aligned_rows(n_ranks, units[0].S, torch.bfloat16, "cuda", 0)
    for t in (1, 2):
        hp = hp_at(t)
        for k in range(1, n_micro + 1):
            g = synthetic.make_grads(units[0].P, n_ranks, 1e-2, ("fu", t, k)).cuda()
            for u in units:
                u.grads.copy_(g)
            a = units[0]
            zf.zero_step(a.grad_rows(), *a.state_rows(), a.accum_rows() if n_micro > 1 else None,
                         k, n_micro, a.param_rows(), a.layout, hp)
            b = units[1]
            zf.zero_reduce_scatter(b.grad_rows(), b.accum_rows(), b.layout, 1 if k > 1 else 0)
            if k == n_micro:
                zf.zero_adamw_shard_step(*b.state_rows(), b.accum_rows(), float(n_micro),
                                         rows(pshards), b.layout, hp)
                zf.zero_all_gather(rows(pshards), b.param_rows(), b.layout)
    torch.cuda.synchronize()
    a, b = units
    for x, y in ((a.master, b.master), (a.m, b.m), (a.v, b.v)):
        assert torch.equal(x.contiguous().view(torch.int32), y.contiguous().view(torch.int32))
    assert torch.equal(a.params.contiguous().view(torch.int16),
                       b.params.contiguous().view(torch.int16))
    assert torch.equal(a.params[0], a.params[1])


def test_flatten_unflatten(oracle):
    shapes = [(33, 7), (0,), (1000,), (5, 5, 5), (1,), (4099,)]
    numels = [int(np.prod(s)) for s in shapes]
    n_ranks = 8
    off, L = zf.zero_flat_layout(numels, n_ranks)
    o_off, P, P_pad, S = oracle.flat_layout(numels, n_ranks)
    assert off == list(o_off)
    gen = torch.Generator().manual_seed(3)
    tens = [torch.randn(s, generator=gen).to(torch.bfloat16).cuda() for s in shapes]
    flat = aligned_rows(1, P_pad, torch.bfloat16, "cuda", 7)  # junk in the padding
    zf.zero_flatten(tens, off, numels, 2, rows(flat), 0, L)
    ref = torch.zeros(P_pad, dtype=torch.bfloat16)
    ref[:P] = torch.cat([t.reshape(-1).cpu() for t in tens])
    torch.cuda.synchronize()
    assert torch.equal(flat[0].cpu().view(torch.int16), ref.view(torch.int16))
    # fp32 into per-rank shards (master weights), then back out
    tens32 = [torch.randn(s, generator=gen).cuda() for s in shapes]
    shards = aligned_rows(n_ranks, S, torch.float32, "cuda", -1.0)
    zf.zero_flatten(tens32, off, numels, 4, rows(shards), 1, L)
    ref32 = torch.zeros(P_pad)
    ref32[:P] = torch.cat([t.reshape(-1).cpu() for t in tens32])
    torch.cuda.synchronize()
    assert torch.equal(shards.cpu().reshape(-1), ref32)
    back = [torch.full_like(t, 9.0) for t in tens32]
    zf.zero_unflatten(rows(shards), 1, off, numels, 4, back, L)
    torch.cuda.synchronize()
    for x, y in zip(back, tens32):
        assert torch.equal(x, y)


def test_misaligned_pointer_rejected_without_launch():
    u = FlatUnit([1000], 4)
    g = u.grad_rows()
    bad = [int(x.data_ptr()) + 2 for x in g]
    with pytest.raises(zf.ZeroError) as ei:
        zf.zero_step(bad, *u.state_rows(), None, 1, 1, u.param_rows(), u.layout, hp_at(1))
    assert ei.value.code == -2


def _units(specs, n_out=1, accum=False, tag="units"):
    out = []
    for i, (numels, n_ranks) in enumerate(specs):
        u = FlatUnit(numels, n_ranks, n_out=n_out, accum=accum)
        u.set_master_flat(synthetic.make_master_flat(u.P, n_ranks, 0.02, (tag, i)).cuda())
        out.append(u)
    return out


def _unit_tuple(u, accum):
    return (u.grad_rows(), *u.state_rows(), u.accum_rows() if accum else None, u.param_rows(),
            u.layout)


@pytest.mark.parametrize("n_micro", [1, 3])
@pytest.mark.parametrize("specs", [
    # GPT-2-small-like: 12 equal blocks + a bigger root unit (scaled down), N_d = 8
    [([768, 768, 9000, 300], 8)] * 12 + [([50000, 7000, 5], 8)],
    # more units than fit one launch, mixed rank counts and ragged shards
    [([1000 + 37 * i], 1 + (i % 9)) for i in range(80)],
    # pointer-limited packing: 64 ranks per unit -> at most 13 units per launch
    [([64 * 53 + i], 64) for i in range(20)],
    # 512-element tails at N_d = 64, 12 units in one launch
    [([64 * 4608 - i], 64) for i in range(12)],
    # tails of 9..453 elements at assorted N_d > 8
    [([n * (4096 + 9 + 37 * i) - i % 3], n)
     for i, n in enumerate([9, 16, 33, 64, 64, 100, 12, 64, 17, 64, 128, 64, 64])],
], ids=["gpt2_like", "80_units_mixed", "pointer_limited", "long_tails_64_ranks",
        "long_tails_mixed"])
def test_step_units_equals_per_unit_steps(kernel, specs, n_micro):
    """zero_step_units over many FlatParameters is bit-identical to one
    zero_step per unit."""
    acc = n_micro > 1
    a_units = _units(specs, n_out=2, accum=acc)
    b_units = _units(specs, n_out=2, accum=acc)
    for t in (1, 2):
        for k in range(1, n_micro + 1):
            for i, (a, b) in enumerate(zip(a_units, b_units)):
                g = synthetic.make_grads(a.P, a.n_ranks, 1e-2, ("su", i, t, k)).cuda()
                a.grads.copy_(g)
                b.grads.copy_(g)
            zf.zero_step_units([_unit_tuple(a, acc) for a in a_units], k, n_micro, hp_at(t))
            for b in b_units:
                zf.zero_step(b.grad_rows(), *b.state_rows(), b.accum_rows() if acc else None, k,
                             n_micro, b.param_rows(), b.layout, hp_at(t))
    torch.cuda.synchronize()
    for a, b in zip(a_units, b_units):
        for x, y in ((a.master, b.master), (a.m, b.m), (a.v, b.v)):
            assert torch.equal(x.contiguous().view(torch.int32), y.contiguous().view(torch.int32))
        assert torch.equal(a.params.contiguous().view(torch.int16),
                           b.params.contiguous().view(torch.int16))


# bf16 bit patterns: -0, +inf, -inf, NaN, the smallest subnormals of both signs
SPECIAL_BF16 = [0x8000, 0x7F80, 0xFF80, 0x7FC0, 0x0001, 0x8001]


@pytest.mark.parametrize("n_ranks", [1, 2, 3, 8, 64])
def test_special_values_staged_equals_direct(monkeypatch, n_ranks):
    """Signed zeros, infinities, NaNs and subnormals, in rank 0 (whose values
    start the staged kernel's sums without a two-sum) and in later ranks, give
    the same bits through the staged kernel and the direct-load kernels, whose
    sums start from (0, 0)."""
    P = n_ranks * (2 * 4096 + 77) + 3
    g = synthetic.make_grads(P, n_ranks, 1e-2, ("special", n_ranks))
    gi = g.view(torch.int16)
    rng = np.random.default_rng(n_ranks)
    for k in sorted({0, n_ranks - 1, n_ranks // 2}):
        pos = rng.choice(P, size=96, replace=False)     # the padding stays zero
        vals = np.array(SPECIAL_BF16 * 16, dtype=np.uint16).view(np.int16)
        gi[k, torch.from_numpy(pos)] = torch.from_numpy(vals)
    # every rank -0 at a few elements (the sum's sign of zero)
    gi[:, :64] = torch.tensor(np.uint16(0x8000).view(np.int16))
    master0 = synthetic.make_master_flat(P, n_ranks, 0.02, ("special-m", n_ranks))
    master0[:32] = -0.0
    runs = {}
    for kern in ("staged", "direct"):
        if kern == "direct":
            monkeypatch.setenv("ZERO_STEP_KERNEL", "direct")
        else:
            monkeypatch.delenv("ZERO_STEP_KERNEL", raising=False)
        u = FlatUnit([P], n_ranks, n_out=1)
        u.set_master_flat(master0.cuda())
        u.grads.copy_(g.cuda())
        for t in (1, 2):
            zf.zero_step(u.grad_rows(), *u.state_rows(), None, 1, 1, u.param_rows(), u.layout,
                         hp_at(t))
        rs = aligned_rows(n_ranks, u.S, torch.float32, "cuda", 0)
        zf.zero_reduce_scatter(u.grad_rows(), rows(rs), u.layout, 0)
        torch.cuda.synchronize()
        runs[kern] = [x.contiguous().view(torch.int32).clone() for x in (u.master, u.m, u.v, rs)] + \
            [u.params.contiguous().view(torch.int16).clone()]
    monkeypatch.delenv("ZERO_STEP_KERNEL", raising=False)
    for x, y in zip(runs["staged"], runs["direct"]):
        assert torch.equal(x, y)
    assert zf.zero_device_status() == zf.zero.ZERO_DEVICE_OK


def test_step_units_against_oracle(oracle):
    """Three units of different shapes stepped together, each checked against
    the oracle."""
    cases = [Case([4099, 17], 4, tag="su0"), Case([100003], 8, tag="su1"),
             Case([64 * 77 + 3], 64, tag="su2")]
    for t in (1, 2, 3):
        grads = []
        for c in cases:
            g = c.grads_for(t, 1)
            c.unit.grads.copy_(g.cuda())
            grads.append(g)
        zf.zero_step_units([_unit_tuple(c.unit, False) for c in cases], 1, 1, hp_at(t))
        for c, g in zip(cases, grads):
            hp = hp_at(t)
            c.o_params = oracle.zero_step(bits(g), c.o_master, c.o_m, c.o_v, lr=hp["lr"],
                                          beta1=hp["beta1"], beta2=hp["beta2"], eps=hp["eps"],
                                          weight_decay=hp["weight_decay"], step=t)
    for c in cases:
        c.compare()


def test_prepared_units_same_as_list():
    """Units marshalled once (prepare_units) step exactly like a fresh list."""
    specs = [([768, 9000], 8), ([50000, 5], 8), ([64 * 33 + 1], 64)]
    a_units, b_units = _units(specs, tag="pu"), _units(specs, tag="pu")
    prepared = zf.zero.prepare_units([_unit_tuple(a, False) for a in a_units])
    for t in (1, 2, 3):
        for i, (a, b) in enumerate(zip(a_units, b_units)):
            g = synthetic.make_grads(a.P, a.n_ranks, 1e-2, ("pu", i, t)).cuda()
            a.grads.copy_(g)
            b.grads.copy_(g)
        zf.zero_step_units(prepared, 1, 1, hp_at(t))
        zf.zero_step_units([_unit_tuple(b, False) for b in b_units], 1, 1, hp_at(t))
    torch.cuda.synchronize()
    for a, b in zip(a_units, b_units):
        assert torch.equal(a.master.contiguous().view(torch.int32),
                           b.master.contiguous().view(torch.int32))
        assert torch.equal(a.params.contiguous().view(torch.int16),
                           b.params.contiguous().view(torch.int16))
