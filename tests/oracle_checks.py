"""Checks that pin the CPU oracle to what the pages and the mathematics fix.

Each ``check_*`` takes an oracle instance and raises AssertionError on a
mismatch.  ``test_oracle_numerics.py`` runs them on the real oracle and
``test_oracle_mutants.py`` runs them on copies of the oracle with a planted
mistake, to show that each plausible mistake is caught by at least one check.

Nothing here re-derives the oracle's formulas: the references are printed
values (golden fixtures), exact rational arithmetic (fractions), closed forms
of Adam on special inputs, identities of the method (reduce-scatter +
all-gather = all-reduce, sharded update = unsharded update, mean of equal
micro-batches), brute-force index scans and library routines (PyTorch's bf16
rounding, torch.optim.AdamW).
"""
from __future__ import annotations

import math
import random
from fractions import Fraction

import numpy as np
import torch

from conftest import read_golden

HP = dict(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.01)


# ----------------------------------------------------------------- helpers --

def torch_bf16_bits(x: np.ndarray) -> np.ndarray:
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def bits_to_f32(bits: np.ndarray) -> np.ndarray:
    return (bits.astype(np.uint32) << 16).view(np.float32)


def random_bf16(rng: np.random.Generator, shape, std) -> np.ndarray:
    return torch_bf16_bits(rng.normal(0.0, std, size=shape).astype(np.float32))


def f32_nearest(q: Fraction) -> np.float32:
    """Correctly rounded (ties to even) fp32 value of an exact rational."""
    c = np.float32(float(q))
    cands = [np.nextafter(c, np.float32(-np.inf)), c, np.nextafter(c, np.float32(np.inf))]
    best = None
    for x in cands:
        d = abs(Fraction(float(x)) - q)
        even = (int(np.array(x, dtype=np.float32).view(np.uint32)) & 1) == 0
        key = (d, not even)
        if best is None or key < best[0]:
            best = (key, x)
    return np.float32(best[1])


def brute_layout(numels, n_ranks):
    """Element-by-element scan: owner tensor of each flat slot, tail padding."""
    slots = []
    starts = []
    for t, n in enumerate(numels):
        starts.append(len(slots))
        slots += [t] * n
    P = len(slots)
    while len(slots) % n_ranks:
        slots.append(-1)
    return starts, P, len(slots), len(slots) // n_ranks, slots


# ------------------------------------------------------------------ checks --

def check_bf16_rounding(o):
    """RNE fp32 -> bf16 equals PyTorch's conversion (a library routine),
    including exact ties, subnormals and overflow to infinity."""
    rng = np.random.default_rng(1)
    raw = rng.integers(0, 1 << 32, size=20000, dtype=np.uint64).astype(np.uint32)
    ties = (rng.integers(0, 1 << 16, size=4000, dtype=np.uint32) << 16) | 0x8000
    near = (rng.integers(0, 1 << 16, size=4000, dtype=np.uint32) << 16) | \
        rng.choice(np.array([0x7FFF, 0x8001, 0x0001, 0xFFFF], dtype=np.uint32), size=4000)
    special = np.array([0, 0x80000000, 0x00000001, 0x007FFFFF, 0x7F7FFFFF, 0x7F7F8000,
                        0x7F800000, 0xFF800000, 0x3F808000, 0x3F818000], dtype=np.uint32)
    bits = np.concatenate([raw, ties, near, special]).view(np.float32)
    finite = ~np.isnan(bits)
    ours = o.round_to_bf16(bits)
    ref = torch_bf16_bits(bits)
    assert np.array_equal(ours[finite], ref[finite]), "bf16 rounding differs from PyTorch"
    assert np.all(np.isnan(bits_to_f32(ours[~finite])))


def check_bf16_widening(o):
    """Every bf16 pattern widens exactly and rounds back to itself."""
    all_bits = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    sample = all_bits[::37]
    wide = o.bf16_to_f32(sample)
    ref = torch.from_numpy(sample.view(np.int16).copy()).view(torch.bfloat16).float().numpy()
    ok = ~np.isnan(ref)
    assert np.array_equal(wide[ok].view(np.uint32), ref[ok].view(np.uint32))
    assert np.array_equal(o.round_to_bf16(wide[ok]), sample[ok])


def check_layout_bruteforce(o):
    """Flatten + tail pad + even split against an element-by-element scan
    for every rank count up to 8 and random small tensor lists."""
    rnd = random.Random(7)
    for _ in range(300):
        n_t = rnd.randint(1, 6)
        numels = [rnd.randint(0, 50) for _ in range(n_t)]
        if sum(numels) == 0:
            numels[0] = 1
        for n_ranks in range(1, 9):
            offsets, P, P_pad, S = o.flat_layout(numels, n_ranks)
            starts, bP, bP_pad, bS, slots = brute_layout(numels, n_ranks)
            assert list(offsets) == starts
            assert (P, P_pad, S) == (bP, bP_pad, bS)
            assert 0 <= P_pad - P < n_ranks
            # the shards tile [0, P_pad) and every slot has exactly one owner
            owners = [e // S for e in range(P_pad)]
            assert owners == sorted(owners) and set(owners) == set(range(n_ranks))
            for r in range(n_ranks):
                seg = slots[r * S:(r + 1) * S]
                assert len(seg) == S


def check_layout_rejects(o):
    import pytest
    for numels, n in (([], 4), ([0, 0], 4), ([3, -1], 2), ([5], 0)):
        with pytest.raises(ValueError):
            o.flat_layout(numels, n)


def check_rank_mean_exact(o):
    """Mean over ranks equals the correctly rounded exact rational mean."""
    rng = np.random.default_rng(2)
    for n_ranks in (1, 2, 3, 4, 5, 7, 8, 16, 64):
        g = random_bf16(rng, (n_ranks, 64), 1e-2)
        # heavy cancellation: rank n-1 cancels the sum of the others in some columns
        if n_ranks > 1:
            g[-1, :8] = torch_bf16_bits(-bits_to_f32(g[0, :8]))
        got = o.rank_mean(g)
        for i in range(g.shape[1]):
            q = sum(Fraction(float(x)) for x in bits_to_f32(g[:, i])) / n_ranks
            assert got[i] == f32_nearest(q), (n_ranks, i)


def check_reduce_scatter_structure(o):
    """Rank r's reduce-scatter output is slice r of the all-reduce, and the
    concatenation of all slices is the all-reduce (RS followed by AG = AR)."""
    rng = np.random.default_rng(3)
    for n_ranks, S in ((1, 5), (2, 7), (4, 3), (8, 9), (64, 2)):
        g = random_bf16(rng, (n_ranks, n_ranks * S), 1e-2)
        # make every column distinct in a way a transposed index would break
        g[:, :] = torch_bf16_bits(bits_to_f32(g) + np.arange(n_ranks * S, dtype=np.float32))
        rs = o.reduce_scatter(g)
        ar = o.all_reduce(g)
        assert rs.shape == (n_ranks, S)
        assert np.array_equal(rs.reshape(-1).view(np.uint32), ar.view(np.uint32))
        # brute force on the owning rank's slice
        for r in range(n_ranks):
            for i in range(S):
                q = sum(Fraction(float(x)) for x in bits_to_f32(g[:, r * S + i])) / n_ranks
                assert rs[r, i] == f32_nearest(q)


def check_all_gather(o):
    rng = np.random.default_rng(4)
    for n_ranks, S in ((1, 4), (3, 5), (8, 1)):
        shards = rng.integers(0, 1 << 16, size=(n_ranks, S)).astype(np.uint16)
        full = o.all_gather(shards)
        for e in range(n_ranks * S):
            assert full[e] == shards[e // S, e % S]


def check_mean_identity(o):
    """Mean of equal-size per-rank mean gradients = global-batch mean gradient;
    with an unequal tail batch the plain mean of rank means is wrong."""
    rng = np.random.default_rng(5)
    n_ranks, b, width = 4, 2, 16
    # per-sample gradients on a grid of 2^-8, small enough that every per-rank
    # mean is exactly a bf16 value
    samples = rng.integers(-64, 64, size=(n_ranks, b, width)) / 256.0
    rank_means = samples.mean(axis=1).astype(np.float32)
    bits = torch_bf16_bits(rank_means)
    assert np.array_equal(bits_to_f32(bits), rank_means)
    got = o.rank_mean(bits)
    for i in range(width):
        exact = sum(Fraction(float(s)) for s in samples[:, :, i].ravel()) / (n_ranks * b)
        assert Fraction(float(got[i])) == exact
    # unequal tail batch: last rank holds one sample, the others two.
    tail = samples.copy()
    tail_means = np.concatenate([tail[:-1].mean(axis=1), tail[-1:, :1].mean(axis=1)])
    tail_bits = torch_bf16_bits(tail_means.astype(np.float32))
    plain = o.rank_mean(tail_bits)
    weighted = (tail[:-1].sum(axis=(0, 1)) + tail[-1, 0]) / (b * (n_ranks - 1) + 1)
    assert np.max(np.abs(plain - weighted)) > 1e-4


def _worked_example():
    rows = {r[0]: r[1:] for r in read_golden("adam_worked_example.txt")}
    world = int(rows["world_size"][0])
    params = [float(x) for x in rows["params"]]
    return world, params, rows


def check_worked_example(o):
    """The pages' 4-rank x 8-parameter Adam step, checked to the printed digits."""
    world, params, rows = _worked_example()
    width = len(params)
    local = np.array([[((r + 1) * (i + 2) - 3) / 100.0 for i in range(width)]
                      for r in range(world)], dtype=np.float32)
    grads = torch_bf16_bits(local)
    S = width // world
    master = np.array(params, dtype=np.float32).reshape(world, S).copy()
    m = np.zeros_like(master)
    v = np.zeros_like(master)
    hp = dict(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.0)
    # averaged gradient: the printed 4-decimal values, up to the bf16 input rounding
    avg = o.all_reduce(grads)
    printed = np.array([float(x) for x in rows["averaged"]])
    bound = np.max(np.abs(bits_to_f32(grads) - local), axis=0) + 5e-5
    assert np.all(np.abs(avg - printed) <= bound + 1e-7)
    full = o.zero_step(grads, master, m, v, step=1, **hp)
    updated = [round(float(x), 6) for x in master.reshape(-1)]
    assert updated == [float(x) for x in rows["updated"]]
    # the gathered bf16 buffer is the rounding of the updated master
    assert np.array_equal(full, o.round_to_bf16(master.reshape(-1)))
    # the unsharded (DDP) path gives the same parameters: max_abs_diff = 0
    theta = np.array(params, dtype=np.float32)
    mm, vv = np.zeros_like(theta), np.zeros_like(theta)
    full_ddp = o.ddp_step(grads, theta, mm, vv, step=1, **hp)
    assert float(np.max(np.abs(theta - master.reshape(-1)))) == float(rows["max_abs_diff"][0])
    assert np.array_equal(full, full_ddp)


def _random_state(rng, n_ranks, P, std_g=1e-2):
    P_pad = -(-P // n_ranks) * n_ranks
    S = P_pad // n_ranks
    grads = np.zeros((n_ranks, P_pad), dtype=np.uint16)
    grads[:, :P] = random_bf16(rng, (n_ranks, P), std_g)
    theta = np.zeros(P_pad, dtype=np.float32)
    theta[:P] = rng.normal(0, 0.02, size=P).astype(np.float32)
    return grads, theta, S


def check_sharded_equals_unsharded(o):
    """ZeRO update == DDP update bit for bit, over several steps, with tail
    padding, for several rank counts; the padded tail stays zero."""
    rng = np.random.default_rng(6)
    for n_ranks, P in ((1, 10), (2, 9), (4, 37), (8, 61), (64, 300), (3, 1)):
        grads, theta, S = _random_state(rng, n_ranks, P)
        master = theta.reshape(n_ranks, S).copy()
        m = np.zeros_like(master)
        v = np.zeros_like(master)
        th, mm, vv = theta.copy(), np.zeros_like(theta), np.zeros_like(theta)
        for step in (1, 2, 3):
            grads_t = grads.copy()
            grads_t[:, :P] = random_bf16(rng, (n_ranks, P), 1e-2)
            full = o.zero_step(grads_t, master, m, v, step=step, **HP)
            full_ddp = o.ddp_step(grads_t, th, mm, vv, step=step, **HP)
            assert np.array_equal(master.reshape(-1).view(np.uint32), th.view(np.uint32))
            assert np.array_equal(m.reshape(-1).view(np.uint32), mm.view(np.uint32))
            assert np.array_equal(v.reshape(-1).view(np.uint32), vv.view(np.uint32))
            assert np.array_equal(full, full_ddp)
            assert np.all(full[P:] == 0) and np.all(master.reshape(-1)[P:] == 0)


def check_adam_first_step_closed_form(o):
    """Step 1 from m = v = 0: m_hat = g and v_hat = g^2, so the update is
    -lr * g / (|g| + eps) on top of the decoupled decay."""
    rng = np.random.default_rng(8)
    n = 512
    g = np.concatenate([rng.normal(0, 1e-3, n - 4), [1e-9, -3e-9, 2.5e-7, 0.0]]).astype(np.float32)
    theta0 = rng.normal(0, 0.02, n).astype(np.float32)
    theta = theta0.copy()
    m = np.zeros(n, np.float32)
    v = np.zeros(n, np.float32)
    o.adamw(theta, m, v, g, step=1, **HP)
    gd = g.astype(np.float64)
    expect = theta0.astype(np.float64) * (1 - HP["lr"] * HP["weight_decay"]) \
        - HP["lr"] * gd / (np.abs(gd) + HP["eps"])
    # m and v are stored in fp32, so m_hat and v_hat carry one fp32 rounding each;
    # the bound is a few fp32 roundings of the terms being combined.
    tol = 2.0 ** -21 * (np.abs(theta0.astype(np.float64)) + HP["lr"])
    assert np.all(np.abs(theta - expect) <= tol)
    assert np.allclose(m, 0.1 * gd, rtol=1e-6, atol=0)
    assert np.allclose(v, 0.001 * gd * gd, rtol=1e-6, atol=0)


def check_adam_constant_gradient(o):
    """With the same gradient every step the bias-corrected moments are exactly
    g and g^2, so theta_T = d^T theta_0 - lr * g/(|g|+eps) * sum_{j<T} d^j with
    d = 1 - lr * wd (decoupled decay)."""
    rng = np.random.default_rng(9)
    n, T = 256, 10
    g = rng.normal(0, 1e-3, n).astype(np.float32)
    theta0 = rng.normal(0, 0.02, n).astype(np.float32)
    theta, m, v = theta0.copy(), np.zeros(n, np.float32), np.zeros(n, np.float32)
    for t in range(1, T + 1):
        o.adamw(theta, m, v, g, step=t, **HP)
    d = 1 - HP["lr"] * HP["weight_decay"]
    gd = g.astype(np.float64)
    expect = d ** T * theta0 - HP["lr"] * gd / (np.abs(gd) + HP["eps"]) * sum(d ** j for j in range(T))
    assert np.max(np.abs(theta - expect)) < 1e-8
    assert np.allclose(m, (1 - 0.9 ** T) * gd, rtol=1e-5)
    assert np.allclose(v, (1 - 0.999 ** T) * gd * gd, rtol=1e-5)


def check_adam_zero_gradient(o):
    """g = 0: the moments stay 0 and theta decays geometrically; eps keeps the
    update finite (0 / (0 + eps) = 0)."""
    theta0 = np.linspace(-0.05, 0.05, 101).astype(np.float32)
    theta, m, v = theta0.copy(), np.zeros(101, np.float32), np.zeros(101, np.float32)
    g = np.zeros(101, np.float32)
    for t in range(1, 6):
        o.adamw(theta, m, v, g, step=t, **HP)
    assert np.all(m == 0) and np.all(v == 0)
    d = 1 - HP["lr"] * HP["weight_decay"]
    assert np.allclose(theta, theta0.astype(np.float64) * d ** 5, rtol=1e-6, atol=0)


def check_single_rank_matches_torch_adamw(o):
    """N_d = 1 (no sharding, the mean of one buffer is itself): ten steps of
    the oracle against torch.optim.AdamW (foreach=False) on the same fp32
    parameter, including gradients far below eps."""
    rng = np.random.default_rng(10)
    n, T = 400, 10
    theta0 = rng.normal(0, 0.02, n).astype(np.float32)
    master = theta0.reshape(1, n).copy()
    m = np.zeros_like(master)
    v = np.zeros_like(master)
    p = torch.nn.Parameter(torch.from_numpy(theta0.astype(np.float64).copy()))
    opt = torch.optim.AdamW([p], lr=HP["lr"], betas=(HP["beta1"], HP["beta2"]), eps=HP["eps"],
                            weight_decay=HP["weight_decay"], foreach=False)
    for t in range(1, T + 1):
        g = random_bf16(rng, (1, n), 1e-3)
        g[0, :20] = torch_bf16_bits(rng.normal(0, 1e-9, 20).astype(np.float32))
        o.zero_step(g, master, m, v, step=t, **HP)
        p.grad = torch.from_numpy(bits_to_f32(g[0]).astype(np.float64))
        opt.step()
        # re-sync torch's float64 state to the fp32 storage the method keeps
        st = opt.state[p]
        with torch.no_grad():
            p.copy_(torch.from_numpy(p.detach().numpy().astype(np.float32).astype(np.float64)))
            st["exp_avg"].copy_(torch.from_numpy(
                st["exp_avg"].numpy().astype(np.float32).astype(np.float64)))
            st["exp_avg_sq"].copy_(torch.from_numpy(
                st["exp_avg_sq"].numpy().astype(np.float32).astype(np.float64)))
    ref = p.detach().numpy()
    # torch keeps the unrounded m, v inside a step while the method stores them
    # in fp32 first: the two differ by a few fp32 roundings of the terms
    # (|theta| and lr), accumulated over the steps.
    assert np.all(np.abs(master[0] - ref) <= 2.0 ** -20 * (np.abs(ref) + HP["lr"]))
    st = opt.state[p]
    em, ev = st["exp_avg"].numpy(), st["exp_avg_sq"].numpy()
    assert np.all(np.abs(m[0] - em) <= 1e-6 * np.abs(em) + 1e-7 * np.max(np.abs(em)))
    assert np.all(np.abs(v[0] - ev) <= 1e-6 * np.abs(ev))


def check_accumulation_invariants(o):
    """Micro-step accumulation: K equal micro-batches give exactly the plain
    step; K = 1 with an accumulator is the plain step; accumulation-only
    micro-steps leave the optimizer state untouched; with exact sums the
    micro-batch order does not matter."""
    rng = np.random.default_rng(11)
    n_ranks, P = 4, 50
    grads, theta, S = _random_state(rng, n_ranks, P)
    base = theta.reshape(n_ranks, S)
    for K in (1, 2, 4):
        ma, mb = base.copy(), base.copy()
        m1, v1, m2, v2 = (np.zeros_like(base) for _ in range(4))
        acc = np.full_like(base, 123.0)     # garbage: step 1 must overwrite it
        for k in range(1, K + 1):
            full = o.zero_step(grads, ma, m1, v1, step=1, accum=acc, micro_step=k, n_micro=K, **HP)
            if k < K:
                assert full is None and np.array_equal(ma, base) and np.all(m1 == 0)
        full_plain = o.zero_step(grads, mb, m2, v2, step=1, **HP)
        assert np.array_equal(full, full_plain)
        assert np.array_equal(ma.view(np.uint32), mb.view(np.uint32))
    # order independence with exactly representable sums (multiples of 2^-10)
    mk = [torch_bf16_bits((rng.integers(-32, 32, size=(n_ranks, n_ranks * S)) / 1024.0)
                          .astype(np.float32)) for _ in range(4)]
    outs = []
    for order in ((0, 1, 2, 3), (3, 1, 0, 2)):
        ma = base.copy()
        m1, v1 = np.zeros_like(base), np.zeros_like(base)
        acc = np.zeros_like(base)
        for k, j in enumerate(order, start=1):
            full = o.zero_step(mk[j], ma, m1, v1, step=1, accum=acc, micro_step=k, n_micro=4, **HP)
        outs.append((full, ma.copy(), m1.copy()))
    assert np.array_equal(outs[0][0], outs[1][0])
    assert np.array_equal(outs[0][1], outs[1][1]) and np.array_equal(outs[0][2], outs[1][2])
    # and the averaged gradient is the exact mean over ranks and micro-batches:
    # m after step 1 is (1 - beta1) * mean, so compare through the oracle's adam
    exact = np.mean([bits_to_f32(x) for x in mk], axis=(0, 1)).astype(np.float32)
    ref_theta, ref_m, ref_v = base.reshape(-1).copy(), np.zeros(n_ranks * S, np.float32), \
        np.zeros(n_ranks * S, np.float32)
    o.adamw(ref_theta, ref_m, ref_v, exact, step=1, **HP)
    assert np.array_equal(outs[0][2].reshape(-1), ref_m)


def check_clip_coefficient_vs_torch(o):
    """The clip coefficient and the clipped gradients against
    torch.nn.utils.clip_grad_norm_ (a library routine), at norms where the
    1e-6 in the denominator matters and where clipping does not apply."""
    rng = np.random.default_rng(12)
    for scale, max_norm in ((1e-4, 1e-5), (1e-2, 0.05), (1.0, 1e3), (1e-3, 7e-4)):
        parts = [rng.normal(0, scale, n).astype(np.float32) for n in (17, 300, 1)]
        params = [torch.nn.Parameter(torch.zeros(len(x))) for x in parts]
        for p, x in zip(params, parts):
            p.grad = torch.from_numpy(x.copy())
        tnorm = float(torch.nn.utils.clip_grad_norm_(params, max_norm))
        total = sum(o.sum_squares(x) for x in parts)
        assert abs(np.sqrt(total) - tnorm) <= 1e-6 * tnorm
        coef = o.clip_coefficient(total, max_norm)
        for p, x in zip(params, parts):
            y = x.copy()
            o.scale(y, coef)
            ref = p.grad.numpy()
            assert np.all(np.abs(y - ref) <= 2e-6 * np.abs(ref) + 1e-30)
            if coef == 1.0:
                assert np.array_equal(y, x)


def check_clip_closed_forms(o):
    """A constant gradient c over n elements has norm |c|*sqrt(n): coef =
    max_norm / (|c| sqrt(n) + 1e-6) and the clipped norm is just under max_norm;
    below the threshold the coefficient is exactly 1."""
    g = np.full(64, 0.5, np.float32)          # norm exactly 4
    total = o.sum_squares(g)
    assert total == 16.0
    coef = o.clip_coefficient(total, 2.0)
    assert coef == np.float32(2.0 / (4.0 + 1e-6))
    y = g.copy()
    o.scale(y, coef)
    assert np.sqrt(o.sum_squares(y)) == pytest_approx(2.0 * 4.0 / (4.0 + 1e-6), 1e-7)
    assert o.clip_coefficient(total, 4.0 + 1e-5) == 1.0
    assert o.clip_coefficient(0.0, 1.0) == 1.0


def pytest_approx(x, rel):
    import pytest
    return pytest.approx(x, rel=rel)


def check_clipped_units_step_vs_torch(o):
    """N_d = 1, three units, ten steps: the oracle's clipped step against
    torch.nn.utils.clip_grad_norm_ over all parameters followed by
    torch.optim.AdamW (foreach=False); the norm spans every unit."""
    rng = np.random.default_rng(13)
    sizes = (33, 200, 7)
    units = []
    for n in sizes:
        theta0 = rng.normal(0, 0.02, n).astype(np.float32)
        units.append(dict(master=theta0.reshape(1, n).copy(), m=np.zeros((1, n), np.float32),
                          v=np.zeros((1, n), np.float32), theta0=theta0))
    params = [torch.nn.Parameter(torch.from_numpy(u["theta0"].astype(np.float64).copy()))
              for u in units]
    opt = torch.optim.AdamW(params, lr=HP["lr"], betas=(HP["beta1"], HP["beta2"]),
                            eps=HP["eps"], weight_decay=HP["weight_decay"], foreach=False)
    max_norm = 5e-3
    clipped_any = False
    for t in range(1, 11):
        for u, p in zip(units, params):
            u["grads"] = random_bf16(rng, (1, u["master"].shape[1]), 1e-3)
            p.grad = torch.from_numpy(bits_to_f32(u["grads"][0]).astype(np.float64))
        outs, norm, coef = o.clipped_units_step(units, max_norm=max_norm, step=t, **HP)
        clipped_any |= coef < 1.0
        tnorm = float(torch.nn.utils.clip_grad_norm_(params, max_norm))
        assert abs(norm - tnorm) <= 1e-9 * tnorm
        # the method clips fp32 gradients: round torch's clipped grads to fp32
        for p in params:
            p.grad.copy_(torch.from_numpy(p.grad.numpy().astype(np.float32).astype(np.float64)))
        opt.step()
        with torch.no_grad():
            for p in params:
                st = opt.state[p]
                p.copy_(torch.from_numpy(p.detach().numpy().astype(np.float32).astype(np.float64)))
                for key in ("exp_avg", "exp_avg_sq"):
                    st[key].copy_(torch.from_numpy(st[key].numpy().astype(np.float32)
                                                   .astype(np.float64)))
        for u, out in zip(units, outs):
            assert np.array_equal(out, o.round_to_bf16(u["master"].reshape(-1)))
    assert clipped_any
    for u, p in zip(units, params):
        ref = p.detach().numpy()
        assert np.all(np.abs(u["master"][0] - ref) <= 2.0 ** -20 * (np.abs(ref) + HP["lr"]))


def check_clip_nonfinite_vs_torch(o):
    """Non-finite gradients against torch.nn.utils.clip_grad_norm_ (no
    error_if_nonfinite): a NaN gradient makes the norm and the coefficient NaN
    and every clipped gradient NaN; an infinite one makes the norm infinite,
    the coefficient 0, its own element NaN (inf * 0) and every other gradient
    0."""
    rng = np.random.default_rng(15)
    for bad in (np.nan, np.inf):
        parts = [rng.normal(0, 1e-2, n).astype(np.float32) for n in (17, 40)]
        parts[1][5] = bad
        params = [torch.nn.Parameter(torch.zeros(len(x))) for x in parts]
        for p, x in zip(params, parts):
            p.grad = torch.from_numpy(x.copy())
        tnorm = float(torch.nn.utils.clip_grad_norm_(params, 1.0))
        total = sum(o.sum_squares(x) for x in parts)
        coef = o.clip_coefficient(total, 1.0)
        if np.isnan(bad):
            assert np.isnan(tnorm) and np.isnan(np.sqrt(total)) and np.isnan(coef)
        else:
            assert np.isinf(tnorm) and np.isinf(total) and coef == 0.0
        for p, x in zip(params, parts):
            y = x.copy()
            o.scale(y, coef)
            ref = p.grad.numpy()
            assert np.array_equal(np.isnan(y), np.isnan(ref))
            assert np.array_equal(y[~np.isnan(y)], ref[~np.isnan(ref)])


def check_zero1_accumulation(o):
    """ZeRO-1 (accumulate full gradients locally, one reduce-scatter at the end):
    with one micro-step it is the plain step; with K equal micro-batches
    (power-of-two K, exact sums) it is the plain step; with exactly
    representable gradients it equals the ZeRO-2 path (reduce-scatter every
    micro-step), because both reach the exact mean."""
    rng = np.random.default_rng(14)
    n_ranks, P = 4, 58
    grads, theta, S = _random_state(rng, n_ranks, P)
    base = theta.reshape(n_ranks, S)
    P_pad = n_ranks * S
    for K in (1, 2, 4):
        acc = np.full((n_ranks, P_pad), 7.0, np.float32)   # garbage: first micro-step resets
        for k in range(1, K + 1):
            o.zero1_accumulate(grads, acc, first=(k == 1))
        ma, m1, v1 = base.copy(), np.zeros_like(base), np.zeros_like(base)
        full = o.zero1_step(acc, ma, m1, v1, n_micro=K, step=1, **HP)
        mb, m2, v2 = base.copy(), np.zeros_like(base), np.zeros_like(base)
        full_plain = o.zero_step(grads, mb, m2, v2, step=1, **HP)
        assert np.array_equal(full, full_plain)
        assert np.array_equal(ma.view(np.uint32), mb.view(np.uint32))
        assert np.array_equal(m1.view(np.uint32), m2.view(np.uint32))
    mk = [torch_bf16_bits((rng.integers(-32, 32, size=(n_ranks, P_pad)) / 1024.0)
                          .astype(np.float32)) for _ in range(4)]
    acc = np.zeros((n_ranks, P_pad), np.float32)
    for k, g in enumerate(mk, start=1):
        o.zero1_accumulate(g, acc, first=(k == 1))
    # each rank's accumulator is the exact sum of its own micro-batches
    assert np.array_equal(acc, np.sum([bits_to_f32(g) for g in mk], axis=0).astype(np.float32))
    ma, m1, v1 = base.copy(), np.zeros_like(base), np.zeros_like(base)
    full1 = o.zero1_step(acc, ma, m1, v1, n_micro=4, step=1, **HP)
    mb, m2, v2 = base.copy(), np.zeros_like(base), np.zeros_like(base)
    acc2 = np.zeros_like(base)
    for k, g in enumerate(mk, start=1):
        full2 = o.zero_step(g, mb, m2, v2, step=1, accum=acc2, micro_step=k, n_micro=4, **HP)
    assert np.array_equal(full1, full2)
    assert np.array_equal(ma.view(np.uint32), mb.view(np.uint32))


def check_sampled_steps_equal_full_steps(o):
    """The sampled forms the full-size GPU tests use (the step on a subset of
    flat elements) give, on every element, the bits of the full step: the plain
    step (sampled_step vs zero_step, 3 steps with padding) and the ZeRO-1 step
    (sampled_zero1_step vs zero1_step, K = 3)."""
    rng = np.random.default_rng(15)
    n_ranks, P = 5, 83
    grads, theta, S = _random_state(rng, n_ranks, P)
    P_pad = n_ranks * S
    ma, m1, v1 = (theta.reshape(n_ranks, S).copy(), np.zeros((n_ranks, S), np.float32),
                  np.zeros((n_ranks, S), np.float32))
    sm, s_m, s_v = theta.copy(), np.zeros(P_pad, np.float32), np.zeros(P_pad, np.float32)
    for t in (1, 2, 3):
        full = o.zero_step(grads, ma, m1, v1, step=t, **HP)
        part = o.sampled_step(grads, sm, s_m, s_v, step=t, **HP)
        assert np.array_equal(full, part)
        assert np.array_equal(ma.reshape(-1).view(np.uint32), sm.view(np.uint32))
        assert np.array_equal(v1.reshape(-1).view(np.uint32), s_v.view(np.uint32))
    K = 3
    acc = np.zeros((n_ranks, P_pad), np.float32)
    for k in range(1, K + 1):
        g = random_bf16(rng, (n_ranks, P_pad), 1e-2)
        o.zero1_accumulate(g, acc, first=(k == 1))
    mb, m2, v2 = (theta.reshape(n_ranks, S).copy(), np.zeros((n_ranks, S), np.float32),
                  np.zeros((n_ranks, S), np.float32))
    full = o.zero1_step(acc, mb, m2, v2, n_micro=K, step=1, **HP)
    cols = np.array([0, 1, 7, S - 1, S, 2 * S + 3, P_pad - 1])
    sm, s_m, s_v = (theta[cols].copy(), np.zeros(cols.size, np.float32),
                    np.zeros(cols.size, np.float32))
    part = o.sampled_zero1_step(np.ascontiguousarray(acc[:, cols]), sm, s_m, s_v, n_micro=K,
                                step=1, **HP)
    assert np.array_equal(full[cols], part)
    assert np.array_equal(mb.reshape(-1)[cols].view(np.uint32), sm.view(np.uint32))
    assert np.array_equal(m2.reshape(-1)[cols].view(np.uint32), s_m.view(np.uint32))


def check_param_shard_bounds_vs_torch_chunk(o):
    """Per-parameter Shard(0): each rank's rows are the chunk torch.chunk gives
    (a library routine), in order, with no padding; chunks past the end are empty."""
    for dim0 in (1, 2, 3, 5, 7, 8, 9, 64, 65, 100, 4096):
        for n_ranks in (1, 2, 3, 4, 8, 64):
            for row in (1, 3, 768):
                sizes = [len(c) for c in torch.arange(dim0).chunk(n_ranks)]
                sizes += [0] * (n_ranks - len(sizes))
                prev = 0
                for r in range(n_ranks):
                    b, e = o.param_shard_bounds(dim0, row, n_ranks, r)
                    assert b == prev and e - b == sizes[r] * row
                    prev = e
                assert prev == dim0 * row


def check_param_sharded_step_equals_flat(o):
    """Per-parameter sharding changes which rank updates which element, not
    the update: the gathered parameters equal the unsharded (DDP) step on the
    same flat vector, bit for bit."""
    rng = np.random.default_rng(15)
    shapes = [(5, 3), (64, 7), (1, 11), (9, 1), (130, 2)]
    for n_ranks in (1, 3, 4, 8):
        params, flat_g, flat_t = [], [], []
        for (d0, row) in shapes:
            n = d0 * row
            g = random_bf16(rng, (n_ranks, n), 1e-2)
            t0 = rng.normal(0, 0.02, n).astype(np.float32)
            prm = dict(dim0=d0, row=row, grads=g, master=[], m=[], v=[])
            for r in range(n_ranks):
                b, e = o.param_shard_bounds(d0, row, n_ranks, r)
                prm["master"].append(t0[b:e].copy())
                prm["m"].append(np.zeros(e - b, np.float32))
                prm["v"].append(np.zeros(e - b, np.float32))
            params.append(prm)
            flat_g.append(g)
            flat_t.append(t0)
        for t in (1, 2):
            outs = o.param_sharded_step(params, step=t, **HP)
            if t == 1:
                G = np.ascontiguousarray(np.concatenate(flat_g, axis=1))
                theta = np.concatenate(flat_t)
                mm, vv = np.zeros_like(theta), np.zeros_like(theta)
                ref = o.ddp_step(G, theta, mm, vv, step=1, **HP)
                assert np.array_equal(np.concatenate(outs), ref)
        # the shards hold exactly the parameter's elements: no padding anywhere
        for prm, (d0, row) in zip(params, shapes):
            assert sum(len(x) for x in prm["master"]) == d0 * row


ALL_CHECKS = [
    check_bf16_rounding,
    check_bf16_widening,
    check_layout_bruteforce,
    check_layout_rejects,
    check_rank_mean_exact,
    check_reduce_scatter_structure,
    check_all_gather,
    check_mean_identity,
    check_worked_example,
    check_sharded_equals_unsharded,
    check_adam_first_step_closed_form,
    check_adam_constant_gradient,
    check_adam_zero_gradient,
    check_single_rank_matches_torch_adamw,
    check_accumulation_invariants,
    check_clip_coefficient_vs_torch,
    check_clip_closed_forms,
    check_clipped_units_step_vs_torch,
    check_clip_nonfinite_vs_torch,
    check_zero1_accumulation,
    check_sampled_steps_equal_full_steps,
    check_param_shard_bounds_vs_torch_chunk,
    check_param_sharded_step_equals_flat,
]
