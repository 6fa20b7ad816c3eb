"""The C-ABI library on the CPU: it loads, exports every function the header
declares, computes the FlatParameter layout bit-exactly like the oracle, and
rejects bad arguments before any launch.  No GPU work is done here."""
import ctypes
import random

import pytest

import fsdp_sharded_mixed_flatten_gb300 as zf
from fsdp_sharded_mixed_flatten_gb300 import synthetic
from fsdp_sharded_mixed_flatten_gb300.zero import header_functions


@pytest.fixture(scope="module")
def lib():
    from fsdp_sharded_mixed_flatten_gb300 import build
    build.build()
    return zf.load()


def test_exports_every_header_function(lib):
    names = header_functions()
    assert len(names) >= 10
    for name in names:
        assert hasattr(lib, name), f"{name} is declared in include/zero_flat.h but not exported"
    assert zf.zero_abi_version() == 1


def test_max_ranks_matches_header():
    import re
    import os
    hdr = open(os.path.join(os.path.dirname(zf.__file__), "..", "include", "zero_flat.h")).read()
    assert int(re.search(r"#define ZERO_MAX_RANKS (\d+)", hdr).group(1)) == zf.ZERO_MAX_RANKS


def test_layout_matches_oracle_bruteforce(lib, oracle):
    rnd = random.Random(11)
    for _ in range(400):
        numels = [rnd.randint(0, 40) for _ in range(rnd.randint(1, 7))]
        if sum(numels) == 0:
            numels[-1] = 3
        n_ranks = rnd.choice([1, 2, 3, 4, 5, 7, 8, 16, 64, 512])
        off, L = zf.zero_flat_layout(numels, n_ranks)
        o_off, P, P_pad, S = oracle.flat_layout(numels, n_ranks)
        assert off == list(o_off)
        assert (L.numel, L.numel_padded, L.shard_numel, L.n_ranks, L.n_tensors) == \
            (P, P_pad, S, n_ranks, len(numels))


@pytest.mark.parametrize("name", ["tiny", "gpt2-small", "llama3-8b-layer", "7.5b"])
def test_layout_of_workloads(lib, oracle, name):
    w = synthetic.workload(name)
    for u in w.units[:2] + w.units[-1:]:
        off, L = zf.zero_flat_layout(u.numels, w.n_ranks)
        o_off, P, P_pad, S = oracle.flat_layout(u.numels, w.n_ranks)
        assert off == list(o_off) and (L.numel, L.numel_padded, L.shard_numel) == (P, P_pad, S)
    if name == "7.5b":
        assert (L.numel, L.numel_padded, L.shard_numel) == (234_375_000, 234_375_040, 3_662_110)
    if name == "llama3-8b-layer":
        assert L.numel == 218_112_000 and L.shard_numel == 3_408_000
    if name == "gpt2-small":
        assert sum(u.numel for u in w.units) == 124_439_808


def test_large_counts_use_64_bit(lib):
    off, L = zf.zero_flat_layout([4 ** 15 + 13] * 3, 64)
    assert L.numel == 3 * (4 ** 15 + 13)
    assert L.numel_padded % 64 == 0 and L.numel_padded - L.numel < 64
    assert off[2] == 2 * (4 ** 15 + 13)


def test_shard_segments_bruteforce(lib):
    rnd = random.Random(12)
    for _ in range(200):
        numels = [rnd.randint(0, 30) for _ in range(rnd.randint(1, 6))]
        if sum(numels) == 0:
            numels[0] = 5
        n_ranks = rnd.randint(1, 9)
        off, L = zf.zero_flat_layout(numels, n_ranks)
        owner = []
        for t, n in enumerate(numels):
            owner += [(t, i) for i in range(n)]
        owner += [(-1, e) for e in range(L.numel, L.numel_padded)]
        for r in range(n_ranks):
            segs = zf.zero_shard_segments(L, off, numels, r)
            got = []
            for t, b, e in segs:
                assert b < e
                got += [(t, i) for i in range(b, e)]
            assert got == owner[r * L.shard_numel:(r + 1) * L.shard_numel]


def test_layout_rejects_bad_input(lib):
    for numels, n in (([], 4), ([0, 0], 4), ([3, -1], 2), ([5], 0), ([5], -3)):
        with pytest.raises(zf.ZeroError) as ei:
            zf.zero_flat_layout(numels, n)
        assert ei.value.code == -1
    with pytest.raises(zf.ZeroError) as ei:
        zf.zero_flat_layout([2 ** 62, 2 ** 62], 2)
    assert ei.value.code == -3


HP = dict(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.01, step=1)


def test_step_rejects_bad_arguments_before_launch(lib):
    """Only argument checks run here: every call below fails validation, so
    nothing reaches CUDA (the addresses are never dereferenced)."""
    off, L = zf.zero_flat_layout([100], 4)
    good = [0x10000 * (i + 1) for i in range(4)]
    bad = [0x10000 * (i + 1) + 2 for i in range(4)]
    cases = [
        (dict(grads=[0] * 4), -1),                      # NULL gradient pointer
        (dict(grads=bad), -2),                          # misaligned gradient pointer
        (dict(master=bad), -2),
        (dict(hp=dict(HP, step=0)), -1),                # step < 1
        (dict(hp=dict(HP, beta2=1.0)), -1),             # beta out of range
        (dict(hp=dict(HP, lr=float("nan"))), -1),       # non-finite
        (dict(micro_step=2, n_micro=4), -1),            # micro-stepping without accumulator
        (dict(full=[]), -1),                            # no output buffer
    ]
    for over, code in cases:
        args = dict(grads=good, master=good, m=good, v=good, full=[0x90000], hp=HP,
                    micro_step=1, n_micro=1)
        args.update(over)
        with pytest.raises(zf.ZeroError) as ei:
            zf.zero_step(args["grads"], args["master"], args["m"], args["v"], None,
                         args["micro_step"], args["n_micro"], args["full"], L, args["hp"],
                         stream=0)
        assert ei.value.code == code, (over, ei.value)


def test_inconsistent_layout_rejected(lib):
    off, L = zf.zero_flat_layout([100], 4)
    good = [0x10000 * (i + 1) for i in range(4)]
    broken = zf.ZeroLayout(L.n_tensors, L.numel, L.numel_padded + 4, L.shard_numel + 1, 4, 0)
    with pytest.raises(zf.ZeroError) as ei:
        zf.zero_reduce_scatter(good, good, broken, 0, stream=0)
    assert ei.value.code == -3
    too_many = zf.ZeroLayout(1, 1024, 1024, 1, 1024, 0)
    with pytest.raises(zf.ZeroError) as ei:
        zf.zero_reduce_scatter(good, good, too_many, 0, stream=0)
    assert ei.value.code == -3


def test_error_message_is_per_call(lib):
    with pytest.raises(zf.ZeroError):
        zf.zero_flat_layout([], 1)
    assert "n_tensors" in zf.zero_last_error()
    zf.zero_flat_layout([3], 1)
    assert zf.zero_last_error() == ""


def test_host_step_rejects_bad_arguments_before_any_copy(lib):
    """zero_step_units_host validates everything before it queues a copy: a
    NULL host gradient row, unknown flags and a broken layout are rejected
    (the fake addresses are never dereferenced)."""
    off, L = zf.zero_flat_layout([100], 4)
    good = [0x10000 * (i + 1) for i in range(4)]
    unit = (good, good, good, good, None, [0x90000], L)
    host_ok = [[0x200000 * (i + 1) for i in range(4)]]
    host_null = [[0x200000, 0, 0x600000, 0x800000]]
    with pytest.raises(zf.ZeroError) as ei:
        zf.zero_step_units_host([unit], (host_null, None), 1, 1, HP, 0, 0, 0, 0)
    assert ei.value.code == -1 and "NULL gradient" in zf.zero_last_error()
    with pytest.raises(zf.ZeroError) as ei:
        zf.zero_step_units_host([unit], (host_ok, None), 1, 1, HP, 6, 0, 0, 0)
    assert ei.value.code == -1 and "flags" in zf.zero_last_error()
    broken = zf.ZeroLayout(L.n_tensors, L.numel, L.numel_padded + 4, L.shard_numel + 1, 4, 0)
    with pytest.raises(zf.ZeroError) as ei:
        zf.zero_step_units_host([(good, good, good, good, None, [0x90000], broken)],
                                (host_ok, None), 1, 1, HP, 0, 0, 0, 0)
    assert ei.value.code == -3
    # the step's own checks also run before any copy is queued
    with pytest.raises(zf.ZeroError) as ei:
        zf.zero_step_units_host([unit], (host_ok, None), 1, 1, dict(HP, step=0), 0, 0, 0, 0)
    assert ei.value.code == -1
    bad = [0x10000 * (i + 1) + 2 for i in range(4)]
    with pytest.raises(zf.ZeroError) as ei:
        zf.zero_step_units_host([(good, bad, good, good, None, [0x90000], L)], (host_ok, None),
                                1, 1, HP, 0, 0, 0, 0)
    assert ei.value.code == -2


def test_injected_cuda_failure_is_reported(lib, monkeypatch):
    """While ZERO_INJECT_FAILURE names a CUDA call, that call is skipped and
    the entry point returns ZERO_ERR_CUDA with the call's label (the fake
    addresses below are checked but never dereferenced)."""
    off, L = zf.zero_flat_layout([100], 4)
    good = [0x10000 * (i + 1) for i in range(4)]
    for kernel, label in (("staged", "staged launch: step"), ("direct", "fused step launch")):
        if kernel == "direct":
            monkeypatch.setenv("ZERO_STEP_KERNEL", "direct")
        monkeypatch.setenv("ZERO_INJECT_FAILURE", label)
        with pytest.raises(zf.ZeroError) as ei:
            zf.zero_step(good, good, good, good, None, 1, 1, [0x90000], L, HP, stream=0)
        assert ei.value.code == -4
        assert zf.zero_last_error() == label + ": injected failure"
    monkeypatch.setenv("ZERO_INJECT_FAILURE", "all-gather")
    with pytest.raises(zf.ZeroError) as ei:
        zf.zero_all_gather(good, [0x90000], L, stream=0)
    assert zf.zero_last_error() == "all-gather launch: injected failure"
    # argument checks still come first
    monkeypatch.setenv("ZERO_INJECT_FAILURE", "launch")
    with pytest.raises(zf.ZeroError) as ei:
        zf.zero_step(good, good, good, [0] * 4, None, 1, 1, [0x90000], L, HP, stream=0)
    assert ei.value.code == -1
