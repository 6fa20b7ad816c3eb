"""Tile order of the staged kernel.

Launches of at least 16 rounds of tiles (all but the norm passes) let the
CTAs claim their tiles after the first from a counter; short launches whose
tiles span several stages run in the fixed order on fewer CTAs than SMs.  The
results must depend on neither the order nor the grid: the same bits as the
direct-load kernels (fixed order, a CTA per SM), eagerly, replayed from a CUDA
graph, and on two streams at once.  Two launches forced onto one counter at
the same time must never corrupt results silently: wrong bits come with
ZERO_DEVICE_SCHED_CONFLICT.
"""
import pytest
import torch

from gpu_harness import hp_at

import fsdp_sharded_mixed_flatten_gb300 as zf
from fsdp_sharded_mixed_flatten_gb300 import synthetic
from fsdp_sharded_mixed_flatten_gb300.buffers import FlatUnit

pytestmark = pytest.mark.gpu

# N_d = 2 with S mod 8 = 7: ceil(S / 4096) * 2 = 4884 tiles, over 16 rounds of
# 152 CTAs, so the launch is dynamically scheduled (LEAD form)
BIG_N2 = ([20_000_013], 2)


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from fsdp_sharded_mixed_flatten_gb300 import build
    build.build()
    zf.load()


def _unit(spec, tag, accum=False):
    numels, n = spec
    u = FlatUnit(numels, n, accum=accum)
    u.set_master_flat(synthetic.make_master_flat(u.P, n, 0.02, (tag,)).cuda())
    return u


def _grads(u, t, tag):
    return synthetic.make_grads(u.P, u.n_ranks, 1e-2, (tag, t)).cuda()


def _bits(u):
    return [x.contiguous().view(torch.int32).clone() for x in (u.master, u.m, u.v)] + \
        [u.params.contiguous().view(torch.int16).clone()]


def _same(a, b):
    return all(torch.equal(x, y) for x, y in zip(a, b))


def _step(u, t, stream=None):
    zf.zero_step(u.grad_rows(), *u.state_rows(), None, 1, 1, u.param_rows(), u.layout, hp_at(t),
                 stream=stream)


def _staged_equals_direct(monkeypatch, spec, tag):
    """3 steps through the staged kernel and through the direct-load kernels
    (fixed order, a CTA per SM), bit for bit."""
    runs = {}
    for kern in ("staged", "direct"):
        if kern == "direct":
            monkeypatch.setenv("ZERO_STEP_KERNEL", "direct")
        else:
            monkeypatch.delenv("ZERO_STEP_KERNEL", raising=False)
        u = _unit(spec, tag)
        for t in (1, 2, 3):
            u.grads.copy_(_grads(u, t, tag))
            _step(u, t)
        torch.cuda.synchronize()
        runs[kern] = _bits(u)
    monkeypatch.delenv("ZERO_STEP_KERNEL", raising=False)
    assert _same(runs["staged"], runs["direct"])
    assert zf.zero_device_status() == zf.zero.ZERO_DEVICE_OK


def test_dynamic_order_equals_fixed_order(monkeypatch):
    """The staged kernel (dynamic order here) against the direct-load kernels."""
    _staged_equals_direct(monkeypatch, BIG_N2, "dyn-vs-fixed")


# Short launches in the fixed order whose tiles span several stages run on a
# balanced grid (fewer CTAs than SMs, every round full but the last):
#   N_d = 64, P = 1,048,589: S = 16,385 (S mod 8 = 1), 4 full tiles per rank
#     plus the tail group = 257 tiles in 2 rounds of 129 CTAs;
#   N_d = 16, P = 1,600,048: S = 100,003, 400 tiles in 3 rounds of 134 CTAs;
#   N_d = 32, P = 2,097,152: S = 65,536 (ALIGNED), 512 tiles in 4 rounds of 128;
#   N_d = 32, P = 1,051,776: S = 32,868 (S mod 8 = 4), 8 full tiles per rank
#     and a 100-element tail tile each = 288 tiles in 2 rounds of 144 CTAs.
SHORT_MULTI_STAGE = [([1_000_000, 48_589], 64), ([1_600_000, 48], 16), ([2_097_152], 32),
                     ([1_051_776], 32)]


@pytest.mark.parametrize("spec", SHORT_MULTI_STAGE,
                         ids=["Nd64_tail_group", "Nd16", "Nd32_aligned", "Nd32_tail100"])
def test_balanced_fixed_order_equals_direct(monkeypatch, spec):
    _staged_equals_direct(monkeypatch, spec, f"balanced-{spec[1]}")


def test_graph_replay_equals_eager():
    """Steps captured into a CUDA graph (capture counters) and replayed twice
    give the bits of the same steps run eagerly."""
    a, b = _unit(BIG_N2, "graph"), _unit(BIG_N2, "graph")
    g = _grads(a, 1, "graph")
    a.grads.copy_(g)
    b.grads.copy_(g)
    _step(a, 1)                       # warm-up outside capture (kernel attributes)
    _step(b, 1)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        for t in (2, 3):
            _step(a, t)
    for _ in range(2):
        graph.replay()
    torch.cuda.synchronize()
    for _ in range(2):
        for t in (2, 3):
            _step(b, t)
    torch.cuda.synchronize()
    assert _same(_bits(a), _bits(b))
    assert zf.zero_device_status() == zf.zero.ZERO_DEVICE_OK


def test_two_streams_at_once_equal_one_after_the_other():
    """Dynamically scheduled launches on two streams at once (each stream has
    its own counter) equal the same launches run one after the other."""
    specs = [BIG_N2, ([12_000_001], 1)]
    conc = [_unit(s, f"two-streams-{i}") for i, s in enumerate(specs)]
    seq = [_unit(s, f"two-streams-{i}") for i, s in enumerate(specs)]
    grads = [[_grads(u, t, f"ts{i}") for t in (1, 2, 3)] for i, u in enumerate(conc)]
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    torch.cuda.synchronize()
    for t in (1, 2, 3):
        for u, s, g in zip(conc, streams, grads):
            with torch.cuda.stream(s):
                u.grads.copy_(g[t - 1])
                _step(u, t, stream=s)
    torch.cuda.synchronize()
    for t in (1, 2, 3):
        for u, g in zip(seq, grads):
            u.grads.copy_(g[t - 1])
            _step(u, t)
    torch.cuda.synchronize()
    for a, b in zip(conc, seq):
        assert _same(_bits(a), _bits(b))
    assert zf.zero_device_status() == zf.zero.ZERO_DEVICE_OK


def test_per_thread_default_stream_from_two_threads():
    """The per-thread default stream handle (cudaStreamPerThread, 2) names a
    different stream in every host thread.  Dynamically scheduled launches
    from two threads on it at once use a counter each: no conflict is
    recorded and the bits equal the same steps run one after the other."""
    import threading
    per_thread = 2
    specs = [BIG_N2, ([12_000_001], 1)]
    conc = [_unit(s, f"per-thread-{i}") for i, s in enumerate(specs)]
    seq = [_unit(s, f"per-thread-{i}") for i, s in enumerate(specs)]
    for i, (a, b) in enumerate(zip(conc, seq)):
        g = _grads(a, 1, f"pt{i}")
        a.grads.copy_(g)
        b.grads.copy_(g)
    torch.cuda.synchronize()
    barrier = threading.Barrier(len(conc))
    errors = []

    def run(u):
        try:
            barrier.wait()
            for t in (1, 2, 3):
                _step(u, t, stream=per_thread)
        except Exception as e:          # reported by the main thread
            errors.append(e)

    threads = [threading.Thread(target=run, args=(u,)) for u in conc]
    for th in threads:
        th.start()
    for th in threads:
        th.join()
    torch.cuda.synchronize()
    assert not errors, errors
    assert zf.zero_device_status() == zf.zero.ZERO_DEVICE_OK
    for u in seq:
        for t in (1, 2, 3):
            _step(u, t)
    torch.cuda.synchronize()
    for a, b in zip(conc, seq):
        assert _same(_bits(a), _bits(b))


def test_shared_counter_conflict_is_reported(monkeypatch):
    """Failure injection: with ZERO_SCHED_SHARED every dynamic launch claims
    from one counter, so launches on two streams at once may take tiles from
    each other.  Wrong results then always come with ZERO_DEVICE_SCHED_CONFLICT
    (never silently); launches that did not overlap are right.  No wait is
    involved: every launch ends."""
    monkeypatch.setenv("ZERO_SCHED_SHARED", "1")
    specs = [BIG_N2, ([12_000_007], 2)]
    conc = [_unit(s, f"conflict-{i}") for i, s in enumerate(specs)]
    ref = [_unit(s, f"conflict-{i}") for i, s in enumerate(specs)]
    grads = [_grads(u, 1, f"cf{i}") for i, u in enumerate(conc)]
    for u, g in zip(conc + ref, grads + grads):
        u.grads.copy_(g)
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    torch.cuda.synchronize()
    for u, s in zip(conc, streams):
        with torch.cuda.stream(s):
            _step(u, 1, stream=s)
    torch.cuda.synchronize()
    status = zf.zero_device_status()
    monkeypatch.delenv("ZERO_SCHED_SHARED", raising=False)
    for u in ref:                      # one after the other, each on its own stream's counter
        _step(u, 1)
    torch.cuda.synchronize()
    right = all(_same(_bits(a), _bits(b)) for a, b in zip(conc, ref))
    assert status in (zf.zero.ZERO_DEVICE_OK, zf.zero.ZERO_DEVICE_SCHED_CONFLICT)
    if not right:
        assert status == zf.zero.ZERO_DEVICE_SCHED_CONFLICT
    assert zf.zero_device_status() == zf.zero.ZERO_DEVICE_OK
