"""Seeded random configurations through the staged and direct fused kernels
and through the unfused entry points, against the oracle: tensor lists with
empty and odd-sized tensors, rank counts from 1 to 130, one to three gathered
outputs, one to three micro-steps."""
import random

import pytest
import torch

from gpu_harness import Case

import fsdp_sharded_mixed_flatten_gb300 as zf

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from fsdp_sharded_mixed_flatten_gb300 import build
    build.build()
    zf.load()


def configs(n, seed):
    rng = random.Random(seed)
    out = []
    for i in range(n):
        n_ranks = rng.choice([1, 2, 3, 4, 5, 7, 8, 9, 16, 31, 64, 65, 130])
        n_tensors = rng.randint(1, 6)
        numels = [rng.choice([0, 1, 7, 8, 13, 4095, 4096, 4097, rng.randint(1, 300000)])
                  for _ in range(n_tensors)]
        if sum(numels) == 0:
            numels[0] = rng.randint(1, 50000)
        out.append((i, numels, n_ranks, rng.randint(1, 3), rng.randint(1, 3)))
    return out


@pytest.mark.parametrize("kernel", ["staged", "direct", "unfused"])
@pytest.mark.parametrize("idx,numels,n_ranks,n_out,n_micro", configs(12, 20261202))
def test_random_configuration(oracle, monkeypatch, kernel, idx, numels, n_ranks, n_out, n_micro):
    if kernel == "direct":
        monkeypatch.setenv("ZERO_STEP_KERNEL", "direct")
    else:
        monkeypatch.delenv("ZERO_STEP_KERNEL", raising=False)
    c = Case(numels, n_ranks, n_out=n_out, n_micro=n_micro, tag=("random", idx),
             path="unfused" if kernel == "unfused" else "fused")
    for t in (1, 2):
        c.step(oracle, t)
    c.compare()
    assert zf.zero_device_status() == zf.zero.ZERO_DEVICE_OK
