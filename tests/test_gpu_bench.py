"""bench.py on the GPU: every variant prints one JSON line with the contract's
keys, on small workloads (seconds each)."""
import json
import os
import subprocess
import sys

import pytest
import torch

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
KEYS = ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
        "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config", "roofline",
        "cpu_baseline", "e2e", "gpu_launches", "clocks")


def _run(*extra):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--steps", "3",
                          "--warmup", "3", "--no-extra", "--no-cpu", *extra],
                         capture_output=True, text=True, timeout=900, cwd=ROOT,
                         env=dict(os.environ, WORLD_SIZE="1", RANK="0", LOCAL_RANK="0"))
    assert out.returncode == 0, out.stderr[-3000:]
    lines = [l for l in out.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    return json.loads(lines[0])


def test_plain_with_host_leg():
    d = _run("--workload", "tiny")
    for k in KEYS:
        assert k in d, k
    assert d["value"] > 0 and d["gpu_launches"] == 3
    assert d["e2e"]["value"] > 0 and d["e2e"]["h2d_bytes_per_step"] > 0
    # the tiny workload: P = 4096*1024 + 1024 + 1000 = P_pad (divisible by N_d = 4);
    # N_d bf16 gradient rows in, one bf16 parameter buffer out, every step
    p_pad = 4196328
    assert d["e2e"]["h2d_bytes_per_step"] == 4 * p_pad * 2
    assert d["e2e"]["d2h_bytes_per_step"] == p_pad * 2
    assert "ZERO_HOST_SM_COPY" in d["e2e"]["transport"]
    assert d["roofline"]["bound"] == "hbm" and d["roofline"]["frac"] > 0


@pytest.mark.parametrize("variant,workload", [("clip", "tiny"), ("per-param", "gpt2-small"),
                                              ("zero1", "sweep:1048576:8")])
def test_variants(variant, workload):
    d = _run("--workload", workload, "--variant", variant, "--no-e2e")
    assert d["config"]["variant"] == variant
    assert d["value"] > 0 and d["roofline"]["achieved"] > 0 and d["gpu_launches"] > 0


def test_streamed_host_leg_byte_counts():
    """The 7.5B model's end-to-end leg (gradients streamed unit by unit from
    host memory through two device buffers) on a small stand-in: 4 units of
    100,003 elements sharing one gradient buffer, N_d = 8."""
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    sys.path.insert(0, ROOT)
    import bench
    from fsdp_sharded_mixed_flatten_gb300 import synthetic
    w = synthetic.Workload("streamed-test", tuple(synthetic.Unit(f"u{i}", (100003,))
                                                  for i in range(4)), 8, 1e-3)
    res = bench.Resident(w, shared_grads=True)
    assert all(fu.grads is res.units[0].grads for fu in res.units)
    p_pad = synthetic.padded(100003, 8)
    el, h2d, d2h, n_rows = bench.time_e2e_streamed(res, 2, 1, 1, torch.device("cuda", 0))
    assert el > 0 and 1 <= n_rows <= 8
    assert h2d == 4 * 8 * p_pad * 2 and d2h == 4 * p_pad * 2
