"""The reference arm of bench.py (the CPU oracle) prints one JSON line with
every key the benchmark contract names; runs on the CPU in a few seconds."""
import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

KEYS = ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
        "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config", "impl",
        "cpu_baseline", "e2e")


def test_reference_arm_json_line():
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                          "--steps", "2", "--warmup", "3"],
                         capture_output=True, text=True, timeout=600, cwd=ROOT,
                         env=dict(os.environ, WORLD_SIZE="1", RANK="0", LOCAL_RANK="0"))
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [l for l in out.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for k in KEYS:
        assert k in d, k
    assert d["impl"] == "reference" and d["steps"] == 2 and d["warmup"] == 3
    assert d["value"] > 0 and d["ms_per_step"] > 0 and d["higher_is_better"] is True
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["d2h_bytes_per_step"] == 0
    # the default workload: the pages' 7.5B model as 32 units over 64 logical ranks
    assert d["config"]["workload"] == "7.5B-32units-Nd64"
    assert "x 64 ranks of the 7.5b workload" in d["cpu_baseline"]["sample"]


def test_threaded_oracle_baseline_computes_the_single_thread_result():
    """The CPU baseline steps one contiguous chunk per thread; the step is
    element-wise, so the chunks together must give the single-chunk bits."""
    import numpy as np
    sys.path.insert(0, ROOT)
    import bench
    runs = [bench.OracleRun(8 * 1024 + 40, t) for t in (1, 4)]
    for r in runs:
        r.step(1)
        r.step(2)
        r.close()
    one = [np.concatenate([c[i] for c in runs[0].chunks]) for i in (1, 2, 3)]
    four = [np.concatenate([c[i] for c in runs[1].chunks]) for i in (1, 2, 3)]
    for x, y in zip(one, four):
        assert x.shape == y.shape and np.array_equal(x.view(np.uint32), y.view(np.uint32))
    assert len(runs[1].chunks) == 4
