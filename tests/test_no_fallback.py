"""The product path has no CPU fallback: with the CUDA library absent, every
entry point raises instead of computing, and nothing under the package
imports the oracle."""
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PKG = os.path.join(ROOT, "fsdp_sharded_mixed_flatten_gb300")

_PROBE = r"""
import sys
import fsdp_sharded_mixed_flatten_gb300 as zf
from fsdp_sharded_mixed_flatten_gb300 import zero as Z
Z.LIB_PATH = "/nonexistent/libzero_gb300.so"
calls = {
    "load": lambda: zf.load(),
    "zero_flat_layout": lambda: zf.zero_flat_layout([10, 6], 4),
    "zero_param_layout": lambda: zf.zero_param_layout(9, 3, 4),
}
for name, fn in calls.items():
    try:
        fn()
    except RuntimeError as e:
        assert "missing" in str(e), (name, str(e))
    else:
        print("NO-RAISE", name)
        sys.exit(1)
assert "oracle" not in sys.modules, "the product package imported the oracle"
print("ok")
"""


def test_entry_points_raise_without_library():
    out = subprocess.run([sys.executable, "-c", _PROBE], capture_output=True, text=True,
                         timeout=300, cwd=ROOT)
    assert out.returncode == 0, out.stdout + out.stderr[-2000:]
    assert out.stdout.strip().endswith("ok")


def test_package_sources_never_name_the_oracle_module():
    for dirpath, _, files in os.walk(PKG):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h", ".cpp")):
                text = open(os.path.join(dirpath, f), encoding="utf-8").read()
                for needle in ("import oracle", "from oracle", "zero_oracle"):
                    assert needle not in text, (f, needle)
