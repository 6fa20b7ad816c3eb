"""Shared test configuration.

Tests marked ``gpu`` need a CUDA device and the compiled CUDA library; the
rest run on the CPU.
"""
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

GOLDEN = os.path.join(ROOT, "tests", "golden")


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU and the compiled CUDA library")
    config.addinivalue_line("markers", "slow: large sizes; still part of the normal runs")


@pytest.fixture(scope="session")
def oracle():
    from oracle import Oracle
    return Oracle()


def read_golden(name):
    """Return the non-comment lines of a golden fixture as lists of tokens."""
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            rows.append(line.split())
    return rows


def pytest_terminal_summary(terminalreporter):
    """Parity margins of the session: per test and array, the worst case over
    every check made (relative error, fp32 / bf16 ulp distance, bit-identical
    fraction, elements passing only through the absolute floor)."""
    try:
        import parity
    except ImportError:
        return
    if not parity.MARGINS:
        return
    import json
    out = os.environ.get("PARITY_MARGINS_JSON")
    if out:
        with open(out, "w") as f:
            for rec in parity.MARGINS:
                f.write(json.dumps(rec) + "\n")
    agg = {}
    for rec in parity.MARGINS:
        key = (rec["test"], rec["kind"], rec["what"])
        a = agg.setdefault(key, dict(n=0, checks=0, max_rel=0.0, max_ulp=0, exact=1.0,
                                     floor_only=0, max_over_tol=0.0, floor_only_max_ulp=0,
                                     floor_only_max_abs_ref=0.0))
        a["checks"] += 1
        a["n"] += rec["n"]
        a["max_rel"] = max(a["max_rel"], rec.get("max_rel", 0.0))
        a["max_ulp"] = max(a["max_ulp"], rec.get("max_ulp", rec.get("max_f32_ulp", 0)))
        a["exact"] = min(a["exact"], rec["exact"])
        a["floor_only"] += rec.get("floor_only", 0)
        a["max_over_tol"] = max(a["max_over_tol"], rec.get("max_over_tol", 0.0))
        a["floor_only_max_ulp"] = max(a["floor_only_max_ulp"], rec.get("floor_only_max_ulp", 0))
        a["floor_only_max_abs_ref"] = max(a["floor_only_max_abs_ref"],
                                          rec.get("floor_only_max_abs_ref", 0.0))
    tr = terminalreporter
    tr.write_sep("=", "parity margins (worst over each test's checks)")
    tr.write_line(f"{'test':60s} {'array':8s} {'elements':>11s} {'max rel':>9s} "
                  f"{'max ulp':>7s} {'min exact':>9s} {'floor-only':>10s} {'d/tol':>6s}")
    for (test, kind, what), a in sorted(agg.items()):
        name = test[-60:]
        tr.write_line(f"{name:60s} {what[:8]:8s} {a['n']:11d} {a['max_rel']:9.2e} "
                      f"{a['max_ulp']:7d} {a['exact']:9.6f} {a['floor_only']:10d} "
                      f"{a['max_over_tol']:6.3f}")
    tot = {}
    for (test, kind, what), a in agg.items():
        t = tot.setdefault(what, dict(n=0, max_rel=0.0, max_ulp=0, exact=1.0, floor_only=0,
                                      max_over_tol=0.0, floor_only_max_ulp=0,
                                      floor_only_max_abs_ref=0.0))
        t["n"] += a["n"]
        for k in ("max_rel", "max_ulp", "max_over_tol", "floor_only_max_ulp",
                  "floor_only_max_abs_ref"):
            t[k] = max(t[k], a[k])
        t["exact"] = min(t["exact"], a["exact"])
        t["floor_only"] += a["floor_only"]
    tr.write_sep("-", "all tests (max rel and max ulp: where the relative criterion binds)")
    for what, t in sorted(tot.items()):
        tr.write_line(f"{what:8s} elements {t['n']:d}  max rel {t['max_rel']:.2e}  "
                      f"max ulp {t['max_ulp']}  min exact {t['exact']:.6f}  "
                      f"max d/tol {t['max_over_tol']:.3f}  floor-only {t['floor_only']} "
                      f"(max ulp {t['floor_only_max_ulp']}, |ref| <= "
                      f"{t['floor_only_max_abs_ref']:.2e})")
