"""Tolerances of the CUDA path against the oracle.

Derivation (restated in the design notes):
* layout, offsets, padding, flatten copies: bit-exact (integer / copy work).
* reduce-scatter mean: the GPU sums the N_d bf16 values in fp32 with an
  error-free two-sum (compensated) and divides once; the oracle forms the
  exact sum in double and rounds once.  The compensated sum is within
  u*|s| + gamma_{N-1}^2 * sum|x| of the exact sum (u = 2^-24,
  gamma_n = n*u/(1-n*u)); with the final rounding and division this gives
  |mean_gpu - mean_ref| <= 2^-23*|mean_ref| + 2^-35 * mean(|x|)   (N_d <= 512).
* AdamW state after T steps: relative 1e-6, with an absolute floor of 1e-7
  for the master weights and of 1e-7 * max|ref| (per tensor) for m and v,
  whose values (~1e-4 and ~1e-9 here) make a literal 1e-7 floor vacuous.
* bf16 parameters: within 1 bf16 ulp (the fp32 masters may sit on either side
  of a rounding boundary), plus the masters' 1e-7 absolute floor where |theta|
  is so small that 1e-7 spans many bf16 ulps; >= 99.9 % bit-identical; and
  always exactly the round-to-nearest-even of the GPU's own fp32 masters.
"""
from __future__ import annotations

import os

import numpy as np

# Margins of every check made in this process, one record per call: printed
# as a table at the end of a pytest session (and written as JSON lines to
# $PARITY_MARGINS_JSON when that is set).
MARGINS = []


def _record(kind, what, **fields):
    test = os.environ.get("PYTEST_CURRENT_TEST", "").split(" ")[0]
    MARGINS.append(dict(test=test, kind=kind, what=what, **fields))


def _fmt(idx, got, ref):
    return f"first bad index {idx}: got {got!r} ref {ref!r}"


def check_mean(got, ref, abs_mean_x, what="mean"):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    tol = 2.0 ** -23 * np.abs(ref) + 2.0 ** -35 * np.asarray(abs_mean_x, dtype=np.float64)
    d = np.abs(got - ref)
    _record("mean", what, n=int(ref.size),
            max_over_tol=float(np.max(d / np.maximum(tol, 1e-300))) if ref.size else 0.0,
            max_f32_ulp=_max_f32_ulp(got, ref), exact=_exact_fraction(got, ref))
    bad = np.nonzero(d > tol)[0]
    assert bad.size == 0, f"{what}: {bad.size} elements out of tolerance; " + \
        _fmt(bad[0], got[bad[0]], ref[bad[0]])


def check_state(name, got, ref, floor_scale=None):
    """master: |d| <= 1e-6|ref| + 1e-7; m, v: |d| <= 1e-6|ref| + 1e-7*max|ref|.
    Records the largest relative error, the largest distance in fp32 ulps, the
    bit-identical fraction and how many elements pass only through the
    absolute floor."""
    got = np.asarray(got, dtype=np.float64).ravel()
    ref = np.asarray(ref, dtype=np.float64).ravel()
    if name == "master":
        floor = 1e-7
    else:
        scale = floor_scale if floor_scale is not None else (np.max(np.abs(ref)) if ref.size else 0)
        floor = 1e-7 * scale
    tol = 1e-6 * np.abs(ref) + floor
    d = np.abs(got - ref)
    # relative regime: elements where 1e-6 |ref| is at least the floor
    rel = 1e-6 * np.abs(ref) >= floor
    _record("state", name, n=int(ref.size), n_relative=int(np.count_nonzero(rel)),
            max_rel=float(np.max(d[rel] / np.abs(ref[rel]))) if rel.any() else 0.0,
            max_f32_ulp=_max_f32_ulp(got[rel], ref[rel]),
            max_abs_below_floor=float(np.max(d[~rel])) if (~rel).any() else 0.0,
            max_over_tol=float(np.max(d / np.maximum(tol, 1e-300))) if ref.size else 0.0,
            floor_only=int(np.count_nonzero((d > 1e-6 * np.abs(ref)) & (d <= tol))),
            exact=_exact_fraction(got, ref))
    bad = np.nonzero(~(d <= tol))[0]
    assert bad.size == 0, f"{name}: {bad.size}/{ref.size} out of tolerance; " + \
        _fmt(bad[0], got[bad[0]], ref[bad[0]])
    return float(np.max(d / np.maximum(tol, 1e-300))) if ref.size else 0.0


def _f32_ordered(x):
    """fp32 values as integers in value order (adjacent floats differ by 1)."""
    b = np.asarray(x, dtype=np.float32).view(np.int32).astype(np.int64)
    return np.where(b < 0, -(b & 0x7FFFFFFF), b)


def _max_f32_ulp(got, ref):
    if np.size(ref) == 0:
        return 0
    return int(np.max(np.abs(_f32_ordered(got) - _f32_ordered(ref))))


def _exact_fraction(got, ref):
    if np.size(ref) == 0:
        return 1.0
    g = np.asarray(got, dtype=np.float32)
    r = np.asarray(ref, dtype=np.float32)
    return float(np.mean(g.view(np.int32) == r.view(np.int32)))


def bf16_ordered(bits):
    b = np.asarray(bits).astype(np.int64) & 0xFFFF
    return np.where(b & 0x8000, -(b & 0x7FFF), b)


def bf16_value(bits):
    return (np.asarray(bits).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def bf16_ulp(bits):
    """Spacing of bf16 values at each element's magnitude (2^(e-7); subnormals 2^-133)."""
    b = np.asarray(bits).astype(np.int64)
    exp = (b >> 7) & 0xFF
    return np.where(exp == 0, 2.0 ** -133, np.ldexp(1.0, (np.maximum(exp, 1) - 127 - 7).astype(int)))


def check_bf16(got_bits, ref_bits, what="params", min_exact=0.999):
    """bf16 parameters: within one bf16 ulp of the reference, plus the master
    weights' absolute floor of 1e-7 (near zero the fp32 masters may differ by
    up to 1e-7, which is many bf16 ulps there); and almost all exactly equal."""
    got_bits = np.asarray(got_bits)
    ref_bits = np.asarray(ref_bits)
    d = np.abs(bf16_value(got_bits) - bf16_value(ref_bits))
    ulp = bf16_ulp(ref_bits)
    tol = ulp + 1e-7
    dist = np.abs(bf16_ordered(got_bits) - bf16_ordered(ref_bits)) if got_bits.size else \
        np.zeros(0, np.int64)
    floor_only = (d > ulp) & (d <= tol)
    _record("bf16", what, n=int(ref_bits.size),
            max_ulp=int(np.max(dist[~floor_only])) if (~floor_only).any() else 0,
            floor_only=int(np.count_nonzero(floor_only)),
            floor_only_max_ulp=int(np.max(dist[floor_only])) if floor_only.any() else 0,
            floor_only_max_abs_ref=float(np.max(np.abs(bf16_value(ref_bits)[floor_only])))
            if floor_only.any() else 0.0,
            exact=float(np.mean(got_bits == ref_bits)) if got_bits.size else 1.0)
    bad = np.nonzero(d > tol)[0]
    assert bad.size == 0, f"{what}: {bad.size} bf16 values out of tolerance; " + \
        _fmt(bad[0], int(got_bits[bad[0]]), int(ref_bits[bad[0]]))
    exact = float(np.mean(got_bits == ref_bits)) if got_bits.size else 1.0
    assert exact >= min_exact, f"{what}: only {exact:.6f} of bf16 values match exactly"
    return int(np.max(np.abs(bf16_ordered(got_bits) - bf16_ordered(ref_bits)))) \
        if got_bits.size else 0


def check_bf16_is_rounded_master(param_bits, master):
    """The gathered parameters are exactly RNE(master) (PyTorch's conversion)."""
    import torch
    m = torch.from_numpy(np.ascontiguousarray(master, dtype=np.float32))
    ref = m.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(np.asarray(param_bits, dtype=np.uint16), ref), \
        "gathered bf16 parameters are not the rounded master weights"
