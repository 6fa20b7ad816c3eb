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
  of a rounding boundary).
"""
from __future__ import annotations

import numpy as np


def _fmt(idx, got, ref):
    return f"first bad index {idx}: got {got!r} ref {ref!r}"


def check_mean(got, ref, abs_mean_x, what="mean"):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    tol = 2.0 ** -23 * np.abs(ref) + 2.0 ** -35 * np.asarray(abs_mean_x, dtype=np.float64)
    bad = np.nonzero(np.abs(got - ref) > tol)[0]
    assert bad.size == 0, f"{what}: {bad.size} elements out of tolerance; " + \
        _fmt(bad[0], got[bad[0]], ref[bad[0]])


def check_state(name, got, ref, floor_scale=None):
    """master: |d| <= 1e-6|ref| + 1e-7; m, v: |d| <= 1e-6|ref| + 1e-7*max|ref|."""
    got = np.asarray(got, dtype=np.float64).ravel()
    ref = np.asarray(ref, dtype=np.float64).ravel()
    if name == "master":
        floor = 1e-7
    else:
        scale = floor_scale if floor_scale is not None else (np.max(np.abs(ref)) if ref.size else 0)
        floor = 1e-7 * scale
    tol = 1e-6 * np.abs(ref) + floor
    d = np.abs(got - ref)
    bad = np.nonzero(~(d <= tol))[0]
    assert bad.size == 0, f"{name}: {bad.size}/{ref.size} out of tolerance; " + \
        _fmt(bad[0], got[bad[0]], ref[bad[0]])
    return float(np.max(d / np.maximum(tol, 1e-300))) if ref.size else 0.0


def bf16_ordered(bits):
    b = np.asarray(bits).astype(np.int64) & 0xFFFF
    return np.where(b & 0x8000, -(b & 0x7FFF), b)


def check_bf16(got_bits, ref_bits, max_ulp=1, what="params"):
    d = np.abs(bf16_ordered(got_bits) - bf16_ordered(ref_bits))
    bad = np.nonzero(d > max_ulp)[0]
    assert bad.size == 0, f"{what}: {bad.size} bf16 values more than {max_ulp} ulp apart; " + \
        _fmt(bad[0], int(np.asarray(got_bits)[bad[0]]), int(np.asarray(ref_bits)[bad[0]]))
    return int(d.max()) if d.size else 0
