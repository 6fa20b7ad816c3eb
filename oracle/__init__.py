"""CPU oracle for the ZeRO / FSDP sharded mixed-precision FlatParameter step.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this package.  The product library
(the CUDA path) never imports it, and the two share no code: the oracle's
arithmetic lives in ``zero_oracle.c`` (plain scalar C, double arithmetic, fp32 /
bf16 stores) and in ``ledger.py`` (pure-Python memory and communication
formulas).  This module only compiles the C file with gcc and marshals numpy
arrays into it.

Sources are cited per function in ``zero_oracle.c`` and ``ledger.py`` by page
title and section.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "zero_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "liboracle.so")

# Exactly the arithmetic that is written: no contraction into fused
# multiply-add and no fast-math reassociation.
CFLAGS = ["-O2", "-fPIC", "-shared", "-std=c11", "-ffp-contract=off", "-fno-fast-math"]

_lock = threading.Lock()
_lib = None


def build(force: bool = False, src: str = _SRC, out: str = _LIB_PATH) -> str:
    """Compile ``zero_oracle.c`` into a shared library (gcc); return its path."""
    os.makedirs(os.path.dirname(out), exist_ok=True)
    stale = force or not os.path.exists(out) or os.path.getmtime(out) < os.path.getmtime(src)
    if stale:
        tmp = out + f".tmp{os.getpid()}"
        cmd = ["gcc", *CFLAGS, "-o", tmp, src, "-lm"]
        subprocess.run(cmd, check=True, capture_output=True, text=True)
        os.replace(tmp, out)
    return out


def _declare(lib: ctypes.CDLL) -> ctypes.CDLL:
    i32, i64, f64 = ctypes.c_int32, ctypes.c_int64, ctypes.c_double
    p = ctypes.c_void_p
    lib.oracle_bf16_to_f32.argtypes = [ctypes.c_uint16]
    lib.oracle_bf16_to_f32.restype = ctypes.c_float
    lib.oracle_f32_to_bf16.argtypes = [ctypes.c_float]
    lib.oracle_f32_to_bf16.restype = ctypes.c_uint16
    lib.oracle_round_to_bf16.argtypes = [p, i64, p]
    lib.oracle_round_to_bf16.restype = None
    lib.oracle_flat_layout.argtypes = [p, i64, i32, p, p]
    lib.oracle_flat_layout.restype = ctypes.c_int
    lib.oracle_rank_mean.argtypes = [p, i32, i64, i64, p]
    lib.oracle_rank_mean.restype = None
    lib.oracle_reduce_scatter.argtypes = [p, i32, i64, p]
    lib.oracle_reduce_scatter.restype = None
    lib.oracle_all_reduce.argtypes = [p, i32, i64, p]
    lib.oracle_all_reduce.restype = None
    lib.oracle_accumulate.argtypes = [p, p, i64, i32]
    lib.oracle_accumulate.restype = None
    lib.oracle_average_micro.argtypes = [p, i64, i32, p]
    lib.oracle_average_micro.restype = None
    lib.oracle_adamw.argtypes = [p, p, p, p, i64, f64, f64, f64, f64, f64, i64]
    lib.oracle_adamw.restype = None
    lib.oracle_all_gather.argtypes = [p, i32, i64, p]
    lib.oracle_all_gather.restype = None
    lib.oracle_param_shard_bounds.argtypes = [i64, i64, i32, i32, p, p]
    lib.oracle_param_shard_bounds.restype = None
    lib.oracle_zero1_accumulate.argtypes = [p, p, i32, i64, i32]
    lib.oracle_zero1_accumulate.restype = None
    lib.oracle_zero1_step.argtypes = [p, i32, i64, i32, p, p, p, p, f64, f64, f64, f64, f64, i64]
    lib.oracle_zero1_step.restype = ctypes.c_int
    lib.oracle_sum_squares.argtypes = [p, i64]
    lib.oracle_sum_squares.restype = f64
    lib.oracle_clip_coefficient.argtypes = [f64, f64]
    lib.oracle_clip_coefficient.restype = ctypes.c_float
    lib.oracle_scale.argtypes = [p, i64, ctypes.c_float]
    lib.oracle_scale.restype = None
    lib.oracle_zero_step.argtypes = [p, p, p, p, p, i32, i32, p, i32, i64,
                                     f64, f64, f64, f64, f64, i64]
    lib.oracle_zero_step.restype = ctypes.c_int
    lib.oracle_ddp_step.argtypes = [p, p, p, p, p, i32, i64, f64, f64, f64, f64, f64, i64]
    lib.oracle_ddp_step.restype = ctypes.c_int
    return lib


def load(path: str | None = None) -> ctypes.CDLL:
    """Load (building first if needed) the oracle library.

    ``path`` loads another build of the same source (tests that plant a
    mistake in a copy of the oracle use it); the default is cached.
    """
    global _lib
    if path is not None:
        return _declare(ctypes.CDLL(path))
    with _lock:
        if _lib is None:
            _lib = _declare(ctypes.CDLL(build()))
        return _lib


def _ptr(a: np.ndarray) -> int:
    assert a.flags["C_CONTIGUOUS"], "oracle arrays must be C-contiguous"
    return a.ctypes.data


def _u16(a) -> np.ndarray:
    a = np.ascontiguousarray(a)
    if a.dtype != np.uint16:
        raise TypeError("bf16 data is passed as uint16 bit patterns")
    return a


def _f32(a) -> np.ndarray:
    a = np.ascontiguousarray(a)
    if a.dtype != np.float32:
        raise TypeError("expected float32")
    return a


class Oracle:
    """numpy-facing wrapper over one build of the C oracle."""

    def __init__(self, lib: ctypes.CDLL | None = None):
        self.lib = lib if lib is not None else load()

    # -- bf16 -------------------------------------------------------------
    def bf16_to_f32(self, bits) -> np.ndarray:
        bits = _u16(bits)
        return np.array([self.lib.oracle_bf16_to_f32(int(b)) for b in bits.ravel()],
                        dtype=np.float32).reshape(bits.shape)

    def round_to_bf16(self, x) -> np.ndarray:
        x = _f32(x)
        out = np.empty(x.shape, dtype=np.uint16)
        self.lib.oracle_round_to_bf16(_ptr(x), x.size, _ptr(out))
        return out

    # -- layout -----------------------------------------------------------
    def flat_layout(self, numels, n_ranks: int):
        """Return (offsets, P, P_pad, S) or raise ValueError."""
        numels = np.ascontiguousarray(np.asarray(numels, dtype=np.int64))
        offsets = np.zeros(max(len(numels), 1), dtype=np.int64)
        out3 = np.zeros(3, dtype=np.int64)
        rc = self.lib.oracle_flat_layout(_ptr(numels), len(numels), int(n_ranks),
                                         _ptr(offsets), _ptr(out3))
        if rc != 0:
            raise ValueError("numels and n_ranks must be positive")
        return offsets[: len(numels)].copy(), int(out3[0]), int(out3[1]), int(out3[2])

    # -- collectives ------------------------------------------------------
    def rank_mean(self, grads) -> np.ndarray:
        """grads: (n_ranks, n) uint16 -> (n,) float32 mean over ranks."""
        grads = _u16(grads)
        n_ranks, n = grads.shape
        out = np.empty(n, dtype=np.float32)
        self.lib.oracle_rank_mean(_ptr(grads), n_ranks, n, n, _ptr(out))
        return out

    def reduce_scatter(self, grads) -> np.ndarray:
        """grads: (n_ranks, P_pad) uint16 -> (n_ranks, S) float32."""
        grads = _u16(grads)
        n_ranks, P_pad = grads.shape
        if P_pad % n_ranks:
            raise ValueError("P_pad must be a multiple of n_ranks")
        S = P_pad // n_ranks
        out = np.empty((n_ranks, S), dtype=np.float32)
        self.lib.oracle_reduce_scatter(_ptr(grads), n_ranks, S, _ptr(out))
        return out

    def all_reduce(self, grads) -> np.ndarray:
        grads = _u16(grads)
        n_ranks, P_pad = grads.shape
        out = np.empty(P_pad, dtype=np.float32)
        self.lib.oracle_all_reduce(_ptr(grads), n_ranks, P_pad, _ptr(out))
        return out

    def all_gather(self, shards) -> np.ndarray:
        shards = _u16(shards)
        n_ranks, S = shards.shape
        out = np.empty(n_ranks * S, dtype=np.uint16)
        self.lib.oracle_all_gather(_ptr(shards), n_ranks, S, _ptr(out))
        return out

    # -- optimizer --------------------------------------------------------
    def accumulate(self, acc, g, first: bool) -> None:
        acc, g = _f32(acc), _f32(g)
        self.lib.oracle_accumulate(_ptr(acc), _ptr(g), acc.size, int(bool(first)))

    def average_micro(self, acc, n_micro: int) -> np.ndarray:
        acc = _f32(acc)
        out = np.empty(acc.shape, dtype=np.float32)
        self.lib.oracle_average_micro(_ptr(acc), acc.size, int(n_micro), _ptr(out))
        return out

    def adamw(self, theta, m, v, g, *, lr, beta1, beta2, eps, weight_decay, step) -> None:
        """In-place AdamW on fp32 arrays of equal size."""
        for a in (theta, m, v, g):
            _f32(a)
        self.lib.oracle_adamw(_ptr(theta), _ptr(m), _ptr(v), _ptr(np.ascontiguousarray(g)),
                              theta.size, lr, beta1, beta2, eps, weight_decay, int(step))

    # -- FSDP2 per-parameter Shard(0) -----------------------------------
    def param_shard_bounds(self, dim0: int, row_numel: int, n_ranks: int, rank: int):
        b, e = ctypes.c_int64(0), ctypes.c_int64(0)
        self.lib.oracle_param_shard_bounds(int(dim0), int(row_numel), int(n_ranks), int(rank),
                                           ctypes.byref(b), ctypes.byref(e))
        return int(b.value), int(e.value)

    def param_sharded_step(self, params, *, lr, beta1, beta2, eps, weight_decay, step):
        """One step over per-parameter Shard(0) shards (no flat buffer, no padding).

        params: list of dicts with 'dim0', 'row', 'grads' ((n_ranks, numel)
        uint16: every rank's full gradient of the parameter) and 'master', 'm',
        'v': lists over ranks of float32 arrays holding that rank's rows (ragged,
        possibly empty), updated in place.  For each parameter and rank: the
        mean over ranks of the gradient rows the rank owns, AdamW on its fp32
        shard, bf16 cast; the gathered parameter is the concatenation of the
        ranks' shards in rank order.  Returns the list of (numel,) uint16.
        """
        outs = []
        for prm in params:
            grads = _u16(prm["grads"])
            n_ranks, numel = grads.shape
            full = np.empty(numel, dtype=np.uint16)
            for r in range(n_ranks):
                b, e = self.param_shard_bounds(prm["dim0"], prm["row"], n_ranks, r)
                if e <= b:
                    continue
                g = self.rank_mean(np.ascontiguousarray(grads[:, b:e]))
                self.adamw(prm["master"][r], prm["m"][r], prm["v"][r], g, lr=lr, beta1=beta1,
                           beta2=beta2, eps=eps, weight_decay=weight_decay, step=step)
                full[b:e] = self.round_to_bf16(prm["master"][r])
            outs.append(full)
        return outs

    # -- ZeRO-1 local accumulation ---------------------------------------
    def zero1_accumulate(self, grads, acc_full, first: bool) -> None:
        """grads: (n_ranks, P_pad) uint16; acc_full: (n_ranks, P_pad) float32, in place."""
        grads = _u16(grads)
        n_ranks, P_pad = grads.shape
        if acc_full.shape != grads.shape or acc_full.dtype != np.float32 or \
                not acc_full.flags["C_CONTIGUOUS"]:
            raise ValueError("acc_full must be C-contiguous float32 (n_ranks, P_pad)")
        self.lib.oracle_zero1_accumulate(_ptr(grads), _ptr(acc_full), n_ranks, P_pad,
                                         int(bool(first)))

    def zero1_step(self, acc_full, master, m, v, *, n_micro, lr, beta1, beta2, eps,
                   weight_decay, step):
        """acc_full: (n_ranks, P_pad) float32; master/m/v: (n_ranks, S) float32,
        updated in place.  Returns the (P_pad,) uint16 gathered parameters."""
        acc_full = _f32(acc_full)
        n_ranks, P_pad = acc_full.shape
        S = P_pad // n_ranks
        full = np.empty(P_pad, dtype=np.uint16)
        rc = self.lib.oracle_zero1_step(_ptr(acc_full), n_ranks, S, int(n_micro), _ptr(master),
                                        _ptr(m), _ptr(v), _ptr(full), lr, beta1, beta2, eps,
                                        weight_decay, int(step))
        if rc != 0:
            raise ValueError("bad arguments to oracle_zero1_step")
        return full

    def sampled_zero1_step(self, acc_at, master_at, m_at, v_at, *, n_micro, lr, beta1, beta2,
                           eps, weight_decay, step):
        """The ZeRO-1 step on gathered sample elements (element-wise, like
        sampled_step): acc_at (n_ranks, n) float32 holds every rank's full fp32
        accumulator at the sampled flat indices; master_at/m_at/v_at (n,) the
        owning rank's state there, updated in place.  Returns the (n,) bf16 bits.
        (Marshalling only: the columns are padded with zeros to a multiple of
        n_ranks so that oracle_zero1_step sees a (n_ranks, S) layout; the step is
        element-wise, so which rank a column is filed under does not matter.)"""
        acc_at = _f32(acc_at)
        n_ranks, n = acc_at.shape
        n_pad = -(-max(n, 1) // n_ranks) * n_ranks
        acc = np.zeros((n_ranks, n_pad), dtype=np.float32)
        acc[:, :n] = acc_at
        st = [np.zeros(n_pad, dtype=np.float32) for _ in range(3)]
        for dst, src in zip(st, (master_at, m_at, v_at)):
            dst[:n] = src
        full = np.empty(n_pad, dtype=np.uint16)
        rc = self.lib.oracle_zero1_step(_ptr(acc), n_ranks, n_pad // n_ranks, int(n_micro),
                                        _ptr(st[0]), _ptr(st[1]), _ptr(st[2]), _ptr(full), lr,
                                        beta1, beta2, eps, weight_decay, int(step))
        if rc != 0:
            raise ValueError("bad arguments to oracle_zero1_step")
        for dst, src in zip((master_at, m_at, v_at), st):
            dst[:] = src[:n]
        return full[:n].copy()

    # -- gradient clipping ----------------------------------------------
    def sum_squares(self, g) -> float:
        g = _f32(g)
        return float(self.lib.oracle_sum_squares(_ptr(g), g.size))

    def clip_coefficient(self, total_sum_squares: float, max_norm: float) -> np.float32:
        return np.float32(self.lib.oracle_clip_coefficient(float(total_sum_squares),
                                                           float(max_norm)))

    def scale(self, g, coef) -> None:
        g = _f32(g)
        self.lib.oracle_scale(_ptr(g), g.size, float(coef))

    def averaged_gradient(self, grads, accum=None, micro_step: int = 1, n_micro: int = 1):
        """The gradient one unit's optimizer step uses: the reduce-scatter mean,
        or, at the last of n_micro micro-steps, the accumulated mean / n_micro.
        grads: (n_ranks, P_pad) uint16 -> (n_ranks, S) float32 (None for an
        accumulation-only micro-step)."""
        g = self.reduce_scatter(grads)
        if accum is not None and n_micro > 1:
            self.accumulate(accum, g, micro_step == 1)
            if micro_step < n_micro:
                return None
            g = self.average_micro(accum, n_micro)
        return g

    def clipped_units_step(self, units, *, max_norm, lr, beta1, beta2, eps, weight_decay, step,
                           micro_step: int = 1, n_micro: int = 1):
        """One step over several units with global gradient-norm clipping.

        units: list of dicts with 'grads' (n_ranks, P_pad) uint16 and 'master',
        'm', 'v' (and 'accum' when micro-stepping) (n_ranks, S) float32,
        updated in place.  Steps: every unit's averaged gradient; the norm over
        all of them; the common clip coefficient; AdamW on each rank's shard
        with the scaled gradient; bf16 cast; all-gather.  Returns (list of
        gathered bf16 buffers or None, total norm, coefficient).
        """
        gs = [self.averaged_gradient(u["grads"], u.get("accum"), micro_step, n_micro)
              for u in units]
        if gs[0] is None:
            return None, None, None
        total = 0.0
        for g in gs:
            total = total + self.sum_squares(g)
        coef = self.clip_coefficient(total, max_norm)
        outs = []
        for u, g in zip(units, gs):
            self.scale(g, coef)
            n_ranks = g.shape[0]
            shards = np.empty(g.shape, dtype=np.uint16)
            for r in range(n_ranks):
                self.adamw(u["master"][r], u["m"][r], u["v"][r], g[r], lr=lr, beta1=beta1,
                           beta2=beta2, eps=eps, weight_decay=weight_decay, step=step)
                shards[r] = self.round_to_bf16(u["master"][r])
            outs.append(self.all_gather(shards))
        return outs, float(np.sqrt(total)), coef

    def zero_step(self, grads, master, m, v, *, lr, beta1, beta2, eps, weight_decay, step,
                  accum=None, micro_step: int = 1, n_micro: int = 1):
        """One sharded step over all logical ranks.

        grads: (n_ranks, P_pad) uint16; master/m/v (and accum): (n_ranks, S)
        float32, updated in place.  Returns the (P_pad,) uint16 gathered
        parameters, or None for an accumulation-only micro-step.
        """
        grads = _u16(grads)
        n_ranks, P_pad = grads.shape
        S = P_pad // n_ranks
        for a in (master, m, v) + ((accum,) if accum is not None else ()):
            if a.shape != (n_ranks, S) or a.dtype != np.float32 or not a.flags["C_CONTIGUOUS"]:
                raise ValueError("state arrays must be C-contiguous float32 (n_ranks, S)")
        full = np.empty(P_pad, dtype=np.uint16)
        rc = self.lib.oracle_zero_step(
            _ptr(grads), _ptr(master), _ptr(m), _ptr(v),
            _ptr(accum) if accum is not None else None,
            int(micro_step), int(n_micro), _ptr(full), n_ranks, S,
            lr, beta1, beta2, eps, weight_decay, int(step))
        if rc < 0:
            raise ValueError("bad arguments to oracle_zero_step")
        return full if rc == 1 else None

    def ddp_step(self, grads, theta, m, v, *, lr, beta1, beta2, eps, weight_decay, step):
        grads = _u16(grads)
        n_ranks, P_pad = grads.shape
        full = np.empty(P_pad, dtype=np.uint16)
        rc = self.lib.oracle_ddp_step(_ptr(grads), _ptr(theta), _ptr(m), _ptr(v), _ptr(full),
                                      n_ranks, P_pad, lr, beta1, beta2, eps, weight_decay,
                                      int(step))
        if rc != 0:
            raise ValueError("bad arguments to oracle_ddp_step")
        return full

    def sampled_step(self, grads_at, master_at, m_at, v_at, *, lr, beta1, beta2, eps,
                     weight_decay, step, acc_at=None, micro_step: int = 1, n_micro: int = 1):
        """The step on gathered sample elements (the method is element-wise).

        grads_at: (n_ranks, n) uint16 — every rank's gradient at the sampled
        flat indices; master_at/m_at/v_at: (n,) float32 state of the owning
        rank at those indices, updated in place.  Returns the (n,) bf16 bits
        of the gathered parameters, or None for an accumulation-only micro-step.
        """
        g = self.rank_mean(grads_at)
        if acc_at is not None and n_micro > 1:
            self.accumulate(acc_at, g, micro_step == 1)
            if micro_step < n_micro:
                return None
            g = self.average_micro(acc_at, n_micro)
        self.adamw(master_at, m_at, v_at, g, lr=lr, beta1=beta1, beta2=beta2, eps=eps,
                   weight_decay=weight_decay, step=step)
        return self.round_to_bf16(master_at)
