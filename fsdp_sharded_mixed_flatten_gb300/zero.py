"""Thin Python binding of the C ABI in include/zero_flat.h (ctypes).

Argument marshalling only: tensors (or raw integer device addresses) are
turned into pointers, lists into pointer tables, and the current torch CUDA
stream is passed by default.  Every step of the computation runs in the CUDA
library; if the library has not been built, every call raises.
"""
from __future__ import annotations

import ctypes
import os
import re
import threading
from typing import Iterable, List, Sequence, Tuple

from .build import LIB_PATH

ZERO_MAX_RANKS = 512
ZERO_OK = 0
ERRORS = {-1: "ZERO_ERR_INVALID_ARG", -2: "ZERO_ERR_MISALIGNED", -3: "ZERO_ERR_SIZE",
          -4: "ZERO_ERR_CUDA"}


class ZeroError(RuntimeError):
    """A non-OK status from the library.  After an argument error
    (ZERO_ERR_INVALID_ARG, ZERO_ERR_MISALIGNED, ZERO_ERR_SIZE) nothing was
    queued; ZERO_ERR_CUDA may follow some launches or copies of the same call."""

    def __init__(self, code: int, message: str, func: str):
        self.code = code
        self.name = ERRORS.get(code, str(code))
        super().__init__(f"{func}: {self.name}: {message}")


class ZeroLayout(ctypes.Structure):
    """zero_layout_t: FlatParameter layout of one FSDP unit."""
    _fields_ = [("n_tensors", ctypes.c_int64), ("numel", ctypes.c_int64),
                ("numel_padded", ctypes.c_int64), ("shard_numel", ctypes.c_int64),
                ("n_ranks", ctypes.c_int32), ("flags", ctypes.c_int32)]

    def __repr__(self):
        return (f"ZeroLayout(n_tensors={self.n_tensors}, numel={self.numel}, "
                f"numel_padded={self.numel_padded}, shard_numel={self.shard_numel}, "
                f"n_ranks={self.n_ranks}, flags={self.flags})")


class ZeroUnit(ctypes.Structure):
    """zero_unit_t: one FlatParameter's layout and buffers for zero_step_units."""
    _fields_ = [("layout", ctypes.POINTER(ZeroLayout)), ("grads", ctypes.c_void_p),
                ("master", ctypes.c_void_p), ("m", ctypes.c_void_p), ("v", ctypes.c_void_p),
                ("accum", ctypes.c_void_p), ("full_params", ctypes.c_void_p),
                ("n_out", ctypes.c_int32), ("reserved", ctypes.c_int32)]


class ZeroAdamW(ctypes.Structure):
    """zero_adamw_t: hyper-parameters of one AdamW step (t >= 1)."""
    _fields_ = [("lr", ctypes.c_double), ("beta1", ctypes.c_double),
                ("beta2", ctypes.c_double), ("eps", ctypes.c_double),
                ("weight_decay", ctypes.c_double), ("step", ctypes.c_int64)]


_lock = threading.Lock()
_lib = None


def library_path() -> str:
    return LIB_PATH


def load() -> ctypes.CDLL:
    """Load the CUDA library; raise if it has not been built."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(
                f"CUDA library {LIB_PATH} is missing: build it with "
                "`python -m fsdp_sharded_mixed_flatten_gb300.build` (needs nvcc)")
        lib = ctypes.CDLL(LIB_PATH)
        p, i32, i64, f32 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_float
        lay, hp = ctypes.POINTER(ZeroLayout), ctypes.POINTER(ZeroAdamW)
        sig = {
            "zero_flat_layout": [p, i64, i32, p, lay],
            "zero_shard_segments": [lay, p, p, i32, p, p, p, i64, p],
            "zero_flatten": [p, p, p, i32, p, i32, lay, p],
            "zero_unflatten": [p, i32, p, p, i32, p, lay, p],
            "zero_reduce_scatter": [p, p, lay, i32, p],
            "zero_adamw_shard_step": [p, p, p, p, f32, p, lay, hp, p],
            "zero_all_gather": [p, p, i32, lay, p],
            "zero_step": [p, p, p, p, p, i32, i32, p, i32, lay, hp, p],
        }
        for name, args in sig.items():
            fn = getattr(lib, name)
            fn.argtypes = args
            fn.restype = ctypes.c_int
        lib.zero_step_units.argtypes = [ctypes.POINTER(ZeroUnit), i32, i32, i32, hp, p]
        lib.zero_step_units.restype = ctypes.c_int
        lib.zero_clip_workspace_bytes.argtypes = [ctypes.POINTER(ZeroUnit), i32, i32,
                                                  ctypes.POINTER(ctypes.c_int64)]
        lib.zero_clip_workspace_bytes.restype = ctypes.c_int
        lib.zero_step_units_clip.argtypes = [ctypes.POINTER(ZeroUnit), i32, i32, i32, hp,
                                             ctypes.c_double, p, i64, p, p]
        lib.zero_step_units_clip.restype = ctypes.c_int
        lib.zero_step_units_clip_noalloc.argtypes = [ctypes.POINTER(ZeroUnit), i32, i32, i32,
                                                     hp, ctypes.c_double, p, p]
        lib.zero_step_units_clip_noalloc.restype = ctypes.c_int
        lib.zero_step_units_host.argtypes = [ctypes.POINTER(ZeroUnit), i32, p, p, i32, i32, hp,
                                             i32, p, p, p]
        lib.zero_step_units_host.restype = ctypes.c_int
        lib.zero1_accumulate.argtypes = [p, p, i32, lay, p]
        lib.zero1_accumulate.restype = ctypes.c_int
        lib.zero1_step.argtypes = [p, i32, p, p, p, p, i32, lay, hp, p]
        lib.zero1_step.restype = ctypes.c_int
        lib.zero_param_layout.argtypes = [i64, i64, i32, lay]
        lib.zero_param_layout.restype = ctypes.c_int
        lib.zero_shard_numel.argtypes = [lay, i32, ctypes.POINTER(ctypes.c_int64)]
        lib.zero_shard_numel.restype = ctypes.c_int
        lib.zero_device_status.argtypes = [p, ctypes.POINTER(ctypes.c_int32), i32]
        lib.zero_device_status.restype = ctypes.c_int
        lib.zero_selftest_wait_timeout.argtypes = [i64, p]
        lib.zero_selftest_wait_timeout.restype = ctypes.c_int
        lib.zero_last_error.argtypes = []
        lib.zero_last_error.restype = ctypes.c_char_p
        lib.zero_abi_version.argtypes = []
        lib.zero_abi_version.restype = ctypes.c_int32
        _lib = lib
        return lib


def header_functions(header: str | None = None) -> List[str]:
    """Names of the functions include/zero_flat.h declares."""
    if header is None:
        header = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                              "include", "zero_flat.h")
    text = re.sub(r"/\*.*?\*/", "", open(header).read(), flags=re.S)
    return sorted(set(re.findall(r"\b(zero_[a-z0-9_]+)\s*\(", text)))


# ------------------------------------------------------------ marshalling --

def _addr(x) -> int:
    if x is None:
        return 0
    if isinstance(x, int):
        return x
    return int(x.data_ptr())


def _ptrs(xs: Sequence):
    arr = (ctypes.c_void_p * max(len(xs), 1))()
    for i, x in enumerate(xs):
        arr[i] = _addr(x) or None
    return arr


def _i64(xs: Iterable[int]):
    xs = [int(x) for x in xs]
    return (ctypes.c_int64 * max(len(xs), 1))(*xs)


def _stream(stream) -> int:
    if stream is None:
        import torch
        if torch.cuda.is_available():
            return int(torch.cuda.current_stream().cuda_stream)
        return 0
    if isinstance(stream, int):
        return stream
    return int(stream.cuda_stream)


def _hp(hp) -> ZeroAdamW:
    if isinstance(hp, ZeroAdamW):
        return hp
    if hp is None:
        return None
    return ZeroAdamW(float(hp["lr"]), float(hp["beta1"]), float(hp["beta2"]), float(hp["eps"]),
                     float(hp["weight_decay"]), int(hp["step"]))


def _check(rc: int, func: str):
    if rc != ZERO_OK:
        raise ZeroError(rc, load().zero_last_error().decode(), func)


# ---------------------------------------------------------------- API ------

def zero_abi_version() -> int:
    return int(load().zero_abi_version())


def zero_last_error() -> str:
    return load().zero_last_error().decode()


def zero_flat_layout(numels: Sequence[int], n_ranks: int) -> Tuple[List[int], ZeroLayout]:
    """Host-only FlatParameter layout: (tensor offsets, layout)."""
    n = len(numels)
    offsets = (ctypes.c_int64 * max(n, 1))()
    layout = ZeroLayout()
    _check(load().zero_flat_layout(_i64(numels), n, int(n_ranks), offsets, ctypes.byref(layout)),
           "zero_flat_layout")
    return [int(offsets[i]) for i in range(n)], layout


def zero_shard_segments(layout: ZeroLayout, offsets, numels, rank: int):
    """Pieces (tensor index or -1 for padding, begin, end) of rank's shard."""
    lib = load()
    count = ctypes.c_int64(0)
    cap = len(numels) + 1
    t, b, e = (ctypes.c_int64 * cap)(), (ctypes.c_int64 * cap)(), (ctypes.c_int64 * cap)()
    _check(lib.zero_shard_segments(ctypes.byref(layout), _i64(offsets), _i64(numels), int(rank),
                                   t, b, e, cap, ctypes.byref(count)), "zero_shard_segments")
    return [(int(t[i]), int(b[i]), int(e[i])) for i in range(count.value)]


def zero_flatten(src, offsets, numels, elem_bytes: int, dst, dst_split: int,
                 layout: ZeroLayout, stream=None):
    _check(load().zero_flatten(_ptrs(src), _i64(offsets), _i64(numels), int(elem_bytes),
                               _ptrs(dst), int(dst_split), ctypes.byref(layout), _stream(stream)),
           "zero_flatten")


def zero_unflatten(src, src_split: int, offsets, numels, elem_bytes: int, dst,
                   layout: ZeroLayout, stream=None):
    _check(load().zero_unflatten(_ptrs(src), int(src_split), _i64(offsets), _i64(numels),
                                 int(elem_bytes), _ptrs(dst), ctypes.byref(layout),
                                 _stream(stream)), "zero_unflatten")


def zero_reduce_scatter(grads, grad_shards, layout: ZeroLayout, accumulate: int = 0, stream=None):
    _check(load().zero_reduce_scatter(_ptrs(grads), _ptrs(grad_shards), ctypes.byref(layout),
                                      int(accumulate), _stream(stream)), "zero_reduce_scatter")


def zero_adamw_shard_step(master, m, v, grad_shards, grad_divisor: float, param_shards,
                          layout: ZeroLayout, hp, stream=None):
    h = _hp(hp)
    _check(load().zero_adamw_shard_step(_ptrs(master), _ptrs(m), _ptrs(v), _ptrs(grad_shards),
                                        float(grad_divisor), _ptrs(param_shards),
                                        ctypes.byref(layout), ctypes.byref(h), _stream(stream)),
           "zero_adamw_shard_step")


def zero_all_gather(param_shards, full_params, layout: ZeroLayout, stream=None):
    _check(load().zero_all_gather(_ptrs(param_shards), _ptrs(full_params), len(full_params),
                                  ctypes.byref(layout), _stream(stream)), "zero_all_gather")


def zero_step(grads, master, m, v, accum, micro_step: int, n_micro: int, full_params,
              layout: ZeroLayout, hp, stream=None):
    h = _hp(hp)
    _check(load().zero_step(_ptrs(grads), _ptrs(master), _ptrs(m), _ptrs(v),
                            _ptrs(accum) if accum is not None else None,
                            int(micro_step), int(n_micro), _ptrs(full_params), len(full_params),
                            ctypes.byref(layout), ctypes.byref(h) if h is not None else None,
                            _stream(stream)), "zero_step")


ZERO_DEVICE_OK = 0
ZERO_DEVICE_TIMEOUT = 1
ZERO_DEVICE_SCHED_CONFLICT = 2


def zero_device_status(stream=None, clear: bool = True) -> int:
    """Synchronise the stream and return (and by default clear) the device
    status word: ZERO_DEVICE_OK, ZERO_DEVICE_TIMEOUT if a kernel's bounded
    wait ran out, or ZERO_DEVICE_SCHED_CONFLICT if two launches claimed tiles
    from one scheduling counter at the same time."""
    v = ctypes.c_int32(0)
    _check(load().zero_device_status(_stream(stream), ctypes.byref(v), int(bool(clear))),
           "zero_device_status")
    return int(v.value)


def zero_selftest_wait_timeout(limit_ns: int, stream=None):
    """Launch a kernel whose bounded barrier wait must run out after limit_ns."""
    _check(load().zero_selftest_wait_timeout(int(limit_ns), _stream(stream)),
           "zero_selftest_wait_timeout")


class PreparedUnits:
    """Units marshalled once into a zero_unit_t array, for calls that step the
    same buffers every iteration (saves rebuilding the pointer tables)."""

    def __init__(self, units):
        self.n = len(units)
        self.array, self._keep = _unit_array(units)

    def __len__(self):
        return self.n


def prepare_units(units) -> PreparedUnits:
    return PreparedUnits(units)


def _units_arg(units):
    if isinstance(units, PreparedUnits):
        return units.array, None, units.n
    arr, keep = _unit_array(units)
    return arr, keep, len(units)


def _unit_array(units):
    """Marshal (grads, master, m, v, accum or None, full_params, layout) tuples
    into a zero_unit_t array; returns (array, keep-alive list)."""
    n = len(units)
    arr = (ZeroUnit * max(n, 1))()
    keep = []
    for i, (grads, master, m, v, accum, full, layout) in enumerate(units):
        tabs = [_ptrs(grads), _ptrs(master), _ptrs(m), _ptrs(v),
                _ptrs(accum) if accum is not None else None, _ptrs(full)]
        keep.append((tabs, layout))
        arr[i].layout = ctypes.pointer(layout)
        arr[i].grads, arr[i].master, arr[i].m, arr[i].v = (ctypes.cast(t, ctypes.c_void_p)
                                                           for t in tabs[:4])
        arr[i].accum = ctypes.cast(tabs[4], ctypes.c_void_p) if tabs[4] is not None else None
        arr[i].full_params = ctypes.cast(tabs[5], ctypes.c_void_p)
        arr[i].n_out = len(full)
    return arr, keep


def zero_step_units(units, micro_step: int, n_micro: int, hp, stream=None):
    """units: sequence of (grads, master, m, v, accum or None, full_params,
    layout), or a PreparedUnits."""
    arr, keep, n = _units_arg(units)
    h = _hp(hp)
    _check(load().zero_step_units(arr, n, int(micro_step), int(n_micro),
                                  ctypes.byref(h) if h is not None else None, _stream(stream)),
           "zero_step_units")


ZERO_HOST_GRADS_FREE = 1
ZERO_HOST_SM_COPY = 2


class HostTables:
    """Host pointer tables of zero_step_units_host, marshalled once:
    host_grads[u][k] (pinned host tensors or addresses) and host_params[u]
    (pinned host tensors, addresses or None; the whole list may be None)."""

    def __init__(self, host_grads, host_params=None):
        self._rows = [_ptrs(g) for g in host_grads]
        self.grads = (ctypes.c_void_p * max(len(self._rows), 1))(
            *[ctypes.cast(r, ctypes.c_void_p) for r in self._rows])
        self.params = _ptrs(host_params) if host_params is not None else None


def zero_step_units_host(units, host, micro_step: int, n_micro: int, hp, flags: int = 0,
                         h2d_stream=None, compute_stream=None, d2h_stream=None):
    """zero_step_units with the gradients copied in from pinned host memory
    and the gathered parameters copied back out.  host: a HostTables, or a
    (host_grads, host_params) pair."""
    arr, keep, n = _units_arg(units)
    if not isinstance(host, HostTables):
        host = HostTables(*host)
    h = _hp(hp)
    _check(load().zero_step_units_host(arr, n, host.grads, host.params, int(micro_step),
                                       int(n_micro), ctypes.byref(h) if h is not None else None,
                                       int(flags), _stream(h2d_stream), _stream(compute_stream),
                                       _stream(d2h_stream)), "zero_step_units_host")


def zero_clip_workspace_bytes(units, n_micro: int = 1) -> int:
    arr, keep, n = _units_arg(units)
    out = ctypes.c_int64(0)
    _check(load().zero_clip_workspace_bytes(arr, n, int(n_micro), ctypes.byref(out)),
           "zero_clip_workspace_bytes")
    return int(out.value)


def zero_step_units_clip(units, micro_step: int, n_micro: int, hp, max_norm: float, workspace,
                         workspace_bytes: int, norm_out=None, stream=None):
    """zero_step_units with global gradient-norm clipping; every unit needs an
    accumulator (it receives the averaged gradient).  workspace: device
    buffer of at least zero_clip_workspace_bytes(units, n_micro) bytes."""
    arr, keep, n = _units_arg(units)
    h = _hp(hp)
    _check(load().zero_step_units_clip(arr, n, int(micro_step), int(n_micro),
                                       ctypes.byref(h) if h is not None else None,
                                       float(max_norm), _addr(workspace) or None,
                                       int(workspace_bytes), _addr(norm_out) or None,
                                       _stream(stream)), "zero_step_units_clip")


ZERO_NOALLOC_CLIP_SLOTS = 4096


def zero_step_units_clip_noalloc(units, micro_step: int, n_micro: int, hp, max_norm: float,
                                 norm_out=None, stream=None):
    """zero_step_units_clip without a caller workspace, for callers that cannot
    allocate device memory: the partial sums live in a fixed 32 KB scratch
    array inside the library, shared by every call (serialise calls that could
    overlap on the GPU)."""
    arr, keep, n = _units_arg(units)
    h = _hp(hp)
    _check(load().zero_step_units_clip_noalloc(arr, n, int(micro_step), int(n_micro),
                                               ctypes.byref(h) if h is not None else None,
                                               float(max_norm), _addr(norm_out) or None,
                                               _stream(stream)), "zero_step_units_clip_noalloc")


def zero1_accumulate(grads, full_accum, first: bool, layout: ZeroLayout, stream=None):
    """ZeRO-1 local accumulation: full_accum[k] = (first ? 0 : full_accum[k]) + grads[k]."""
    _check(load().zero1_accumulate(_ptrs(grads), _ptrs(full_accum), int(bool(first)),
                                   ctypes.byref(layout), _stream(stream)), "zero1_accumulate")


def zero1_step(full_accum, n_micro: int, master, m, v, full_params, layout: ZeroLayout, hp,
               stream=None):
    """ZeRO-1 step: one reduce-scatter of the accumulated fp32 gradients / n_micro,
    then AdamW, bf16 cast and all-gather."""
    h = _hp(hp)
    _check(load().zero1_step(_ptrs(full_accum), int(n_micro), _ptrs(master), _ptrs(m), _ptrs(v),
                             _ptrs(full_params), len(full_params), ctypes.byref(layout),
                             ctypes.byref(h), _stream(stream)), "zero1_step")


ZERO_LAYOUT_UNPADDED = 1


def zero_param_layout(dim0: int, row_numel: int, n_ranks: int) -> ZeroLayout:
    """FSDP2 per-parameter Shard(0) layout of one parameter (no padding)."""
    layout = ZeroLayout()
    _check(load().zero_param_layout(int(dim0), int(row_numel), int(n_ranks),
                                    ctypes.byref(layout)), "zero_param_layout")
    return layout


def zero_shard_numel(layout: ZeroLayout, rank: int) -> int:
    out = ctypes.c_int64(0)
    _check(load().zero_shard_numel(ctypes.byref(layout), int(rank), ctypes.byref(out)),
           "zero_shard_numel")
    return int(out.value)
