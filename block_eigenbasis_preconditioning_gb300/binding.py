"""ctypes binding of the C ABI in include/dobb.h.

Argument marshalling only: every step of the optimizer runs in the CUDA
library.  PyTorch supplies device memory (the state buffer, parameters,
gradients, activations) and the current stream.  If the library cannot be
loaded the binding raises: there is no fallback implementation.
"""
from __future__ import annotations

import ctypes
import os
from typing import List, Optional, Sequence, Tuple

from . import build as _build

_LIB = None

DOBB_OK = 0
STATUS_NAMES = {0: "DOBB_OK", 1: "DOBB_ERR_INVALID_ARG", 2: "DOBB_ERR_CUDA",
                3: "DOBB_ERR_NONFINITE", 4: "DOBB_ERR_NOT_CONVERGED", 5: "DOBB_ERR_STATE",
                6: "DOBB_ERR_UNSUPPORTED"}
DTYPES = {"f32": 0, "bf16": 1}
REFRESH_METHODS = {"eigh": 0, "orth": 1}
NORMS = {"sign": 0, "l2": 1}
SIDES = {"input": 0, "output": 1}
TENSORS = {"moments": 0, "bases": 1, "eigvals": 2, "momentum": 3, "flags": 4, "stats": 5,
           "error": 6}
FLAG_NONFINITE_X = 1
FLAG_NONFINITE_G = 2
FLAG_NONFINITE_A = 4
FLAG_NOT_CONVERGED = 8

# (name, restype, argtypes) of every exported symbol
_c = ctypes
_VP = _c.c_void_p
_I64P = _c.POINTER(_c.c_int64)
SIGNATURES = [
    ("dobb_state_bytes", _c.c_size_t, [_c.c_int, _I64P, _I64P, _c.c_int]),
    ("dobb_create", _c.c_int, [_c.POINTER(_VP), _c.c_int, _I64P, _I64P, _c.c_int, _c.c_float,
                               _c.c_float, _c.c_int, _c.c_float, _c.c_int, _c.c_int, _VP,
                               _c.c_size_t, _VP]),
    ("dobb_destroy", _c.c_int, [_VP]),
    ("dobb_last_error", _c.c_char_p, []),
    ("dobb_accumulate_moments", _c.c_int, [_VP, _c.POINTER(_VP), _I64P, _VP]),
    ("dobb_refresh_bases", _c.c_int, [_VP, _VP]),
    ("dobb_step", _c.c_int, [_VP, _c.POINTER(_VP), _c.POINTER(_VP), _c.c_float, _VP]),
    ("dobb_step_with_signs", _c.c_int, [_VP, _c.POINTER(_VP), _c.POINTER(_VP), _c.c_float,
                                        _c.POINTER(_VP), _VP]),
    ("dobb_get_step", _c.c_int, [_VP, _I64P]),
    ("dobb_set_step", _c.c_int, [_VP, _c.c_int64]),
    ("dobb_set_basis_dtype", _c.c_int, [_VP, _c.c_int, _VP]),
    ("dobb_set_refresh", _c.c_int, [_VP, _c.c_int, _c.c_int]),
    ("dobb_set_normalization", _c.c_int, [_VP, _c.c_int]),
    ("dobb_set_side", _c.c_int, [_VP, _c.c_int, _c.c_int, _VP]),
    ("dobb_set_jacobi", _c.c_int, [_VP, _c.c_int, _c.c_float]),
    ("dobb_set_refresh_period", _c.c_int, [_VP, _c.c_int]),
    ("dobb_set_eig_grid", _c.c_int, [_VP, _c.c_int, _c.c_int64]),
    ("dobb_state_tensor", _c.c_int, [_VP, _c.c_int, _c.c_int, _c.POINTER(_VP),
                                     _c.POINTER(_c.c_size_t)]),
    ("dobb_num_blocks", _c.c_int64, [_VP]),
    ("dobb_block_offset", _c.c_int64, [_VP, _c.c_int]),
    ("dobb_get_block_flags", _c.c_int, [_VP, _c.POINTER(_c.c_uint32), _VP]),
    ("dobb_clear_block_flags", _c.c_int, [_VP, _VP]),
    ("dobb_get_block_stats", _c.c_int, [_VP, _c.POINTER(_c.c_float), _VP]),
    ("dobb_check_bases", _c.c_int, [_VP, _c.POINTER(_c.c_float), _VP]),
    ("dobb_checkpoint_bytes", _c.c_size_t, [_VP]),
    ("dobb_get_state", _c.c_int, [_VP, _VP, _c.c_size_t, _I64P, _VP]),
    ("dobb_set_state", _c.c_int, [_VP, _VP, _c.c_size_t, _c.c_int64, _VP]),
    ("dobb_launch_count", _c.c_int64, [_VP]),
    ("dobb_describe_work", _c.c_int64, [_c.c_int, _I64P, _I64P, _c.c_int, _c.c_int, _I64P,
                                        _c.c_int64]),
    ("dobb_set_step_path", _c.c_int, [_VP, _c.c_int]),
    ("dobb_sync_bases", _c.c_int, [_VP, _VP]),
    ("dobb_peak_probe", _c.c_int, [_c.c_int, _VP, _c.c_size_t, _c.c_int,
                                   _c.POINTER(_c.c_float), _c.POINTER(_c.c_double), _VP]),
    ("dobb_selftest_wait_timeout", _c.c_int, [_c.POINTER(_c.c_uint32), _c.c_uint64, _VP]),
    ("dobb_eigh_noalloc", _c.c_int, [_VP, _VP, _VP, _c.c_int, _c.c_int, _c.c_int,
                                     _c.POINTER(_c.c_uint32), _VP]),
    ("dobb_eigh_noalloc_last_error", _c.c_char_p, []),
]


class DobbError(RuntimeError):
    def __init__(self, status: int, msg: str):
        super().__init__(f"{STATUS_NAMES.get(status, status)}: {msg}")
        self.status = status


def library_path() -> str:
    return _build.LIB


def load_library(build_if_missing: bool = True):
    """Load libdobb.so (building it first if missing or stale)."""
    global _LIB
    if _LIB is not None:
        return _LIB
    path = _build.build() if build_if_missing else _build.LIB
    if not os.path.exists(path):
        raise RuntimeError(f"libdobb.so not found at {path}; run build() first")
    lib = ctypes.CDLL(path)
    for name, res, args in SIGNATURES:
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _LIB = lib
    return lib


def check(status: int) -> None:
    if status != DOBB_OK:
        msg = _LIB.dobb_last_error().decode() if _LIB is not None else ""
        raise DobbError(status, msg)


def _i64(vals: Sequence[int]):
    return (ctypes.c_int64 * len(vals))(*[int(v) for v in vals])


def _ptrs(vals):
    return (ctypes.c_void_p * len(vals))(*[None if v is None else int(v) for v in vals])


def describe_work(shapes: Sequence[Tuple[int, int]], B: int, phase: int):
    """The scheduler's work list of one phase (see dobb_describe_work) as a
    list of (launch, kind, mat_base, matrix, block, a, b) tuples."""
    lib = load_library()
    ms = _i64([s[0] for s in shapes])
    ns = _i64([s[1] for s in shapes])
    cnt = lib.dobb_describe_work(len(shapes), ms, ns, B, phase, None, 0)
    if cnt < 0:
        raise DobbError(1, lib.dobb_last_error().decode())
    buf = (ctypes.c_int64 * (7 * max(cnt, 1)))()
    lib.dobb_describe_work(len(shapes), ms, ns, B, phase, buf, cnt)
    return [tuple(buf[7 * i:7 * i + 7]) for i in range(cnt)]


PEAK_PROBES = {"ffma": 0, "mma_sync_tf32": 1, "tc_tf32": 2, "tc_bf16": 3}


def peak_probe(which: str, scratch_ptr: int, scratch_bytes: int, iters: int, stream_ptr=None):
    """One run of a throughput probe (see dobb_peak_probe): (ms, flops)."""
    lib = load_library()
    ms = ctypes.c_float()
    fl = ctypes.c_double()
    st = lib.dobb_peak_probe(PEAK_PROBES[which], ctypes.c_void_p(scratch_ptr),
                             ctypes.c_size_t(scratch_bytes), int(iters), ctypes.byref(ms),
                             ctypes.byref(fl), ctypes.c_void_p(stream_ptr) if stream_ptr else None)
    if st != DOBB_OK:
        raise DobbError(st, f"peak probe {which} failed")
    return float(ms.value), float(fl.value)


def state_bytes(shapes: Sequence[Tuple[int, int]], B: int) -> int:
    lib = load_library()
    ms = _i64([s[0] for s in shapes])
    ns = _i64([s[1] for s in shapes])
    nb = lib.dobb_state_bytes(len(shapes), ms, ns, B)
    if nb == 0:
        raise DobbError(1, lib.dobb_last_error().decode())
    return int(nb)
