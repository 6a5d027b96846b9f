"""ctypes loader of libpcg.so (the C ABI declared in include/pcg.h).

The library is built in-tree by ``particle_cell_grid_gb300.build``; loading
fails loudly when it is missing.  There is no fallback implementation.
"""
from __future__ import annotations

import ctypes
import os
import threading

from . import build as _build

_lock = threading.Lock()
_lib = None

PCG_OK = 0
STATUS_NAMES = {
    0: "PCG_OK", 1: "PCG_ERR_INVALID_ARG", 2: "PCG_ERR_WORKSPACE", 3: "PCG_ERR_UNSUPPORTED",
    4: "PCG_ERR_CUDA", 5: "PCG_ERR_TIMEOUT", 6: "PCG_ERR_DOMAIN",
}

# every entry point the header declares, with (restype, argtypes)
_i32, _i64, _dbl, _vp, _sz = ctypes.c_int32, ctypes.c_int64, ctypes.c_double, ctypes.c_void_p, ctypes.c_size_t
_P = ctypes.POINTER
SIGNATURES = {
    "pcg_version": (ctypes.c_int, []),
    "pcg_status_string": (ctypes.c_char_p, [ctypes.c_int]),
    "pcg_stats_check": (ctypes.c_int, [_vp]),
    "pcg_bounds_check_failures": (ctypes.c_int, [_P(ctypes.c_uint64), _P(_i32)]),
    "pcg_deposit_cic1d": (ctypes.c_int, [_vp, _vp, _i64, _vp, _i32, _i32, _dbl, _dbl, _vp, _vp, _vp]),
    "pcg_deposit_cic1d_grad": (ctypes.c_int, [_vp, _vp, _i64, _vp, _i32, _i32, _dbl, _dbl, _vp, _vp, _vp, _vp]),
    "pcg_tile_sort_workspace_size": (ctypes.c_int, [_i32, _vp, _i32, _i64, _i32, _P(_sz)]),
    "pcg_tile_sort": (ctypes.c_int, [_i32, _vp, _i32, _i64, _vp, _i32, _vp, _vp, _vp, _vp, _vp, _sz, _vp]),
    "pcg_deposit_current_workspace_size": (ctypes.c_int, [_i32, _vp, _i32, _i64, _P(_sz)]),
    "pcg_deposit_current": (ctypes.c_int, [_i32, _vp, _i32, _i32, _i32, _i32, _i64, _vp, _vp, _vp, _vp,
                                           _vp, _vp, _vp, _sz, _vp]),
    "pcg_deposit_current_noalloc": (ctypes.c_int, [_i32, _vp, _i32, _i32, _i32, _i32, _i64, _vp, _vp, _vp,
                                                   _vp, _vp, _vp, _vp]),
    "pcg_deposit_zigzag": (ctypes.c_int, [_vp, _i32, _i64, _vp, _vp, _vp, _dbl, _vp, _vp, _vp, _vp, _sz, _vp]),
    "pcg_profile_enable": (ctypes.c_int, [_i32]),
    "pcg_profile_collect": (ctypes.c_int, [_i32, _vp, _vp, _vp, _P(_i32)]),
    "pcg_assemble_mass_matrix_workspace_size": (ctypes.c_int, [_vp, _i64, _P(_sz)]),
    "pcg_assemble_mass_matrix_scalar": (ctypes.c_int, [_vp, _i32, _i32, _i64, _vp, _vp, _vp, _vp, _vp, _vp]),
    "pcg_assemble_mass_matrix": (ctypes.c_int, [_vp, _i32, _i32, _i64, _vp, _vp, _vp, _vp, _vp, _vp,
                                                _vp, _sz, _vp]),
}


class PcgError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {STATUS_NAMES.get(status, status)} ({describe(status)})")


def library_path() -> str:
    """libpcg.so of this package; PCG_LIBRARY selects another build of the same
    library (e.g. the checked build, particle_cell_grid_gb300/_build_checked)."""
    return os.environ.get("PCG_LIBRARY") or _build.LIB


def load() -> ctypes.CDLL:
    """Load libpcg.so; raises when it has not been built."""
    global _lib
    with _lock:
        if _lib is None:
            path = library_path()
            if not os.path.exists(path):
                raise RuntimeError(
                    f"{path} is missing: build it first with "
                    "`python -c 'import __graft_entry__ as g; g.build()'`")
            lib = ctypes.CDLL(path)
            for name, (res, args) in SIGNATURES.items():
                fn = getattr(lib, name)
                fn.restype = res
                fn.argtypes = args
            _lib = lib
    return _lib


def describe(status: int) -> str:
    try:
        return load().pcg_status_string(int(status)).decode()
    except Exception:  # pragma: no cover - only when the library cannot load
        return "?"


def check(status: int, where: str) -> None:
    if status != PCG_OK:
        raise PcgError(status, where)
