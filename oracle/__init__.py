"""fp64 CPU oracle for the particle-to-grid deposit path.

TEST INFRASTRUCTURE ONLY: imported by ``tests/``, ``__graft_entry__.smoke()``
and the CPU-baseline leg of ``bench.py``, never by the product package.  It
shares no code with the CUDA library; the two meet only through the seeded
input generators in ``synth``.

The arithmetic lives in ``pcg_oracle.c`` (plain C, double precision, compiled
with ``-ffp-contract=off``).  This module compiles it on first use if needed
and marshals numpy arrays through ctypes.

Sources, by page title and section:
  * "03. Compaction and scatter-add" (WEANJ): 1D windowed CIC histogram.
  * Pennati & Markidis, "Mass Matrix Assembly on Tensor Cores for Implicit
    Particle-In-Cell Methods": Eqs. (4)-(6) mass matrix and alpha tensor,
    Eq. (12) B-spline shape, Sec. 3.4 offset storage.
  * "Tiled current deposit" (Entity wiki): tile key and tile_offsets.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "pcg_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_SO = os.path.join(_BUILD_DIR, "liboracle.so")
_lock = threading.Lock()
_lib = None

CFLAGS = ["-O2", "-fPIC", "-shared", "-std=c11", "-ffp-contract=off",
          "-fno-fast-math"]


def build(force: bool = False) -> str:
    """Compile the oracle into ``oracle/_build/liboracle.so`` (gcc)."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    stale = (not os.path.exists(_SO)) or os.path.getmtime(_SO) < os.path.getmtime(_SRC)
    if force or stale:
        tmp = _SO + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", *CFLAGS, "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _SO)
    return _SO


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            i32, i64, dbl, vp = ctypes.c_int32, ctypes.c_int64, ctypes.c_double, ctypes.c_void_p
            lib.oracle_version.restype = ctypes.c_int
            lib.oracle_cic1d.restype = i64
            lib.oracle_cic1d.argtypes = [vp, vp, i64, vp, i32, i32, dbl, dbl, vp, vp]
            lib.oracle_cic1d_grad.restype = i64
            lib.oracle_cic1d_grad.argtypes = [vp, vp, i64, vp, i32, i32, dbl, dbl, vp, vp, vp]
            lib.oracle_axis_support.restype = ctypes.c_int
            lib.oracle_axis_support.argtypes = [i32, dbl, vp, vp]
            lib.oracle_deposit_current.restype = i64
            lib.oracle_deposit_current.argtypes = [i32, vp, i32, i64, vp, vp, vp, vp]
            lib.oracle_mass_matrix_scalar.restype = i64
            lib.oracle_mass_matrix_scalar.argtypes = [vp, i64, vp, vp, vp]
            lib.oracle_mass_matrix_tsc.restype = i64
            lib.oracle_mass_matrix_tsc.argtypes = [vp, i64, vp, vp, vp, vp]
            lib.oracle_deposit_zigzag.restype = i64
            lib.oracle_deposit_zigzag.argtypes = [vp, i64, vp, vp, vp, dbl, vp]
            lib.oracle_alpha.restype = None
            lib.oracle_alpha.argtypes = [vp, vp]
            lib.oracle_mass_matrix.restype = i64
            lib.oracle_mass_matrix.argtypes = [vp, i64, vp, vp, vp, vp]
            lib.oracle_tile_keys.restype = i64
            lib.oracle_tile_keys.argtypes = [i32, vp, i32, i64, vp, vp, vp]
            _lib = lib
    return _lib


def _f32(a):
    return np.ascontiguousarray(a, dtype=np.float32)


def _ptr(a):
    return a.ctypes.data_as(ctypes.c_void_p)


def _ptr_array(arrs):
    t = (ctypes.c_void_p * 3)()
    for i, a in enumerate(arrs):
        t[i] = a.ctypes.data
    return t


def cic1d(x0, v, target, nbins=1024, nsteps=50, dt=0.01, halfwidth=0.005):
    """1D windowed CIC histogram; returns (H float64[nbins], loss, n_deposits)."""
    lib = _load()
    x0, v, target = _f32(x0), _f32(v), _f32(target)
    assert x0.shape == v.shape and target.shape == (nbins,)
    H = np.zeros(nbins, dtype=np.float64)
    loss = np.zeros(1, dtype=np.float64)
    nsel = lib.oracle_cic1d(_ptr(x0), _ptr(v), x0.size, _ptr(target), nbins, nsteps,
                            float(dt), float(halfwidth), _ptr(H), _ptr(loss))
    return H, float(loss[0]), int(nsel)


def cic1d_grad(x0, v, target, nbins=1024, nsteps=50, dt=0.01, halfwidth=0.005):
    """Gradient of the 1D loss with respect to x0 (the page's d L / d x0).

    Returns (dx0 float64[n], H float64[nbins], loss, n_deposits); follows
    "03. Compaction and scatter-add", "The problem" and "Code" (reverse pass
    seeded with dL/dH = 2 (H - target))."""
    lib = _load()
    x0, v, target = _f32(x0), _f32(v), _f32(target)
    assert x0.shape == v.shape and target.shape == (nbins,)
    H = np.zeros(nbins, dtype=np.float64)
    loss = np.zeros(1, dtype=np.float64)
    dx0 = np.zeros(x0.size, dtype=np.float64)
    nsel = lib.oracle_cic1d_grad(_ptr(x0), _ptr(v), x0.size, _ptr(target), nbins, nsteps, float(dt),
                                 float(halfwidth), _ptr(H), _ptr(loss), _ptr(dx0))
    return dx0, H, float(loss[0]), int(nsel)


def axis_support(order, x):
    """First node and weights of the 1D B-spline support of coordinate x."""
    lib = _load()
    first = np.zeros(1, dtype=np.int64)
    w = np.zeros(3, dtype=np.float64)
    k = lib.oracle_axis_support(int(order), float(x), _ptr(first), _ptr(w))
    if k < 0:
        raise ValueError("order must be 1 or 2")
    return int(first[0]), w[:k].copy()


def deposit_current(grid, order, pos, vel, q):
    """J (float64[3, *grid reversed]) = sum_p q v W, periodic; returns (J, n_invalid).

    grid = (Nx, Ny) or (Nx, Ny, Nz); pos = list of dim arrays; vel = 3 arrays.
    The returned array has shape (3, Ny, Nx) or (3, Nz, Ny, Nx).
    """
    lib = _load()
    dim = len(grid)
    pos = [_f32(p) for p in pos]
    vel = [_f32(v) for v in vel]
    q = _f32(q)
    n = q.size
    g = np.array(list(grid) + [1] * (3 - dim), dtype=np.int32)
    ncells = int(np.prod(grid))
    J = np.zeros(3 * ncells, dtype=np.float64)
    posp = _ptr_array(pos + [pos[0]] * (3 - dim))
    velp = _ptr_array(vel)
    ninv = lib.oracle_deposit_current(dim, _ptr(g), int(order), n, posp, velp, _ptr(q), _ptr(J))
    return J.reshape((3,) + tuple(reversed(grid))), int(ninv)


def deposit_zigzag(grid, pos_prev, pos, q, dt):
    """Charge-conserving zigzag current (Umeda et al. 2003; the O == 0 deposit of
    "Tiled current deposit", "Halo sizing") of the moves pos_prev -> pos on a 3D
    periodic grid.  Returns (J float64[3, Nz, Ny, Nx], n_invalid); J[c] lives on
    the edges from each node towards +e_c."""
    lib = _load()
    assert len(grid) == 3
    pp = [_f32(a) for a in pos_prev]
    pc = [_f32(a) for a in pos]
    q = _f32(q)
    g = np.array(grid, dtype=np.int32)
    J = np.zeros(3 * int(np.prod(grid)), dtype=np.float64)
    ninv = lib.oracle_deposit_zigzag(_ptr(g), q.size, _ptr_array(pp), _ptr_array(pc), _ptr(q), float(dt),
                                     _ptr(J))
    return J.reshape((3,) + tuple(reversed(grid))), int(ninv)


def alpha(omega):
    """Rotation-response tensor alpha (3x3) of one magnetisation vector."""
    lib = _load()
    w = np.ascontiguousarray(omega, dtype=np.float64)
    a = np.zeros(9, dtype=np.float64)
    lib.oracle_alpha(_ptr(w), _ptr(a))
    return a.reshape(3, 3)


def mass_matrix(grid, pos, wq, omega):
    """M (float64[Nz, Ny, Nx, 27, 3, 3]) for CIC shapes; returns (M, n_invalid)."""
    lib = _load()
    pos = [_f32(p) for p in pos]
    omega = [_f32(o) for o in omega]
    wq = _f32(wq)
    g = np.array(grid, dtype=np.int32)
    ncells = int(np.prod(grid))
    M = np.zeros(ncells * 243, dtype=np.float64)
    ninv = lib.oracle_mass_matrix(_ptr(g), wq.size, _ptr_array(pos), _ptr(wq),
                                  _ptr_array(omega), _ptr(M))
    return M.reshape(tuple(reversed(grid)) + (27, 3, 3)), int(ninv)


def mass_matrix_tsc(grid, pos, wq, omega):
    """M (float64[Nz, Ny, Nx, 125, 3, 3]) for second-order (TSC) shapes, every
    offset in {-2..2}^3 kept (Pennati & Markidis, Sec. 2.3, 3.3-3.4); returns
    (M, n_invalid).  Every grid edge must be >= 5."""
    lib = _load()
    assert all(N >= 5 for N in grid)
    pos = [_f32(p) for p in pos]
    omega = [_f32(o) for o in omega]
    wq = _f32(wq)
    g = np.array(grid, dtype=np.int32)
    M = np.zeros(int(np.prod(grid)) * 1125, dtype=np.float64)
    ninv = lib.oracle_mass_matrix_tsc(_ptr(g), wq.size, _ptr_array(pos), _ptr(wq), _ptr_array(omega), _ptr(M))
    return M.reshape(tuple(reversed(grid)) + (125, 3, 3)), int(ninv)


def mass_matrix_scalar(grid, pos, w):
    """Scalar (MPM) mass matrix M (float64[Nz, Ny, Nx, 27]) = sum_p w W_pg W_pg' for
    CIC shapes (Pennati & Markidis, Sec. 2.1, the scalar case of Eq. (6));
    returns (M, n_invalid)."""
    lib = _load()
    pos = [_f32(p) for p in pos]
    w = _f32(w)
    g = np.array(grid, dtype=np.int32)
    M = np.zeros(int(np.prod(grid)) * 27, dtype=np.float64)
    ninv = lib.oracle_mass_matrix_scalar(_ptr(g), w.size, _ptr_array(pos), _ptr(w), _ptr(M))
    return M.reshape(tuple(reversed(grid)) + (27,)), int(ninv)


def tile_keys(grid, tile, pos):
    """Per-particle tile keys (uint32, sentinel = ntiles) and tile_offsets[ntiles+1]."""
    lib = _load()
    dim = len(grid)
    pos = [_f32(p) for p in pos]
    n = pos[0].size
    g = np.array(list(grid) + [1] * (3 - dim), dtype=np.int32)
    nt = 1
    for N in grid:
        nt *= -(-N // tile)
    keys = np.zeros(n, dtype=np.uint32)
    offs = np.zeros(nt + 1, dtype=np.uint32)
    total = lib.oracle_tile_keys(dim, _ptr(g), int(tile), n, _ptr_array(pos + [pos[0]] * (3 - dim)),
                                 _ptr(keys), _ptr(offs))
    assert total == nt
    return keys, offs
