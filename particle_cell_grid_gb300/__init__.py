"""GB300-native particle-to-grid deposit: thin Python binding of libpcg.so.

Every function here only marshals arguments (torch CUDA tensors -> device
pointers, the current CUDA stream) and calls the C ABI of ``include/pcg.h``;
every step of the computation runs in the library's sm_103a kernels.  PyTorch
provides device memory and streams.  Outputs not supplied by the caller are
allocated with torch; workspaces likewise.

Entry points (same names as the C ABI without the ``pcg_`` prefix):
  deposit_cic1d, deposit_cic1d_grad, tile_sort, deposit_current, deposit_zigzag,
  assemble_mass_matrix, assemble_mass_matrix_scalar,
  plus the *_workspace_size queries and stats helpers.
"""
from __future__ import annotations

import ctypes

import torch

from . import _lib
from ._lib import PcgError, check

__all__ = [
    "PcgError", "version", "deposit_cic1d", "deposit_cic1d_grad", "tile_sort", "tile_sort_workspace_size",
    "deposit_current", "deposit_current_workspace_size", "deposit_zigzag", "assemble_mass_matrix",
    "assemble_mass_matrix_scalar",
    "assemble_mass_matrix_workspace_size", "new_stats", "read_stats", "n_tiles",
    "profile_enable", "profile_collect",
]

STATS_BYTES = 24
PRECISION = {"tf32": 0, "bf16": 1, "simt": 2}


def version() -> int:
    return int(_lib.load().pcg_version())


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else ctypes.c_void_p(0)


def _dev(t, dtype=None, name="tensor"):
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError(f"{name} must be a CUDA tensor")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must have dtype {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return t


def _stream(stream):
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _grid_arr(grid):
    return (ctypes.c_int32 * 3)(*(list(grid) + [1] * (3 - len(grid))))


def _ptr_arr(ts, n=None):
    n = len(ts) if n is None else n
    arr = (ctypes.c_void_p * max(n, 1))()
    for i, t in enumerate(ts):
        arr[i] = t.data_ptr()
    return arr


def n_tiles(grid, tile) -> int:
    nt = 1
    for N in grid:
        nt *= -(-int(N) // int(tile))
    return nt


def new_stats(device=None) -> torch.Tensor:
    """A zeroed device pcg_stats (24 bytes) as a uint8 tensor."""
    return torch.zeros(STATS_BYTES, dtype=torch.uint8, device=device or "cuda")


def read_stats(stats: torch.Tensor) -> dict:
    raw = stats.cpu().numpy().tobytes()
    esc, inv = int.from_bytes(raw[0:8], "little"), int.from_bytes(raw[8:16], "little")
    flags = int.from_bytes(raw[16:20], "little")
    return {"n_escaped": esc, "n_invalid": inv, "error_flags": flags}


def _workspace(nbytes, device, workspace):
    if nbytes == 0:
        return workspace
    if workspace is not None:
        if workspace.numel() * workspace.element_size() < nbytes:
            raise ValueError(f"workspace needs {nbytes} bytes")
        return workspace
    return torch.empty(nbytes, dtype=torch.uint8, device=device)


def _ws_bytes(t):
    return 0 if t is None else t.numel() * t.element_size()


# ---------------------------------------------------------------------------
def deposit_cic1d(x0, v, target, nsteps=50, dt=0.01, halfwidth=0.005, H=None, loss=None, stream=None):
    """1D windowed CIC histogram H (float32[nbins]) and loss (float64[1])."""
    _dev(x0, torch.float32, "x0")
    _dev(v, torch.float32, "v")
    _dev(target, torch.float32, "target")
    nb = target.numel()
    H = torch.empty(nb, dtype=torch.float32, device=target.device) if H is None else _dev(H, torch.float32, "H")
    loss = torch.empty(1, dtype=torch.float64, device=target.device) if loss is None else _dev(loss, torch.float64, "loss")
    st = _lib.load().pcg_deposit_cic1d(_ptr(x0), _ptr(v), x0.numel(), _ptr(target), nb, int(nsteps),
                                       float(dt), float(halfwidth), _ptr(H), _ptr(loss), _stream(stream))
    check(st, "pcg_deposit_cic1d")
    return H, loss


def deposit_cic1d_grad(x0, v, target, nsteps=50, dt=0.01, halfwidth=0.005, H=None, loss=None, dx0=None,
                       stream=None):
    """Forward (H, loss) and dL/dx0 (float64[n]) of the 1D windowed CIC loss."""
    _dev(x0, torch.float32, "x0")
    _dev(v, torch.float32, "v")
    _dev(target, torch.float32, "target")
    nb = target.numel()
    H = torch.empty(nb, dtype=torch.float32, device=target.device) if H is None else _dev(H, torch.float32, "H")
    loss = torch.empty(1, dtype=torch.float64, device=target.device) if loss is None else _dev(loss, torch.float64, "loss")
    dx0 = torch.empty(x0.numel(), dtype=torch.float64, device=target.device) if dx0 is None else _dev(dx0, torch.float64, "dx0")
    st = _lib.load().pcg_deposit_cic1d_grad(_ptr(x0), _ptr(v), x0.numel(), _ptr(target), nb, int(nsteps),
                                            float(dt), float(halfwidth), _ptr(H), _ptr(loss), _ptr(dx0),
                                            _stream(stream))
    check(st, "pcg_deposit_cic1d_grad")
    return H, loss, dx0


# ---------------------------------------------------------------------------
def tile_sort_workspace_size(grid, tile, n, n_payload=7) -> int:
    out = ctypes.c_size_t(0)
    check(_lib.load().pcg_tile_sort_workspace_size(len(grid), _grid_arr(grid), int(tile), int(n), int(n_payload),
                                                    ctypes.byref(out)), "pcg_tile_sort_workspace_size")
    return out.value


def tile_sort(grid, tile, key_pos, payload, out=None, tile_offsets=None, stats=None, workspace=None,
              stream=None):
    """Counting sort of particles into tiles.

    key_pos: list of dim float32 tensors; payload: list of 4-byte tensors of the
    same length.  Returns (permuted payload list, tile_offsets uint32-as-int32
    tensor of n_tiles + 1 entries).
    """
    dim = len(grid)
    n = key_pos[0].numel()
    for i, k in enumerate(key_pos):
        _dev(k, torch.float32, f"key_pos[{i}]")
    for i, p in enumerate(payload):
        _dev(p, None, f"payload[{i}]")
        if p.element_size() != 4 or p.numel() != n:
            raise ValueError("payload arrays must hold n 4-byte elements")
    dev = key_pos[0].device
    if out is None:
        out = [torch.empty_like(p) for p in payload]
    nt = n_tiles(grid, tile)
    if tile_offsets is None:
        tile_offsets = torch.empty(nt + 1, dtype=torch.int32, device=dev)
    if tile_offsets.numel() != nt + 1 or tile_offsets.element_size() != 4:
        raise ValueError("tile_offsets must hold n_tiles + 1 32-bit entries")
    ws = _workspace(tile_sort_workspace_size(grid, tile, n, len(payload)), dev, workspace)
    st = _lib.load().pcg_tile_sort(dim, _grid_arr(grid), int(tile), n, _ptr_arr(key_pos, 3),
                                   len(payload), _ptr_arr(payload), _ptr_arr(out), _ptr(tile_offsets),
                                   _ptr(stats), _ptr(ws), _ws_bytes(ws), _stream(stream))
    check(st, "pcg_tile_sort")
    return out, tile_offsets


# ---------------------------------------------------------------------------
def deposit_current_workspace_size(grid, tile, n) -> int:
    out = ctypes.c_size_t(0)
    check(_lib.load().pcg_deposit_current_workspace_size(len(grid), _grid_arr(grid), int(tile), int(n),
                                                          ctypes.byref(out)),
          "pcg_deposit_current_workspace_size")
    return out.value


def deposit_current(grid, order, pos, vel, q, tile_offsets=None, tile=8, halo=1, block=0, J=None,
                    stats=None, workspace=None, stream=None):
    """J = sum_p q v W (float32[3, *reversed(grid)]); tiled when tile_offsets is given."""
    dim = len(grid)
    n = q.numel()
    for i, t in enumerate(pos):
        _dev(t, torch.float32, f"pos[{i}]")
    for i, t in enumerate(vel):
        _dev(t, torch.float32, f"vel[{i}]")
    _dev(q, torch.float32, "q")
    dev = q.device
    shape = (3,) + tuple(int(N) for N in reversed(grid))
    J = torch.empty(shape, dtype=torch.float32, device=dev) if J is None else _dev(J, torch.float32, "J")
    if tile_offsets is not None:
        _dev(tile_offsets, None, "tile_offsets")
        ws = _workspace(deposit_current_workspace_size(grid, tile, n), dev, workspace)
    else:
        ws = workspace
    st = _lib.load().pcg_deposit_current(dim, _grid_arr(grid), int(order), int(tile), int(halo),
                                         int(block), n, _ptr_arr(pos, 3), _ptr_arr(vel, 3), _ptr(q),
                                         _ptr(tile_offsets), _ptr(J), _ptr(stats), _ptr(ws),
                                         _ws_bytes(ws), _stream(stream))
    check(st, "pcg_deposit_current")
    return J


def deposit_zigzag(grid, pos_prev, pos, q, dt, tile_offsets=None, tile=8, J=None, stats=None, workspace=None,
                   stream=None):
    """Charge-conserving zigzag current of the moves pos_prev -> pos
    (float32[3, Nz, Ny, Nx], J[c] on the edges from each node towards +e_c);
    tiled when tile_offsets (a tile sort keyed on pos_prev) is given."""
    assert len(grid) == 3
    n = q.numel()
    for i, t in enumerate(pos_prev):
        _dev(t, torch.float32, f"pos_prev[{i}]")
    for i, t in enumerate(pos):
        _dev(t, torch.float32, f"pos[{i}]")
    _dev(q, torch.float32, "q")
    dev = q.device
    shape = (3,) + tuple(int(N) for N in reversed(grid))
    J = torch.empty(shape, dtype=torch.float32, device=dev) if J is None else _dev(J, torch.float32, "J")
    if tile_offsets is not None:
        _dev(tile_offsets, None, "tile_offsets")
        ws = _workspace(deposit_current_workspace_size(grid, tile, n), dev, workspace)
    else:
        ws = workspace
    st = _lib.load().pcg_deposit_zigzag(_grid_arr(grid), int(tile), n, _ptr_arr(pos_prev, 3), _ptr_arr(pos, 3),
                                        _ptr(q), float(dt), _ptr(tile_offsets), _ptr(J), _ptr(stats), _ptr(ws),
                                        _ws_bytes(ws), _stream(stream))
    check(st, "pcg_deposit_zigzag")
    return J


# ---------------------------------------------------------------------------
def assemble_mass_matrix_workspace_size(grid, n) -> int:
    out = ctypes.c_size_t(0)
    check(_lib.load().pcg_assemble_mass_matrix_workspace_size(_grid_arr(grid), int(n), ctypes.byref(out)),
          "pcg_assemble_mass_matrix_workspace_size")
    return out.value


def assemble_mass_matrix(grid, pos, w, omega, cell_offsets, precision="tf32", M=None, stats=None,
                         workspace=None, stream=None, order=1):
    """M[g][o][i][j] from cell-sorted particles: float32[Nz, Ny, Nx, 27, 3, 3] for
    order 1 (CIC), float32[Nz, Ny, Nx, 125, 3, 3] for order 2 (TSC, CUDA cores)."""
    n = w.numel()
    for i, t in enumerate(pos):
        _dev(t, torch.float32, f"pos[{i}]")
    for i, t in enumerate(omega):
        _dev(t, torch.float32, f"omega[{i}]")
    _dev(w, torch.float32, "w")
    _dev(cell_offsets, None, "cell_offsets")
    dev = w.device
    shape = tuple(int(N) for N in reversed(grid)) + ((27 if order == 1 else 125), 3, 3)
    M = torch.empty(shape, dtype=torch.float32, device=dev) if M is None else _dev(M, torch.float32, "M")
    ws = _workspace(assemble_mass_matrix_workspace_size(grid, n), dev, workspace)
    prec = PRECISION[precision] if isinstance(precision, str) else int(precision)
    st = _lib.load().pcg_assemble_mass_matrix(_grid_arr(grid), int(order), prec, n, _ptr_arr(pos, 3), _ptr(w),
                                              _ptr_arr(omega, 3), _ptr(cell_offsets), _ptr(M), _ptr(stats),
                                              _ptr(ws), _ws_bytes(ws), _stream(stream))
    check(st, "pcg_assemble_mass_matrix")
    return M


def assemble_mass_matrix_scalar(grid, pos, w, cell_offsets, precision="tf32", M=None, stats=None, stream=None):
    """Scalar mass matrix M[g][o] (float32[Nz, Ny, Nx, 27]) = sum_p w W_pg W_pg' from
    cell-sorted particles."""
    n = w.numel()
    for i, t in enumerate(pos):
        _dev(t, torch.float32, f"pos[{i}]")
    _dev(w, torch.float32, "w")
    _dev(cell_offsets, None, "cell_offsets")
    shape = tuple(int(N) for N in reversed(grid)) + (27,)
    M = torch.empty(shape, dtype=torch.float32, device=w.device) if M is None else _dev(M, torch.float32, "M")
    st = _lib.load().pcg_assemble_mass_matrix_scalar(_grid_arr(grid), 1, PRECISION[precision], n, _ptr_arr(pos, 3),
                                                     _ptr(w), _ptr(cell_offsets), _ptr(M), _ptr(stats),
                                                     _stream(stream))
    check(st, "pcg_assemble_mass_matrix_scalar")
    return M


# ---------------------------------------------------------------------------
def profile_enable(on: bool = True) -> None:
    """Start / stop recording an event pair around every library kernel launch."""
    check(_lib.load().pcg_profile_enable(1 if on else 0), "pcg_profile_enable")


def profile_collect(max_entries: int = 64) -> dict:
    """{kernel name: (launches, total ms)} for the launches recorded so far (then cleared)."""
    names = ctypes.create_string_buffer(64 * max_entries)
    launches = (ctypes.c_int64 * max_entries)()
    total = (ctypes.c_double * max_entries)()
    count = ctypes.c_int32(0)
    check(_lib.load().pcg_profile_collect(max_entries, names, launches, total, ctypes.byref(count)),
          "pcg_profile_collect")
    out = {}
    for i in range(min(count.value, max_entries)):
        nm = names.raw[64 * i:64 * (i + 1)].split(b"\0", 1)[0].decode()
        out[nm] = (int(launches[i]), float(total[i]))
    return out
