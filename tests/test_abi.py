"""The C-ABI library builds, loads and exports every symbol include/pcg.h declares;
host-side argument validation rejects bad requests before any launch.

CPU only: the calls below return from the host checks, no kernel is launched.
"""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "pcg.h")


@pytest.fixture(scope="module")
def lib():
    from particle_cell_grid_gb300 import _lib, build
    build.build()
    return _lib.load()


def declared_symbols():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"PCG_API\s+[\w\s\*]*?\b(pcg_\w+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = declared_symbols()
    for want in ("pcg_deposit_cic1d", "pcg_deposit_cic1d_grad", "pcg_deposit_zigzag", "pcg_tile_sort", "pcg_deposit_current", "pcg_assemble_mass_matrix"):
        assert want in names


def test_library_exports_every_declared_symbol(lib):
    from particle_cell_grid_gb300 import _lib
    for name in declared_symbols():
        assert hasattr(lib, name), name
        assert name in _lib.SIGNATURES, f"binding misses {name}"


def test_status_strings_and_version(lib):
    assert lib.pcg_version() >= 100
    assert lib.pcg_status_string(0) == b"ok"
    assert lib.pcg_status_string(2) == b"workspace too small"


def _grid(*g):
    return (ctypes.c_int32 * 3)(*(list(g) + [1] * (3 - len(g))))


def test_stats_check(lib):
    raw = (ctypes.c_uint8 * 24)()
    assert lib.pcg_stats_check(raw) == 0
    raw[8] = 1  # n_invalid = 1
    assert lib.pcg_stats_check(raw) == 6
    assert lib.pcg_stats_check(None) == 1


def test_cic1d_rejects_bad_arguments(lib):
    vp = ctypes.c_void_p(16)
    # nbins out of range, nsteps < 1, halfwidth <= 0, null outputs
    assert lib.pcg_deposit_cic1d(vp, vp, 10, vp, 0, 50, 0.01, 0.005, vp, vp, None) == 1
    assert lib.pcg_deposit_cic1d(vp, vp, 10, vp, 20000, 50, 0.01, 0.005, vp, vp, None) == 1
    assert lib.pcg_deposit_cic1d(vp, vp, 10, vp, 1024, 0, 0.01, 0.005, vp, vp, None) == 1
    assert lib.pcg_deposit_cic1d(vp, vp, 10, vp, 1024, 50, 0.01, 0.0, vp, vp, None) == 1
    assert lib.pcg_deposit_cic1d(vp, vp, 10, vp, 1024, 50, 0.01, 0.005, None, vp, None) == 1
    assert lib.pcg_deposit_cic1d(vp, vp, -1, vp, 1024, 50, 0.01, 0.005, vp, vp, None) == 1


def test_zigzag_rejects_bad_arguments(lib):
    vp = ctypes.c_void_p(4096)
    arr = (ctypes.c_void_p * 3)(4096, 4096, 4096)
    f = lib.pcg_deposit_zigzag
    g = _grid(8, 8, 8)
    assert f(_grid(8, 2, 8), 8, 10, arr, arr, vp, 1.0, None, vp, None, None, 0, None) == 1  # grid < 3
    assert f(g, 8, 10, arr, arr, vp, 0.0, None, vp, None, None, 0, None) == 1              # dt <= 0
    assert f(g, 8, 10, arr, arr, vp, float("nan"), None, vp, None, None, 0, None) == 1
    assert f(g, 8, 10, None, arr, vp, 1.0, None, vp, None, None, 0, None) == 1             # no pos_prev
    assert f(g, 8, 10, arr, arr, vp, 1.0, None, None, None, None, 0, None) == 1            # no J
    assert f(g, 8, 10, arr, arr, vp, 1.0, None, ctypes.c_void_p(4100), None, None, 0, None) == 1  # J unaligned
    assert f(g, 4, 10, arr, arr, vp, 1.0, vp, vp, None, vp, 1 << 20, None) == 3            # tile 4: unsupported
    assert f(g, 8, 10, arr, arr, vp, 1.0, vp, vp, None, None, 0, None) == 2                # tiled, no workspace


def test_cic1d_grad_rejects_bad_arguments(lib):
    vp = ctypes.c_void_p(16)
    f = lib.pcg_deposit_cic1d_grad
    assert f(vp, vp, 10, vp, 0, 50, 0.01, 0.005, vp, vp, vp, None) == 1
    assert f(vp, vp, 10, vp, 1024, 0, 0.01, 0.005, vp, vp, vp, None) == 1
    assert f(vp, vp, 10, vp, 1024, 50, 0.01, -1.0, vp, vp, vp, None) == 1
    assert f(vp, vp, 10, vp, 1024, 50, float("nan"), 0.005, vp, vp, vp, None) == 1
    assert f(vp, vp, 10, vp, 1024, 50, 0.01, 0.005, vp, vp, None, None) == 1  # no dx0
    assert f(vp, vp, 10, vp, 1024, 50, 0.01, 0.005, vp, None, vp, None) == 1  # no loss


def test_workspace_queries(lib):
    out = ctypes.c_size_t(0)
    # 3D 256^3 with tile 8: 32768 tiles + sentinel, block-private counters
    assert lib.pcg_tile_sort_workspace_size(3, _grid(256, 256, 256), 8, 268435456, 7, ctypes.byref(out)) == 0
    assert out.value > 268435456 * 8 * 4  # two-pass: intermediate payload + key
    # one bin per cell of 64^3: global counters (two arrays of 262145 entries)
    assert lib.pcg_tile_sort_workspace_size(3, _grid(64, 64, 64), 1, 100000, 7, ctypes.byref(out)) == 0
    assert out.value == 2 * ((262145 * 4 + 255) // 256 * 256)
    assert lib.pcg_tile_sort_workspace_size(4, _grid(8, 8, 8), 8, 10, 1, ctypes.byref(out)) == 1
    assert lib.pcg_tile_sort_workspace_size(3, _grid(8, 0, 8), 8, 10, 1, ctypes.byref(out)) == 1
    assert lib.pcg_tile_sort_workspace_size(3, _grid(8, 8, 8), 0, 10, 1, ctypes.byref(out)) == 1
    assert lib.pcg_tile_sort_workspace_size(3, _grid(8, 8, 8), 8, 10, 0, ctypes.byref(out)) == 1
    assert lib.pcg_deposit_current_workspace_size(3, _grid(16, 16, 16), 8, 100000, ctypes.byref(out)) == 0
    assert out.value >= 4 and out.value % 256 == 0
    assert lib.pcg_assemble_mass_matrix_workspace_size(_grid(64, 64, 64), 16, ctypes.byref(out)) == 0


def test_tile_sort_rejects_bad_arguments(lib):
    vp = ctypes.c_void_p(256)
    ptrs = (ctypes.c_void_p * 3)(256, 256, 256)
    g = _grid(16, 16, 16)
    # n_payload out of range
    assert lib.pcg_tile_sort(3, g, 8, 10, ptrs, 0, ptrs, ptrs, vp, None, vp, 1 << 20, None) == 1
    assert lib.pcg_tile_sort(3, g, 8, 10, ptrs, 17, ptrs, ptrs, vp, None, vp, 1 << 20, None) == 1
    # workspace too small / misaligned
    assert lib.pcg_tile_sort(3, g, 8, 10, ptrs, 1, ptrs, ptrs, vp, None, vp, 0, None) == 2
    assert lib.pcg_tile_sort(3, g, 8, 10, ptrs, 1, ptrs, ptrs, vp, None, ctypes.c_void_p(260), 1 << 20, None) == 2
    # missing tile_offsets
    assert lib.pcg_tile_sort(3, g, 8, 10, ptrs, 1, ptrs, ptrs, None, None, vp, 1 << 20, None) == 1


def test_deposit_current_rejects_bad_arguments(lib):
    vp = ctypes.c_void_p(256)
    ptrs = (ctypes.c_void_p * 3)(256, 256, 256)
    g = _grid(16, 16, 16)
    args = lambda **k: dict(dim=3, grid=g, order=1, tile=8, halo=1, block=0, n=10, pos=ptrs, vel=ptrs,
                            q=vp, offs=vp, J=vp, stats=None, ws=vp, wsb=1 << 20, s=None) | k
    call = lambda a: lib.pcg_deposit_current(a["dim"], a["grid"], a["order"], a["tile"], a["halo"], a["block"],
                                             a["n"], a["pos"], a["vel"], a["q"], a["offs"], a["J"], a["stats"],
                                             a["ws"], a["wsb"], a["s"])
    assert call(args(order=3)) == 1
    assert call(args(dim=1)) == 1
    assert call(args(block=100)) == 1
    assert call(args(J=ctypes.c_void_p(260))) == 1          # J must be 16-byte aligned
    assert call(args(tile=6)) == 3                           # valid tile without a compiled kernel
    assert call(args(halo=3)) == 3
    assert call(args(halo=-1)) == 1
    assert call(args(wsb=0)) == 2
    assert call(args(q=None)) == 1


def test_mass_matrix_rejects_bad_arguments(lib):
    vp = ctypes.c_void_p(256)
    ptrs = (ctypes.c_void_p * 3)(256, 256, 256)
    call = lambda grid=_grid(8, 8, 8), order=1, prec=0, M=vp: lib.pcg_assemble_mass_matrix(
        grid, order, prec, 10, ptrs, vp, ptrs, vp, M, None, None, 0, None)
    assert call(grid=_grid(2, 8, 8)) == 1                    # 27 offsets need an edge >= 3
    assert call(order=3) == 1
    assert call(grid=_grid(8, 4, 8), order=2) == 1           # 125 offsets need an edge >= 5
    assert call(grid=_grid(5, 5, 5), order=2, prec=3) == 1
    assert call(prec=3) == 1
    assert call(M=ctypes.c_void_p(260)) == 1


def test_scalar_mass_rejects_bad_arguments(lib):
    vp = ctypes.c_void_p(4096)
    arr = (ctypes.c_void_p * 3)(4096, 4096, 4096)
    f = lib.pcg_assemble_mass_matrix_scalar
    g = _grid(8, 8, 8)
    assert f(g, 2, 0, 10, arr, vp, vp, vp, None, None) == 1           # order 2
    assert f(g, 1, 3, 10, arr, vp, vp, vp, None, None) == 1           # precision
    assert f(_grid(8, 2, 8), 1, 0, 10, arr, vp, vp, vp, None, None) == 1
    assert f(g, 1, 0, 10, None, vp, vp, vp, None, None) == 1          # no positions
    assert f(g, 1, 0, 10, arr, vp, None, vp, None, None) == 1         # no cell offsets
    assert f(g, 1, 0, 10, arr, vp, vp, ctypes.c_void_p(4100), None, None) == 1  # M unaligned


def test_tsc_mass_rejects_small_grids_and_bad_precisions(lib):
    vp = ctypes.c_void_p(4096)
    arr = (ctypes.c_void_p * 3)(4096, 4096, 4096)
    f = lib.pcg_assemble_mass_matrix
    assert f(_grid(8, 4, 8), 2, 2, 10, arr, vp, arr, vp, vp, None, None, 0, None) == 1  # order 2 needs >= 5
    assert f(_grid(8, 8, 8), 3, 2, 10, arr, vp, arr, vp, vp, None, None, 0, None) == 1  # order 3
    assert f(_grid(8, 8, 8), 2, -1, 10, arr, vp, arr, vp, vp, None, None, 0, None) == 1  # precision
    assert f(_grid(8, 8, 8), 2, 0, 10, arr, vp, arr, vp, ctypes.c_void_p(4100), None, None, 0, None) == 1  # M align


def test_bounds_check_query_of_the_unchecked_build(lib):
    failures = ctypes.c_uint64(7)
    checked = ctypes.c_int32(-1)
    assert lib.pcg_bounds_check_failures(ctypes.byref(failures), ctypes.byref(checked)) == 0
    assert checked.value == 0 and failures.value == 0
    assert lib.pcg_bounds_check_failures(None, None) == 1
