"""pcg_deposit_current_noalloc: the deposit for callers that cannot allocate.

Such callers (a host callback, a plugin handed only its buffers, a pool that
forbids run-time allocation) get the tiled deposit with its scratch in a fixed
device array inside the library.  The result must match pcg_deposit_current,
the entry point that takes a workspace, on consecutive calls that share the
array.  This file is collected last so that a run stopping at its first failure
has already run every other test.
"""
import ctypes

import numpy as np
import pytest

import synth
from helpers import DEPOSIT_TOL, dev, host, need_gpu

PCG_ERR_INVALID_ARG = 1
PCG_ERR_WORKSPACE = 2


def _grid(g):
    return (ctypes.c_int32 * 3)(*(list(g) + [1] * (3 - len(g))))


def _ptrs(ts):
    arr = (ctypes.c_void_p * 3)()
    for i, t in enumerate(ts):
        arr[i] = t.data_ptr()
    return arr


def test_noalloc_rejects_more_chunks_than_its_array_holds():
    from particle_cell_grid_gb300 import _lib, build
    build.build()
    lib = _lib.load()
    vp = ctypes.c_void_p(256)
    p3 = (ctypes.c_void_p * 3)(256, 256, 256)
    # 2^30 + 1 particles need 65537 chunks of 16384: one more than the array holds
    st = lib.pcg_deposit_current_noalloc(3, _grid((64, 64, 64)), 1, 8, 2, 0, (1 << 30) + 1, p3, p3, vp, vp,
                                         vp, None, None)
    assert st == PCG_ERR_WORKSPACE


def test_noalloc_checks_arguments_before_its_size_limit():
    from particle_cell_grid_gb300 import _lib, build
    build.build()
    lib = _lib.load()
    vp = ctypes.c_void_p(256)
    p3 = (ctypes.c_void_p * 3)(256, 256, 256)
    big = (1 << 30) + 1  # beyond the array's chunk limit
    # an invalid order, tile size or grid is reported as such, not as a workspace shortfall
    assert lib.pcg_deposit_current_noalloc(3, _grid((64, 64, 64)), 3, 8, 2, 0, big, p3, p3, vp, vp, vp,
                                           None, None) == PCG_ERR_INVALID_ARG
    assert lib.pcg_deposit_current_noalloc(3, _grid((64, 64, 64)), 1, 0, 2, 0, big, p3, p3, vp, vp, vp,
                                           None, None) == PCG_ERR_INVALID_ARG
    assert lib.pcg_deposit_current_noalloc(3, _grid((64, 0, 64)), 1, 8, 2, 0, big, p3, p3, vp, vp, vp,
                                           None, None) == PCG_ERR_INVALID_ARG
    # an unaligned J as well
    assert lib.pcg_deposit_current_noalloc(3, _grid((64, 64, 64)), 1, 8, 2, 0, big, p3, p3, vp, vp,
                                           ctypes.c_void_p(260), None, None) == PCG_ERR_INVALID_ARG


@pytest.mark.gpu
def test_noalloc_matches_workspace_entry_point_on_consecutive_calls():
    pcg = need_gpu()
    import torch
    lib = pcg._lib.load()
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    # a large case, then a smaller one: the second call reuses the array the
    # first one filled with more entries
    for grid, ppc in (((64, 64, 64), 16), ((24, 24, 24), 4)):
        d = synth.cic3d_drift(grid=grid, ppc=ppc)
        payload = [dev(a) for a in d["pos"] + d["vel"] + [d["q"]]]
        out, offs = pcg.tile_sort(grid, 8, [dev(k) for k in d["key_pos"]], payload)
        want = pcg.deposit_current(grid, 1, out[:3], out[3:6], out[6], tile_offsets=offs, tile=8, halo=2)
        J = torch.full_like(want, np.nan)
        st = lib.pcg_deposit_current_noalloc(3, _grid(grid), 1, 8, 2, 0, d["n"], _ptrs(out[:3]),
                                             _ptrs(out[3:6]), ctypes.c_void_p(out[6].data_ptr()),
                                             ctypes.c_void_p(offs.data_ptr()), ctypes.c_void_p(J.data_ptr()),
                                             None, stream)
        assert st == 0, pcg._lib.describe(st)
        got, ref = host(J).astype(np.float64), host(want).astype(np.float64)
        for c in range(3):
            assert np.abs(got[c] - ref[c]).max() <= DEPOSIT_TOL * np.abs(ref[c]).max()
