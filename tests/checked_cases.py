"""Small cases of every kernel family, run against the library selected by
PCG_LIBRARY (the checked build in tests/test_gpu_checked.py): each result is
compared with the oracle at the tolerances of the parity tests, then the
index-check failures are read back.  Prints one JSON line; exits non-zero on a
mismatch."""
import ctypes
import json
import os
import sys

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(HERE))
sys.path.insert(0, HERE)

import oracle  # noqa: E402
import particle_cell_grid_gb300 as pcg  # noqa: E402
import synth  # noqa: E402
from helpers import DEPOSIT_TOL, MASS_TOL, assert_deposit_close, dev, host, rel_frobenius  # noqa: E402


def main():
    lib = pcg._lib.load()
    assert os.path.realpath(pcg._lib.library_path()) == os.path.realpath(os.environ["PCG_LIBRARY"])
    cases = []
    # 1D histogram and gradient, the single-cluster and the full-grid paths
    for n in (2000, 40000):
        d = synth.cic1d(n=n)
        H, loss, gx = pcg.deposit_cic1d_grad(dev(d["x0"]), dev(d["v"]), dev(d["target"]), d["nsteps"], d["dt"],
                                             d["halfwidth"])
        gr, Hr, Lr, _ = oracle.cic1d_grad(d["x0"], d["v"], d["target"], d["nbins"], d["nsteps"], d["dt"],
                                          d["halfwidth"])
        assert np.abs(host(H) - Hr).max() <= DEPOSIT_TOL * np.abs(Hr).max()
        assert np.abs(host(gx) - gr).max() <= DEPOSIT_TOL * np.abs(gr).max()
        cases.append(f"cic1d n={n}")
    # tile sort + current deposit: 2D and 3D, both orders, every halo, flat, drift and escapes
    d = synth.cic3d_drift(grid=(24, 20, 28), ppc=4)
    g = d["grid"]
    payload = [dev(a) for a in d["pos"] + d["vel"] + [d["q"]]]
    out, offs = pcg.tile_sort(g, 8, [dev(k) for k in d["key_pos"]], payload)
    for order in (1, 2):
        Jr, _ = oracle.deposit_current(g, order, d["pos"], d["vel"], d["q"])
        for halo in ((0, 1, 2) if order == 1 else (2,)):
            J = pcg.deposit_current(g, order, out[:3], out[3:6], out[6], tile_offsets=offs, tile=8, halo=halo)
            assert_deposit_close(host(J), Jr, where=f"3D order {order} halo {halo}")
        J = pcg.deposit_current(g, order, out[:3], out[3:6], out[6])
        assert_deposit_close(host(J), Jr, where=f"3D order {order} flat")
        cases.append(f"deposit 3D order {order}")
    d = synth.cic2d(grid=(40, 36), ppc=8)
    g = d["grid"]
    payload = [dev(a) for a in d["pos"] + d["vel"] + [d["q"]]]
    out, offs = pcg.tile_sort(g, 8, [dev(k) for k in d["key_pos"]], payload)
    for order in (1, 2):
        Jr, _ = oracle.deposit_current(g, order, d["pos"], d["vel"], d["q"])
        J = pcg.deposit_current(g, order, out[:2], out[2:5], out[5], tile_offsets=offs, tile=8, halo=1 + order - 1)
        assert_deposit_close(host(J), Jr, where=f"2D order {order}")
        cases.append(f"deposit 2D order {order}")
    # the sort's other paths: global counters (more bins than shared memory
    # holds) and the partition (outputs above 96 MB: 7 M x 4 fields), one pass
    # and two
    rng = np.random.default_rng(5)
    for grid, tile, n in (((64, 64, 64), 1, 40000), ((64, 64, 64), 8, 7_000_001), ((128, 128, 128), 4, 7_000_001)):
        pos = [rng.uniform(0, N, n).astype(np.float32) for N in grid]
        ids = np.arange(n, dtype=np.int32)
        out, offs = pcg.tile_sort(grid, tile, [dev(p) for p in pos], [dev(p) for p in pos] + [dev(ids)])
        keys, want = oracle.tile_keys(grid, tile, pos)
        assert np.array_equal(host(offs).astype(np.uint32), want), f"sort offsets {grid} t{tile}"
        oid = host(out[-1]).astype(np.int64)
        assert np.array_equal(np.sort(oid), ids), f"sort permutation {grid} t{tile}"
        slot_tile = np.searchsorted(want, np.arange(n), side="right") - 1
        assert np.array_equal(keys[oid], slot_tile.astype(np.uint32)), f"sort tiles {grid} t{tile}"
        cases.append(f"sort {grid} t{tile} n={n}")
    # the zigzag deposit, flat and tiled
    d = synth.zigzag3d(grid=(16, 12, 20), ppc=4, sigma_v=0.3)
    g = d["grid"]
    pp = [dev(a) for a in d["pos_prev"]]
    out, offs = pcg.tile_sort(g, 8, pp, pp + [dev(a) for a in d["pos"]] + [dev(d["q"])])
    Jr, _ = oracle.deposit_zigzag(g, d["pos_prev"], d["pos"], d["q"], d["dt"])
    for tiled in (True, False):
        J = pcg.deposit_zigzag(g, out[0:3], out[3:6], out[6], d["dt"], tile_offsets=offs if tiled else None)
        assert_deposit_close(host(J), Jr, where=f"zigzag tiled={tiled}")
    cases.append("zigzag")
    # mass matrices: CIC tensor and scalar, TSC tensor, every precision
    d = synth.mass3d(grid=(9, 8, 10), ppc=40)
    g = d["grid"]
    dp = [dev(p) for p in d["pos"]]
    out, offs = pcg.tile_sort(g, 1, dp, dp + [dev(d["w"])] + [dev(o) for o in d["omega"]])
    Mr, _ = oracle.mass_matrix(g, d["pos"], d["w"], d["omega"])
    Msr, _ = oracle.mass_matrix_scalar(g, d["pos"], d["w"])
    Mtr, _ = oracle.mass_matrix_tsc(g, d["pos"], d["w"], d["omega"])
    for prec in ("tf32", "bf16", "simt"):
        tol = MASS_TOL if prec != "simt" else 1e-5
        M = pcg.assemble_mass_matrix(g, out[:3], out[3], out[4:7], offs, precision=prec)
        assert rel_frobenius(host(M), Mr) <= tol, prec
        Ms = pcg.assemble_mass_matrix_scalar(g, out[:3], out[3], offs, precision=prec)
        assert rel_frobenius(host(Ms), Msr) <= tol, prec
        Mt = pcg.assemble_mass_matrix(g, out[:3], out[3], out[4:7], offs, precision=prec, order=2)
        assert rel_frobenius(host(Mt), Mtr) <= tol, prec
        cases.append(f"mass {prec}")
    failures = ctypes.c_uint64(0)
    checked = ctypes.c_int32(-1)
    st = lib.pcg_bounds_check_failures(ctypes.byref(failures), ctypes.byref(checked))
    assert st == 0
    print(json.dumps({"checked_build": checked.value, "failures": failures.value, "cases": cases}))


if __name__ == "__main__":
    main()
