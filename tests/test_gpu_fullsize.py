"""Full-size workloads, in the launch configuration the benchmark times.

The oracle cannot afford the whole 256^3 / 192^3 grids one particle at a time in
a test, so it computes exact values on sampled boxes of nodes: every particle
whose stencil can reach a box is fed to the oracle, which is then exact inside
the box.  Boxes include the periodic corner and, for the density bump, its peak.
Whole-grid invariants (sum_g J = sum_p q v) are checked everywhere.
"""
import numpy as np
import pytest

import oracle
import synth
from helpers import DEPOSIT_TOL, MASS_TOL, dev, host, need_gpu, rel_frobenius, stats_dict

pytestmark = [pytest.mark.gpu, pytest.mark.slow]


def _near_box(pos, grid, lo, hi, margin=3):
    """Particles whose cell lies within `margin` cells of the box [lo, hi) (periodic)."""
    sel = np.ones(pos[0].size, bool)
    for mu, N in enumerate(grid):
        c = np.floor(pos[mu]).astype(np.int64)
        d = (c - (lo[mu] - margin)) % N
        sel &= d < (hi[mu] - lo[mu] + 2 * margin)
    return np.nonzero(sel)[0]


def _box_index(grid, lo, hi):
    axes = [np.arange(l, h) % N for l, h, N in zip(lo, hi, grid)]
    return np.ix_(*reversed(axes))  # (z, y, x)


def _run_current(pcg, d):
    grid, dim = d["grid"], len(d["grid"])
    pos_d = [dev(p) for p in d["pos"]]
    vel_d = [dev(v) for v in d["vel"]]
    q_d = dev(d["q"])
    kp = [dev(k) for k in d["key_pos"]] if d["key_pos"] is not d["pos"] else pos_d
    out, offs = pcg.tile_sort(grid, d["tile"], kp, pos_d + vel_d + [q_d])
    del pos_d, vel_d, q_d, kp
    stats = pcg.new_stats()
    J = pcg.deposit_current(grid, d["order"], out[:dim], out[dim:dim + 3], out[dim + 3], tile_offsets=offs,
                            tile=d["tile"], halo=d["halo"], stats=stats)
    return host(J), stats_dict(stats)


def _check_boxes(d, J, boxes):
    grid = d["grid"]
    for lo, hi in boxes:
        idx = _near_box(d["pos"], grid, lo, hi)
        Jr, _ = oracle.deposit_current(grid, d["order"], [p[idx] for p in d["pos"]],
                                       [v[idx] for v in d["vel"]], d["q"][idx])
        box = _box_index(grid, lo, hi)
        for c in range(3):
            ref = Jr[c][box]
            got = J[c][box].astype(np.float64)
            # tolerance scale: the whole grid's max |J| (computed from the GPU
            # result, checked separately against the invariants)
            scale = max(np.abs(ref).max(), 1e-30)
            assert np.abs(got - ref).max() <= DEPOSIT_TOL * scale, (lo, c)


def _check_totals(d, J):
    for c in range(3):
        want = np.sum(d["q"].astype(np.float64) * d["vel"][c].astype(np.float64))
        got = J[c].astype(np.float64).sum()
        bound = 1e-6 * np.abs(d["q"] * d["vel"][c]).astype(np.float64).sum()
        assert abs(got - want) <= bound


def test_cic2d_512():
    pcg = need_gpu()
    d = synth.cic2d()
    J, st = _run_current(pcg, d)
    Jr, _ = oracle.deposit_current(d["grid"], 1, d["pos"], d["vel"], d["q"])
    for c in range(3):
        assert np.abs(J[c] - Jr[c]).max() <= DEPOSIT_TOL * np.abs(Jr[c]).max()
    assert st["n_escaped"] == 0 and st["n_invalid"] == 0


def test_cic3d_256_drift():
    pcg = need_gpu()
    d = synth.cic3d_drift()
    J, st = _run_current(pcg, d)
    assert st["n_invalid"] == 0
    # a displacement U[-3, 3] per axis leaves the 2-cell halo with probability
    # 5/96 per axis for a uniform in-tile position (~15 % over three axes)
    assert 0.10 * d["displaced"].size <= st["n_escaped"] <= 0.25 * d["displaced"].size
    _check_totals(d, J)
    _check_boxes(d, J, [((0, 0, 0), (12, 12, 12)), ((120, 64, 250), (136, 80, 262)),
                        ((200, 7, 99), (213, 21, 110))])


def test_quad3d_192_bump():
    pcg = need_gpu()
    d = synth.quad3d_bump()
    J, st = _run_current(pcg, d)
    assert st["n_invalid"] == 0 and st["n_escaped"] == 0
    _check_totals(d, J)
    _check_boxes(d, J, [((90, 90, 90), (102, 102, 102)), ((186, 0, 5), (198, 10, 15))])


def test_mass3d_64():
    pcg = need_gpu()
    d = synth.mass3d()
    grid = d["grid"]
    dp = [dev(p) for p in d["pos"]]
    out, offs = pcg.tile_sort(grid, 1, dp, dp + [dev(d["w"])] + [dev(o) for o in d["omega"]])
    for precision in ("tf32", "bf16"):
        stats = pcg.new_stats()
        M = host(pcg.assemble_mass_matrix(grid, out[:3], out[3], out[4:7], offs, precision=precision,
                                          stats=stats))
        assert stats_dict(stats)["error_flags"] == 0
        for lo, hi in [((0, 0, 0), (6, 6, 6)), ((30, 41, 60), (38, 47, 66))]:
            idx = _near_box(d["pos"], grid, lo, hi, margin=2)
            Mr, _ = oracle.mass_matrix(grid, [p[idx] for p in d["pos"]], d["w"][idx],
                                       [o[idx] for o in d["omega"]])
            box = _box_index(grid, lo, hi)
            assert rel_frobenius(M[box], Mr[box]) <= MASS_TOL, (precision, lo)


def test_mass3d_tsc_64():
    """Second-order (TSC) mass matrix at 64^3 x 64 ppc on tcgen05 (TF32, BF16):
    sampled node boxes against the oracle fed every particle that can reach them."""
    pcg = need_gpu()
    d = synth.mass3d()
    grid = d["grid"]
    dp = [dev(p) for p in d["pos"]]
    out, offs = pcg.tile_sort(grid, 1, dp, dp + [dev(d["w"])] + [dev(o) for o in d["omega"]])
    del dp
    refs = []
    for lo, hi in [((0, 0, 0), (5, 5, 5)), ((30, 41, 59), (36, 46, 64))]:
        idx = _near_box(d["pos"], grid, lo, hi, margin=3)
        Mr, _ = oracle.mass_matrix_tsc(grid, [p[idx] for p in d["pos"]], d["w"][idx], [o[idx] for o in d["omega"]])
        box = _box_index(grid, lo, hi)
        refs.append((box, Mr[box].copy()))
        del Mr
    for precision in ("tf32", "bf16"):
        stats = pcg.new_stats()
        M = host(pcg.assemble_mass_matrix(grid, out[:3], out[3], out[4:7], offs, precision=precision,
                                          stats=stats, order=2))
        st = stats_dict(stats)
        assert st["error_flags"] == 0 and st["n_invalid"] == 0
        for box, Mb in refs:
            assert rel_frobenius(M[box], Mb) <= MASS_TOL, precision
        del M


def test_cic1d_grad_ten_million():
    """The gradient at N = 10^7 (the size the pages time it at), checked whole."""
    pcg = need_gpu()
    d = synth.cic1d(n=10_000_000, seed=1003)
    H, L, g = pcg.deposit_cic1d_grad(dev(d["x0"]), dev(d["v"]), dev(d["target"]), d["nsteps"], d["dt"],
                                     d["halfwidth"])
    gr, Hr, Lr, nsel = oracle.cic1d_grad(d["x0"], d["v"], d["target"], d["nbins"], d["nsteps"], d["dt"],
                                         d["halfwidth"])
    H, g = host(H), host(g)
    assert np.abs(H - Hr).max() <= DEPOSIT_TOL * np.abs(Hr).max()
    assert abs(float(host(L)[0]) - Lr) <= 1e-5 * Lr
    assert np.abs(g - gr).max() <= DEPOSIT_TOL * np.abs(gr).max()
    assert np.array_equal(g == 0.0, gr == 0.0)
    assert nsel > 4_000_000


def test_zigzag3d_256():
    """Charge-conserving zigzag deposit on 256^3 x 16 ppc moves, in the bench's
    launch configuration: sampled boxes against the oracle, and the total
    current of every component against sum_p q (x - x_prev) / dt."""
    pcg = need_gpu()
    d = synth.zigzag3d()
    grid = d["grid"]
    pp = [dev(a) for a in d["pos_prev"]]
    pc = [dev(a) for a in d["pos"]]
    qd = dev(d["q"])
    out, offs = pcg.tile_sort(grid, 8, pp, pp + pc + [qd])
    del pc, qd
    stats = pcg.new_stats()
    J = host(pcg.deposit_zigzag(grid, out[0:3], out[3:6], out[6], d["dt"], tile_offsets=offs, stats=stats))
    del out, offs, pp
    st = stats_dict(stats)
    assert st["n_invalid"] == 0 and st["n_escaped"] == 0
    for lo, hi in [((0, 0, 0), (6, 6, 6)), ((250, 120, 60), (256, 128, 67)), ((128, 255, 3), (134, 258, 9))]:
        idx = _near_box(d["pos"], grid, lo, hi)
        Jr, _ = oracle.deposit_zigzag(grid, [a[idx] for a in d["pos_prev"]], [a[idx] for a in d["pos"]],
                                      d["q"][idx], d["dt"])
        box = _box_index(grid, lo, hi)
        for c in range(3):
            ref = Jr[c][box]
            assert np.abs(J[c][box].astype(np.float64) - ref).max() <= DEPOSIT_TOL * np.abs(ref).max(), (lo, c)
    for c, N in enumerate(grid):
        dx = d["pos"][c].astype(np.float64) - d["pos_prev"][c].astype(np.float64)
        dx -= N * np.round(dx / N)
        qd = d["q"].astype(np.float64) * dx / d["dt"]
        assert abs(J[c].astype(np.float64).sum() - qd.sum()) <= 1e-6 * np.abs(qd).sum()
