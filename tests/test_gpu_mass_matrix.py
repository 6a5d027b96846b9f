"""GPU ECSIM mass matrix (tcgen05 TF32 / BF16 and the CUDA-core baseline) against
the fp64 oracle: relative Frobenius error <= 2e-3 on the tensor cores; the fp32
CUDA-core path must be far tighter (1e-5)."""
import numpy as np
import pytest

import oracle
import synth
from helpers import MASS_TOL, dev, host, need_gpu, rel_frobenius, stats_dict

pytestmark = pytest.mark.gpu

TOL = {"tf32": MASS_TOL, "bf16": MASS_TOL, "simt": 1e-5}


def _assemble(pcg, grid, pos, w, omega, precision):
    dp = [dev(p) for p in pos]
    out, offs = pcg.tile_sort(grid, 1, dp, dp + [dev(w)] + [dev(o) for o in omega])
    stats = pcg.new_stats()
    M = pcg.assemble_mass_matrix(grid, out[:3], out[3], out[4:7], offs, precision=precision, stats=stats)
    return host(M), stats_dict(stats)


@pytest.mark.parametrize("precision", ["tf32", "bf16", "simt"])
def test_workload_recipe_small(precision):
    pcg = need_gpu()
    d = synth.mass3d(grid=(16, 16, 16), ppc=64)
    M, st = _assemble(pcg, d["grid"], d["pos"], d["w"], d["omega"], precision)
    Mr, _ = oracle.mass_matrix(d["grid"], d["pos"], d["w"], d["omega"])
    assert rel_frobenius(M, Mr) <= TOL[precision]
    assert st["error_flags"] == 0


@pytest.mark.parametrize("precision", ["tf32", "bf16", "simt"])
@pytest.mark.parametrize("grid", [(3, 3, 3), (5, 4, 6), (9, 7, 8)])
def test_variable_occupancy(precision, grid):
    # 0..200 particles per cell: empty cells, several batches per cell, padding
    pcg = need_gpu()
    rng = np.random.default_rng(sum(grid))
    ncell = int(np.prod(grid))
    counts = rng.integers(0, 200, ncell)
    counts[::5] = 0
    cell = np.repeat(np.arange(ncell), counts)
    n = cell.size
    coords = [cell % grid[0], (cell // grid[0]) % grid[1], cell // (grid[0] * grid[1])]
    pos = [synth._inside_cell_f32(c, rng.random(n)) for c in coords]
    perm = rng.permutation(n)
    pos = [p[perm] for p in pos]
    w = rng.uniform(0.5, 1.5, n).astype(np.float32)
    omega = [rng.normal(0, 0.8, n).astype(np.float32) for _ in range(3)]
    M, st = _assemble(pcg, grid, pos, w, omega, precision)
    Mr, _ = oracle.mass_matrix(grid, pos, w, omega)
    assert rel_frobenius(M, Mr) <= TOL[precision]
    # symmetry per component holds exactly in structure: M[g][d] ~ M[g+d][-d]
    assert st["error_flags"] == 0


def test_listed_cell_mismatch_is_still_exact():
    # cell_offsets describing other particles than the arrays hold: every
    # misplaced particle goes through the slow global path and is flagged
    pcg = need_gpu()
    grid = (6, 6, 6)
    d = synth.mass3d(grid=grid, ppc=8, seed=3)
    dp = [dev(p) for p in d["pos"]]
    out, offs = pcg.tile_sort(grid, 1, dp, dp + [dev(d["w"])] + [dev(o) for o in d["omega"]])
    # shuffle the sorted arrays so that the layout no longer matches
    perm = np.random.default_rng(1).permutation(d["n"])
    arrs = [host(t)[perm] for t in out]
    stats = pcg.new_stats()
    M = pcg.assemble_mass_matrix(grid, [dev(a) for a in arrs[:3]], dev(arrs[3]), [dev(a) for a in arrs[4:7]],
                                 offs, precision="tf32", stats=stats)
    Mr, _ = oracle.mass_matrix(grid, d["pos"], d["w"], d["omega"])
    assert rel_frobenius(host(M), Mr) <= MASS_TOL
    assert stats_dict(stats)["error_flags"] & 2


def test_empty():
    pcg = need_gpu()
    grid = (4, 4, 4)
    z = np.zeros(0, np.float32)
    offs = np.zeros(65, np.int32)
    M = pcg.assemble_mass_matrix(grid, [dev(z)] * 3, dev(z), [dev(z)] * 3, dev(offs))
    assert np.all(host(M) == 0)


# ---------------------------------------------------------------------------
# scalar (MPM) mass matrix: the same assembly with one component
def _assemble_scalar(pcg, grid, pos, w, precision):
    dp = [dev(p) for p in pos]
    out, offs = pcg.tile_sort(grid, 1, dp, dp + [dev(w)])
    stats = pcg.new_stats()
    M = pcg.assemble_mass_matrix_scalar(grid, out[:3], out[3], offs, precision=precision, stats=stats)
    return host(M), stats_dict(stats)


@pytest.mark.parametrize("precision", ["tf32", "bf16", "simt"])
@pytest.mark.parametrize("grid,ppc", [((16, 16, 16), 64), ((5, 4, 6), 100), ((3, 3, 3), 7)])
def test_scalar_matches_oracle(precision, grid, ppc):
    pcg = need_gpu()
    d = synth.mass3d(grid=grid, ppc=ppc, seed=sum(grid) + ppc)
    M, st = _assemble_scalar(pcg, grid, d["pos"], d["w"], precision)
    Mr, _ = oracle.mass_matrix_scalar(grid, d["pos"], d["w"])
    assert M.shape == Mr.shape
    assert rel_frobenius(M, Mr) <= TOL[precision]
    assert st["error_flags"] == 0


@pytest.mark.parametrize("precision", ["tf32", "simt"])
def test_scalar_variable_occupancy_and_mismatch(precision):
    pcg = need_gpu()
    grid = (9, 7, 8)
    rng = np.random.default_rng(11)
    ncell = int(np.prod(grid))
    counts = rng.integers(0, 200, ncell)
    counts[::5] = 0
    cell = np.repeat(np.arange(ncell), counts)
    n = cell.size
    coords = [cell % grid[0], (cell // grid[0]) % grid[1], cell // (grid[0] * grid[1])]
    pos = [synth._inside_cell_f32(c, rng.random(n))[rng.permutation(n)] for c in coords]
    w = rng.uniform(0.5, 1.5, n).astype(np.float32)
    M, st = _assemble_scalar(pcg, grid, pos, w, precision)
    Mr, _ = oracle.mass_matrix_scalar(grid, pos, w)
    assert rel_frobenius(M, Mr) <= TOL[precision]
    # arrays that no longer match their cell layout: exact through the slow path, flagged
    dp = [dev(p) for p in pos]
    out, offs = pcg.tile_sort(grid, 1, dp, dp + [dev(w)])
    perm = np.random.default_rng(2).permutation(n)
    arrs = [host(t)[perm] for t in out]
    stats = pcg.new_stats()
    M = pcg.assemble_mass_matrix_scalar(grid, [dev(a) for a in arrs[:3]], dev(arrs[3]), offs,
                                        precision=precision, stats=stats)
    assert rel_frobenius(host(M), Mr) <= TOL[precision]
    assert stats_dict(stats)["error_flags"] & 2


# ---------------------------------------------------------------------------
# second-order (TSC) matrix on CUDA cores: 125 offsets, support groups
def _assemble_tsc(pcg, grid, pos, w, omega, precision="simt", stats=None):
    dp = [dev(p) for p in pos]
    out, offs = pcg.tile_sort(grid, 1, dp, dp + [dev(w)] + [dev(o) for o in omega])
    return pcg.assemble_mass_matrix(grid, out[:3], out[3], out[4:7], offs, precision=precision, stats=stats,
                                    order=2)


@pytest.mark.parametrize("precision", ["tf32", "bf16", "simt"])
@pytest.mark.parametrize("grid,ppc", [((5, 6, 5), 20), ((8, 8, 8), 64), ((7, 5, 9), 3), ((9, 6, 5), 130)])
def test_tsc_matches_oracle(grid, ppc, precision):
    pcg = need_gpu()
    d = synth.mass3d(grid=grid, ppc=ppc, seed=sum(grid) + ppc + 7)
    stats = pcg.new_stats()
    M = host(_assemble_tsc(pcg, grid, d["pos"], d["w"], d["omega"], stats=stats, precision=precision))
    Mr, _ = oracle.mass_matrix_tsc(grid, d["pos"], d["w"], d["omega"])
    assert M.shape == Mr.shape
    assert rel_frobenius(M, Mr) <= TOL[precision]
    st = stats_dict(stats)
    assert st["error_flags"] == 0 and st["n_invalid"] == 0


@pytest.mark.parametrize("precision", ["tf32", "bf16", "simt"])
def test_tsc_variable_occupancy_and_mismatch(precision):
    pcg = need_gpu()
    grid = (6, 7, 5)
    rng = np.random.default_rng(12)
    ncell = int(np.prod(grid))
    counts = rng.integers(0, 150, ncell)
    counts[::4] = 0
    cell = np.repeat(np.arange(ncell), counts)
    n = cell.size
    coords = [cell % grid[0], (cell // grid[0]) % grid[1], cell // (grid[0] * grid[1])]
    perm = rng.permutation(n)
    pos = [synth._inside_cell_f32(c, rng.random(n))[perm] for c in coords]
    w = rng.uniform(0.5, 1.5, n).astype(np.float32)
    omega = [rng.normal(0, 0.8, n).astype(np.float32) for _ in range(3)]
    Mr, _ = oracle.mass_matrix_tsc(grid, pos, w, omega)
    assert rel_frobenius(host(_assemble_tsc(pcg, grid, pos, w, omega, precision=precision)), Mr) <= TOL[precision]
    # arrays that no longer match their cell layout: exact through the slow path, flagged
    dp = [dev(p) for p in pos]
    out, offs = pcg.tile_sort(grid, 1, dp, dp + [dev(w)] + [dev(o) for o in omega])
    perm2 = np.random.default_rng(3).permutation(n)
    arrs = [host(t)[perm2] for t in out]
    stats = pcg.new_stats()
    M = pcg.assemble_mass_matrix(grid, [dev(a) for a in arrs[:3]], dev(arrs[3]), [dev(a) for a in arrs[4:7]], offs,
                                 precision=precision, stats=stats, order=2)
    assert rel_frobenius(host(M), Mr) <= TOL[precision]
    assert stats_dict(stats)["error_flags"] & 2


@pytest.mark.parametrize("precision,order", [("tf32", 1), ("bf16", 1), ("simt", 1), ("tf32", 2), ("bf16", 2),
                                             ("simt", 2)])
def test_invalid_particles_are_skipped_and_counted(precision, order):
    # NaN and x = N before the sort (parked in the sentinel bin after the last
    # cell: the tail pass), and coordinates made invalid after the sort while
    # still listed under a cell: all are skipped and counted in n_invalid
    pcg = need_gpu()
    grid = (6, 6, 6)
    d = synth.mass3d(grid=grid, ppc=8, seed=5)
    pos = [p.copy() for p in d["pos"]]
    rng = np.random.default_rng(7)
    bad = rng.choice(d["n"], 12, replace=False)
    pos[0][bad[:6]] = np.nan
    pos[1][bad[6:]] = np.float32(grid[1])
    dp = [dev(p) for p in pos]
    out, offs = pcg.tile_sort(grid, 1, dp, dp + [dev(d["w"])] + [dev(o) for o in d["omega"]])
    arrs = [host(t).copy() for t in out]
    listed = int(host(offs)[-1])
    assert listed == d["n"] - 12
    idx = rng.choice(listed, 10, replace=False)
    arrs[2][idx[:5]] = np.float32(-0.5)
    arrs[0][idx[5:]] = np.float32(np.inf)
    stats = pcg.new_stats()
    M = pcg.assemble_mass_matrix(grid, [dev(a) for a in arrs[:3]], dev(arrs[3]), [dev(a) for a in arrs[4:7]],
                                 offs, precision=precision, stats=stats, order=order)
    ref = oracle.mass_matrix if order == 1 else oracle.mass_matrix_tsc
    Mr, ninv = ref(grid, arrs[:3], arrs[3], arrs[4:7])
    assert ninv == 22
    assert stats_dict(stats)["n_invalid"] == 22
    assert rel_frobenius(host(M), Mr) <= TOL[precision]


def test_scalar_invalid_particles_are_skipped_and_counted():
    pcg = need_gpu()
    grid = (5, 4, 6)
    d = synth.mass3d(grid=grid, ppc=9, seed=8)
    pos = [p.copy() for p in d["pos"]]
    pos[2][:7] = np.nan
    dp = [dev(p) for p in pos]
    out, offs = pcg.tile_sort(grid, 1, dp, dp + [dev(d["w"])])
    stats = pcg.new_stats()
    M = pcg.assemble_mass_matrix_scalar(grid, out[:3], out[3], offs, precision="tf32", stats=stats)
    Mr, ninv = oracle.mass_matrix_scalar(grid, pos, d["w"])
    assert ninv == 7 and stats_dict(stats)["n_invalid"] == 7
    assert rel_frobenius(host(M), Mr) <= MASS_TOL
