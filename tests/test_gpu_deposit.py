"""GPU current deposit (flat and tiled) against the fp64 oracle.

Per component, max |J_gpu - J_oracle| <= 1e-5 * max |J_oracle|.  The tiled path
must give the oracle's result for any halo, with drifted or unsorted particles
(the escape valve), with invalid particles, partial tiles and a ragged tail.
"""
import numpy as np
import pytest

import oracle
import synth
from helpers import assert_deposit_close, dev, host, need_gpu, stats_dict

pytestmark = pytest.mark.gpu


def _deposit(pcg, grid, order, pos, vel, q, tile=None, halo=1, key_pos=None, block=0):
    """Flat when tile is None, else sort (keys from key_pos) then tiled deposit."""
    stats = pcg.new_stats()
    pos_d = [dev(p) for p in pos]
    vel_d = [dev(v) for v in vel]
    q_d = dev(q)
    if tile is None:
        J = pcg.deposit_current(grid, order, pos_d, vel_d, q_d, stats=stats)
        return host(J), stats_dict(stats)
    kp = [dev(k) for k in (key_pos if key_pos is not None else pos)]
    out, offs = pcg.tile_sort(grid, tile, kp, pos_d + vel_d + [q_d], stats=pcg.new_stats())
    dim = len(grid)
    J = pcg.deposit_current(grid, order, out[:dim], out[dim:dim + 3], out[dim + 3], tile_offsets=offs,
                            tile=tile, halo=halo, block=block, stats=stats)
    return host(J), stats_dict(stats)


def _random(rng, grid, n, sigma=0.2):
    pos = [rng.uniform(0, N, n).astype(np.float32) for N in grid]
    vel = [rng.normal(0, sigma, n).astype(np.float32) for _ in range(3)]
    q = rng.choice([-1.0, 1.0], n).astype(np.float32)
    return pos, vel, q


@pytest.mark.parametrize("grid", [(64, 64), (37, 21), (24, 24, 24), (19, 13, 11)])
@pytest.mark.parametrize("order", [1, 2])
def test_flat(grid, order):
    pcg = need_gpu()
    rng = np.random.default_rng(len(grid) * 10 + order)
    pos, vel, q = _random(rng, grid, 30001)
    J, st = _deposit(pcg, grid, order, pos, vel, q)
    Jr, _ = oracle.deposit_current(grid, order, pos, vel, q)
    assert_deposit_close(J, Jr)
    assert st["n_invalid"] == 0


@pytest.mark.parametrize("grid,tile", [((64, 64), 8), ((37, 21), 8), ((20, 20), 4), ((32, 32, 32), 8),
                                       ((19, 13, 11), 4), ((24, 17, 9), 8)])
@pytest.mark.parametrize("order,halo", [(1, 0), (1, 1), (1, 2), (2, 0), (2, 1), (2, 2)])
def test_tiled_any_halo(grid, tile, order, halo):
    pcg = need_gpu()
    rng = np.random.default_rng(hash((grid, tile, order, halo)) % 2 ** 32)
    pos, vel, q = _random(rng, grid, 60001)
    J, st = _deposit(pcg, grid, order, pos, vel, q, tile=tile, halo=halo)
    Jr, _ = oracle.deposit_current(grid, order, pos, vel, q)
    assert_deposit_close(J, Jr, where=f"{grid} t{tile} o{order} h{halo}")
    if halo >= 2 or (halo >= 1 and order == 1):
        assert st["n_escaped"] == 0  # deposit at the sort positions always fits


@pytest.mark.parametrize("order", [1, 2])
def test_tiled_drift_and_escape(order):
    # sort on x_s, deposit at x = x_s + drift: small drifts stay in the halo,
    # the displaced particles escape to global atomics
    pcg = need_gpu()
    grid = (40, 36, 32)
    rng = np.random.default_rng(77 + order)
    n = 80000
    xs = [rng.uniform(0, N, n).astype(np.float32) for N in grid]
    pos = []
    for mu, N in enumerate(grid):
        d = rng.normal(0, 0.3, n)
        d[:500] += rng.uniform(-5, 5, 500)
        pos.append(synth.to_cell_f32(xs[mu].astype(np.float64) + d, N))
    vel = [rng.normal(0, 0.1, n).astype(np.float32) for _ in range(3)]
    q = rng.choice([-1.0, 1.0], n).astype(np.float32)
    J, st = _deposit(pcg, grid, order, pos, vel, q, tile=8, halo=2, key_pos=xs)
    Jr, _ = oracle.deposit_current(grid, order, pos, vel, q)
    assert_deposit_close(J, Jr)
    assert st["n_escaped"] > 0


@pytest.mark.parametrize("order", [1, 2])
def test_tiled_one_dense_cell(order):
    # ~3500 particles in one cell (about half of each round of that tile): its
    # support group overflows the per-round lists and the excess takes the
    # general path.  (Many more in one cell would put the fp32 sum of the
    # node's contributions, in any order, beyond the 1e-5 relative tolerance.)
    pcg = need_gpu()
    grid = (32, 24, 16)
    rng = np.random.default_rng(19 + order)
    n = 70001
    pos, vel, q = _random(rng, grid, n)
    hot = rng.random(n) < 0.05
    for mu, c in enumerate((13, 6, 9)):
        pos[mu][hot] = (c + rng.random(int(hot.sum()))).astype(np.float32)
    J, st = _deposit(pcg, grid, order, pos, vel, q, tile=8, halo=2)
    Jr, _ = oracle.deposit_current(grid, order, pos, vel, q)
    assert_deposit_close(J, Jr)
    assert st["n_escaped"] == 0 and st["n_invalid"] == 0


def test_tiled_stale_layout_unsorted_input():
    # a layout whose ranges do not match the particles at all: everything that
    # does not fit escapes, and the result is still exact
    pcg = need_gpu()
    grid = (32, 32, 32)
    rng = np.random.default_rng(5)
    pos, vel, q = _random(rng, grid, 40000)
    keys, offs = oracle.tile_keys(grid, 8, pos)          # counts right, order wrong
    stats = pcg.new_stats()
    J = pcg.deposit_current(grid, 1, [dev(p) for p in pos], [dev(v) for v in vel], dev(q),
                            tile_offsets=dev(offs.view(np.int32)), tile=8, halo=1, stats=stats)
    Jr, _ = oracle.deposit_current(grid, 1, pos, vel, q)
    assert_deposit_close(host(J), Jr)
    assert stats_dict(stats)["n_escaped"] > 30000


def test_invalid_particles_skipped_and_tail_pass():
    pcg = need_gpu()
    grid = (24, 24, 24)
    rng = np.random.default_rng(8)
    pos, vel, q = _random(rng, grid, 20000)
    pos[1][:40] = np.nan
    pos[2][40:60] = 24.0
    for tiled in (False, True):
        J, st = _deposit(pcg, grid, 1, pos, vel, q, tile=8 if tiled else None, halo=1)
        Jr, ninv = oracle.deposit_current(grid, 1, pos, vel, q)
        assert_deposit_close(J, Jr)
        assert st["n_invalid"] == ninv == 60


@pytest.mark.parametrize("halo", [1, 2])
def test_drift_out_of_domain_in_a_partial_last_tile(halo):
    # grid edges not multiples of the tile: the last tile along each axis sticks
    # out of the grid; particles sorted inside it whose deposit position drifted
    # past N (or below 0 in the first tile) are invalid, not deposited
    pcg = need_gpu()
    grid = (20, 19, 21)
    rng = np.random.default_rng(31)
    n = 30000
    kp = [rng.uniform(0, N, n).astype(np.float32) for N in grid]
    vel = [rng.normal(0, 0.05, n).astype(np.float32) for _ in range(3)]
    q = rng.choice([-1.0, 1.0], n).astype(np.float32)
    pos = [k.copy() for k in kp]
    for mu, N in enumerate(grid):
        hi = np.flatnonzero(kp[mu] > N - 1)[:50]
        pos[mu][hi] = np.float32(N) + rng.uniform(0, 0.9, hi.size).astype(np.float32)  # drifted past N
        lo = np.flatnonzero(kp[mu] < 1)[:50]
        pos[mu][lo] = -rng.uniform(0.01, 0.9, lo.size).astype(np.float32)  # drifted below 0
    J, st = _deposit(pcg, grid, 1, pos, vel, q, tile=8, halo=halo, key_pos=kp)
    Jr, ninv = oracle.deposit_current(grid, 1, pos, vel, q)
    assert ninv > 200
    assert_deposit_close(J, Jr)
    assert st["n_invalid"] == ninv


def test_tail_pass_deposits_particles_that_were_invalid_at_sort_time():
    # keys from positions that were out of the domain at sort time, deposit
    # positions inside: those slots form the tail and go through the flat path
    pcg = need_gpu()
    grid = (16, 16, 16)
    rng = np.random.default_rng(12)
    pos, vel, q = _random(rng, grid, 10000)
    kp = [p.copy() for p in pos]
    kp[0][:123] = -1.0
    J, st = _deposit(pcg, grid, 2, pos, vel, q, tile=4, halo=2, key_pos=kp)
    Jr, _ = oracle.deposit_current(grid, 2, pos, vel, q)
    assert_deposit_close(J, Jr)
    assert st["n_invalid"] == 0


@pytest.mark.parametrize("block", [128, 256, 512])
def test_block_sizes(block):
    pcg = need_gpu()
    grid = (48, 40, 16)
    rng = np.random.default_rng(block)
    pos, vel, q = _random(rng, grid, 50000)
    J, _ = _deposit(pcg, grid, 2, pos, vel, q, tile=8, halo=2, block=block)
    Jr, _ = oracle.deposit_current(grid, 2, pos, vel, q)
    assert_deposit_close(J, Jr)


def test_empty_and_tiny_grids():
    pcg = need_gpu()
    for grid, tile in (((8, 8, 8), 8), ((3, 2), 4), ((2, 2, 3), 4), ((1, 5), 4)):
        rng = np.random.default_rng(sum(grid))
        pos, vel, q = _random(rng, grid, 300)
        for order in (1, 2):
            J, _ = _deposit(pcg, grid, order, pos, vel, q, tile=tile, halo=2)
            Jr, _ = oracle.deposit_current(grid, order, pos, vel, q)
            assert_deposit_close(J, Jr, where=f"{grid}")
    z = np.zeros(0, np.float32)
    J, st = _deposit(pcg, (8, 8, 8), 1, [z] * 3, [z] * 3, z, tile=8)
    assert np.all(J == 0)


def test_workload_recipes_small():
    # the three current-deposit workloads at reduced sizes, same recipes
    pcg = need_gpu()
    for d in (synth.cic2d(grid=(64, 64)), synth.cic3d_drift(grid=(32, 32, 32)),
              synth.quad3d_bump(grid=(48, 48, 48), sigma_bump=4.0)):
        J, st = _deposit(pcg, d["grid"], d["order"], d["pos"], d["vel"], d["q"], tile=d["tile"],
                         halo=d["halo"], key_pos=d["key_pos"])
        Jr, _ = oracle.deposit_current(d["grid"], d["order"], d["pos"], d["vel"], d["q"])
        assert_deposit_close(J, Jr, where=str(d["grid"]))
        assert st["n_invalid"] == 0
