"""GPU tile counting sort: tile_offsets bit-exact against the oracle, the output a
permutation of the input grouped by tile (order inside a tile is free)."""
import numpy as np
import pytest

import oracle
from helpers import dev, host, need_gpu, stats_dict

pytestmark = pytest.mark.gpu


def _particles(rng, grid, n, invalid=0):
    pos = [rng.uniform(0, N, n).astype(np.float32) for N in grid]
    if invalid:
        idx = rng.choice(n, invalid, replace=False)
        bad = np.array([np.nan, -0.5, np.float32(grid[0]), 1e9], np.float32)
        pos[0][idx] = bad[np.arange(invalid) % 4]
    return pos


def _check_sort(pcg, grid, tile, pos, extra_payload=True):
    n = pos[0].size
    ids = np.arange(n, dtype=np.int32)
    payload = [dev(p) for p in pos] + [dev(ids)]
    stats = pcg.new_stats()
    out, offs = pcg.tile_sort(grid, tile, [dev(p) for p in pos], payload, stats=stats)
    offs = host(offs).astype(np.uint32)
    keys, want_offs = oracle.tile_keys(grid, tile, pos)
    assert np.array_equal(offs, want_offs)
    oid = host(out[-1]).astype(np.int64)
    assert np.array_equal(np.sort(oid), ids)                      # a permutation
    for k, p in enumerate(pos):                                    # payload rows travel together
        assert np.array_equal(host(out[k]).view(np.uint32), p[oid].view(np.uint32))
    nt = len(want_offs) - 1
    slot_tile = np.searchsorted(want_offs, np.arange(n), side="right") - 1
    slot_tile[np.arange(n) >= want_offs[-1]] = nt                  # sentinel tail
    assert np.array_equal(keys[oid], slot_tile.astype(np.uint32))  # every slot holds its tile
    assert stats_dict(stats)["n_invalid"] == int((keys == nt).sum())
    return out, offs


@pytest.mark.parametrize("grid,tile,n", [((64, 64), 8, 50000), ((20, 13), 8, 3001), ((16, 16, 16), 4, 70001),
                                         ((37, 29, 21), 8, 90001), ((12, 10, 9), 8, 5), ((8, 8), 8, 1)])
def test_sort_chunked_path(grid, tile, n):
    pcg = need_gpu()
    rng = np.random.default_rng(n)
    _check_sort(pcg, grid, tile, _particles(rng, grid, n))


@pytest.mark.parametrize("grid,tile,n", [((64, 64, 64), 1, 200000), ((40, 36, 33), 1, 100003),
                                         ((300, 300), 1, 50000)])
def test_sort_global_path(grid, tile, n):
    # more than 32769 bins: global-memory counters
    pcg = need_gpu()
    rng = np.random.default_rng(n + 1)
    _check_sort(pcg, grid, tile, _particles(rng, grid, n))


@pytest.mark.parametrize("grid,tile", [((64, 64, 64), 8), ((128, 128, 128), 4), ((64, 64, 64), 1),
                                       ((700, 700), 8)])
def test_sort_partition_passes(grid, tile):
    # outputs larger than L2 (9 M particles x 3-4 fields here): one partition
    # pass for <= 2048 bins, else two passes (coarse buckets, then tiles)
    pcg = need_gpu()
    rng = np.random.default_rng(sum(grid) + tile)
    _check_sort(pcg, grid, tile, _particles(rng, grid, 9_000_001, invalid=1001))


@pytest.mark.parametrize("grid,tile", [((32, 32, 32), 8), ((50, 50, 50), 1)])
def test_sort_invalid_particles_go_to_the_tail(grid, tile):
    pcg = need_gpu()
    rng = np.random.default_rng(3)
    _check_sort(pcg, grid, tile, _particles(rng, grid, 20000, invalid=37))


def test_sort_empty():
    pcg = need_gpu()
    grid = (16, 16, 16)
    z = np.zeros(0, np.float32)
    out, offs = pcg.tile_sort(grid, 8, [dev(z)] * 3, [dev(z)])
    assert np.all(host(offs) == 0) and host(offs).size == 9


def test_sort_skewed_density():
    # every particle in one tile plus a few elsewhere: one bin takes almost all
    pcg = need_gpu()
    rng = np.random.default_rng(9)
    n = 100000
    pos = [rng.uniform(0, 8, n).astype(np.float32) for _ in range(3)]
    pos[0][:10] = rng.uniform(8, 64, 10).astype(np.float32)
    _check_sort(pcg, (64, 64, 64), 8, pos)


@pytest.mark.parametrize("grid,tile", [((128, 128, 128), 4), ((64, 64, 64), 8)])
def test_sort_partition_skewed(grid, tile):
    # partition sizes with 90% of the particles in one tile: the bucket (and,
    # in one pass, the tile) that holds them spans many chunks of the count
    pcg = need_gpu()
    rng = np.random.default_rng(11)
    n = 9_000_003
    pos = _particles(rng, grid, n, invalid=17)
    hot = rng.random(n) < 0.9
    for mu in range(3):
        pos[mu][hot] = rng.uniform(tile, 2 * tile, int(hot.sum())).astype(np.float32)
    _check_sort(pcg, grid, tile, pos)

