"""The zigzag current regrouped as the GPU kernel regroups it, against the oracle.

The tiled zigzag kernel does not add each segment's 12 edge values as it meets
them: every cell keeps four sums per component over the segments that lie in it,
  S0 = sum F^c, Su = sum F^c m^u, Sv = sum F^c m^v,
  Q  = sum F^c (m^u m^v + D^u D^v / 12),
(m the segment's midpoint relative to its cell, D its move, F = q D / dt, u and v
the two axes after c), and turns them into the cell's c-edges at
cell + a e_u + b e_v once: S0 - Su - Sv + Q, Su - Q, Sv - Q, Q.  A particle that
stays in its cell is one straight segment; one that crosses a face is its two
relay segments ("Tiled current deposit" (Entity wiki), "Halo sizing": the O == 0
zigzag deposit).  This test rebuilds J that way in fp64 and compares it with the
oracle, which adds every segment's edge weights directly."""
import numpy as np
import pytest

import oracle
import synth


def _relay(x1, x2, N):
    """Per axis: lower cell of the move, the two segments' cells (0 or 1 above
    it), moves and midpoints (relative to their cells)."""
    i1, i2 = np.floor(x1).astype(np.int64), np.floor(x2).astype(np.int64)
    di = i2 - i1
    di = np.where(2 * di > N, di - N, di)
    di = np.where(2 * di < -N, di + N, di)
    assert np.all(np.abs(di) <= 1)
    lo = np.minimum(di, 0)
    a, b = -lo, di - lo
    X1, X2 = a + (x1 - i1), b + (x2 - i2)
    xr = np.minimum(1.0, np.maximum(np.maximum(a, b).astype(np.float64), 0.5 * (X1 + X2)))
    return i1 + lo, (a, b), (xr - X1, X2 - xr), (0.5 * (X1 + xr) - a, 0.5 * (xr + X2) - b)


def _add_cells(J, grid, cell, m, D, qdt):
    """Four sums per cell and component, then the cell's 12 edges."""
    N = np.array(grid)
    F = qdt[:, None] * D
    for c in range(3):
        u, v = (c + 1) % 3, (c + 2) % 3
        S0 = F[:, c]
        Su, Sv = F[:, c] * m[:, u], F[:, c] * m[:, v]
        Q = F[:, c] * (m[:, u] * m[:, v] + D[:, u] * D[:, v] / 12.0)
        for (a, b), val in {(0, 0): S0 - Su - Sv + Q, (1, 0): Su - Q, (0, 1): Sv - Q, (1, 1): Q}.items():
            node = cell.copy()
            node[:, u] += a
            node[:, v] += b
            node %= N
            np.add.at(J[c], (node[:, 2], node[:, 1], node[:, 0]), val)


def _cell_sums_current(grid, prev, pos, q, dt):
    x1 = np.stack([p.astype(np.float64) for p in prev], 1)
    x2 = np.stack([p.astype(np.float64) for p in pos], 1)
    qdt = q.astype(np.float64) / dt
    J = np.zeros((3,) + tuple(reversed(grid)))
    same = np.all(np.floor(x1) == np.floor(x2), axis=1)
    # particles that stay in their cell: one straight segment
    cell = np.floor(x1[same]).astype(np.int64)
    f1, f2 = x1[same] - cell, x2[same] - cell
    _add_cells(J, grid, cell, 0.5 * (f1 + f2), f2 - f1, qdt[same])
    # the others: their two relay segments
    sp = [_relay(x1[~same, mu], x2[~same, mu], grid[mu]) for mu in range(3)]
    for s in range(2):
        cell = np.stack([sp[mu][0] + sp[mu][1][s] for mu in range(3)], 1)
        D = np.stack([sp[mu][2][s] for mu in range(3)], 1)
        m = np.stack([sp[mu][3][s] for mu in range(3)], 1)
        _add_cells(J, grid, cell, m, D, qdt[~same])
    return J


@pytest.mark.parametrize("grid,ppc,sigma_v", [((16, 16, 16), 4, 0.4), ((3, 4, 5), 8, 0.4), ((9, 8, 17), 2, 0.3),
                                              ((12, 10, 8), 4, 0.05)])
def test_zigzag_cell_sums_equal_the_oracle(grid, ppc, sigma_v):
    d = synth.zigzag3d(grid=grid, ppc=ppc, sigma_v=sigma_v, seed=sum(grid) + ppc)
    Jr, ninv = oracle.deposit_zigzag(d["grid"], d["pos_prev"], d["pos"], d["q"], d["dt"])
    assert ninv == 0
    J = _cell_sums_current(d["grid"], d["pos_prev"], d["pos"], d["q"], d["dt"])
    assert np.abs(J - Jr).max() <= 1e-12 * np.abs(Jr).max()
