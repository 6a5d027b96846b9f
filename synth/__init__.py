"""Seeded synthetic inputs for the deposit workloads.

This module holds no deposit, shape-function or mass-matrix arithmetic: it only
draws particles (positions, velocities, charges, weights, magnetisation
vectors) with numpy's PCG64 generator.  Both the CUDA path and the CPU oracle
consume its arrays; neither is imported here.

Each generator takes the workload's sizes as arguments, so the tests can draw
small cases with the same recipe as the full-size workloads:

  cic1d          N particles on [0,1), x0 ~ U[0,1), v ~ N(0, 0.1^2),
                 target ~ U[0,1) per bin.                     (seed 1001)
  cic2d          2D periodic grid, exactly ppc particles per cell placed
                 uniformly inside it, globally shuffled; v ~ N(0, 0.1^2) per
                 component, redrawn until |v| < 1; q = +1 / -1 half and half.
                                                               (seed 1002)
  cic3d_drift    3D periodic grid, exactly ppc per cell, shuffled; sort-time
                 positions x_s; v ~ N(0, 0.05^2); deposit-time positions
                 x = wrap(x_s + v * 1.0); a 0.1 % subset is displaced by a
                 further U[-3, 3] cells per axis.              (seed 1003)
  quad3d_bump    3D periodic grid, per-cell count floor(rho(centre) + u) with
                 rho = rho0 + rho1 exp(-r^2 / (2 * 16^2)), r the periodic
                 distance to the box centre, rho0 + rho1 = 10 x mean;
                 v ~ N(0, 0.1^2).                               (seed 1004)
  zigzag3d       3D periodic grid, exactly ppc per cell at the previous
                 positions, shuffled; v ~ N(0, 0.05^2) clipped to |v dt| <= 0.95;
                 pos = wrap(pos_prev + v dt); optionally a subset moved by whole
                 tiles so that stale sort keys leave them outside their tile.
                                                               (seed 1006)
  mass3d         3D periodic grid, exactly ppc per cell, shuffled;
                 w ~ U[0.5, 1.5]; b a random unit vector, beta ~ U(0, 1),
                 omega = beta b.                                (seed 1005)

Positions are fp32 in cell units and always satisfy 0 <= x < N.
"""
from __future__ import annotations

import numpy as np

F32 = np.float32


def _rng(seed):
    return np.random.Generator(np.random.PCG64(seed))


def to_cell_f32(x64, N):
    """Round fp64 positions to fp32 and keep them inside [0, N) after rounding."""
    x = np.asarray(x64, dtype=np.float64) % float(N)
    x32 = x.astype(F32)
    hi = np.nextafter(F32(N), F32(0))
    np.minimum(x32, hi, out=x32)
    x32[x32 < 0] = 0
    return x32


def _inside_cell_f32(cell, u64):
    """fp32 position cell + u with u in [0,1), never rounded up into the next cell."""
    x32 = (cell.astype(np.float64) + u64).astype(F32)
    top = np.nextafter((cell + 1).astype(F32), F32(0))
    np.minimum(x32, top, out=x32)
    return x32


def _halves(n):
    """Charges: +1 on even indices, -1 on odd ones (the order is already random)."""
    q = np.ones(n, dtype=F32)
    q[1::2] = -1
    return q


def _cells_uniform(rng, grid, ppc):
    """Cell coordinates for exactly ppc particles per cell, in shuffled order."""
    ncell = int(np.prod(grid))
    n = ncell * ppc
    cell = rng.permutation(n) // ppc
    coords = []
    rem = cell
    for N in grid:
        coords.append(rem % N)
        rem = rem // N
    return n, coords


def cic1d(n=2000, nbins=1024, nsteps=50, dt=0.01, halfwidth=0.005, sigma_v=0.1, seed=1001):
    rng = _rng(seed)
    x0 = rng.random(n, dtype=np.float64).astype(F32)
    x0[x0 >= 1] = np.nextafter(F32(1), F32(0))
    v = (rng.standard_normal(n) * sigma_v).astype(F32)
    target = rng.random(nbins, dtype=np.float64).astype(F32)
    return dict(x0=x0, v=v, target=target, nbins=nbins, nsteps=nsteps, dt=dt,
                halfwidth=halfwidth, n=n)


def _maxwellian(rng, n, sigma, vmax=None):
    v = rng.standard_normal((3, n)) * sigma
    if vmax is not None:
        bad = np.sqrt((v * v).sum(0)) >= vmax
        while bad.any():
            v[:, bad] = rng.standard_normal((3, int(bad.sum()))) * sigma
            bad = np.sqrt((v * v).sum(0)) >= vmax
    return [v[c].astype(F32) for c in range(3)]


def cic2d(grid=(512, 512), ppc=8, sigma_v=0.1, seed=1002, tile=8, halo=1):
    rng = _rng(seed)
    n, coords = _cells_uniform(rng, grid, ppc)
    pos = [_inside_cell_f32(c, rng.random(n)) for c in coords]
    vel = _maxwellian(rng, n, sigma_v, vmax=1.0)
    return dict(grid=tuple(grid), order=1, tile=tile, halo=halo, n=n,
                key_pos=pos, pos=pos, vel=vel, q=_halves(n))


def cic3d_drift(grid=(256, 256, 256), ppc=16, sigma_v=0.05, dt=1.0, displaced_frac=0.001,
                max_disp=3.0, seed=1003, tile=8, halo=2):
    rng = _rng(seed)
    n, coords = _cells_uniform(rng, grid, ppc)
    xs = [_inside_cell_f32(c, rng.random(n)) for c in coords]
    del coords
    vel = _maxwellian(rng, n, sigma_v)
    k = int(round(displaced_frac * n))
    idx = rng.choice(n, size=k, replace=False) if k > 0 else np.zeros(0, dtype=np.int64)
    pos = []
    for mu, N in enumerate(grid):
        x64 = xs[mu].astype(np.float64) + vel[mu].astype(np.float64) * dt
        if k:
            x64[idx] += rng.uniform(-max_disp, max_disp, size=k)
        pos.append(to_cell_f32(x64, N))
        del x64
    return dict(grid=tuple(grid), order=1, tile=tile, halo=halo, n=n,
                key_pos=xs, pos=pos, vel=vel, q=_halves(n), displaced=idx)


def zigzag3d(grid=(256, 256, 256), ppc=16, sigma_v=0.05, dt=1.0, vmax=0.95, escaped_frac=0.0, seed=1006,
             tile=8):
    """Moves pos_prev -> pos for the charge-conserving deposit: exactly ppc
    particles per cell at pos_prev (the sort-time positions), v ~ N(0, sigma^2)
    per component clipped to |v| dt <= vmax (< 1 cell: the scheme's CFL limit),
    pos = wrap(pos_prev + v dt).  escaped_frac of the particles are first moved
    by a further whole number of tiles (1..3 per axis) in both pos_prev and pos,
    so that they sit far outside the tile they are sorted under only when the
    caller sorts with stale keys (key_pos_stale)."""
    rng = _rng(seed)
    n, coords = _cells_uniform(rng, grid, ppc)
    prev = [_inside_cell_f32(c, rng.random(n)) for c in coords]
    del coords
    vel = _maxwellian(rng, n, sigma_v)
    pos = []
    for mu, N in enumerate(grid):
        d = np.clip(vel[mu].astype(np.float64) * dt, -vmax, vmax)
        pos.append(to_cell_f32(prev[mu].astype(np.float64) + d, N))
    k = int(round(escaped_frac * n))
    stale = prev
    if k:
        idx = rng.choice(n, size=k, replace=False)
        stale = [a.copy() for a in prev]
        for mu, N in enumerate(grid):
            shift = rng.integers(1, 4, size=k) * tile * rng.choice([-1, 1], size=k)
            prev[mu][idx] = to_cell_f32(prev[mu][idx].astype(np.float64) + shift, N)
            pos[mu][idx] = to_cell_f32(pos[mu][idx].astype(np.float64) + shift, N)
    return dict(grid=tuple(grid), tile=tile, n=n, dt=dt, pos_prev=prev, pos=pos, q=_halves(n),
                key_pos=prev, key_pos_stale=stale)


def bump_density(grid, mean=32.0, peak=320.0, sigma=16.0):
    """rho at cell centres: rho0 + rho1 exp(-r^2/(2 sigma^2)), periodic r to the centre.

    rho1 is chosen so that the average over all cells is `mean` and the peak is
    rho0 + rho1 = `peak`.
    """
    axes = []
    for N in grid:
        c = np.arange(N, dtype=np.float64) + 0.5
        d = c - N / 2.0
        d = d - N * np.round(d / N)
        axes.append(np.exp(-d * d / (2 * sigma * sigma)))
    g = axes[0][None, None, :] * axes[1][None, :, None] * axes[2][:, None, None]
    gbar = g.mean()
    rho1 = (peak - mean) / (1.0 - gbar)
    rho0 = peak - rho1
    return rho0 + rho1 * g  # shape (Nz, Ny, Nx)


def quad3d_bump(grid=(192, 192, 192), mean=32.0, peak=320.0, sigma_bump=16.0, sigma_v=0.1,
                seed=1004, tile=8, halo=2):
    rng = _rng(seed)
    rho = bump_density(grid, mean, peak, sigma_bump).ravel()
    counts = np.floor(rho + rng.random(rho.size)).astype(np.int64)
    n = int(counts.sum())
    cell = np.repeat(np.arange(rho.size, dtype=np.int64), counts)
    cell = cell[rng.permutation(n)]
    coords = []
    rem = cell
    for N in grid:
        coords.append(rem % N)
        rem = rem // N
    del cell, rem
    pos = [_inside_cell_f32(c, rng.random(n)) for c in coords]
    del coords
    vel = _maxwellian(rng, n, sigma_v)
    return dict(grid=tuple(grid), order=2, tile=tile, halo=halo, n=n,
                key_pos=pos, pos=pos, vel=vel, q=_halves(n), counts=counts)


def mass3d(grid=(64, 64, 64), ppc=64, seed=1005):
    rng = _rng(seed)
    n, coords = _cells_uniform(rng, grid, ppc)
    pos = [_inside_cell_f32(c, rng.random(n)) for c in coords]
    del coords
    w = rng.uniform(0.5, 1.5, size=n).astype(F32)
    b = rng.standard_normal((3, n))
    b /= np.sqrt((b * b).sum(0))
    beta = rng.random(n)
    omega = [(beta * b[c]).astype(F32) for c in range(3)]
    return dict(grid=tuple(grid), n=n, pos=pos, w=w, omega=omega)


WORKLOADS = {
    "cic1d": cic1d,
    "cic2d": cic2d,
    "cic3d_drift": cic3d_drift,
    "quad3d_bump": quad3d_bump,
    "mass3d": mass3d,
}
