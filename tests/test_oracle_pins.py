"""Pins of the fp64 CPU oracle to things other than itself.

Each test checks the oracle against a brute-force formulation written
differently (all-node sums with B-splines built from box convolutions, a dense
W S W^T product, numpy bincount), a hand-worked fixture under tests/golden, a
closed form, or an invariant of the method.  A dropped term, a wrong sign or a
transposed index in the oracle fails at least one of them.
"""
from fractions import Fraction

import numpy as np
import pytest

import oracle
import synth
from conftest import read_golden

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")


# ---------------------------------------------------------------------------
# B-splines built from their definition: repeated convolution with the unit box
# (Pennati & Markidis, Sec. 2.3, Eq. (12)).  phi_n(s) = int_{s-1/2}^{s+1/2} phi_{n-1}.
# The antiderivative of the previous order is evaluated in closed form, so none
# of the oracle's piecewise formulas or node-selection logic is reused here.
# ---------------------------------------------------------------------------
def _box_cdf(t):
    return np.clip(t + 0.5, 0.0, 1.0)


def _tent(s):  # order 1 = box * box
    return _box_cdf(s + 0.5) - _box_cdf(s - 0.5)


def _tent_cdf(t):  # integral of the tent from -inf to t
    t = np.asarray(t, dtype=np.float64)
    return np.where(t < -1, 0.0,
           np.where(t < 0, 0.5 * (t + 1) ** 2,
           np.where(t < 1, 1.0 - 0.5 * (1 - t) ** 2, 1.0)))


def _quad(s):  # order 2 = tent * box
    return _tent_cdf(s + 0.5) - _tent_cdf(s - 0.5)


def _phi(order, s):
    return _tent(s) if order == 1 else _quad(s)


def _minimg(s, N):
    return s - N * np.round(s / N)


def test_bspline_from_convolution_matches_numeric_integral():
    # the convolution construction itself, against a midpoint Riemann sum
    s = np.linspace(-2, 2, 41)
    h = 1e-4
    t = np.arange(-3, 3, h) + h / 2
    tent_num = np.array([np.sum((np.abs(t) <= 0.5) & (np.abs(x - t) <= 0.5)) * h for x in s])
    assert np.allclose(tent_num, _tent(s), atol=2e-4)
    quad_num = np.array([np.sum(_tent(t) * (np.abs(x - t) <= 0.5)) * h for x in s])
    assert np.allclose(quad_num, _quad(s), atol=2e-4)


@pytest.mark.parametrize("row", read_golden("bspline_weights.txt"))
def test_axis_support_golden(row):
    order, x, first = int(row[0]), float(row[1]), int(row[2])
    want = [float(Fraction(w)) for w in row[3:]]
    got_first, got_w = oracle.axis_support(order, x)
    assert got_first == first
    assert np.allclose(got_w, want, rtol=0, atol=1e-15)


def test_axis_support_against_convolution_spline():
    rng = np.random.default_rng(7)
    for order in (1, 2):
        for x in list(rng.uniform(0, 50, 200)) + [0.0, 0.5, 1.0, 7.5, 7.25]:
            first, w = oracle.axis_support(order, x)
            nodes = first + np.arange(len(w))
            assert np.allclose(w, _phi(order, x - nodes), atol=1e-14)
            # the support holds every node with a non-zero weight
            around = np.arange(int(np.floor(x)) - 3, int(np.floor(x)) + 4)
            outside = np.setdiff1d(around, nodes)
            assert np.allclose(_phi(order, x - outside), 0.0, atol=1e-14)


# ---------------------------------------------------------------------------
# current deposit: brute force over every node of small periodic grids
# ---------------------------------------------------------------------------
def _brute_J(grid, order, pos, vel, q):
    dim = len(grid)
    shape = tuple(reversed(grid))
    J = np.zeros((3,) + shape)
    axes = np.meshgrid(*[np.arange(N) for N in reversed(grid)], indexing="ij")  # z,y,x order
    node = list(reversed(axes))  # node[mu] has coordinate mu
    for p in range(len(q)):
        x = [float(pos[mu][p]) for mu in range(dim)]
        if not all(0 <= x[mu] < grid[mu] for mu in range(dim)):
            continue
        W = np.ones(shape)
        for mu in range(dim):
            W = W * _phi(order, _minimg(x[mu] - node[mu], grid[mu]))
        for c in range(3):
            J[c] += float(q[p]) * float(vel[c][p]) * W
    return J


def _small_particles(rng, grid, n):
    pos = [rng.uniform(0, N, n).astype(np.float32) for N in grid]
    # special positions: on nodes, on half-cells, next to the upper edge, at 0
    for mu, N in enumerate(grid):
        pos[mu][0] = 0.0
        pos[mu][1] = np.float32(N) - np.float32(2 ** -20)
        pos[mu][2] = 1.5
        pos[mu][3] = 2.0
    vel = [rng.normal(0, 0.3, n).astype(np.float32) for _ in range(3)]
    q = rng.choice([-1.0, 1.0, 0.5], n).astype(np.float32)
    return pos, vel, q


@pytest.mark.parametrize("grid", [(5, 4), (3, 7), (4, 5, 3), (6, 3, 4)])
@pytest.mark.parametrize("order", [1, 2])
def test_deposit_bruteforce_all_nodes(grid, order):
    rng = np.random.default_rng(hash((grid, order)) % 2 ** 32)
    pos, vel, q = _small_particles(rng, grid, 24)
    J, ninv = oracle.deposit_current(grid, order, pos, vel, q)
    assert ninv == 0
    Jb = _brute_J(grid, order, pos, vel, q)
    scale = np.abs(Jb).max()
    assert np.abs(J - Jb).max() <= 1e-12 * scale


@pytest.mark.parametrize("order", [1, 2])
def test_deposit_partition_of_unity_and_moments(order):
    grid = (9, 8, 7)
    rng = np.random.default_rng(11)
    n = 500
    pos = [rng.uniform(0, N, n).astype(np.float32) for N in grid]
    vel = [rng.normal(0, 0.2, n).astype(np.float32) for _ in range(3)]
    q = rng.choice([-1.0, 1.0], n).astype(np.float32)
    J, _ = oracle.deposit_current(grid, order, pos, vel, q)
    for c in range(3):
        want = np.sum(q.astype(np.float64) * vel[c].astype(np.float64))
        assert abs(J[c].sum() - want) <= 1e-11 * max(1.0, np.abs(q * vel[c]).sum())
    # single particle: first moment zero, second moment = variance of the spline
    for x in [(3.3, 4.71, 2.05), (0.2, 7.9, 6.5), (4.0, 4.0, 4.0)]:
        J1, _ = oracle.deposit_current(grid, order, [np.array([v], np.float32) for v in x],
                                       [np.array([1.0], np.float32), np.zeros(1, np.float32), np.zeros(1, np.float32)],
                                       np.ones(1, np.float32))
        W = J1[0]  # (z, y, x)
        xs = [float(np.float32(v)) for v in x]
        for mu, N in enumerate(grid):
            axis = 2 - mu
            marg = W.sum(axis=tuple(a for a in range(3) if a != axis))
            d = _minimg(np.arange(N) - xs[mu], N)
            assert abs((marg * d).sum()) < 1e-12
            if order == 2:
                assert abs((marg * d * d).sum() - 0.25) < 1e-12
            else:
                xi = xs[mu] - np.floor(xs[mu])
                assert abs((marg * d * d).sum() - xi * (1 - xi)) < 1e-12


def test_deposit_node_closed_forms():
    grid = (6, 6, 6)
    one = np.ones(1, np.float32)
    z = np.zeros(1, np.float32)
    # CIC on a node: all weight on that node
    J, _ = oracle.deposit_current(grid, 1, [np.array([2.0], np.float32)] * 3, [one, z, z], one)
    assert J[0][2, 2, 2] == 1.0 and np.count_nonzero(J[0]) == 1
    # quadratic on a node: 1/8, 3/4, 1/8 per axis
    J, _ = oracle.deposit_current(grid, 2, [np.array([2.0], np.float32)] * 3, [one, z, z], one)
    w = np.array([1 / 8, 3 / 4, 1 / 8])
    assert np.allclose(J[0][1:4, 1:4, 1:4], np.einsum("i,j,k->ijk", w, w, w), atol=1e-15)
    assert np.count_nonzero(J[0]) == 27


def test_deposit_invalid_particles_skipped_and_counted():
    grid = (4, 4)
    pos = [np.array([1.5, 4.0, -0.25, np.nan, 2.5], np.float32),
           np.array([1.5, 1.0, 1.0, 1.0, 3.99], np.float32)]
    vel = [np.ones(5, np.float32)] * 3
    q = np.ones(5, np.float32)
    J, ninv = oracle.deposit_current(grid, 1, pos, vel, q)
    assert ninv == 3
    Jv, _ = oracle.deposit_current(grid, 1, [p[[0, 4]] for p in pos], [v[[0, 4]] for v in vel], q[[0, 4]])
    assert np.array_equal(J, Jv)


# ---------------------------------------------------------------------------
# 1D windowed CIC histogram
# ---------------------------------------------------------------------------
def _golden_cic1d():
    rows = {r[0]: r[1:] for r in read_golden("cic1d_worked.txt")}
    f = lambda k: [float(v) for v in rows[k]]
    return rows, f


def test_cic1d_worked_example():
    rows, f = _golden_cic1d()
    H, loss, nsel = oracle.cic1d(np.array(f("x0"), np.float32), np.array(f("v"), np.float32),
                                 np.array(f("target"), np.float32), nbins=int(rows["nbins"][0]),
                                 nsteps=int(rows["nsteps"][0]), dt=f("dt")[0], halfwidth=f("halfwidth")[0])
    want = np.array(f("H_num")) / f("H_den")[0]
    assert np.allclose(H, want, rtol=0, atol=1e-15)
    assert abs(loss - f("loss_num")[0] / f("loss_den")[0]) < 1e-15
    assert nsel == int(rows["n_deposits"][0])


def _tent_hist(x, w, nb):
    """Histogram by the periodic tent at bin centres (b + 1/2)/nb: no floor, no mod."""
    b = (np.arange(nb) + 0.5) / nb
    d = x[:, None] - b[None, :]
    d = d - np.round(d)
    return (w[:, None] * np.maximum(0.0, 1.0 - np.abs(d) * nb)).sum(0)


def test_cic1d_all_selected_matches_tent_bruteforce():
    # a half-width above 1/2 selects every particle at every step (|minimg| <= 1/2)
    rng = np.random.default_rng(3)
    n, nb, T, dt, h = 40, 16, 7, 0.013, 0.8
    x0 = rng.random(n).astype(np.float32)
    v = rng.normal(0, 0.3, n).astype(np.float32)
    target = rng.random(nb).astype(np.float32)
    H, loss, nsel = oracle.cic1d(x0, v, target, nb, T, dt, h)
    assert nsel == n * T
    Hb = np.zeros(nb)
    for t in range(1, T + 1):
        x = np.mod(x0.astype(np.float64) + v.astype(np.float64) * (t * dt), 1.0)
        r = np.mod(x - t / T, 1.0)
        dist = np.minimum(r, 1.0 - r)            # circular distance to the window centre
        Hb += _tent_hist(x, (1.0 - dist / h) ** 2, nb)
    assert np.allclose(H, Hb, rtol=0, atol=1e-12)
    assert abs(loss - np.sum((Hb - target.astype(np.float64)) ** 2)) < 1e-10


def test_cic1d_selection_count_and_mass():
    d = synth.cic1d()
    H, loss, nsel = oracle.cic1d(d["x0"], d["v"], d["target"], d["nbins"], d["nsteps"], d["dt"], d["halfwidth"])
    # independent count of (particle, step) pairs inside the window: circular distance
    x0 = d["x0"].astype(np.float64)
    v = d["v"].astype(np.float64)
    tot_w = 0.0
    cnt = 0
    per_step = []
    ever = np.zeros(x0.size, bool)
    for t in range(1, d["nsteps"] + 1):
        x = np.mod(x0 + v * (t * d["dt"]), 1.0)
        r = np.mod(x - t / d["nsteps"], 1.0)
        dist = np.minimum(r, 1.0 - r)
        sel = dist < d["halfwidth"] * (1 - 1e-9)
        near = np.abs(dist - d["halfwidth"]) < 1e-12
        assert not near.any()  # no pair sits on the window edge for this seed
        cnt += sel.sum()
        per_step.append(sel.sum())
        ever |= sel
        tot_w += ((1 - dist[sel] / d["halfwidth"]) ** 2).sum()
    assert nsel == cnt
    assert abs(H.sum() - tot_w) < 1e-9                # CIC weights sum to one
    assert (H >= 0).all()
    # loose sanity check of the generator against the page's printed statistics
    # (capacity 30 and 983 of 2000 particles ever selected, other inputs): same regime
    assert 15 <= max(per_step) <= 45
    assert 0.35 <= ever.mean() <= 0.65


@pytest.mark.parametrize("seed,nb,T,hw", [(5, 64, 20, 0.05), (6, 256, 50, 0.01), (7, 32, 8, 0.2)])
def test_cic1d_gradient_matches_central_differences(seed, nb, T, hw):
    # the gradient against central differences of the (separately pinned) loss;
    # a step of 2^-20 is exact in fp32 for x0 in [0.5, 1)
    rng = np.random.default_rng(seed)
    n, dt = 48, 0.01
    x0 = (0.5 + 0.5 * rng.random(n)).astype(np.float32)
    v = rng.normal(0, 0.1, n).astype(np.float32)
    target = rng.random(nb).astype(np.float32)
    g, H, loss, nsel = oracle.cic1d_grad(x0, v, target, nb, T, dt, hw)
    H1, loss1, nsel1 = oracle.cic1d(x0, v, target, nb, T, dt, hw)
    assert nsel == nsel1 and loss == loss1 and np.array_equal(H, H1)
    eps = np.float32(2.0 ** -20)
    fd = np.zeros(n)
    for i in range(n):
        xp, xm = x0.copy(), x0.copy()
        xp[i] += eps
        xm[i] -= eps
        fd[i] = (oracle.cic1d(xp, v, target, nb, T, dt, hw)[1] -
                 oracle.cic1d(xm, v, target, nb, T, dt, hw)[1]) / (float(xp[i]) - float(xm[i]))
    assert nsel > 0
    # a particle within one step of a bin boundary sits on a kink of the loss
    # (the CIC weight derivatives switch bins there) and the central difference
    # averages the two sides; a wrong term would spoil nearly every particle
    ok = np.abs(fd - g) <= 1e-6 * max(np.abs(g).max(), 1.0)
    assert ok.mean() >= 0.95


def test_cic1d_gradient_zero_for_unselected_and_linear_in_residual():
    d = synth.cic1d()
    args = (d["nbins"], d["nsteps"], d["dt"], d["halfwidth"])
    g, H, loss, nsel = oracle.cic1d_grad(d["x0"], d["v"], d["target"], *args)
    # particles never inside the window have an exactly zero gradient
    x0 = d["x0"].astype(np.float64)
    v = d["v"].astype(np.float64)
    ever = np.zeros(x0.size, bool)
    for t in range(1, d["nsteps"] + 1):
        r = np.mod(np.mod(x0 + v * (t * d["dt"]), 1.0) - t / d["nsteps"], 1.0)
        ever |= np.minimum(r, 1.0 - r) < d["halfwidth"]
    assert (g[~ever] == 0).all() and (g[ever] != 0).sum() > 0.9 * ever.sum()
    # dL/dx0 = sum_b 2 (H_b - target_b) dH_b/dx0 is affine in the target: the
    # gradients at targets t_a and t_b average to the gradient at (t_a + t_b)/2
    # (dyadic targets, so that the midpoint is exact in fp32)
    rng = np.random.default_rng(1)
    ta = (rng.integers(0, 1024, d["nbins"]) / 1024.0).astype(np.float32)
    tb = (rng.integers(0, 1024, d["nbins"]) / 1024.0).astype(np.float32)
    tm = ((ta.astype(np.float64) + tb) / 2).astype(np.float32)
    assert np.array_equal(tm.astype(np.float64), (ta.astype(np.float64) + tb) / 2)
    ga = oracle.cic1d_grad(d["x0"], d["v"], ta, *args)[0]
    gb = oracle.cic1d_grad(d["x0"], d["v"], tb, *args)[0]
    gm = oracle.cic1d_grad(d["x0"], d["v"], tm, *args)[0]
    assert np.abs((ga + gb) / 2 - gm).max() <= 1e-9 * np.abs(ga).max()


# ---------------------------------------------------------------------------
# mass matrix: dense W S W^T on tiny grids, alpha closed forms and invariants
# ---------------------------------------------------------------------------
def _cross_matrix(w):
    return np.array([[0, -w[2], w[1]], [w[2], 0, -w[0]], [-w[1], w[0], 0]], dtype=np.float64)


@pytest.mark.parametrize("row", read_golden("alpha_closed_form.txt"))
def test_alpha_closed_form(row):
    vals = [float(v) for v in row]
    a = oracle.alpha(vals[:3])
    assert np.allclose(a, np.array(vals[3:]).reshape(3, 3), atol=1e-15)


def test_alpha_is_inverse_of_one_plus_cross():
    rng = np.random.default_rng(5)
    for _ in range(50):
        w = rng.normal(0, 1.5, 3)
        a = oracle.alpha(w)
        want = np.linalg.solve(np.eye(3) + _cross_matrix(w), np.eye(3))
        assert np.allclose(a, want, atol=1e-13)
        # the cross operator really is w x u
        u = rng.normal(size=3)
        assert np.allclose(_cross_matrix(w) @ u, np.cross(w, u))


def _dense_mass(grid, pos, wq, omega):
    """M^{ij} = W S^{ij} W^T with W the dense node-by-particle weight matrix (Eq. (10))."""
    Nx, Ny, Nz = grid
    ng = Nx * Ny * Nz
    n = len(wq)
    gz, gy, gx = np.meshgrid(np.arange(Nz), np.arange(Ny), np.arange(Nx), indexing="ij")
    W = np.zeros((ng, n))
    for p in range(n):
        Wp = (_tent(_minimg(float(pos[0][p]) - gx, Nx)) * _tent(_minimg(float(pos[1][p]) - gy, Ny))
              * _tent(_minimg(float(pos[2][p]) - gz, Nz)))
        W[:, p] = Wp.ravel()
    S = np.zeros((3, 3, n))
    for p in range(n):
        w = np.array([float(omega[c][p]) for c in range(3)])
        a = np.linalg.solve(np.eye(3) + _cross_matrix(w), np.eye(3))   # Eq. (5) in closed form
        S[:, :, p] = float(wq[p]) * a
    Md = np.einsum("gp,ijp,hp->ijgh", W, S, W)
    return Md  # [i][j][g][g']


def _offset_layout(Md, grid):
    Nx, Ny, Nz = grid
    ng = Nx * Ny * Nz
    out = np.zeros((ng, 27, 3, 3))
    for g in range(ng):
        x, y, z = g % Nx, (g // Nx) % Ny, g // (Nx * Ny)
        for dz in (-1, 0, 1):
            for dy in (-1, 0, 1):
                for dx in (-1, 0, 1):
                    h = (((z + dz) % Nz) * Ny + (y + dy) % Ny) * Nx + (x + dx) % Nx
                    o = (dz + 1) * 9 + (dy + 1) * 3 + (dx + 1)
                    out[g, o] = Md[:, :, g, h]
    return out


@pytest.mark.parametrize("grid", [(3, 4, 5), (4, 3, 3), (5, 5, 4)])
def test_mass_matrix_dense_product(grid):
    rng = np.random.default_rng(sum(grid))
    n = 30
    pos = [rng.uniform(0, N, n).astype(np.float32) for N in grid]
    pos[0][0] = np.float32(grid[0]) - np.float32(1e-5)  # wraps in x
    pos[1][1] = 0.0
    wq = rng.uniform(0.5, 1.5, n).astype(np.float32)
    omega = [rng.normal(0, 0.6, n).astype(np.float32) for _ in range(3)]
    M, ninv = oracle.mass_matrix(grid, pos, wq, omega)
    assert ninv == 0
    want = _offset_layout(_dense_mass(grid, pos, wq, omega), grid)
    got = M.reshape(-1, 27, 3, 3)
    assert np.abs(got - want).max() <= 1e-12 * np.abs(want).max()


@pytest.mark.parametrize("grid", [(3, 4, 5), (5, 3, 4)])
def test_scalar_mass_matrix_dense_product(grid):
    """M = W diag(w) W^T (Eq. (10) with S = diag(w)), built densely."""
    rng = np.random.default_rng(sum(grid) + 100)
    n = 30
    pos = [rng.uniform(0, N, n).astype(np.float32) for N in grid]
    pos[2][0] = np.float32(grid[2]) - np.float32(1e-5)  # wraps in z
    w = rng.uniform(0.5, 1.5, n).astype(np.float32)
    zero = [np.zeros(n, np.float32)] * 3
    M, ninv = oracle.mass_matrix_scalar(grid, pos, w)
    assert ninv == 0
    want = _offset_layout(_dense_mass(grid, pos, w, zero), grid)[:, :, 0, 0]
    assert np.abs(M.reshape(-1, 27) - want).max() <= 1e-12 * np.abs(want).max()
    # and the tensor matrix with omega = 0 (alpha = I) carries it on its diagonal
    Mt, _ = oracle.mass_matrix(grid, pos, w, zero)
    for i in range(3):
        assert np.abs(Mt[..., i, i] - M).max() <= 1e-12 * np.abs(M).max()


def test_scalar_mass_matrix_row_sums_and_symmetry():
    """sum_o M[g][o] = sum_p w W_pg (partition of unity), and M[g][o] = M[g+d][-o]."""
    grid = (6, 5, 4)
    rng = np.random.default_rng(7)
    n = 400
    pos = [rng.uniform(0, N, n).astype(np.float32) for N in grid]
    w = rng.uniform(0.5, 1.5, n).astype(np.float32)
    M, _ = oracle.mass_matrix_scalar(grid, pos, w)
    ones, zeros = np.ones(n, np.float32), np.zeros(n, np.float32)
    rho = oracle.deposit_current(grid, 1, pos, [ones, zeros, zeros], w)[0][0]
    assert np.abs(M.sum(axis=-1) - rho).max() <= 1e-12 * np.abs(rho).max()
    for o in range(27):
        dz, dy, dx = o // 9 - 1, (o // 3) % 3 - 1, o % 3 - 1
        mirrored = np.roll(M[..., 26 - o], shift=(-dz, -dy, -dx), axis=(0, 1, 2))
        assert np.abs(M[..., o] - mirrored).max() <= 1e-12 * np.abs(M).max()


def test_mass_matrix_invariants():
    grid = (6, 5, 4)
    Nx, Ny, Nz = grid
    rng = np.random.default_rng(9)
    n = 400
    pos = [rng.uniform(0, N, n).astype(np.float32) for N in grid]
    wq = rng.uniform(0.5, 1.5, n).astype(np.float32)
    omega = [rng.normal(0, 0.7, n).astype(np.float32) for _ in range(3)]
    M, _ = oracle.mass_matrix(grid, pos, wq, omega)
    M = M.reshape(-1, 27, 3, 3)
    # symmetry per component (Eq. (11)): M[g][delta] = M[g+delta][-delta]
    for g in range(M.shape[0]):
        x, y, z = g % Nx, (g // Nx) % Ny, g // (Nx * Ny)
        for o in range(27):
            dx, dy, dz = o % 3 - 1, (o // 3) % 3 - 1, o // 9 - 1
            h = (((z + dz) % Nz) * Ny + (y + dy) % Ny) * Nx + (x + dx) % Nx
            assert np.allclose(M[g, o], M[h, 26 - o], atol=1e-13)
    # row sums = deposited weight sum_p s_p W_pg; total = sum_p s_p
    s = np.stack([float(wq[p]) * oracle.alpha([float(omega[c][p]) for c in range(3)]) for p in range(n)])
    gz, gy, gx = np.meshgrid(np.arange(Nz), np.arange(Ny), np.arange(Nx), indexing="ij")
    dep = np.zeros((M.shape[0], 3, 3))
    for p in range(n):
        Wp = (_tent(_minimg(float(pos[0][p]) - gx, Nx)) * _tent(_minimg(float(pos[1][p]) - gy, Ny))
              * _tent(_minimg(float(pos[2][p]) - gz, Nz)))
        dep += Wp.ravel()[:, None, None] * s[p][None]
    assert np.allclose(M.sum(axis=1), dep, atol=1e-12)
    assert np.allclose(M.sum(axis=(0, 1)), s.sum(0), atol=1e-10)


def test_mass_matrix_closed_forms():
    grid = (4, 4, 4)
    one = np.ones(1, np.float32)
    zero = np.zeros(1, np.float32)
    # cell-centre particle, omega = 0: every one of the 64 pairs gets w/64 * I
    M, _ = oracle.mass_matrix(grid, [np.array([1.5], np.float32)] * 3, np.array([2.0], np.float32), [zero] * 3)
    M = M.reshape(-1, 27, 3, 3)
    nz = np.argwhere(np.abs(M[..., 0, 0]) > 0)
    assert len(nz) == 64
    for g, o in nz:
        assert np.allclose(M[g, o], 2.0 / 64 * np.eye(3), atol=1e-16)
    # particle on a node with omega = (0, 0, 1/2): one block, w * alpha, at offset 13
    M, _ = oracle.mass_matrix(grid, [np.array([2.0], np.float32)] * 3, one,
                              [zero, zero, np.array([0.5], np.float32)])
    M = M.reshape(-1, 27, 3, 3)
    g = (2 * 4 + 2) * 4 + 2
    assert np.allclose(M[g, 13], [[0.8, 0.4, 0], [-0.4, 0.8, 0], [0, 0, 1]], atol=1e-15)
    assert np.count_nonzero(M) == 5


# ---------------------------------------------------------------------------
# tile keys and tile_offsets
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("grid,tile", [((16, 16), 8), ((20, 13), 8), ((12, 10, 9), 4), ((16, 16, 16), 8), ((7, 5, 6), 1)])
def test_tile_keys_against_bincount(grid, tile):
    rng = np.random.default_rng(len(grid) * 100 + tile)
    n = 3000
    pos = [rng.uniform(0, N, n).astype(np.float32) for N in grid]
    pos[0][:3] = [np.nan, -1.0, float(grid[0])]
    keys, offs = oracle.tile_keys(grid, tile, pos)
    nt = [-(-N // tile) for N in grid]
    tc = [np.floor(np.nan_to_num(p, nan=-1.0)).astype(np.int64) // tile for p in pos]
    ok = np.ones(n, bool)
    for mu, N in enumerate(grid):
        ok &= (pos[mu] >= 0) & (pos[mu] < N)
    k = np.zeros(n, np.int64)
    stride = 1
    for mu in range(len(grid)):
        k += np.where(ok, tc[mu], 0) * stride
        stride *= nt[mu]
    total = stride
    k[~ok] = total
    assert np.array_equal(keys, k.astype(np.uint32))
    counts = np.bincount(k, minlength=total + 1)[:total]
    assert np.array_equal(offs, np.concatenate([[0], np.cumsum(counts)]).astype(np.uint32))
    assert offs[-1] == ok.sum()


# ---------------------------------------------------------------------------
# Charge-conserving zigzag current deposit (the O == 0 deposit named in "Tiled
# current deposit", "Halo sizing"; scheme of Umeda et al. 2003).  Pins: hand-
# worked values, the discrete continuity equation against a CIC charge density
# built here from its definition, the total current, and time reversal.
# ---------------------------------------------------------------------------
def _zigzag_moves(grid, n, seed, dmax=0.95):
    rng = np.random.default_rng(seed)
    x1 = [synth.to_cell_f32(rng.random(n) * N, N) for N in grid]
    x2 = [synth.to_cell_f32(a.astype(np.float64) + rng.uniform(-dmax, dmax, n), N) for a, N in zip(x1, grid)]
    q = rng.choice([-1.0, 1.0, 0.5], n).astype(np.float32)
    return x1, x2, q


def _cic_rho(grid, pos, q):
    """Charge on the nodes: every particle gives q (1 - f) / q f to the two nodes
    around it along each axis (the product over axes), periodic."""
    import itertools
    rho = np.zeros(tuple(reversed(grid)))
    for corner in itertools.product((0, 1), repeat=3):
        w = q.astype(np.float64).copy()
        idx = []
        for mu, N in enumerate(grid):
            x = pos[mu].astype(np.float64)
            i = np.floor(x)
            f = x - i
            w *= f if corner[mu] else 1.0 - f
            idx.append(((i + corner[mu]) % N).astype(np.int64))
        np.add.at(rho, (idx[2], idx[1], idx[0]), w)
    return rho


def _div_backward(J):
    # J[c] on the edge from node g towards +e_c: (div J)_g = sum_c J_c(g) - J_c(g - e_c);
    # array axes are (z, y, x), so component c differences along axis 2 - c
    return sum(J[c] - np.roll(J[c], 1, axis=2 - c) for c in range(3))


def _golden_zigzag():
    rows = read_golden("zigzag_worked.txt")
    grid = tuple(int(v) for v in rows[0][1:])
    dt = float(rows[1][1])
    parts, cur = {}, None
    for r in rows[2:]:
        if r[0] == "particle":
            cur = r[1]
            parts[cur] = ([float(v) for v in r[2:5]], [float(v) for v in r[5:8]], {})
        else:
            c, i, j, k, num = (int(v) for v in r[1:])
            parts[cur][2][(c, k, j, i)] = Fraction(num, 384)
    return grid, dt, parts


@pytest.mark.parametrize("name", ["A", "C", "D", "E"])
def test_zigzag_worked_examples(name):
    grid, dt, parts = _golden_zigzag()
    x1, x2, want = parts[name]
    J, ninv = oracle.deposit_zigzag(grid, [np.array([v], np.float32) for v in x1],
                                    [np.array([v], np.float32) for v in x2], np.ones(1, np.float32), dt)
    assert ninv == 0
    got = {tuple(int(v) for v in ix): float(J[ix]) for ix in zip(*np.nonzero(J))}
    assert set(got) == set(want)
    # thirds (the /12 terms) are not binary fractions: allow the rounding of a few operations
    for k, v in want.items():
        assert abs(got[k] - float(v)) <= 4e-16, (k, got[k], v)


@pytest.mark.parametrize("grid,dt,seed", [((3, 3, 3), 1.0, 1), ((5, 6, 7), 0.5, 2), ((8, 4, 5), 0.3, 3),
                                          ((4, 9, 3), 2.0, 4)])
def test_zigzag_continuity_equation(grid, dt, seed):
    x1, x2, q = _zigzag_moves(grid, 3000, seed)
    J, ninv = oracle.deposit_zigzag(grid, x1, x2, q, dt)
    assert ninv == 0
    res = (_cic_rho(grid, x2, q) - _cic_rho(grid, x1, q)) / dt + _div_backward(J)
    assert np.abs(res).max() <= 1e-11 * max(1.0, np.abs(J).max())
    # and the current is not trivially zero
    assert np.abs(J).max() > 1.0


def test_zigzag_total_current_and_time_reversal():
    grid, dt = (6, 5, 7), 0.25
    x1, x2, q = _zigzag_moves(grid, 2000, 11)
    J, _ = oracle.deposit_zigzag(grid, x1, x2, q, dt)
    for c, N in enumerate(grid):
        d = x2[c].astype(np.float64) - x1[c].astype(np.float64)
        d -= N * np.round(d / N)  # the periodic minimum image of the move
        assert abs(J[c].sum() - np.sum(q * d) / dt) <= 1e-10 * np.abs(q * d / dt).sum()
    Jr, _ = oracle.deposit_zigzag(grid, x2, x1, q, dt)
    assert np.abs(J + Jr).max() <= 1e-12 * np.abs(J).max()


def test_zigzag_invalid_moves_skipped_and_counted():
    grid, dt = (6, 6, 6), 1.0
    x1, x2, q = _zigzag_moves(grid, 500, 12)
    J_ok, _ = oracle.deposit_zigzag(grid, x1, x2, q, dt)
    bad1 = [np.array([1.5, 0.5, 2.5, 3.5], np.float32), np.array([1.5, 0.5, 2.5, np.nan], np.float32),
            np.array([1.5, 0.5, 2.5, 1.0], np.float32)]
    bad2 = [np.array([3.5, 0.5, 2.5, 3.5], np.float32),   # two cells along x
            np.array([1.5, 6.0, 2.5, 1.0], np.float32),   # y outside [0, 6)
            np.array([1.5, 0.5, -0.25, 1.0], np.float32)]  # z below 0
    a = [np.concatenate([u, v]) for u, v in zip(x1, bad1)]
    b = [np.concatenate([u, v]) for u, v in zip(x2, bad2)]
    J, ninv = oracle.deposit_zigzag(grid, a, b, np.concatenate([q, np.ones(4, np.float32)]), dt)
    assert ninv == 4
    assert np.array_equal(J, J_ok)


# ---------------------------------------------------------------------------
# TSC (second-order) mass matrix (Pennati & Markidis, Sec. 2.3, 3.3-3.4):
# the dense W S W^T with W from the convolution-built quadratic spline
# ---------------------------------------------------------------------------
def _dense_mass_order(grid, pos, wq, omega, order):
    Nx, Ny, Nz = grid
    ng = Nx * Ny * Nz
    n = len(wq)
    gz, gy, gx = np.meshgrid(np.arange(Nz), np.arange(Ny), np.arange(Nx), indexing="ij")
    W = np.zeros((ng, n))
    for p in range(n):
        Wp = (_phi(order, _minimg(float(pos[0][p]) - gx, Nx)) * _phi(order, _minimg(float(pos[1][p]) - gy, Ny))
              * _phi(order, _minimg(float(pos[2][p]) - gz, Nz)))
        W[:, p] = Wp.ravel()
    S = np.zeros((3, 3, n))
    for p in range(n):
        w = np.array([float(omega[c][p]) for c in range(3)])
        S[:, :, p] = float(wq[p]) * np.linalg.solve(np.eye(3) + _cross_matrix(w), np.eye(3))
    return np.einsum("gp,ijp,hp->ijgh", W, S, W)


def _offset_layout_125(Md, grid):
    Nx, Ny, Nz = grid
    ng = Nx * Ny * Nz
    out = np.zeros((ng, 125, 3, 3))
    for g in range(ng):
        x, y, z = g % Nx, (g // Nx) % Ny, g // (Nx * Ny)
        for dz in range(-2, 3):
            for dy in range(-2, 3):
                for dx in range(-2, 3):
                    h = (((z + dz) % Nz) * Ny + (y + dy) % Ny) * Nx + (x + dx) % Nx
                    out[g, (dz + 2) * 25 + (dy + 2) * 5 + (dx + 2)] = Md[:, :, g, h]
    return out


@pytest.mark.parametrize("grid", [(5, 6, 5), (7, 5, 6)])
def test_tsc_mass_matrix_dense_product(grid):
    rng = np.random.default_rng(sum(grid) + 200)
    n = 25
    pos = [rng.uniform(0, N, n).astype(np.float32) for N in grid]
    # fractional parts either side of 1/2, on a node, at the top edge (wraps)
    pos[0][0], pos[1][0], pos[2][0] = 1.5, 2.25, 3.75
    pos[0][1] = np.float32(grid[0]) - np.float32(1e-5)
    pos[2][2] = 0.0
    wq = rng.uniform(0.5, 1.5, n).astype(np.float32)
    omega = [rng.normal(0, 0.6, n).astype(np.float32) for _ in range(3)]
    M, ninv = oracle.mass_matrix_tsc(grid, pos, wq, omega)
    assert ninv == 0
    want = _offset_layout_125(_dense_mass_order(grid, pos, wq, omega, 2), grid)
    assert np.abs(M.reshape(-1, 125, 3, 3) - want).max() <= 1e-12 * np.abs(want).max()


def test_tsc_mass_matrix_symmetry_and_groups():
    """Each component block is symmetric in (g, g') (Eq. (11)); a particle's 27
    nodes follow the base-offset rule, so a cell holds at most 8 node sets."""
    grid = (6, 5, 7)
    rng = np.random.default_rng(31)
    n = 300
    pos = [rng.uniform(0, N, n).astype(np.float32) for N in grid]
    wq = rng.uniform(0.5, 1.5, n).astype(np.float32)
    omega = [rng.normal(0, 0.6, n).astype(np.float32) for _ in range(3)]
    M, _ = oracle.mass_matrix_tsc(grid, pos, wq, omega)
    for o in range(125):
        dz, dy, dx = o // 25 - 2, (o // 5) % 5 - 2, o % 5 - 2
        mirrored = np.roll(M[:, :, :, 124 - o], shift=(-dz, -dy, -dx), axis=(0, 1, 2))
        assert np.abs(M[:, :, :, o] - mirrored).max() <= 1e-12 * np.abs(M).max()
    firsts = set()
    for p in range(n):
        cell = tuple(int(np.floor(pos[mu][p])) for mu in range(3))
        f = tuple(oracle.axis_support(2, float(pos[mu][p]))[0] - cell[mu] for mu in range(3))
        assert all(v in (-1, 0) for v in f)
        firsts.add(f)
    assert len(firsts) == 8


def test_zigzag_translation_covariance():
    """Moving every particle (before and after its move) by whole cells along an
    axis shifts J by the same number of nodes, periodically."""
    grid, dt = (6, 5, 7), 0.5
    x1, x2, q = _zigzag_moves(grid, 800, 21)
    # positions on multiples of 2^-16, so that whole-cell shifts are exact in fp32
    x1 = [(np.floor(a.astype(np.float64) * 65536) / 65536).astype(np.float32) for a in x1]
    x2 = [(np.floor(a.astype(np.float64) * 65536) / 65536).astype(np.float32) for a in x2]
    J, _ = oracle.deposit_zigzag(grid, x1, x2, q, dt)
    for mu, shift in ((0, 2), (1, 4), (2, 3)):
        N = grid[mu]
        s1 = [a.copy() for a in x1]
        s2 = [a.copy() for a in x2]
        s1[mu] = ((x1[mu].astype(np.float64) + shift) % N).astype(np.float32)
        s2[mu] = ((x2[mu].astype(np.float64) + shift) % N).astype(np.float32)
        Js, ninv = oracle.deposit_zigzag(grid, s1, s2, q, dt)
        assert ninv == 0
        assert np.abs(Js - np.roll(J, shift, axis=3 - mu)).max() <= 1e-12 * np.abs(J).max()
