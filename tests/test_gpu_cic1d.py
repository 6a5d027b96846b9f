"""GPU parity of the 1D windowed CIC histogram, loss and gradient against the
fp64 oracle."""
import numpy as np
import pytest

import oracle
import synth
from conftest import read_golden
from helpers import DEPOSIT_TOL, dev, host, need_gpu

pytestmark = pytest.mark.gpu


def _run(pcg, x0, v, target, nsteps, dt, hw):
    H, loss = pcg.deposit_cic1d(dev(x0), dev(v), dev(target), nsteps=nsteps, dt=dt, halfwidth=hw)
    return host(H), float(host(loss)[0])


def _check(H, L, x0, v, target, nsteps, dt, hw):
    Hr, Lr, _ = oracle.cic1d(x0, v, target, target.size, nsteps, dt, hw)
    scale = max(np.abs(Hr).max(), 1e-30)
    assert np.abs(H - Hr).max() <= DEPOSIT_TOL * scale
    # the loss is accumulated in fp64 from the fp32 histogram: its error is
    # bounded by sum 2|H - t| |dH|, far below 1e-6 relative here
    assert abs(L - Lr) <= 1e-6 * max(abs(Lr), 1.0)


def test_workload_full_size():
    pcg = need_gpu()
    d = synth.cic1d()
    H, L = _run(pcg, d["x0"], d["v"], d["target"], d["nsteps"], d["dt"], d["halfwidth"])
    _check(H, L, d["x0"], d["v"], d["target"], d["nsteps"], d["dt"], d["halfwidth"])
    assert (H > 0).sum() > 100


def test_worked_example():
    pcg = need_gpu()
    rows = {r[0]: r[1:] for r in read_golden("cic1d_worked.txt")}
    f = lambda k: np.array([float(x) for x in rows[k]], np.float32)
    H, L = _run(pcg, f("x0"), f("v"), f("target"), int(rows["nsteps"][0]), float(rows["dt"][0]),
                float(rows["halfwidth"][0]))
    want = np.array([float(x) for x in rows["H_num"]]) / float(rows["H_den"][0])
    assert np.allclose(H, want, rtol=0, atol=1e-6)
    assert abs(L - float(rows["loss_num"][0]) / float(rows["loss_den"][0])) < 1e-6


# n = 16384 is the largest input of the single-cluster path, 16385 the smallest
# of the full-grid path (memset, grid of CTAs with global reductions, loss)
SIZES = [(1, 1024, 50, 0.005), (7, 4, 3, 0.3), (5000, 16384, 20, 0.01), (3000, 1000, 9, 0.6),
         (16384, 1024, 50, 0.005), (16385, 1024, 50, 0.005), (40000, 512, 50, 0.002),
         (300001, 1024, 50, 0.005), (100000, 16384, 7, 0.05)]


@pytest.mark.parametrize("n,nb,T,hw", SIZES)
def test_sizes_and_windows(n, nb, T, hw):
    pcg = need_gpu()
    rng = np.random.default_rng(n + nb)
    x0 = rng.random(n).astype(np.float32)
    v = rng.normal(0, 0.3, n).astype(np.float32)
    target = rng.random(nb).astype(np.float32)
    H, L = _run(pcg, x0, v, target, T, 0.013, hw)
    _check(H, L, x0, v, target, T, 0.013, hw)


def test_positions_outside_unit_interval_wrap():
    pcg = need_gpu()
    rng = np.random.default_rng(5)
    x0 = rng.uniform(-30, 30, 4000).astype(np.float32)
    v = rng.normal(0, 2.0, 4000).astype(np.float32)
    target = np.zeros(256, np.float32)
    H, L = _run(pcg, x0, v, target, 40, 0.01, 0.01)
    _check(H, L, x0, v, target, 40, 0.01, 0.01)


def test_empty_input():
    pcg = need_gpu()
    target = np.linspace(0, 1, 64).astype(np.float32)
    H, L = _run(pcg, np.zeros(0, np.float32), np.zeros(0, np.float32), target, 10, 0.01, 0.005)
    assert np.all(H == 0)
    assert abs(L - float(np.sum(target.astype(np.float64) ** 2))) < 1e-9


def test_repeat_calls_overwrite():
    pcg = need_gpu()
    d = synth.cic1d(n=500, seed=7)
    a = _run(pcg, d["x0"], d["v"], d["target"], 50, 0.01, 0.005)
    b = _run(pcg, d["x0"], d["v"], d["target"], 50, 0.01, 0.005)
    assert np.abs(a[0] - b[0]).max() <= 1e-6 * max(np.abs(a[0]).max(), 1e-30)


# ---------------------------------------------------------------------------
# gradient dL/dx0
def _run_grad(pcg, x0, v, target, nsteps, dt, hw):
    H, loss, g = pcg.deposit_cic1d_grad(dev(x0), dev(v), dev(target), nsteps=nsteps, dt=dt, halfwidth=hw)
    return host(H), float(host(loss)[0]), host(g)


def _check_grad(H, L, g, x0, v, target, nsteps, dt, hw):
    _check(H, L, x0, v, target, nsteps, dt, hw)
    gr, _, _, _ = oracle.cic1d_grad(x0, v, target, target.size, nsteps, dt, hw)
    assert g.dtype == np.float64 and g.shape == gr.shape
    # G = 2 (H - target) is taken from the fp32 histogram on the GPU and from
    # the fp64 one in the oracle: the gradient inherits the histogram's
    # tolerance relative to its largest entry
    scale = max(np.abs(gr).max(), 1e-30)
    assert np.abs(g - gr).max() <= DEPOSIT_TOL * scale
    # particles that are never selected get exactly zero on both sides
    assert np.array_equal(g == 0.0, gr == 0.0)


def test_grad_workload_full_size():
    pcg = need_gpu()
    d = synth.cic1d()
    H, L, g = _run_grad(pcg, d["x0"], d["v"], d["target"], d["nsteps"], d["dt"], d["halfwidth"])
    _check_grad(H, L, g, d["x0"], d["v"], d["target"], d["nsteps"], d["dt"], d["halfwidth"])
    # about half of the particles cross a window in 50 steps
    assert 500 < np.count_nonzero(g) < 1500


@pytest.mark.parametrize("n,nb,T,hw", SIZES)
def test_grad_sizes_and_windows(n, nb, T, hw):
    pcg = need_gpu()
    rng = np.random.default_rng(n + nb + 1)
    x0 = rng.random(n).astype(np.float32)
    v = rng.normal(0, 0.3, n).astype(np.float32)
    target = rng.random(nb).astype(np.float32)
    H, L, g = _run_grad(pcg, x0, v, target, T, 0.013, hw)
    _check_grad(H, L, g, x0, v, target, T, 0.013, hw)


def test_grad_positions_outside_unit_interval_wrap():
    pcg = need_gpu()
    rng = np.random.default_rng(6)
    x0 = rng.uniform(-30, 30, 30000).astype(np.float32)
    v = rng.normal(0, 2.0, 30000).astype(np.float32)
    target = rng.random(256).astype(np.float32)
    H, L, g = _run_grad(pcg, x0, v, target, 40, 0.01, 0.01)
    _check_grad(H, L, g, x0, v, target, 40, 0.01, 0.01)


def test_grad_empty_input():
    pcg = need_gpu()
    target = np.linspace(0, 1, 64).astype(np.float32)
    H, L, g = _run_grad(pcg, np.zeros(0, np.float32), np.zeros(0, np.float32), target, 10, 0.01, 0.005)
    assert g.shape == (0,)
    assert np.all(H == 0)
    assert abs(L - float(np.sum(target.astype(np.float64) ** 2))) < 1e-9


def test_grad_overwrites_stale_output():
    """dx0 is fully written: a buffer holding garbage gives the same result."""
    pcg = need_gpu()
    import torch
    d = synth.cic1d(n=20000, seed=9)
    g = torch.full((20000,), float("nan"), dtype=torch.float64, device="cuda")
    pcg.deposit_cic1d_grad(dev(d["x0"]), dev(d["v"]), dev(d["target"]), 50, 0.01, 0.005, dx0=g)
    gr = oracle.cic1d_grad(d["x0"], d["v"], d["target"], d["nbins"], 50, 0.01, 0.005)[0]
    g = host(g)
    assert np.isfinite(g).all()
    assert np.abs(g - gr).max() <= DEPOSIT_TOL * np.abs(gr).max()


@pytest.mark.parametrize("n", [3000, 40000])
def test_particles_moving_with_the_window(n):
    """Velocities near 1/(T dt), where a particle keeps pace with the window and
    stays selected for many consecutive steps, mixed with ordinary and fast
    ones: the candidate-step enumeration and its fallback must both cover
    every step the fp64 test selects."""
    pcg = need_gpu()
    rng = np.random.default_rng(n)
    T, dt, hw = 50, 0.01, 0.005
    x0 = rng.random(n).astype(np.float32)
    v = np.where(rng.random(n) < 0.5, 1.0 / (T * dt) + rng.normal(0, 0.02, n), rng.normal(0, 0.1, n))
    v[: n // 10] = 1.0 / (T * dt)
    v[n // 10: n // 5] = rng.normal(0, 30.0, n // 5 - n // 10)
    v = v.astype(np.float32)
    target = rng.random(1024).astype(np.float32)
    H, L, g = _run_grad(pcg, x0, v, target, T, dt, hw)
    _check_grad(H, L, g, x0, v, target, T, dt, hw)
