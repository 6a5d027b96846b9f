"""GPU charge-conserving zigzag deposit (flat and tiled) against the fp64 oracle.

Per component, max |J_gpu - J_oracle| <= 1e-5 * max |J_oracle|.  The tiled path
must give the oracle's result with partial tiles, grids smaller than the
scratch window, particles crossing the periodic boundary, particles sorted
under stale keys (the escape valve) and invalid moves; and the GPU current must
satisfy the continuity equation with the CIC charge to fp32 accuracy.
"""
import numpy as np
import pytest

import oracle
import synth
from helpers import assert_deposit_close, dev, host, need_gpu, stats_dict

pytestmark = pytest.mark.gpu


def _zigzag(pcg, d, tiled=True, key=None, extra=None):
    """Deposit the moves of d (plus extra = (prev, pos, q) appended)."""
    prev, pos, q = d["pos_prev"], d["pos"], d["q"]
    if extra is not None:
        prev = [np.concatenate([a, b]) for a, b in zip(prev, extra[0])]
        pos = [np.concatenate([a, b]) for a, b in zip(pos, extra[1])]
        q = np.concatenate([q, extra[2]])
        if key is not None:
            key = [np.concatenate([a, b]) for a, b in zip(key, extra[0])]
    stats = pcg.new_stats()
    pp, pc, qd = [dev(a) for a in prev], [dev(a) for a in pos], dev(q)
    if not tiled:
        J = pcg.deposit_zigzag(d["grid"], pp, pc, qd, d["dt"], stats=stats)
    else:
        kp = [dev(a) for a in (key if key is not None else prev)]
        out, offs = pcg.tile_sort(d["grid"], 8, kp, pp + pc + [qd])
        J = pcg.deposit_zigzag(d["grid"], out[0:3], out[3:6], out[6], d["dt"], tile_offsets=offs, stats=stats)
    Jr, ninv = oracle.deposit_zigzag(d["grid"], prev, pos, q, d["dt"])
    return host(J), Jr, stats_dict(stats), ninv


@pytest.mark.parametrize("grid,ppc", [((16, 16, 16), 8), ((20, 19, 21), 4), ((3, 4, 5), 16), ((9, 8, 17), 3)])
@pytest.mark.parametrize("tiled", [False, True])
def test_zigzag_matches_oracle(grid, ppc, tiled):
    pcg = need_gpu()
    d = synth.zigzag3d(grid=grid, ppc=ppc, sigma_v=0.4, seed=sum(grid) + ppc)
    J, Jr, st, ninv = _zigzag(pcg, d, tiled)
    assert ninv == 0 and st["n_invalid"] == 0
    assert_deposit_close(J, Jr, where=f"{grid} tiled={tiled}")
    if tiled and min(grid) >= 8:
        assert st["n_escaped"] == 0


def test_zigzag_stale_keys_take_the_escape_valve():
    pcg = need_gpu()
    d = synth.zigzag3d(grid=(24, 16, 32), ppc=6, sigma_v=0.3, escaped_frac=0.03, seed=61)
    J, Jr, st, _ = _zigzag(pcg, d, key=d["key_pos_stale"])
    assert st["n_escaped"] > 0.02 * d["n"]
    assert_deposit_close(J, Jr)


def test_zigzag_invalid_moves_are_counted_and_skipped():
    pcg = need_gpu()
    d = synth.zigzag3d(grid=(16, 12, 8), ppc=4, sigma_v=0.3, seed=62)
    f = lambda *v: np.array(v, np.float32)
    # two cells along x; z outside [0, N); NaN; y exactly N
    bad_prev = [f(3.5, 1.5, 2.5, 1.5), f(1.5, 1.5, 2.5, 1.5), f(1.5, 1.5, np.nan, 1.5)]
    bad_pos = [f(5.5, 1.5, 2.5, 1.5), f(1.5, 1.5, 2.5, 12.0), f(1.5, -0.5, 2.5, 1.5)]
    for tiled in (False, True):
        J, Jr, st, ninv = _zigzag(pcg, d, tiled, extra=(bad_prev, bad_pos, np.ones(4, np.float32)))
        assert ninv == 4 and st["n_invalid"] == 4
        assert_deposit_close(J, Jr)


def test_zigzag_continuity_on_the_gpu_current():
    """(rho(pos) - rho(pos_prev)) / dt + div J = 0 with the GPU's J and the CIC
    charge from the oracle: a property that holds at any size."""
    pcg = need_gpu()
    d = synth.zigzag3d(grid=(32, 24, 16), ppc=8, sigma_v=0.4, dt=0.5, seed=63)
    J, _, _, _ = _zigzag(pcg, d)
    ones, zeros = np.ones(d["n"], np.float32), np.zeros(d["n"], np.float32)
    rho2 = oracle.deposit_current(d["grid"], 1, d["pos"], [ones, zeros, zeros], d["q"])[0][0]
    rho1 = oracle.deposit_current(d["grid"], 1, d["pos_prev"], [ones, zeros, zeros], d["q"])[0][0]
    J = J.astype(np.float64)
    div = sum(J[c] - np.roll(J[c], 1, axis=2 - c) for c in range(3))
    res = (rho2 - rho1) / d["dt"] + div
    assert np.abs(res).max() <= 1e-5 * np.abs(J).max() * 6


def test_zigzag_empty_input_zeroes_J():
    pcg = need_gpu()
    import torch
    J = torch.full((3, 8, 8, 8), 7.0, device="cuda")
    e = [torch.zeros(0, device="cuda") for _ in range(3)]
    pcg.deposit_zigzag((8, 8, 8), e, e, torch.zeros(0, device="cuda"), 1.0, J=J)
    assert float(J.abs().max()) == 0.0
