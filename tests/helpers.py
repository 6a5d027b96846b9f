"""Shared helpers of the GPU parity tests (no arithmetic of the method here)."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

# tolerances stated for the workloads: per-node |err| <= 1e-5 * max|ref| for the
# fp32 deposits (per component), relative Frobenius error <= 2e-3 for the mass
# matrix on TF32/BF16 tensor cores
DEPOSIT_TOL = 1e-5
MASS_TOL = 2e-3


def dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def host(t):
    return t.detach().cpu().numpy()


def stats_dict(stats):
    import particle_cell_grid_gb300 as pcg
    return pcg.read_stats(stats)


def assert_deposit_close(J_gpu, J_ref, tol=DEPOSIT_TOL, where=""):
    """Per component: max |J_gpu - J_ref| <= tol * max |J_ref|."""
    J_gpu = np.asarray(J_gpu, dtype=np.float64)
    assert J_gpu.shape == J_ref.shape, (J_gpu.shape, J_ref.shape)
    for c in range(3):
        scale = np.abs(J_ref[c]).max()
        err = np.abs(J_gpu[c] - J_ref[c]).max()
        assert err <= tol * max(scale, 1e-30), f"{where} component {c}: err {err:.3e} vs scale {scale:.3e}"


def rel_frobenius(a, b):
    a = np.asarray(a, dtype=np.float64)
    return float(np.linalg.norm((a - b).ravel()) / max(np.linalg.norm(b.ravel()), 1e-300))


def need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import particle_cell_grid_gb300 as pcg
    pcg._lib.load()  # fails loudly when the library is missing
    return pcg
