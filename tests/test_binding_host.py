"""The Python binding on a host without a GPU: host tensors and wrong dtypes
are refused before anything reaches the library (there is no CPU fallback),
and a missing library is reported, not worked around."""
import os
import sys

import pytest

torch = pytest.importorskip("torch")
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import particle_cell_grid_gb300 as pcg  # noqa: E402


def test_host_tensors_are_refused():
    x = torch.zeros(8)
    with pytest.raises(TypeError, match="CUDA tensor"):
        pcg.deposit_cic1d(x, x, torch.zeros(16))
    with pytest.raises(TypeError, match="CUDA tensor"):
        pcg.deposit_cic1d_grad(x, x, torch.zeros(16))
    with pytest.raises(TypeError, match="CUDA tensor"):
        pcg.deposit_zigzag((8, 8, 8), [x] * 3, [x] * 3, x, 1.0)
    with pytest.raises(TypeError, match="CUDA tensor"):
        pcg.deposit_current((8, 8, 8), 1, [x] * 3, [x] * 3, x)
    with pytest.raises(TypeError, match="CUDA tensor"):
        pcg.assemble_mass_matrix_scalar((8, 8, 8), [x] * 3, x, torch.zeros(513, dtype=torch.int32))


def test_dtype_and_layout_checks():
    dev = pcg._dev
    fake = torch.zeros(4, dtype=torch.float64)
    with pytest.raises(TypeError):
        dev(fake, torch.float32, "x")
    with pytest.raises(TypeError):
        dev([1.0, 2.0], torch.float32, "x")


def test_missing_library_is_reported(monkeypatch, tmp_path):
    from particle_cell_grid_gb300 import _lib
    monkeypatch.setattr(_lib, "_lib", None)
    monkeypatch.setattr(_lib, "library_path", lambda: str(tmp_path / "libpcg.so"))
    with pytest.raises(RuntimeError, match="missing"):
        _lib.load()
