"""Host logic of bench.py that needs no GPU: recorded DRAM traffic is used only
while the sources of its own kernel are unchanged."""
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def _tree(tmp_path, files):
    csrc = tmp_path / "particle_cell_grid_gb300" / "csrc"
    csrc.mkdir(parents=True)
    for name, text in files.items():
        (csrc / name).write_text(text)
    (tmp_path / "profiles").mkdir()
    return csrc


def test_kernel_hashes_cover_their_own_sources(tmp_path, monkeypatch):
    files = {n: n for n in ("tile_sort.cu", "tcgen05.cuh", "common.cuh", "checked.cuh", "profile.cuh",
                            "deposit_tiled.cuh", "deposit_quad3d.cuh", "deposit.cuh", "deposit.cu", "deposit_2d.cu",
                            "deposit_3d.cu", "cic1d.cu")}
    csrc = _tree(tmp_path, files)
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    sort_h, dep_h = bench.source_hash("sort_partition1"), bench.source_hash("deposit_tiled")
    assert bench.source_hash("sort_count") == sort_h  # same sources
    assert sort_h != dep_h
    (csrc / "cic1d.cu").write_text("changed")  # another kernel's file
    assert bench.source_hash("sort_partition1") == sort_h
    assert bench.source_hash("deposit_tiled") == dep_h
    (csrc / "tile_sort.cu").write_text("changed")  # the sort's own file
    assert bench.source_hash("sort_partition1") != sort_h
    assert bench.source_hash("deposit_tiled") == dep_h


def test_stale_traffic_entries_are_ignored(tmp_path, monkeypatch):
    files = {n: n for n in ("tile_sort.cu", "tcgen05.cuh", "common.cuh", "checked.cuh", "profile.cuh",
                            "deposit_tiled.cuh", "deposit_quad3d.cuh", "deposit.cuh", "deposit.cu", "deposit_2d.cu",
                            "deposit_3d.cu")}
    _tree(tmp_path, files)
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    lines = [
        "# comment line",
        f"sort_partition1 1000 10 {bench.source_hash('sort_partition1')}",
        "deposit_tiled 2000 10 000000000000",  # taken with other sources
    ]
    (tmp_path / "profiles" / "ncu_traffic.txt").write_text("\n".join(lines) + "\n")
    assert bench.load_traffic() == {"sort_partition1": (1000.0, 10.0)}


def test_roofline_entry_scales_traffic_to_a_full_launch():
    prof = {"k": (4, 8.0)}  # 4 launches, 8 ms in total
    e = bench.roofline_entry("k", prof, 2e9, 1000.0, {"k": (1e8, 1e6)}, 4e6)
    assert e["avg_ms"] == 2.0
    assert e["achieved"] == 1000.0 and e["frac"] == 1.0  # 2 GB in 2 ms against a 1000 GB/s peak
    assert e["traffic"] == 4e8  # captured on 1e6 units, reported for 4e6
    assert bench.roofline_entry("k", prof, 2e9, 1000.0, {}, 4e6)["traffic"] is None


def test_all_core_oracle_leg_sums_private_grids():
    """The all-core CPU leg splits the particles over threads, one private J
    each: the summed grid equals one call over every particle (up to the order
    of the fp64 sums)."""
    import numpy as np
    import oracle
    import synth
    d = synth.cic3d_drift(grid=(16, 16, 16), ppc=4)
    n = d["n"]
    ranges = [(0, n // 3), (n // 3, n // 2), (n // 2, n)]
    J = bench.oracle_on_threads(d, ranges, 3)
    Jr, _ = oracle.deposit_current(d["grid"], d["order"], d["pos"], d["vel"], d["q"])
    assert np.abs(J - Jr).max() <= 1e-12 * np.abs(Jr).max()
    threads, cpu = bench.cpu_threads_for(d)
    assert 1 <= threads <= cpu["usable"] and cpu["model"]
