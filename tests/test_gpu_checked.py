"""The index-checked build (-DPCG_CHECKED): every data-dependent index of the
kernels is range-checked before its access and a failure is counted, not
trapped.  The small cases of every kernel family (tests/checked_cases.py) run
against that build in a subprocess: the results must match the oracle and the
failure count must be zero."""
import json
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

HERE = os.path.dirname(os.path.abspath(__file__))


def test_checked_build_has_no_index_failures():
    from helpers import need_gpu
    need_gpu()
    from particle_cell_grid_gb300 import build
    lib = build.build(checked=True)
    env = dict(os.environ, PCG_LIBRARY=lib)
    r = subprocess.run([sys.executable, os.path.join(HERE, "checked_cases.py")], env=env, capture_output=True,
                       text=True, timeout=1200)
    assert r.returncode == 0, r.stdout[-2000:] + r.stderr[-4000:]
    line = json.loads(r.stdout.strip().splitlines()[-1])
    assert line["checked_build"] == 1
    assert line["failures"] == 0, line
    assert len(line["cases"]) >= 10
