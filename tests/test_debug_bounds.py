"""The debug-bounds build (-DNVFP4_DEBUG_BOUNDS, libnvfp4_gemv_debug.so) on
the GPU: its device checks of the computed workspace indices (partial tiles,
split-row counters) never fire on the paths the release library takes --
whole row blocks, row blocks summed in clusters, uneven splits through the
workspace, stream-K grids, the tcgen05 reduction, the streaming kernels --
and its outputs match the oracle.  Run in a child process so that this
process keeps the release library."""
from __future__ import annotations

import json
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu
HERE = os.path.dirname(os.path.abspath(__file__))


def test_debug_bounds_build_checks_pass():
    r = subprocess.run([sys.executable, os.path.join(HERE, "_debug_bounds_child.py")], capture_output=True,
                       text=True, timeout=900)
    assert r.returncode == 0, r.stderr[-3000:]
    rows = [json.loads(line) for line in r.stdout.splitlines() if line.startswith("{")]
    assert len(rows) == 9, r.stdout
    for row in rows:
        assert row["error_word"] == 0, row
        assert row["worst_over_tol"] <= 1.0, row
