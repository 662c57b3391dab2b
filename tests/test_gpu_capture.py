"""The step entry points can be captured in a CUDA graph from their first call in a
process: the per-context preparation they do on first use (kernel attributes, occupancy
and cluster-occupancy queries) runs inside the capture.  Run in a child process, so that
no earlier test has warmed the library up."""

import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

HERE = os.path.dirname(os.path.abspath(__file__))


def test_first_calls_inside_a_graph_capture():
    import __graft_entry__

    __graft_entry__.build()
    r = subprocess.run([sys.executable, os.path.join(HERE, "gpu_capture_child.py")], capture_output=True, text=True,
                       timeout=600, env=dict(os.environ))
    assert r.returncode == 0 and r.stdout.strip().endswith("OK"), (r.stdout[-2000:], r.stderr[-2000:])
