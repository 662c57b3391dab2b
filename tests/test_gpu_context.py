"""The library's per-context state: a call in a second CUDA context of the same device
(created with the driver API and made current by the caller) prepares its kernels and
looks the fixed top-k scratch up in that context, and calls alternating between the
two contexts give the oracle's selection in each.  Run in a child process, which owns
both contexts and uses no torch CUDA state."""

import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

HERE = os.path.dirname(os.path.abspath(__file__))


def test_static_topk_alternates_between_two_contexts():
    import __graft_entry__

    __graft_entry__.build()
    env = dict(os.environ)
    r = subprocess.run([sys.executable, os.path.join(HERE, "gpu_context_child.py")], capture_output=True, text=True,
                       timeout=600, env=env)
    assert r.returncode == 0 and r.stdout.strip().endswith("OK"), (r.stdout[-2000:], r.stderr[-2000:])
