"""The library's host-side caches (kernel attributes and the static-scratch
address, kept per CUDA context behind a lock) under concurrent first use: a
fresh process whose first library calls come from six host threads at once,
each on its own stream, must give the same bits as the same calls made one
after the other (tests/threads_case.py)."""
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_first_calls_from_several_threads():
    import __graft_entry__
    __graft_entry__.build()
    r = subprocess.run([sys.executable, "-m", "tests.threads_case"], cwd=ROOT, capture_output=True, text=True,
                       timeout=900)
    assert r.returncode == 0, r.stdout[-2000:] + r.stderr[-4000:]
