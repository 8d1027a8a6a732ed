"""The bounds-checked build (-DGDN_CHECKED=1) on every verify mode, the
rollbacks and the layer step: no access falls outside its buffer (the status
word stays GDN_OK) and the results are bit-identical to the ordinary build."""
import os
import subprocess
import sys

import numpy as np
import pytest
import torch

import gated_deltanet_verify_gb300 as gdn

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_checked_build_runs_clean_and_matches(tmp_path):
    import __graft_entry__
    __graft_entry__.build()
    from gated_deltanet_verify_gb300 import _build
    _build.build(checked=True)
    out = tmp_path / "checked.npz"
    r = subprocess.run([sys.executable, "-m", "tests.checked_cases", str(out)], cwd=ROOT, capture_output=True,
                       text=True, timeout=600)
    assert r.returncode == 0, r.stdout + r.stderr
    chk = dict(np.load(out))
    assert "checked" in bytes(chk.pop("version")).decode()
    assert int(chk["status"][0]) == gdn.GDN_OK, f"checked build reported status {int(chk['status'][0])}"
    from tests.checked_cases import run_all
    torch.cuda.set_device(0)
    ref = run_all()
    assert "checked" not in gdn.gdn_version()
    assert set(ref) == set(chk)
    for k in ref:
        assert np.array_equal(ref[k], chk[k]), k
