"""The test build (-DGDN_CHECKED=1): bounds checks on every verify mode, the
rollbacks and the layer step -- no access falls outside its buffer (the status
word stays GDN_OK) and the results are bit-identical to the ordinary build --
and its host-side fault injection of the prefill's ring-flag wait."""
import numpy as np
import pytest
import torch

import gated_deltanet_verify_gb300 as gdn
from tests.gpu_util import run_test_build

pytestmark = pytest.mark.gpu


def test_checked_build_runs_clean_and_matches(tmp_path):
    chk = run_test_build(tmp_path, "all")
    assert "checked" in bytes(chk.pop("version")).decode()
    assert int(chk["status"][0]) == gdn.GDN_OK, f"checked build reported status {int(chk['status'][0])}"
    from tests.checked_cases import run_all
    torch.cuda.set_device(0)
    ref = run_all()
    assert "checked" not in gdn.gdn_version()
    assert set(ref) == set(chk)
    for k in ref:
        assert np.array_equal(ref[k], chk[k]), k


def test_prefill_lost_chunk_reports_timeout(tmp_path):
    # fault injected on the host (test build only): chunk 2 is never published to the state CTA, whose
    # bounded wait (about a second) then gives up and writes GDN_ERR_TIMEOUT to the status word; the
    # device stays usable and the next clean call matches the oracle
    import oracle
    from tests.checked_cases import LOST_CHUNK_SHAPE
    from tests.tolerance import assert_act_close, assert_f32_close
    from workloads.synth import make_inputs
    r = run_test_build(tmp_path, "lost_chunk")
    assert int(r["status_dropped"][0]) == gdn.GDN_ERR_TIMEOUT
    assert int(r["status_clean"][0]) == gdn.GDN_OK
    shape = LOST_CHUNK_SHAPE
    ref = oracle.verify(shape, make_inputs(shape).as_f64(), capture=False, n_threads=8)
    assert_f32_close(r["state"], ref["state"], "state after recovery")
    assert_act_close(r["out"], ref["out"], shape.act, "out after recovery")


def test_ordinary_build_ignores_the_fault_switch(monkeypatch):
    # the ordinary library never reads the environment: with the switch set, a prefill still runs clean
    import __graft_entry__
    import oracle
    from tests.checked_cases import LOST_CHUNK_SHAPE, _prefill
    from tests.gpu_util import upload
    from tests.tolerance import assert_f32_close
    from workloads.synth import make_inputs
    __graft_entry__.build()
    torch.cuda.set_device(0)
    monkeypatch.setenv("GDN_FAULT_DROP_CHUNK", "2")
    shape = LOST_CHUNK_SHAPE.with_(n_tokens=200)
    inp = make_inputs(shape)
    x = upload(inp)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    _prefill(shape, x, status)
    assert int(status.item()) == gdn.GDN_OK
    ref = oracle.verify(shape, inp.as_f64(), capture=False, n_threads=8)
    assert_f32_close(x["state"].double().cpu().numpy(), ref["state"], "state")
