"""gdn_prefill_chunked_static (scratch from the library's built-in array, no
caller workspace) against gdn_prefill_chunked (caller workspace), through the
C ABI on the GPU.  Collected last so that it also runs after every other GPU
test has used the device."""
import numpy as np
import pytest
import torch

import gated_deltanet_verify_gb300 as gdn
from tests.gpu_util import as_f64, dims_of, params_of, run_test_build, upload
from tests.tolerance import assert_act_close, assert_f32_close
from workloads.device import act_torch_dtype
from workloads.synth import Shape, make_inputs

pytestmark = pytest.mark.gpu

SHAPE = Shape("prefill_static", n_slots=1, n_qk_heads=2, n_v_heads=6, d_k=128, d_v=128, n_tokens=200,
              act="bf16", seed=47)


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()
    torch.cuda.set_device(0)


def _out(shape):
    return torch.empty((shape.n_slots, shape.n_tokens, shape.n_v_heads * shape.d_v), dtype=act_torch_dtype(shape),
                       device="cuda")


def _with_workspace(shape, inp):
    x = upload(inp)
    d = dims_of(shape)
    ws_bytes = gdn.gdn_prefill_workspace_bytes(d)
    ws = torch.empty(max(ws_bytes, 1), dtype=torch.uint8, device="cuda")
    out = _out(shape)
    gdn.gdn_prefill_chunked(d, params_of(x), x["qkv"], x["z"], x["alpha"], x["beta_raw"], x["state"],
                            x["conv_state"], out, ws, ws_bytes)
    torch.cuda.synchronize()
    return as_f64({"state": x["state"], "conv_state": x["conv_state"], "out": out})


def _static(shape, inp, status):
    x = upload(inp)
    out = _out(shape)
    gdn.gdn_prefill_chunked_static(dims_of(shape), params_of(x), x["qkv"], x["z"], x["alpha"], x["beta_raw"],
                                   x["state"], x["conv_state"], out, status)
    torch.cuda.synchronize()
    return as_f64({"state": x["state"], "conv_state": x["conv_state"], "out": out})


def test_static_scratch_prefill_matches_workspace_prefill_on_two_calls():
    assert gdn.gdn_prefill_workspace_bytes(dims_of(SHAPE)) <= gdn.prefill_static_scratch_bytes()
    inp = make_inputs(SHAPE)
    ref = _with_workspace(SHAPE, inp)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    for call in range(2):           # the second call reuses the scratch the first one left behind
        got = _static(SHAPE, inp, status)
        assert_f32_close(got["state"], ref["state"], f"call {call} state")
        assert_act_close(got["out"], ref["out"], SHAPE.act, f"call {call} out")
        assert np.array_equal(got["conv_state"], ref["conv_state"])
    assert int(status.item()) == gdn.GDN_OK


def test_static_scratch_rejects_dims_beyond_its_size():
    big = SHAPE.with_(n_slots=400, n_qk_heads=16, n_v_heads=48)
    d = dims_of(big)
    assert gdn.gdn_prefill_workspace_bytes(d) > gdn.prefill_static_scratch_bytes()
    with pytest.raises(gdn.GdnError) as ei:
        # rejected on the host before any pointer is looked at or any work is enqueued
        gdn.gdn_prefill_chunked_static(d, gdn.LayerParams(), None, None, None, None, None, None, None)
    assert ei.value.status == gdn.GDN_ERR_WORKSPACE


def test_static_scratch_address_is_looked_up_per_context(tmp_path):
    # the address is cached per CUDA context: a second context on the same device gets its own copy of
    # the array (a different address), and the first context keeps its cached one; only the lookup runs
    # in the second context, no kernel
    a = [int(v) for v in run_test_build(tmp_path, "scratch_contexts")["addr"]]
    assert all(a), a
    assert a[0] == a[1] == a[4]
    assert a[2] == a[3]
    assert a[2] != a[0]
