"""Prefill -> verify -> rollback on the same state buffers (the serving path: a
prompt is prefilled without capture, then speculative steps verify K+1 tokens
with capture and roll back the rejected tail), against one sequential run of
the fp64 oracle over the prompt plus each slot's accepted tokens."""
import numpy as np
import pytest
import torch

import gated_deltanet_verify_gb300 as gdn
import oracle
from tests.gpu_util import as_f64, dims_of, params_of, upload
from tests.tolerance import assert_act_close, assert_f32_close
from workloads.device import act_torch_dtype, empty_outputs
from workloads.synth import Shape, make_inputs

pytestmark = pytest.mark.gpu

L, T = 150, 16


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()
    torch.cuda.set_device(0)


def _part(x, lo, hi):
    y = dict(x)
    for k in ("qkv", "z", "alpha", "beta_raw"):
        y[k] = x[k][:, lo:hi].clone(memory_format=torch.contiguous_format)
    return y


def _slot(x, s, n):
    return {k: (v[s:s + 1, :n] if k in ("qkv", "z", "alpha", "beta_raw") else
                v[s:s + 1] if k in ("state", "conv_state") else v) for k, v in x.items()}


def test_prefill_then_verify_then_rollback_matches_sequential_oracle():
    full = Shape("handoff", n_slots=3, n_qk_heads=2, n_v_heads=6, d_k=128, d_v=128, n_tokens=L + T, act="bf16",
                 seed=51)
    inp = make_inputs(full)
    trims = np.array([0, 5, 15], dtype=np.int32)
    x = upload(inp)
    params = params_of(x)

    # prefill the prompt
    pre = _part(x, 0, L)
    ps = full.with_(n_tokens=L)
    dp = dims_of(ps)
    ws_bytes = gdn.gdn_prefill_workspace_bytes(dp)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device="cuda")
    out_p = torch.empty((full.n_slots, L, full.value_dim), dtype=act_torch_dtype(full), device="cuda")
    gdn.gdn_prefill_chunked(dp, params, pre["qkv"], pre["z"], pre["alpha"], pre["beta_raw"], x["state"],
                            x["conv_state"], out_p, ws, ws_bytes)
    # verify K+1 = 16 tokens with capture, then roll back each slot's rejected tail
    ver = _part(x, L, L + T)
    vs = full.with_(n_tokens=T)
    o = empty_outputs(vs, "cuda", capture=True)
    gdn.gdn_verify_forward(dims_of(vs), params, ver["qkv"], ver["z"], ver["alpha"], ver["beta_raw"], x["state"],
                           x["conv_state"], o["cap_state"], o["cap_conv"], o["out"], None)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    gdn.gdn_rollback(dims_of(vs), torch.from_numpy(trims).cuda(), x["state"], x["conv_state"], o["cap_state"],
                     o["cap_conv"], status)
    torch.cuda.synchronize()
    assert int(status.item()) == gdn.GDN_OK
    got = as_f64({"state": x["state"], "conv_state": x["conv_state"], "out_p": out_p, "out_v": o["out"]})

    xf = inp.as_f64()
    ref_all = oracle.verify(full, xf, capture=False, n_threads=8)          # prompt + all 16 tokens
    assert_act_close(got["out_p"], ref_all["out"][:, :L], full.act, "prefill out")
    assert_act_close(got["out_v"], ref_all["out"][:, L:], full.act, "verify out")
    for s in range(full.n_slots):
        n = L + T - int(trims[s])                                           # prompt + accepted tokens
        one = full.with_(n_slots=1, n_tokens=n)
        ref = oracle.verify(one, _slot(xf, s, n), capture=False, n_threads=8)
        assert_f32_close(got["state"][s:s + 1], ref["state"], f"slot {s} state")
        assert np.array_equal(got["conv_state"][s:s + 1], ref["conv_state"]), f"slot {s} conv state"
