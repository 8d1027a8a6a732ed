"""GPU parity of gdn_prefill_chunked against the fp64 oracle (sequential form)."""
import numpy as np
import pytest
import torch

import gated_deltanet_verify_gb300 as gdn
import oracle
from tests.gpu_util import as_f64, dims_of, params_of, upload
from tests.tolerance import assert_act_close, assert_f32_close
from workloads.device import act_torch_dtype
from workloads.synth import WORKLOADS, Shape, make_inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()
    torch.cuda.set_device(0)


def run_prefill(shape, x, status=None, q_scale=1.0):
    d = dims_of(shape, q_scale=q_scale)
    ws_bytes = gdn.gdn_prefill_workspace_bytes(d)
    ws = torch.empty(max(ws_bytes, 1), dtype=torch.uint8, device="cuda") if ws_bytes else None
    out = torch.empty((shape.n_slots, shape.n_tokens, shape.n_v_heads * shape.d_v), dtype=act_torch_dtype(shape),
                      device="cuda")
    gdn.gdn_prefill_chunked(d, params_of(x), x["qkv"], x["z"], x["alpha"], x["beta_raw"], x["state"],
                            x["conv_state"], out, ws, ws_bytes, status)
    torch.cuda.synchronize()
    return as_f64({"state": x["state"], "conv_state": x["conv_state"], "out": out})


def _shape(**kw):
    base = dict(n_slots=1, n_qk_heads=2, n_v_heads=6, d_k=128, d_v=128, n_tokens=300, act="bf16", seed=41)
    base.update(kw)
    return Shape("prefill_small", **base)


CASES = {
    "L300_ragged": _shape(),
    "L64_one_chunk": _shape(n_tokens=64),
    "L1": _shape(n_tokens=1),
    "L2_conv_tail": _shape(n_tokens=2),
    "L129_two_slots": _shape(n_tokens=129, n_slots=2),
    "L200_f32": _shape(n_tokens=200, act="f32"),
    "L520_r1": _shape(n_tokens=520, n_qk_heads=3, n_v_heads=3, seed=42),
    "L190_r8": _shape(n_tokens=190, n_qk_heads=1, n_v_heads=8, seed=43),
}


@pytest.mark.parametrize("case", list(CASES))
def test_prefill_matches_sequential_oracle(case):
    shape = CASES[case]
    inp = make_inputs(shape)
    gpu = run_prefill(shape, upload(inp))
    ref = oracle.verify(shape, inp.as_f64(), capture=False, n_threads=8)
    assert_f32_close(gpu["state"], ref["state"], f"{case} state")
    assert_act_close(gpu["out"], ref["out"], shape.act, f"{case} out")
    assert np.array_equal(gpu["conv_state"], ref["conv_state"])


def test_prefill_full_size_all_heads():
    # the 8192-token layer as the bench runs it, every head (so every key-head group of the work split)
    # against the sequential oracle
    shape = WORKLOADS["prefill"]
    inp = make_inputs(shape)
    gpu = run_prefill(shape, upload(inp))
    ref = oracle.verify(shape, inp.as_f64(), capture=False, n_threads=16)
    assert_f32_close(gpu["state"], ref["state"], "state")
    assert_act_close(gpu["out"], ref["out"], shape.act, "out")
    for h in range(shape.n_v_heads):      # per head as well: each head's state at its own scale
        assert_f32_close(gpu["state"][:, h], ref["state"][:, h], f"state h{h}")
    assert np.array_equal(gpu["conv_state"], ref["conv_state"])


def test_prefill_q_scale():
    shape = _shape(n_tokens=150, seed=44)
    inp = make_inputs(shape)
    qs = 1.0 / np.sqrt(128.0)
    gpu = run_prefill(shape, upload(inp), q_scale=qs)
    ref = oracle.verify(shape, inp.as_f64(), capture=False, n_threads=8, q_scale=qs)
    assert_f32_close(gpu["state"], ref["state"], "state")
    assert_act_close(gpu["out"], ref["out"], shape.act, "out")


def test_prefill_more_pairs_than_one_launch():
    # 2 slots x 48 value heads = 96 (slot, head) pairs: more than one cooperative launch holds on the
    # GPU (three CTAs per pair), so the call spans several launches
    shape = Shape("prefill_pairs", n_slots=2, n_qk_heads=16, n_v_heads=48, d_k=128, d_v=128, n_tokens=130,
                  act="bf16", seed=45)
    inp = make_inputs(shape)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    gpu = run_prefill(shape, upload(inp), status=status)
    ref = oracle.verify(shape, inp.as_f64(), capture=False, n_threads=16)
    assert_f32_close(gpu["state"], ref["state"], "state")
    assert_act_close(gpu["out"], ref["out"], shape.act, "out")
    assert np.array_equal(gpu["conv_state"], ref["conv_state"])
    assert int(status.item()) == gdn.GDN_OK
