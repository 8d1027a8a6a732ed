"""The 48-layer hybrid-stack workload at full size (8 slots, 16/48 heads, d=128,
T=16): every layer's verify + rollback captured in one CUDA graph, as the
bench times it; every layer and head checked against the fp64 oracle."""
import numpy as np
import pytest
import torch

import gated_deltanet_verify_gb300 as gdn
import oracle
from tests.gpu_util import dims_of, params_of
from tests.tolerance import assert_act_close, assert_f32_close
from workloads.device import empty_outputs, to_device, to_f64
from workloads.synth import WORKLOADS, make_inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()
    torch.cuda.set_device(0)


def test_stack_graph_matches_oracle_on_every_layer():
    shape = WORKLOADS["stack_verify"]
    one = shape.with_(n_layers=1)
    layers = []
    host = []
    for li in range(shape.n_layers):
        inp = make_inputs(one, layer=li)
        host.append(inp)
        x = to_device(inp, "cuda")
        x.update(empty_outputs(one, "cuda"))
        x["status"] = torch.zeros(1, dtype=torch.int32, device="cuda")
        layers.append(x)
    d = dims_of(one)
    stream = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        sp = torch.cuda.current_stream().cuda_stream
        for x in layers:
            gdn.gdn_verify_forward(d, params_of(x), x["qkv"], x["z"], x["alpha"], x["beta_raw"], x["state"],
                                   x["conv_state"], x["cap_state"], x["cap_conv"], x["out"], x["status"], sp)
            gdn.gdn_rollback(d, x["trim"], x["state"], x["conv_state"], x["cap_state"], x["cap_conv"],
                             x["status"], sp)
    g.replay()
    torch.cuda.synchronize()
    # every layer and every head: the rolled-back state, the outputs and the conv state; the captures of
    # every head on three layers (each is 400 MB of fp32 per layer)
    cap_layers = (0, 23, shape.n_layers - 1)
    for li, (x, inp) in enumerate(zip(layers, host)):
        assert int(x["status"].item()) == 0, li
        ref = oracle.verify(one, inp.as_f64(), n_threads=16)
        st, cs, status = oracle.rollback(one, inp.trim, ref["state"], ref["conv_state"], ref["cap_state"],
                                         ref["cap_conv"])
        assert np.all(status == 0)
        assert_f32_close(to_f64(x["state"]), st, f"layer {li} rolled-back state")
        assert_act_close(to_f64(x["out"]), ref["out"], one.act, f"layer {li} out")
        assert np.array_equal(to_f64(x["conv_state"]), cs), li
        if li in cap_layers:
            for s in range(one.n_slots):
                assert_f32_close(to_f64(x["cap_state"][s]), ref["cap_state"][s], f"layer {li} capture slot {s}")
        del ref
