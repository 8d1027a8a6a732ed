"""The 48-layer hybrid-stack workload at full size (8 slots, 16/48 heads, d=128,
T=16): every layer's verify + rollback captured in one CUDA graph, as the
bench times it; sampled layers and heads checked against the fp64 oracle."""
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


def test_stack_graph_matches_oracle_on_sampled_layers():
    shape = WORKLOADS["stack_verify"]
    one = shape.with_(n_layers=1)
    layers = []
    host = {}
    check_layers = (0, 23, shape.n_layers - 1)
    for li in range(shape.n_layers):
        inp = make_inputs(one, layer=li)
        if li in check_layers:
            host[li] = inp
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
    heads = [0, 31]
    for li in check_layers:
        x, inp = layers[li], host[li]
        assert int(x["status"].item()) == 0
        ref = oracle.verify(one, inp.as_f64(), head_mask=heads, n_threads=8)
        st, cs, status = oracle.rollback(one, inp.trim, ref["state"], ref["conv_state"], ref["cap_state"],
                                         ref["cap_conv"])
        assert np.all(status == 0)
        gs, gc, gout = to_f64(x["state"]), to_f64(x["conv_state"]), to_f64(x["out"])
        gcap = to_f64(x["cap_state"])
        for h in heads:
            assert_f32_close(gs[:, h], st[:, h], f"layer {li} rolled-back state h{h}")
            assert_f32_close(gcap[:, :, h], ref["cap_state"][:, :, h], f"layer {li} capture h{h}")
            sl = slice(h * one.d_v, (h + 1) * one.d_v)
            assert_act_close(gout[:, :, sl], ref["out"][:, :, sl], one.act, f"layer {li} out h{h}")
        assert np.array_equal(gc, cs)
