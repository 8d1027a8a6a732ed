"""gdn_rollback_layers (every layer of a step rolled back in one launch, the
layers' buffers from device pointer tables) against gdn_rollback called layer
by layer: bit-identical states and conv states, through the C ABI."""
import ctypes

import pytest
import torch

import gated_deltanet_verify_gb300 as gdn
from tests.gpu_util import dims_of, params_of, upload
from workloads.device import empty_outputs
from workloads.synth import Shape, make_inputs

pytestmark = pytest.mark.gpu

SHAPE = Shape("rb_layers", n_slots=4, n_qk_heads=2, n_v_heads=4, d_k=64, d_v=64, n_tokens=6, act="bf16", seed=71)
LAYERS = 3


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()
    torch.cuda.set_device(0)


def _verified_layers():
    """LAYERS layers of seeded inputs, each verified with capture (state and conv state advanced)."""
    d = dims_of(SHAPE)
    layers = []
    for li in range(LAYERS):
        x = upload(make_inputs(SHAPE, layer=li))
        o = empty_outputs(SHAPE, "cuda")
        gdn.gdn_verify_forward(d, params_of(x), x["qkv"], x["z"], x["alpha"], x["beta_raw"], x["state"],
                               x["conv_state"], o["cap_state"], o["cap_conv"], o["out"])
        layers.append({"state": x["state"], "conv_state": x["conv_state"], "cap_state": o["cap_state"],
                       "cap_conv": o["cap_conv"]})
    torch.cuda.synchronize()
    return layers


def _copy(layers):
    return [{k: v.clone() for k, v in layer.items()} for layer in layers]


def _tables(layers):
    return [gdn.pointer_table([layer[k] for layer in layers]) for k in ("state", "conv_state", "cap_state", "cap_conv")]


def test_rollback_layers_is_per_layer_rollback_bit_for_bit():
    d = dims_of(SHAPE)
    trim = torch.tensor([0, 1, 3, SHAPE.n_tokens - 1], dtype=torch.int32, device="cuda")   # no-op .. maximum
    a = _verified_layers()
    post = _copy(a)
    b = _copy(a)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    for layer in b:
        gdn.gdn_rollback(d, trim, layer["state"], layer["conv_state"], layer["cap_state"], layer["cap_conv"], status)
    tabs = _tables(a)
    gdn.gdn_rollback_layers(d, LAYERS, trim, *tabs, status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    for la, lb in zip(a, b):
        assert torch.equal(la["state"], lb["state"]) and torch.equal(la["conv_state"], lb["conv_state"])
    for la, lp in zip(a, post):
        assert torch.equal(la["state"][0], lp["state"][0])              # trim 0: the state after the verify
        assert torch.equal(la["state"][3], lp["cap_state"][3, 0])       # trim T-1: the state after token 0


def test_rollback_layers_skips_a_bad_table_entry():
    d = dims_of(SHAPE)
    trim = torch.tensor([2, 2, 2, 2], dtype=torch.int32, device="cuda")
    a = _verified_layers()
    before = _copy(a)
    ref = _copy(a)
    for layer in ref:
        gdn.gdn_rollback(d, trim, layer["state"], layer["conv_state"], layer["cap_state"], layer["cap_conv"])
    tabs = _tables(a)
    tabs[0][1] = 0                           # layer 1: no state buffer
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    gdn.gdn_rollback_layers(d, LAYERS, trim, *tabs, status)
    torch.cuda.synchronize()
    assert int(status.item()) == gdn.GDN_ERR_ARG
    assert torch.equal(a[0]["state"], ref[0]["state"]) and torch.equal(a[2]["state"], ref[2]["state"])
    assert torch.equal(a[1]["state"], before[1]["state"]) and torch.equal(a[1]["conv_state"], before[1]["conv_state"])


def test_rollback_layers_host_checks():
    d = dims_of(SHAPE)
    trim = torch.zeros(SHAPE.n_slots, dtype=torch.int32, device="cuda")
    L = gdn.lib()
    t = gdn.pointer_table([trim] * 2)
    d = ctypes.byref(d)
    assert L.gdn_rollback_layers(d, 0, trim.data_ptr(), *([t.data_ptr()] * 4), None, None) == gdn.GDN_ERR_SHAPE
    assert L.gdn_rollback_layers(d, 2, trim.data_ptr(), None, t.data_ptr(), t.data_ptr(), t.data_ptr(), None,
                                 None) == gdn.GDN_ERR_ARG
    assert L.gdn_rollback_layers(d, 2, trim.data_ptr(), t.data_ptr(), t.data_ptr(), None, t.data_ptr(), None,
                                 None) == gdn.GDN_ERR_NO_CAPTURE


def test_rollback_tree_layers_is_per_layer_tree_rollback_bit_for_bit():
    from workloads.synth import make_parents
    d = dims_of(SHAPE)
    acc = torch.tensor([-1, 0, 3, SHAPE.n_tokens - 1], dtype=torch.int32, device="cuda")   # nothing .. last node
    layers = []
    for li in range(LAYERS):
        x = upload(make_inputs(SHAPE, layer=li))
        o = empty_outputs(SHAPE, "cuda")
        cap_conv = torch.empty((SHAPE.n_slots, SHAPE.n_tokens, 3, SHAPE.conv_channels), dtype=torch.float32,
                               device="cuda")
        par = torch.from_numpy(make_parents(SHAPE, "random", layer=li).astype("int32")).to("cuda")
        gdn.gdn_verify_tree(d, params_of(x), x["qkv"], x["z"], x["alpha"], x["beta_raw"], par, x["state"],
                            x["conv_state"], o["cap_state"], cap_conv, o["out"])
        layers.append({"state": x["state"], "conv_state": x["conv_state"], "cap_state": o["cap_state"],
                       "cap_conv": cap_conv})
    torch.cuda.synchronize()
    ref = _copy(layers)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    for layer in ref:
        gdn.gdn_rollback_tree(d, acc, layer["state"], layer["conv_state"], layer["cap_state"], layer["cap_conv"],
                              status)
    gdn.gdn_rollback_tree_layers(d, LAYERS, acc, *_tables(layers), status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    for la, lr in zip(layers, ref):
        assert torch.equal(la["state"], lr["state"]) and torch.equal(la["conv_state"], lr["conv_state"])
