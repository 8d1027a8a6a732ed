"""Tree (DDTree) verify and rollback on the GPU against the fp64 oracle."""
import numpy as np
import pytest
import torch

import gated_deltanet_verify_gb300 as gdn
import oracle
from tests.test_fuzz_shapes_gpu import supported_draws
from tests.gpu_util import as_f64, dims_of, params_of, run_verify, upload
from tests.tolerance import assert_act_close, assert_f32_close
from workloads.device import act_torch_dtype
from workloads.synth import WORKLOADS, Shape, make_inputs, make_parents

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()
    torch.cuda.set_device(0)


def run_tree(shape, x, parents, q_scale=1.0, status=None):
    B, T, Hv = shape.n_slots, shape.n_tokens, shape.n_v_heads
    cap_state = torch.empty((B, T, Hv, shape.d_v, shape.d_k), dtype=torch.float32, device="cuda")
    cap_conv = torch.empty((B, T, shape.conv_width - 1, shape.conv_channels), dtype=torch.float32, device="cuda")
    out = torch.empty((B, T, Hv * shape.d_v), dtype=act_torch_dtype(shape), device="cuda")
    par = torch.from_numpy(np.ascontiguousarray(parents, dtype=np.int32)).cuda()
    gdn.gdn_verify_tree(dims_of(shape, q_scale=q_scale), params_of(x), x["qkv"], x["z"], x["alpha"], x["beta_raw"],
                        par, x["state"], x["conv_state"], cap_state, cap_conv, out, status)
    torch.cuda.synchronize()
    return {"cap_state": cap_state, "cap_conv": cap_conv, "out": out}


def _shape(**kw):
    base = dict(n_slots=2, n_qk_heads=2, n_v_heads=6, d_k=128, d_v=128, n_tokens=16, act="bf16", seed=61)
    base.update(kw)
    return Shape("tree_small", **base)


CASES = {
    "random_T16": (_shape(), "random"),
    "spine_T16": (_shape(seed=62), "spine"),
    "star_T16": (_shape(seed=63), "star"),
    "random_T33_f32": (_shape(n_tokens=33, act="f32", seed=64), "random"),
    "random_T64": (_shape(n_tokens=64, n_slots=1, seed=65), "random"),
    "random_dk32_tiny": (WORKLOADS["tiny"].with_(n_slots=3, n_tokens=7), "random"),
    "random_dk64": (_shape(d_k=64, d_v=64, seed=66), "random"),
}
for _s, _kind in zip(supported_draws(3, 300), ("random", "spine", "star")):   # random shapes the verify accepts
    CASES[_s.name] = (_s, _kind)


@pytest.mark.parametrize("case", list(CASES))
def test_tree_verify_matches_oracle(case):
    shape, kind = CASES[case]
    inp = make_inputs(shape)
    par = make_parents(shape, kind, seed=shape.seed + 100)
    x = upload(inp)
    st0, cs0 = x["state"].clone(), x["conv_state"].clone()
    got = as_f64(run_tree(shape, x, par))
    ref = oracle.verify_tree(shape, inp.as_f64(), par, n_threads=8)
    assert_f32_close(got["cap_state"], ref["cap_state"], f"{case} cap_state")
    assert np.array_equal(got["cap_conv"], ref["cap_conv"]), f"{case} cap_conv"
    assert_act_close(got["out"], ref["out"], shape.act, f"{case} out")
    # a tree verify only reads the state
    assert torch.equal(x["state"], st0) and torch.equal(x["conv_state"], cs0)


def test_tree_q_scale():
    shape = _shape(seed=67)
    inp = make_inputs(shape)
    par = make_parents(shape, "random", seed=3)
    qs = 1.0 / np.sqrt(128.0)
    got = as_f64(run_tree(shape, upload(inp), par, q_scale=qs))
    ref = oracle.verify_tree(shape, inp.as_f64(), par, n_threads=8, q_scale=qs)
    assert_f32_close(got["cap_state"], ref["cap_state"], "cap_state")
    assert_act_close(got["out"], ref["out"], shape.act, "out")


def test_chain_tree_is_bit_identical_to_the_chain_kernel():
    shape = WORKLOADS["layer_verify"].with_(n_slots=2)
    inp = make_inputs(shape)
    tree = as_f64(run_tree(shape, upload(inp), make_parents(shape, "chain")))
    chain = as_f64(run_verify(shape, upload(inp), capture=True))
    assert np.array_equal(tree["cap_state"], chain["cap_state"])
    assert np.array_equal(tree["out"], chain["out"])
    for t in range(shape.n_tokens):
        assert np.array_equal(tree["cap_conv"][:, t], chain["cap_conv"][:, t + 1:t + 4])


def test_tree_full_layer_sampled_heads():
    shape = WORKLOADS["multislot_verify"].with_(n_slots=4)
    inp = make_inputs(shape)
    par = make_parents(shape, "spine", seed=5)
    got = as_f64(run_tree(shape, upload(inp), par))
    heads = [0, 25, 47]
    ref = oracle.verify_tree(shape, inp.as_f64(), par, head_mask=heads, n_threads=8)
    for h in heads:
        assert_f32_close(got["cap_state"][:, :, h], ref["cap_state"][:, :, h], f"cap_state h{h}")
        sl = slice(h * shape.d_v, (h + 1) * shape.d_v)
        assert_act_close(got["out"][:, :, sl], ref["out"][:, :, sl], shape.act, f"out h{h}")
    assert np.array_equal(got["cap_conv"], ref["cap_conv"])


def test_tree_rollback_moves_slots_to_their_accepted_nodes():
    shape = _shape(n_slots=4, seed=68)
    inp = make_inputs(shape)
    par = make_parents(shape, "random", seed=9)
    x = upload(inp)
    caps = run_tree(shape, x, par)
    accept = np.array([-1, 0, 15, 7], dtype=np.int32)
    st0, cs0 = x["state"].clone(), x["conv_state"].clone()
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    gdn.gdn_rollback_tree(dims_of(shape), torch.from_numpy(accept).cuda(), x["state"], x["conv_state"],
                          caps["cap_state"], caps["cap_conv"], status)
    torch.cuda.synchronize()
    assert int(status.item()) == gdn.GDN_OK
    assert torch.equal(x["state"][0], st0[0]) and torch.equal(x["conv_state"][0], cs0[0])
    for s in (1, 2, 3):
        assert torch.equal(x["state"][s], caps["cap_state"][s, accept[s]])
        assert torch.equal(x["conv_state"][s], caps["cap_conv"][s, accept[s]])
    ref_st, ref_cs, ref_status = oracle.rollback_tree(shape, accept, inp.as_f64()["state"], inp.as_f64()["conv_state"],
                                                      *oracle_caps(shape, inp, par))
    assert_f32_close(as_f64({"s": x["state"]})["s"], ref_st, "rolled-back state")
    assert np.array_equal(as_f64({"c": x["conv_state"]})["c"], ref_cs)


def oracle_caps(shape, inp, par):
    r = oracle.verify_tree(shape, inp.as_f64(), par, n_threads=8)
    return r["cap_state"], r["cap_conv"]


def test_tree_rollback_out_of_range_leaves_slot():
    shape = _shape(n_slots=2, seed=69)
    inp = make_inputs(shape)
    x = upload(inp)
    caps = run_tree(shape, x, make_parents(shape, "random", seed=2))
    st0 = x["state"].clone()
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    gdn.gdn_rollback_tree(dims_of(shape), torch.tensor([16, -2], dtype=torch.int32, device="cuda"), x["state"],
                          x["conv_state"], caps["cap_state"], caps["cap_conv"], status)
    torch.cuda.synchronize()
    assert int(status.item()) == gdn.GDN_ERR_TRIM_RANGE
    assert torch.equal(x["state"], st0)


def test_tree_bad_parent_is_reported():
    shape = _shape(n_slots=1, seed=70)
    inp = make_inputs(shape)
    par = make_parents(shape, "chain")
    par[0, 5] = 9                                     # a parent after the token
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    run_tree(shape, upload(inp), par, status=status)
    assert int(status.item()) == gdn.GDN_ERR_TREE
