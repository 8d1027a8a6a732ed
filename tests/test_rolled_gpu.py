"""GPU tests of gdn_verify_after_rollback (the previous batch's rollback folded
into the next verify): bit-identity with gdn_rollback + gdn_verify_forward over
several steps, parity with the oracle, refused trims, CUDA-graph replay."""
import numpy as np
import pytest
import torch

import gated_deltanet_verify_gb300 as gdn
import oracle
from tests.test_fuzz_shapes_gpu import supported_draws
from tests.gpu_util import dims_of, params_of, run_verify, upload
from tests.tolerance import assert_act_close, assert_f32_close
from workloads.device import empty_outputs, to_f64
from workloads.synth import WORKLOADS, Shape, make_inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()
    torch.cuda.set_device(0)


def _shape(**kw):
    base = dict(name="rolled", n_slots=4, n_qk_heads=2, n_v_heads=6, d_k=128, d_v=128, n_tokens=16, act="bf16",
                seed=61)
    base.update(kw)
    return Shape(**base)


def _batch(shape, x, seed):
    nxt = upload(make_inputs(shape, seed=seed))
    y = dict(x)
    for k in ("qkv", "z", "alpha", "beta_raw"):
        y[k] = nxt[k]
    return y


def _rolled(shape, x, o, trims, status=None):
    d_trim = torch.tensor(trims, dtype=torch.int32, device="cuda")
    gdn.gdn_verify_after_rollback(dims_of(shape), params_of(x), d_trim, x["qkv"], x["z"], x["alpha"], x["beta_raw"],
                                  x["state"], x["conv_state"], o["cap_state"], o["cap_conv"], o["out"], status)
    torch.cuda.synchronize()


CASES = {
    "slots4_T16": (_shape(), [[0, 1, 7, 15], [15, 3, 0, 8], [2, 2, 2, 2]]),
    "layer": (WORKLOADS["layer_verify"], [[5], [0], [15]]),
    "tiny_f32": (WORKLOADS["tiny"].with_(n_slots=2), [[3, 0], [1, 2]]),
    "T7_dk64_r4": (_shape(n_slots=3, n_tokens=7, d_k=64, d_v=64, n_qk_heads=2, n_v_heads=8), [[6, 0, 3], [1, 5, 2]]),
    "dv72_unequal": (_shape(n_slots=2, n_tokens=6, d_k=64, d_v=72, n_qk_heads=2, n_v_heads=4), [[5, 1], [0, 3]]),
}
for _s in supported_draws(3, 100):            # random shapes the verify accepts, two steps of random trims
    _rng = np.random.default_rng(_s.seed)
    CASES[_s.name] = (_s, [[int(t) for t in _rng.integers(0, _s.n_tokens, _s.n_slots)] for _ in range(2)])


@pytest.mark.parametrize("case", list(CASES))
def test_rolled_steps_equal_rollback_then_verify(case):
    shape, trims = CASES[case]
    inp = make_inputs(shape)
    xa, xb = upload(inp), upload(inp)            # a: verify + rollback per step; b: rolled verify per step
    oa = run_verify(shape, xa)
    ob = empty_outputs(shape, "cuda")
    gdn.gdn_verify_forward(dims_of(shape), params_of(xb), xb["qkv"], xb["z"], xb["alpha"], xb["beta_raw"],
                           xb["state"], xb["conv_state"], ob["cap_state"], ob["cap_conv"], ob["out"])
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    xo = inp.as_f64()
    ref = oracle.verify(shape, xo, n_threads=8)
    for i, tr in enumerate(trims):
        d_trim = torch.tensor(tr, dtype=torch.int32, device="cuda")
        gdn.gdn_rollback(dims_of(shape), d_trim, xa["state"], xa["conv_state"], oa["cap_state"], oa["cap_conv"],
                         status)
        ba = _batch(shape, xa, 200 + i)
        oa = run_verify(shape, ba)
        bb = _batch(shape, xb, 200 + i)
        _rolled(shape, bb, ob, tr, status)
        for k in ("out", "cap_state", "cap_conv"):
            assert torch.equal(oa[k], ob[k]), f"step {i}: {k}"
        assert torch.equal(xa["state"], xb["state"]) and torch.equal(xa["conv_state"], xb["conv_state"])
        # the oracle: rollback of the previous batch, then the new batch
        st, cs, _ = oracle.rollback(shape, tr, ref["state"], ref["conv_state"], ref["cap_state"], ref["cap_conv"])
        nxt = make_inputs(shape, seed=200 + i).as_f64()
        xo = dict(xo, state=st, conv_state=cs, **{k: nxt[k] for k in ("qkv", "z", "alpha", "beta_raw")})
        ref = oracle.verify(shape, xo, n_threads=8)
        assert_act_close(to_f64(ob["out"]), ref["out"], shape.act, f"step {i} out")
        assert_f32_close(to_f64(xb["state"]), ref["state"], f"step {i} state")
        assert np.array_equal(to_f64(xb["conv_state"]), ref["conv_state"])
    assert int(status.item()) == 0


def test_rolled_refused_trim_skips_the_slot():
    shape = _shape(n_slots=3, n_tokens=6)
    inp = make_inputs(shape)
    x = upload(inp)
    o = run_verify(shape, x)
    s0, c0 = to_f64(x["state"]).copy(), to_f64(x["conv_state"]).copy()
    cap0 = to_f64(o["cap_state"]).copy()
    b2 = _batch(shape, x, 91)
    o["out"].fill_(3.0)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    _rolled(shape, b2, o, [6, 1, -1], status)
    assert int(status.item()) == gdn.GDN_ERR_TRIM_RANGE
    st, cs, out, cap = to_f64(x["state"]), to_f64(x["conv_state"]), to_f64(o["out"]), to_f64(o["cap_state"])
    for b in (0, 2):
        assert np.array_equal(st[b], s0[b]) and np.array_equal(cs[b], c0[b]) and np.all(out[b] == 3.0)
        assert np.array_equal(cap[b], cap0[b])
    assert not np.array_equal(st[1], s0[1])


def test_rolled_step_in_a_cuda_graph():
    shape = _shape(n_slots=2, n_tokens=8)
    inp = make_inputs(shape)
    xg, xe = upload(inp), upload(inp)
    og, oe = run_verify(shape, xg), run_verify(shape, xe)
    trims = torch.tensor([4, 0], dtype=torch.int32, device="cuda")
    warm = upload(inp)
    ow = run_verify(shape, warm)
    _rolled(shape, warm, ow, [4, 0])              # attributes set before the capture
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        gdn.gdn_verify_after_rollback(dims_of(shape), params_of(xg), trims, xg["qkv"], xg["z"], xg["alpha"],
                                      xg["beta_raw"], xg["state"], xg["conv_state"], og["cap_state"], og["cap_conv"],
                                      og["out"], None, s)
    torch.cuda.synchronize()
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    for _ in range(3):
        _rolled(shape, xe, oe, [4, 0])
    for k in ("out", "cap_state", "cap_conv"):
        assert torch.equal(og[k], oe[k]), k
    assert torch.equal(xg["state"], xe["state"]) and torch.equal(xg["conv_state"], xe["conv_state"])


def test_rolled_needs_captures():
    shape = _shape(n_slots=1, n_tokens=2)
    x = upload(make_inputs(shape))
    o = empty_outputs(shape, "cuda")
    with pytest.raises(gdn.GdnError) as ei:
        gdn.gdn_verify_after_rollback(dims_of(shape), params_of(x), torch.zeros(1, dtype=torch.int32, device="cuda"),
                                      x["qkv"], x["z"], x["alpha"], x["beta_raw"], x["state"], x["conv_state"],
                                      None, None, o["out"])
    assert ei.value.status == gdn.GDN_ERR_NO_CAPTURE
