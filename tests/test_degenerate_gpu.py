"""Degenerate inputs through the CUDA path, against the fp64 oracle: gates at
their limits (beta -> 0 with g -> 1, where the state must hold; g -> 0 through
the large-argument branch of softplus, where only the last token's write
survives), all-zero activations and conv state (q^, k^ and the outputs are
exactly zero through the eps of both norms), z -> -inf (SiLU(z) -> 0) and
large-magnitude activations.  The verify, its rollback and the prefill."""
import numpy as np
import pytest
import torch

import oracle
from tests.gpu_util import as_f64, run_verify, upload
from tests.test_prefill_gpu import run_prefill
from tests.tolerance import assert_act_close, assert_f32_close
from workloads.synth import Shape, make_inputs, to_bf16_bits

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()
    torch.cuda.set_device(0)


def _shape(**kw):
    base = dict(name="degenerate", n_slots=2, n_qk_heads=2, n_v_heads=6, d_k=128, d_v=128, n_tokens=9, act="bf16",
                seed=81)
    base.update(kw)
    return Shape(**base)


def _set(inp, name, value):
    """Overwrite an activation of the seeded inputs with a constant or an array of values."""
    a = getattr(inp, name)
    v = np.broadcast_to(np.asarray(value, dtype=np.float64), a.shape)
    a[...] = to_bf16_bits(v) if inp.shape.act == "bf16" else v.astype(np.float32)


def _verify_both(shape, inp):
    gpu = as_f64(run_verify(shape, upload(inp)))
    ref = oracle.verify(shape, inp.as_f64(), n_threads=8)
    assert_f32_close(gpu["state"], ref["state"], "state")
    assert_f32_close(gpu["cap_state"], ref["cap_state"], "cap_state")
    assert_act_close(gpu["out"], ref["out"], shape.act, "out")
    assert np.array_equal(gpu["conv_state"], ref["conv_state"])
    return gpu, ref


@pytest.mark.parametrize("act", ["bf16", "f32"])
def test_no_write_no_decay_keeps_the_state(act):
    shape = _shape(act=act)
    inp = make_inputs(shape)
    _set(inp, "beta_raw", -60.0)          # beta = sigmoid(-60) ~ 1e-26
    _set(inp, "alpha", -60.0)             # softplus(-60 + dt_bias) ~ 1e-26: g = 1 to fp32
    gpu, ref = _verify_both(shape, inp)
    s0 = inp.state.astype(np.float64)
    np.testing.assert_allclose(gpu["state"], s0, rtol=0, atol=1e-6)
    np.testing.assert_allclose(ref["state"], s0, rtol=0, atol=1e-12)


def test_full_decay_keeps_only_the_last_write():
    shape = _shape()
    inp = make_inputs(shape)
    _set(inp, "alpha", 60.0)              # softplus's large branch: g = exp(-exp(A_log) 60) ~ 0
    gpu, ref = _verify_both(shape, inp)
    # with g = 0 each state is beta_t k_t v_t^T: rank one per value head
    for h in range(shape.n_v_heads):
        sv = np.linalg.svd(ref["state"][0, h], compute_uv=False)
        assert sv[1] < 1e-9 * sv[0]


def test_zero_activations_give_zero_outputs():
    shape = _shape()
    inp = make_inputs(shape)
    _set(inp, "qkv", 0.0)
    inp.conv_state[...] = 0.0
    gpu, ref = _verify_both(shape, inp)
    assert np.all(gpu["out"] == 0.0) and np.all(ref["out"] == 0.0)


def test_gate_z_off_gives_zero_outputs():
    shape = _shape()
    inp = make_inputs(shape)
    _set(inp, "z", -200.0)                # SiLU(-200) = -200 / (1 + e^200): below bf16's smallest subnormal
    gpu, _ = _verify_both(shape, inp)
    assert np.max(np.abs(gpu["out"])) < 1e-30


def test_large_activations():
    shape = _shape(act="f32")
    inp = make_inputs(shape)
    inp.qkv[...] = inp.qkv * 300.0
    inp.z[...] = inp.z * 30.0
    _verify_both(shape, inp)


def test_rollback_after_degenerate_gates():
    # the capture with g = 1 and beta = 0 holds the same state at every position: any trim restores it
    shape = _shape()
    inp = make_inputs(shape)
    _set(inp, "beta_raw", -60.0)
    _set(inp, "alpha", -60.0)
    x = upload(inp)
    o = run_verify(shape, x)
    cap = as_f64(o)["cap_state"]
    for t in range(1, shape.n_tokens):
        assert np.array_equal(cap[:, t], cap[:, 0])


def test_prefill_zero_activations():
    shape = Shape("degenerate_prefill", 1, 2, 6, 128, 128, 150, "bf16", seed=82)
    inp = make_inputs(shape)
    _set(inp, "qkv", 0.0)
    inp.conv_state[...] = 0.0
    gpu = run_prefill(shape, upload(inp))
    ref = oracle.verify(shape, inp.as_f64(), capture=False, n_threads=8)
    assert np.all(gpu["out"] == 0.0)
    assert_f32_close(gpu["state"], ref["state"], "state")
    assert np.array_equal(gpu["conv_state"], ref["conv_state"])


def test_prefill_full_decay():
    shape = Shape("degenerate_prefill", 1, 2, 6, 128, 128, 150, "bf16", seed=83)
    inp = make_inputs(shape)
    _set(inp, "alpha", 60.0)
    gpu = run_prefill(shape, upload(inp))
    ref = oracle.verify(shape, inp.as_f64(), capture=False, n_threads=8)
    assert_f32_close(gpu["state"], ref["state"], "state")
    assert_act_close(gpu["out"], ref["out"], shape.act, "out")
