"""GPU parity of the layer step with its projections (gdn_project_in,
gdn_layer_verify, gdn_project_out) against the fp64 oracle, and bit-identity
of the verify inside it with gdn_verify_forward on the same activations."""
import numpy as np
import pytest
import torch

import gated_deltanet_verify_gb300 as gdn
import oracle
from tests.gpu_util import dims_of, params_of, run_verify, upload
from tests.tolerance import assert_act_close, assert_f32_close
from workloads.device import act_host, to_f64
from workloads.synth import WORKLOADS, Shape, bf16_bits_to_f64, make_inputs, make_proj, proj_in_rows

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()
    torch.cuda.set_device(0)


def _shape(**kw):
    base = dict(name="proj", n_slots=2, n_qk_heads=2, n_v_heads=8, d_k=64, d_v=64, n_tokens=5, act="bf16", seed=51,
                n_embd=256)
    base.update(kw)
    return Shape(**base)


def _run_layer(shape, x, p, capture=True):
    """gdn_layer_verify on device tensors; returns (y, act, out, captures) with act and
    out read from the documented places in the workspace."""
    dims = dims_of(shape)
    w = gdn.proj_weights(shape.n_embd, p["w_in"], p["w_out"])
    ws_bytes = gdn.gdn_layer_workspace_bytes(dims, shape.n_embd)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device="cuda")
    M = shape.n_slots * shape.n_tokens
    y = torch.empty((shape.n_slots, shape.n_tokens, shape.n_embd), dtype=torch.bfloat16, device="cuda")
    cap = {}
    if capture:
        cap["cap_state"] = torch.empty((shape.n_slots, shape.n_tokens, shape.n_v_heads, shape.d_v, shape.d_k),
                                       dtype=torch.float32, device="cuda")
        cap["cap_conv"] = torch.empty((shape.n_slots, 3 + shape.n_tokens, shape.conv_channels), dtype=torch.float32,
                                      device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    gdn.gdn_layer_verify(dims, params_of(x), w, p["x"], x["state"], x["conv_state"], cap.get("cap_state"),
                         cap.get("cap_conv"), y, ws, ws_bytes, status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    ld = gdn.gdn_proj_in_ld(dims)
    act_bytes = M * ld * 2
    act = ws[:act_bytes].view(torch.bfloat16).view(M, ld)
    off = (act_bytes + 255) // 256 * 256
    out = ws[off:off + M * shape.value_dim * 2].view(torch.bfloat16).view(shape.n_slots, shape.n_tokens, -1)
    return y, act, out, cap


def _upload_proj(p):
    return {k: act_host(v, WORKLOADS["layer_verify"]).to("cuda") for k, v in p.items()}


def _check_act(shape, act_gpu, hidden, w_in):
    """The projected activations: fp32 accumulation then one bf16 rounding, so
    |gpu - ref| <= 2^-8 |ref| + K 2^-23 sum_k |x_k w_k| (bf16 half-ulp is 2^-9
    relative; the fp32 sum's error bound taken with a factor 2 to spare)."""
    N = proj_in_rows(shape)
    ref = oracle.project(hidden, w_in).reshape(-1, N)
    bound = 2.0 ** -8 * np.abs(ref) + shape.n_embd * 2.0 ** -23 * (np.abs(hidden).reshape(-1, shape.n_embd)
                                                                   @ np.abs(w_in).T)
    got = to_f64(act_gpu)[:, :N]
    bad = np.abs(got - ref) > bound
    assert not bad.any(), f"{bad.sum()} projected activations outside the bound"


def _check_y(y_gpu, y_ref, what):
    """The oracle stores the activation matrix and the block's output in bf16 as
    the layer does, so what separates the two is y's own rounding (<= 2^-9 |y|),
    fp32 against fp64 sums, and the rare stored value whose fp32 sum lies on the
    other side of a bf16 rounding boundary: one ulp in one input, which a gate
    can carry into a whole head (d log g = -exp(A_log) sigmoid(.) d alpha, a
    gain up to e^2).  Bounds: every element within 2^-8 |y| + 2.5e-2 RMS(y);
    the RMS of the error within 3e-3 RMS(y)."""
    y = to_f64(y_gpu)
    rms = np.sqrt(np.mean(y_ref ** 2))
    err = np.abs(y - y_ref)
    assert np.all(err <= 2.0 ** -8 * np.abs(y_ref) + 2.5e-2 * rms), f"{what}: max err {err.max() / rms:.3g} RMS"
    assert np.sqrt(np.mean(err ** 2)) <= 3e-3 * rms, f"{what}: RMS err {np.sqrt(np.mean(err ** 2)) / rms:.3g}"


@pytest.mark.parametrize("kw", [{}, dict(n_slots=1, n_tokens=1), dict(d_k=128, d_v=128, n_tokens=16, n_embd=512),
                                dict(n_qk_heads=1, n_v_heads=8, d_k=32, d_v=32, n_tokens=9, n_embd=8)])
def test_layer_matches_oracle(kw):
    shape = _shape(**kw)
    inp = make_inputs(shape)
    pr = make_proj(shape)
    x, p = upload(inp), _upload_proj(pr)
    y, act, out, cap = _run_layer(shape, x, p)
    hidden, w_in, w_out = (bf16_bits_to_f64(pr[k]) for k in ("x", "w_in", "w_out"))
    _check_act(shape, act, hidden, w_in)
    ref = oracle.layer_verify(shape, inp.as_f64(), hidden, w_in, w_out, n_threads=8)
    _check_y(y, ref["y"], "y")
    _check_y(out, ref["out"], "block output")


@pytest.mark.parametrize("kw", [{}, dict(d_k=128, d_v=128, n_tokens=16, n_embd=512), "full"])
def test_layer_stages_each_within_the_bar(kw):
    # every stage of the layer against the oracle fed with that stage's own GPU input: the projected
    # activations (the GEMM bound), the block on the layer's own activation matrix (the 2e-3 bar of every
    # verify: outputs, state, captures), and y from the block's own output (the GEMM bound).  The end-to-end
    # bound of test_layer_matches_oracle is looser only because one stored bf16 value on the other side of a
    # rounding boundary propagates through the gates; stage by stage the layer meets the verify's bar.
    shape = WORKLOADS["proj_verify"] if kw == "full" else _shape(**kw)
    inp = make_inputs(shape)
    pr = make_proj(shape)
    x, p = upload(inp), _upload_proj(pr)
    y, act, out, cap = _run_layer(shape, x, p)
    hidden, w_in, w_out = (bf16_bits_to_f64(pr[k]) for k in ("x", "w_in", "w_out"))
    _check_act(shape, act, hidden, w_in)
    C, V, H = shape.conv_channels, shape.value_dim, shape.n_v_heads
    a = to_f64(act).reshape(shape.n_slots, shape.n_tokens, -1)
    xin = inp.as_f64()
    xin["qkv"], xin["z"] = a[:, :, :C], a[:, :, C:C + V]
    xin["alpha"], xin["beta_raw"] = a[:, :, C + V:C + V + H], a[:, :, C + V + H:C + V + 2 * H]
    ref = oracle.verify(shape, xin, n_threads=8)
    assert_act_close(to_f64(out), ref["out"], "bf16", "block output on the layer's activations")
    assert_f32_close(to_f64(x["state"]), ref["state"], "state")
    assert_f32_close(to_f64(cap["cap_state"]), ref["cap_state"], "captured states")
    M = shape.n_slots * shape.n_tokens
    o64 = to_f64(out).reshape(M, -1)
    y_ref = oracle.project(o64, w_out)
    bound = 2.0 ** -8 * np.abs(y_ref) + V * 2.0 ** -23 * (np.abs(o64) @ np.abs(w_out).T)
    assert np.all(np.abs(to_f64(y).reshape(M, -1) - y_ref) <= bound), "y from the block's own output"


def test_verify_inside_the_layer_is_the_verify_kernel_bit_for_bit():
    # the strided reads of the activation matrix give exactly what gdn_verify_forward gives on contiguous copies
    shape = _shape(n_tokens=7)
    inp = make_inputs(shape)
    pr = make_proj(shape)
    x, p = upload(inp), _upload_proj(pr)
    xc = upload(inp)
    y, act, out, cap = _run_layer(shape, x, p)
    C, V, H = shape.conv_channels, shape.value_dim, shape.n_v_heads
    a = act.view(shape.n_slots, shape.n_tokens, -1)
    for k, sl in (("qkv", slice(0, C)), ("z", slice(C, C + V)), ("alpha", slice(C + V, C + V + H)),
                  ("beta_raw", slice(C + V + H, C + V + 2 * H))):
        xc[k] = a[:, :, sl].contiguous()
    o = run_verify(shape, xc)
    assert torch.equal(o["out"], out)
    assert torch.equal(o["cap_state"], cap["cap_state"]) and torch.equal(o["cap_conv"], cap["cap_conv"])
    assert torch.equal(xc["state"], x["state"]) and torch.equal(xc["conv_state"], x["conv_state"])


def test_project_calls_alone():
    shape = _shape()
    pr = make_proj(shape)
    p = _upload_proj(pr)
    dims = dims_of(shape)
    w = gdn.proj_weights(shape.n_embd, p["w_in"], p["w_out"])
    M = shape.n_slots * shape.n_tokens
    ws = torch.empty(32 << 20, dtype=torch.uint8, device="cuda")
    act = torch.empty((M, gdn.gdn_proj_in_ld(dims)), dtype=torch.bfloat16, device="cuda")
    gdn.gdn_project_in(dims, w, p["x"], act, ws, ws.numel())
    out = torch.from_numpy(np.ascontiguousarray(make_inputs(shape).z)).view(torch.bfloat16).to("cuda")
    y = torch.empty((M, shape.n_embd), dtype=torch.bfloat16, device="cuda")
    gdn.gdn_project_out(dims, w, out, y, ws, ws.numel())
    torch.cuda.synchronize()
    hidden, w_in, w_out = (bf16_bits_to_f64(pr[k]) for k in ("x", "w_in", "w_out"))
    _check_act(shape, act, hidden, w_in)
    o64 = to_f64(out).reshape(M, -1)
    ref = oracle.project(o64, w_out)
    bound = 2.0 ** -8 * np.abs(ref) + shape.value_dim * 2.0 ** -23 * (np.abs(o64) @ np.abs(w_out).T)
    assert np.all(np.abs(to_f64(y) - ref) <= bound)


@pytest.mark.parametrize("kw", [
    dict(n_slots=1, n_tokens=1, n_embd=72),                  # one activation row; K below one pipeline stage
    dict(n_slots=3, n_tokens=7, n_embd=200),                 # ragged M (21), K not a multiple of 64
    dict(n_slots=20, n_tokens=15, n_embd=136),               # 300 rows: two blocks of activation rows
    dict(n_slots=1, n_tokens=16, n_qk_heads=16, n_v_heads=48, d_k=128, d_v=128, n_embd=1024),   # split K on out
    # two K blocks split two ways: every split holds one stage, so only the even stages' MMA thread has work
    dict(n_slots=2, n_tokens=8, n_qk_heads=2, n_v_heads=8, d_k=32, d_v=32, n_embd=256),
    # 256 activation rows in one block: both accumulators fill the 512 tensor-memory columns
    dict(n_slots=16, n_tokens=16, n_embd=128),
])
def test_projection_gemm_shapes(kw):
    # both projections on their own against the fp64 product, over the tilings the GEMM kernel uses: weight
    # tiles with a ragged last tile, 16-row activation blocks (M padded), one or two blocks of up to 256
    # rows, K tails, and K split across a cluster when the output tiles are few
    shape = _shape(**kw)
    pr = make_proj(shape)
    p = _upload_proj(pr)
    dims = dims_of(shape)
    w = gdn.proj_weights(shape.n_embd, p["w_in"], p["w_out"])
    M = shape.n_slots * shape.n_tokens
    act = torch.empty((M, gdn.gdn_proj_in_ld(dims)), dtype=torch.bfloat16, device="cuda")
    gdn.gdn_project_in(dims, w, p["x"], act, None, 0)
    out = torch.from_numpy(np.ascontiguousarray(make_inputs(shape).z)).view(torch.bfloat16).to("cuda")
    y = torch.empty((M, shape.n_embd), dtype=torch.bfloat16, device="cuda")
    gdn.gdn_project_out(dims, w, out, y, None, 0)
    torch.cuda.synchronize()
    hidden, w_in, w_out = (bf16_bits_to_f64(pr[k]) for k in ("x", "w_in", "w_out"))
    _check_act(shape, act, hidden, w_in)
    o64 = to_f64(out).reshape(M, -1)
    ref = oracle.project(o64, w_out)
    bound = 2.0 ** -8 * np.abs(ref) + shape.value_dim * 2.0 ** -23 * (np.abs(o64) @ np.abs(w_out).T)
    assert np.all(np.abs(to_f64(y) - ref) <= bound)


def test_layer_full_size():
    # one slot of the layer shape with hidden 5120: all of y and the state against the oracle
    shape = WORKLOADS["proj_verify"]
    inp = make_inputs(shape)
    pr = make_proj(shape)
    x, p = upload(inp), _upload_proj(pr)
    y, act, out, cap = _run_layer(shape, x, p)
    hidden, w_in, w_out = (bf16_bits_to_f64(pr[k]) for k in ("x", "w_in", "w_out"))
    _check_act(shape, act, hidden, w_in)
    ref = oracle.layer_verify(shape, inp.as_f64(), hidden, w_in, w_out, n_threads=16)
    _check_y(y, ref["y"], "y")
    # the state carries the bf16 rounding of the activations too (same bounds)
    _check_y(x["state"], ref["state"], "state")


def test_layer_argument_checks():
    shape = _shape()
    inp = make_inputs(shape)
    x = upload(inp)
    p = _upload_proj(make_proj(shape))
    dims = dims_of(shape)
    w = gdn.proj_weights(shape.n_embd, p["w_in"], p["w_out"])
    need = gdn.gdn_layer_workspace_bytes(dims, shape.n_embd)
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    y = torch.empty((shape.n_slots, shape.n_tokens, shape.n_embd), dtype=torch.bfloat16, device="cuda")

    def call(d=dims, ww=w, n=need):
        gdn.gdn_layer_verify(d, params_of(x), ww, p["x"], x["state"], x["conv_state"], None, None, y, ws, n)

    for d, ww, n, code in ((dims, w, need - 1, gdn.GDN_ERR_WORKSPACE),
                           (dims_of(shape.with_(act="f32")), w, need, gdn.GDN_ERR_DTYPE),
                           (dims_of(shape.with_(n_v_heads=6, n_qk_heads=2)), w, need, gdn.GDN_ERR_SHAPE),
                           (dims, gdn.proj_weights(12, p["w_in"], p["w_out"]), need, gdn.GDN_ERR_SHAPE)):
        with pytest.raises(gdn.GdnError) as ei:
            call(d, ww, n)
        assert ei.value.status == code
