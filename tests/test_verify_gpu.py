"""GPU parity of gdn_verify_forward / gdn_rollback against the fp64 oracle,
plus the bit-identity properties the rollback contract needs."""
import numpy as np
import pytest
import torch

import gated_deltanet_verify_gb300 as gdn
import oracle
from tests.gpu_util import as_f64, dims_of, prefix, run_verify, upload
from tests.tolerance import assert_act_close, assert_f32_close
from workloads.device import to_f64
from workloads.synth import WORKLOADS, Shape, make_inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()
    torch.cuda.set_device(0)


def _shape(name="v", **kw):
    base = dict(n_slots=2, n_qk_heads=2, n_v_heads=6, d_k=128, d_v=128, n_tokens=16, act="bf16", seed=7)
    base.update(kw)
    return Shape(name, **base)


def _compare(shape, gpu, ref, what=""):
    assert_f32_close(gpu["state"], ref["state"], f"{what} state")
    assert_act_close(gpu["out"], ref["out"], shape.act, f"{what} out")
    assert np.array_equal(gpu["conv_state"], ref["conv_state"]), f"{what} conv_state"
    if "cap_state" in gpu and "cap_state" in ref:
        assert_f32_close(gpu["cap_state"], ref["cap_state"], f"{what} cap_state")
        assert np.array_equal(gpu["cap_conv"], ref["cap_conv"]), f"{what} cap_conv"


CASES = {
    "tiny": WORKLOADS["tiny"],
    "layer_verify": WORKLOADS["layer_verify"],
    "T1": _shape(n_tokens=1),
    "T2": _shape(n_tokens=2),
    "T3": _shape(n_tokens=3),
    "T5_ragged": _shape(n_tokens=5, n_slots=3),
    "T64_max": _shape(n_tokens=64, n_slots=1),
    "dk64_dv64": _shape(d_k=64, d_v=64, n_qk_heads=4, n_v_heads=8),
    "dk32_dv16": _shape(d_k=32, d_v=16, n_qk_heads=3, n_v_heads=3),
    "dv256_r1": _shape(d_v=256, n_qk_heads=2, n_v_heads=2, n_tokens=7),
    "r4_f32": _shape(n_qk_heads=2, n_v_heads=8, act="f32", n_tokens=9),
    "r8": _shape(d_k=64, d_v=32, n_qk_heads=1, n_v_heads=8, n_tokens=6),
    "r12_nonportable": _shape(d_k=32, d_v=32, n_qk_heads=1, n_v_heads=12, n_tokens=4, n_slots=1),
    # d_v/8 warps with no power-of-two split of at most 8 warps: parts of unequal width (5 + 4, 8 + 7 + 8 + 7)
    "dv72_unequal": _shape(d_k=64, d_v=72, n_qk_heads=2, n_v_heads=4, n_tokens=6, n_slots=2),
    "dv240_unequal": _shape(d_v=240, n_qk_heads=2, n_v_heads=2, n_tokens=11, n_slots=2),
    # one warp per CTA (8 value rows) and more tokens than threads: the RMSNorm's per-token sums in rounds
    "dv16_T53_one_warp": _shape(d_v=16, n_qk_heads=2, n_v_heads=8, n_tokens=53, n_slots=2, act="f32"),
    "dv8_T64_one_warp": _shape(d_k=64, d_v=8, n_qk_heads=1, n_v_heads=2, n_tokens=64, n_slots=1),
}


@pytest.mark.parametrize("case", list(CASES))
def test_verify_matches_oracle(case):
    shape = CASES[case]
    inp = make_inputs(shape)
    gpu = as_f64(run_verify(shape, upload(inp)))
    ref = oracle.verify(shape, inp.as_f64(), n_threads=8)
    _compare(shape, gpu, ref, case)


def test_verify_q_scale():
    shape = _shape(n_tokens=4)
    inp = make_inputs(shape)
    qs = 1.0 / np.sqrt(shape.d_k)
    gpu = as_f64(run_verify(shape, upload(inp), q_scale=qs))
    ref = oracle.verify(shape, inp.as_f64(), q_scale=qs)
    _compare(shape, gpu, ref, "q_scale")


def test_multislot_full_size_all_heads():
    # the 32-slot workload as the bench runs it: every slot, every head, every captured position
    shape = WORKLOADS["multislot_verify"]
    inp = make_inputs(shape)
    x = upload(inp)
    o = run_verify(shape, x)
    ref = oracle.verify(shape, inp.as_f64(), n_threads=16)
    assert_f32_close(to_f64(o["state"]), ref["state"], "state")
    assert_act_close(to_f64(o["out"]), ref["out"], shape.act, "out")
    assert np.array_equal(to_f64(o["conv_state"]), ref["conv_state"])
    assert np.array_equal(to_f64(o["cap_conv"]), ref["cap_conv"])
    for s in range(shape.n_slots):            # one slot at a time: 100 MB of fp64 each
        assert_f32_close(to_f64(o["cap_state"][s]), ref["cap_state"][s], f"cap_state slot {s}")


def test_capture_off_is_bit_identical():
    shape = _shape(n_slots=3, n_tokens=11)
    inp = make_inputs(shape)
    a = as_f64(run_verify(shape, upload(inp), capture=True))
    b = as_f64(run_verify(shape, upload(inp), capture=False))
    for k in ("state", "conv_state", "out"):
        assert np.array_equal(a[k], b[k]), k
    assert np.array_equal(a["cap_state"][:, -1], a["state"])


def test_slot_isolation_bitwise():
    shape = _shape(n_slots=4, n_tokens=9)
    inp = make_inputs(shape)
    x = upload(inp)
    full = as_f64(run_verify(shape, {k: v.clone() for k, v in x.items()}))
    one = shape.with_(n_slots=1)
    for b in range(4):
        # fresh allocations: a slice of a slot would not be 16-byte aligned in general
        xb = {k: (v[b:b + 1].clone() if k in ("qkv", "z", "alpha", "beta_raw", "state", "conv_state", "trim")
                  else v) for k, v in x.items()}
        rb = as_f64(run_verify(one, xb))
        for k in ("state", "conv_state", "out", "cap_state", "cap_conv"):
            assert np.array_equal(rb[k][0], full[k][b]), (b, k)


def test_dense_launch_is_bit_identical_to_one_slot_launches():
    # 8 slots of the layer shape launch 768 CTAs (more than two per SM: the three-per-SM build of the
    # kernel); one slot launches 96 (the two-per-SM build).  Every result must be the same bits.
    shape = WORKLOADS["layer_verify"].with_(n_slots=8, seed=17)
    inp = make_inputs(shape)
    x = upload(inp)
    full = as_f64(run_verify(shape, {k: v.clone() for k, v in x.items()}))
    one = shape.with_(n_slots=1)
    for b in (0, 5, 7):
        xb = {k: (v[b:b + 1].clone() if k in ("qkv", "z", "alpha", "beta_raw", "state", "conv_state", "trim")
                  else v) for k, v in x.items()}
        rb = as_f64(run_verify(one, xb))
        for k in ("state", "conv_state", "out", "cap_state", "cap_conv"):
            assert np.array_equal(rb[k][0], full[k][b]), (b, k)


def _rollback(shape, x, o, trims, status=None):
    d_trim = torch.tensor(trims, dtype=torch.int32, device=x["qkv"].device)
    gdn.gdn_rollback(dims_of(shape), d_trim, x["state"], x["conv_state"], o["cap_state"], o["cap_conv"], status)
    torch.cuda.synchronize()


def test_rollback_bit_identical_to_capture_and_prefix_rerun():
    shape = _shape(n_slots=4, n_tokens=16)
    inp = make_inputs(shape)
    x0 = upload(inp)
    x = {k: v.clone() for k, v in x0.items()}
    o = run_verify(shape, x)
    cap = to_f64(o["cap_state"])
    capc = to_f64(o["cap_conv"])
    final = to_f64(x["state"]).copy()
    trims = [0, 1, 7, 15]
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    _rollback(shape, x, o, trims, status)
    assert int(status.item()) == 0
    st = to_f64(x["state"])
    cs = to_f64(x["conv_state"])
    T = shape.n_tokens
    for b, tr in enumerate(trims):
        idx = T - 1 - tr
        if tr == 0:
            assert np.array_equal(st[b], final[b])
        assert np.array_equal(st[b], cap[b, idx])
        assert np.array_equal(cs[b], capc[b, idx + 1: idx + 4])
        # a GPU re-run of only the accepted prefix from the pre-verify state
        one = shape.with_(n_slots=1)
        xb = {k: (v[b:b + 1].clone() if k in ("qkv", "z", "alpha", "beta_raw", "state", "conv_state")
                  else v) for k, v in x0.items()}
        rr = as_f64(run_verify(one, prefix(xb, idx + 1), capture=False, n_tokens=idx + 1))
        assert np.array_equal(rr["state"][0], st[b]), f"slot {b}: prefix re-run differs"
        assert np.array_equal(rr["conv_state"][0], cs[b])
        assert np.array_equal(rr["out"][0], to_f64(o["out"])[b, :idx + 1])


def test_rollback_matches_oracle_full_layer():
    shape = WORKLOADS["layer_verify"]
    inp = make_inputs(shape)
    inp.trim[:] = 5
    x = upload(inp)
    o = run_verify(shape, x)
    _rollback(shape, x, o, [5])
    ref = oracle.verify(shape, inp.as_f64(), n_threads=8)
    st, cs, status = oracle.rollback(shape, [5], ref["state"], ref["conv_state"], ref["cap_state"], ref["cap_conv"])
    assert status[0] == 0
    assert_f32_close(to_f64(x["state"]), st, "rolled-back state")
    assert np.array_equal(to_f64(x["conv_state"]), cs)


def test_rollback_out_of_range_trims_leave_slots_untouched():
    shape = _shape(n_slots=4, n_tokens=6)
    inp = make_inputs(shape)
    x = upload(inp)
    o = run_verify(shape, x)
    before_s = to_f64(x["state"]).copy()
    before_c = to_f64(x["conv_state"]).copy()
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    _rollback(shape, x, o, [6, -1, 2, 100], status)
    assert int(status.item()) == gdn.GDN_ERR_TRIM_RANGE
    st, cs = to_f64(x["state"]), to_f64(x["conv_state"])
    for b in (0, 1, 3):
        assert np.array_equal(st[b], before_s[b]) and np.array_equal(cs[b], before_c[b])
    assert np.array_equal(st[2], to_f64(o["cap_state"])[2, 6 - 1 - 2])


def test_device_pointer_misaligned_is_rejected():
    shape = _shape(n_slots=1, n_tokens=2)
    inp = make_inputs(shape)
    x = upload(inp)
    flat = torch.empty(x["state"].numel() + 1, dtype=torch.float32, device="cuda")
    x["state"] = flat[1:].view_as(x["state"])
    with pytest.raises(gdn.GdnError) as ei:
        run_verify(shape, x)
    assert ei.value.status == gdn.GDN_ERR_ALIGN


def test_repeated_calls_on_the_same_stream_agree():
    # two verify steps back to back (state carried on the device) vs the oracle run twice
    shape = _shape(n_slots=2, n_tokens=8)
    inp = make_inputs(shape)
    x = upload(inp)
    run_verify(shape, x, capture=False)
    inp2 = make_inputs(shape, seed=99)
    x2 = upload(inp2)
    x2["state"], x2["conv_state"] = x["state"], x["conv_state"]
    for k in ("conv_w", "A_log", "dt_bias", "norm_w"):
        x2[k] = x[k]
    gpu = as_f64(run_verify(shape, x2, capture=False))
    r1 = oracle.verify(shape, inp.as_f64(), capture=False)
    x2f = inp2.as_f64()
    x2f["state"], x2f["conv_state"] = r1["state"], r1["conv_state"]
    for k in ("conv_w", "A_log", "dt_bias", "norm_w"):
        x2f[k] = inp.as_f64()[k]
    r2 = oracle.verify(shape, x2f, capture=False)
    _compare(shape, gpu, r2, "second step")
