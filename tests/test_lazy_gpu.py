"""GPU parity of lazy capture (gdn_verify_lazy, with and without a pending
batch, and gdn_commit_lazy): outputs and committed states against the fp64
oracle, and bit-identity with the per-position capture path (verify with
capture, then rollback)."""
import numpy as np
import pytest
import torch

import gated_deltanet_verify_gb300 as gdn
import oracle
from tests.test_fuzz_shapes_gpu import supported_draws
from tests.gpu_util import as_f64, dims_of, params_of, run_verify, upload
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
    base = dict(name="lazy", n_slots=4, n_qk_heads=2, n_v_heads=6, d_k=128, d_v=128, n_tokens=16, act="bf16",
                seed=31)
    base.update(kw)
    return Shape(**base)


def _lazy(shape, x, status=None, prev=None, prev_trims=None, out=None):
    """Lazy verify of the batch in x; with prev (a dict holding the pending batch's
    qkv, alpha, beta_raw) and prev_trims it commits that batch first."""
    if out is None:
        out = empty_outputs(shape, x["qkv"].device, capture=False)["out"]
    kw = {}
    if prev is not None:
        kw = dict(prev_trim=torch.tensor(prev_trims, dtype=torch.int32, device=x["qkv"].device),
                  prev_qkv=prev["qkv"], prev_alpha=prev["alpha"], prev_beta_raw=prev["beta_raw"])
    gdn.gdn_verify_lazy(dims_of(shape), params_of(x), x["qkv"], x["z"], x["alpha"], x["beta_raw"], x["state"],
                        x["conv_state"], out, status, **kw)
    torch.cuda.synchronize()
    return out


def _next_batch(shape, x, seed):
    """The activations of another batch (seeded) over x's parameters and state."""
    nxt = upload(make_inputs(shape, seed=seed))
    y = dict(x)
    for k in ("qkv", "z", "alpha", "beta_raw"):
        y[k] = nxt[k]
    return y


def _host_batch(x_host, seed, shape):
    nxt = make_inputs(shape, seed=seed).as_f64()
    y = dict(x_host)
    for k in ("qkv", "z", "alpha", "beta_raw"):
        y[k] = nxt[k]
    return y


def _commit(shape, x, trims, status=None):
    d_trim = torch.tensor(trims, dtype=torch.int32, device=x["qkv"].device)
    gdn.gdn_commit_lazy(dims_of(shape), params_of(x), d_trim, x["qkv"], x["alpha"], x["beta_raw"], x["state"],
                        x["conv_state"], status)
    torch.cuda.synchronize()


CASES = {
    "layer": (WORKLOADS["layer_verify"], None),
    "slots4_T16": (_shape(), [0, 1, 7, 15]),
    "tiny_f32": (WORKLOADS["tiny"].with_(n_slots=3), [3, 0, 2]),
    "T1": (_shape(n_slots=2, n_tokens=1), [0, 0]),
    "T5_dk64_r4": (_shape(n_slots=3, n_tokens=5, d_k=64, d_v=64, n_qk_heads=2, n_v_heads=8), [4, 2, 0]),
    "T64_max": (_shape(n_slots=1, n_tokens=64), [17]),
    "dv240_unequal": (_shape(n_slots=2, n_tokens=9, d_v=240, n_qk_heads=2, n_v_heads=2), [3, 0]),
}
for _s in supported_draws(3, 200):            # random shapes the verify accepts, their own drawn trims
    CASES[_s.name] = (_s, None)


@pytest.mark.parametrize("case", list(CASES))
def test_lazy_matches_oracle_and_capture_path(case):
    shape, trims = CASES[case]
    inp = make_inputs(shape)
    if trims is None:
        trims = [int(t) for t in inp.trim]
    x = upload(inp)
    state0, conv0 = to_f64(x["state"]).copy(), to_f64(x["conv_state"]).copy()
    status = torch.zeros(1, dtype=torch.int32, device="cuda")

    out = to_f64(_lazy(shape, x, status))
    # the lazy verify writes nothing but its outputs
    assert np.array_equal(to_f64(x["state"]), state0) and np.array_equal(to_f64(x["conv_state"]), conv0)
    _commit(shape, x, trims, status)
    assert int(status.item()) == 0

    ref = oracle.verify(shape, inp.as_f64(), capture=False, n_threads=8)
    assert_act_close(out, ref["out"], shape.act, "lazy out")
    st, cs, ost = oracle.commit_lazy(shape, inp.as_f64(), trims, n_threads=8)
    assert np.all(ost == 0)
    assert_f32_close(to_f64(x["state"]), st, "committed state")
    assert np.array_equal(to_f64(x["conv_state"]), cs), "committed conv_state"

    # bit-identity with the per-position capture path on the same inputs
    xc = upload(inp)
    o = run_verify(shape, xc)
    assert np.array_equal(to_f64(o["out"]), out), "lazy out differs from the capture verify's"
    d_trim = torch.tensor(trims, dtype=torch.int32, device="cuda")
    gdn.gdn_rollback(dims_of(shape), d_trim, xc["state"], xc["conv_state"], o["cap_state"], o["cap_conv"], status)
    torch.cuda.synchronize()
    assert np.array_equal(to_f64(xc["state"]), to_f64(x["state"])), "commit differs from capture + rollback"
    assert np.array_equal(to_f64(xc["conv_state"]), to_f64(x["conv_state"]))


FUSED = {
    "slots4_T16": (_shape(), [[0, 1, 7, 15], [15, 3, 0, 8], [2, 2, 2, 2]]),
    "layer": (WORKLOADS["layer_verify"], [[5], [0], [15]]),
    "tiny_f32": (WORKLOADS["tiny"].with_(n_slots=2), [[3, 0], [1, 2], [0, 3]]),
    "T32_dk64": (_shape(n_slots=2, n_tokens=32, d_k=64, d_v=64, n_qk_heads=1, n_v_heads=3), [[31, 0], [9, 20]]),
}
for _s in supported_draws(3, 400):            # random shapes the verify accepts, three steps of random trims
    _rng = np.random.default_rng(_s.seed)
    FUSED[_s.name] = (_s, [[int(t) for t in _rng.integers(0, _s.n_tokens, _s.n_slots)] for _ in range(3)])


@pytest.mark.parametrize("case", list(FUSED))
def test_pending_commit_rides_in_the_next_verify(case):
    # steps of (verify batch i, accept) with the commit of batch i inside the verify of batch i+1, against
    # (a) the capture path: verify with capture + rollback per step, bit for bit, and (b) the oracle
    shape, trims = FUSED[case]
    inp = make_inputs(shape)
    xl, xc = upload(inp), upload(inp)
    xo = inp.as_f64()
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    prev_l = None
    for i, tr in enumerate(trims):
        bl = xl if i == 0 else _next_batch(shape, xl, 100 + i)
        bc = xc if i == 0 else _next_batch(shape, xc, 100 + i)
        bo = xo if i == 0 else _host_batch(xo, 100 + i, shape)
        out_l = _lazy(shape, bl, status, prev=prev_l, prev_trims=trims[i - 1] if i else None)
        o = run_verify(shape, bc)
        assert np.array_equal(to_f64(out_l), to_f64(o["out"])), f"step {i}: outputs differ from the capture path"
        ref = oracle.verify(shape, bo, capture=False, n_threads=8)
        assert_act_close(to_f64(out_l), ref["out"], shape.act, f"step {i} out")
        d_trim = torch.tensor(tr, dtype=torch.int32, device="cuda")
        gdn.gdn_rollback(dims_of(shape), d_trim, bc["state"], bc["conv_state"], o["cap_state"], o["cap_conv"],
                         status)
        torch.cuda.synchronize()
        st, cs, ost = oracle.commit_lazy(shape, bo, tr, n_threads=8)
        assert np.all(ost == 0)
        xo = dict(xo, state=st, conv_state=cs)
        prev_l = bl
    assert int(status.item()) == 0
    # commit the last pending batch on its own: the stored state is the capture path's
    _commit(shape, prev_l, trims[-1], status)
    assert np.array_equal(to_f64(xl["state"]), to_f64(xc["state"]))
    assert np.array_equal(to_f64(xl["conv_state"]), to_f64(xc["conv_state"]))
    assert_f32_close(to_f64(xl["state"]), xo["state"], "final state")
    assert np.array_equal(to_f64(xl["conv_state"]), xo["conv_state"])


def test_pending_trim_out_of_range_skips_the_slot():
    shape = _shape(n_slots=3, n_tokens=6)
    inp = make_inputs(shape)
    x = upload(inp)
    s0, c0 = to_f64(x["state"]).copy(), to_f64(x["conv_state"]).copy()
    b2 = _next_batch(shape, x, 77)
    out = torch.full_like(empty_outputs(shape, "cuda", capture=False)["out"], 7.0)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    _lazy(shape, b2, status, prev=x, prev_trims=[6, 2, -3], out=out)
    assert int(status.item()) == gdn.GDN_ERR_TRIM_RANGE
    st, cs, o = to_f64(x["state"]), to_f64(x["conv_state"]), to_f64(out)
    for b in (0, 2):                                   # untouched, no outputs
        assert np.array_equal(st[b], s0[b]) and np.array_equal(cs[b], c0[b])
        assert np.all(o[b] == 7.0)
    ref, rcs, _ = oracle.commit_lazy(shape, inp.as_f64(), [6, 2, -3])
    assert_f32_close(st[1], ref[1], "slot 1")
    assert np.array_equal(cs[1], rcs[1])


def test_commit_out_of_range_trims_leave_slots_untouched():
    shape = _shape(n_slots=4, n_tokens=6)
    inp = make_inputs(shape)
    x = upload(inp)
    s0, c0 = to_f64(x["state"]).copy(), to_f64(x["conv_state"]).copy()
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    _commit(shape, x, [6, -1, 2, 100], status)
    assert int(status.item()) == gdn.GDN_ERR_TRIM_RANGE
    st, cs = to_f64(x["state"]), to_f64(x["conv_state"])
    for b in (0, 1, 3):
        assert np.array_equal(st[b], s0[b]) and np.array_equal(cs[b], c0[b])
    ref, rcs, _ = oracle.commit_lazy(shape, inp.as_f64(), [6, -1, 2, 100])
    assert_f32_close(st[2], ref[2], "slot 2")
    assert np.array_equal(cs[2], rcs[2])


def test_lazy_steps_in_a_cuda_graph():
    # verify + commit captured once and replayed over a changing state: two replays equal two eager steps
    shape = _shape(n_slots=2, n_tokens=8)
    inp = make_inputs(shape)
    warm, xg, xe = upload(inp), upload(inp), upload(inp)
    _lazy(shape, warm)                        # the kernels' attributes are set before the capture
    _lazy(shape, warm, prev=warm, prev_trims=[3, 0])
    _commit(shape, warm, [3, 0])
    trims = torch.tensor([3, 0], dtype=torch.int32, device="cuda")
    out_g = empty_outputs(shape, "cuda", capture=False)["out"]
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        gdn.gdn_verify_lazy(dims_of(shape), params_of(xg), xg["qkv"], xg["z"], xg["alpha"], xg["beta_raw"],
                            xg["state"], xg["conv_state"], out_g, None, s)
        gdn.gdn_commit_lazy(dims_of(shape), params_of(xg), trims, xg["qkv"], xg["alpha"], xg["beta_raw"],
                            xg["state"], xg["conv_state"], None, s)
    torch.cuda.synchronize()
    g.replay()
    g.replay()
    torch.cuda.synchronize()
    for _ in range(2):
        out_e = _lazy(shape, xe)
        _commit(shape, xe, [3, 0])
    assert np.array_equal(to_f64(out_g), to_f64(out_e))
    assert np.array_equal(to_f64(xg["state"]), to_f64(xe["state"]))
    assert np.array_equal(to_f64(xg["conv_state"]), to_f64(xe["conv_state"]))


def test_pending_batch_in_a_cuda_graph():
    # one launch per step, replayed: each replay commits the pending batch (the same buffers) and verifies
    shape = _shape(n_slots=2, n_tokens=8)
    inp = make_inputs(shape)
    warm, xg, xe = upload(inp), upload(inp), upload(inp)
    _lazy(shape, warm, prev=warm, prev_trims=[5, 1])
    trims = torch.tensor([5, 1], dtype=torch.int32, device="cuda")
    out_g = empty_outputs(shape, "cuda", capture=False)["out"]
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        gdn.gdn_verify_lazy(dims_of(shape), params_of(xg), xg["qkv"], xg["z"], xg["alpha"], xg["beta_raw"],
                            xg["state"], xg["conv_state"], out_g, None, s, prev_trim=trims, prev_qkv=xg["qkv"],
                            prev_alpha=xg["alpha"], prev_beta_raw=xg["beta_raw"])
    torch.cuda.synchronize()
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    for _ in range(3):
        out_e = _lazy(shape, xe, prev=xe, prev_trims=[5, 1])
    assert np.array_equal(to_f64(out_g), to_f64(out_e))
    assert np.array_equal(to_f64(xg["state"]), to_f64(xe["state"]))
    assert np.array_equal(to_f64(xg["conv_state"]), to_f64(xe["conv_state"]))


def test_commit_needs_trims():
    shape = _shape(n_slots=1, n_tokens=2)
    x = upload(make_inputs(shape))
    with pytest.raises(gdn.GdnError) as ei:
        gdn.gdn_commit_lazy(dims_of(shape), params_of(x), None, x["qkv"], x["alpha"], x["beta_raw"], x["state"],
                            x["conv_state"])
    assert ei.value.status == gdn.GDN_ERR_ARG
