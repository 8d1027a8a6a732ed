"""Seeded random shapes through the chain verify, the rollback, the tree verify
and the chunkwise prefill, against the fp64 oracle: slot counts, head counts and ratios, d_k,
d_v, batch lengths and activation dtypes drawn from everything the verify
accepts (d_k 32/64/128, d_v a multiple of 8 up to 256, T up to 64, H_v/H_k up
to 12), so that launch shapes the fixed cases do not reach (parts per head,
cluster sizes, shared-memory layouts, ragged slot and token counts) meet the
same bar."""
import numpy as np
import pytest
import torch

import gated_deltanet_verify_gb300 as gdn
import oracle
from tests.gpu_util import as_f64, dims_of, run_verify, upload
from tests.tolerance import assert_act_close, assert_f32_close
from workloads.device import empty_outputs, to_f64
from workloads.synth import Shape, make_inputs, make_parents

pytestmark = pytest.mark.gpu

N_CASES = 24


def _draw(i):
    rng = np.random.default_rng(1000 + i)
    hk = int(rng.integers(1, 5))
    r = int(rng.choice([1, 2, 3, 4, 6, 8, 12]))
    while hk * r > 24:
        hk -= 1
    dk = int(rng.choice([32, 64, 128]))
    dv = int(8 * rng.integers(1, 33))
    B, T = int(rng.integers(1, 6)), int(rng.integers(1, 65))
    act = str(rng.choice(["bf16", "f32"]))
    while B * T * hk * r * dv * dk > 12_000_000:      # the oracle's fp64 captures stay below ~100 MB
        if T > 8:
            T //= 2
        elif B > 1:
            B -= 1
        else:
            dv = max(8, dv // 2)
    return Shape(f"fuzz{i}", n_slots=B, n_qk_heads=hk, n_v_heads=hk * r, d_k=dk, d_v=dv, n_tokens=T, act=act,
                 seed=2000 + i)


def verify_parts(r, dv):
    """CTAs per value head the library picks for a ratio r and d_v (its host rule, restated); 0: refused."""
    w = dv // 8
    best, p = 0, 1
    while p <= w:
        if w % p == 0 and w // p <= 8 and r * p <= 8:
            best = p
        p *= 2
    if best:
        return best
    p = 1
    while p <= w:
        if w % p == 0 and w // p <= 8 and r * p <= 16:
            return p
        p *= 2
    p = (w + 7) // 8
    return p if r * p <= 16 else 0


def supported_draws(n, first):
    """n random shapes the verify accepts, drawn from seeds first, first + 1, ..."""
    out, i = [], first
    while len(out) < n:
        s = _draw(i)
        if verify_parts(s.n_v_heads // s.n_qk_heads, s.d_v):
            out.append(s)
        i += 1
    return out


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()
    torch.cuda.set_device(0)


@pytest.mark.parametrize("i", range(N_CASES))
def test_random_shape_verify_rollback_tree(i):
    shape = _draw(i)
    inp = make_inputs(shape)
    x = upload(inp)
    try:
        o = run_verify(shape, x)
    except RuntimeError as e:
        # the library refuses only what it documents (e.g. a head group too wide for one cluster)
        assert "GDN_ERR_SHAPE" in str(e), e
        pytest.skip(f"{shape}: {e}")
    gpu = as_f64(o)
    ref = oracle.verify(shape, inp.as_f64(), n_threads=8)
    what = f"{shape.name} B{shape.n_slots} Hk{shape.n_qk_heads} Hv{shape.n_v_heads} dk{shape.d_k} dv{shape.d_v} " \
           f"T{shape.n_tokens} {shape.act}"
    assert_f32_close(gpu["state"], ref["state"], f"{what} state")
    assert_act_close(gpu["out"], ref["out"], shape.act, f"{what} out")
    assert np.array_equal(gpu["conv_state"], ref["conv_state"]), what
    assert_f32_close(gpu["cap_state"], ref["cap_state"], f"{what} cap_state")
    assert np.array_equal(gpu["cap_conv"], ref["cap_conv"]), what
    # rollback with the drawn trims: bit-identical to the capture, conv state to the window rows
    trims = np.asarray(inp.trim, dtype=np.int32) % shape.n_tokens
    d_trim = torch.tensor(trims, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    gdn.gdn_rollback(dims_of(shape), d_trim, x["state"], x["conv_state"], o["cap_state"], o["cap_conv"], status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    st, cs = to_f64(x["state"]), to_f64(x["conv_state"])
    for s, tr in enumerate(trims):
        if tr == 0:
            continue
        acc = shape.n_tokens - 1 - tr
        assert np.array_equal(st[s], gpu["cap_state"][s, acc]), (what, s)
        assert np.array_equal(cs[s], gpu["cap_conv"][s, acc + 1:acc + 4]), (what, s)
    # a random draft tree over the same inputs (state and conv state as before the batch)
    xt = upload(inp)
    par = make_parents(shape, "random", seed=3000 + i).astype(np.int32)
    ot = empty_outputs(shape, "cuda")
    cap_conv_t = torch.empty((shape.n_slots, shape.n_tokens, 3, shape.conv_channels), dtype=torch.float32,
                             device="cuda")
    gdn.gdn_verify_tree(dims_of(shape), gdn.layer_params(xt["conv_w"], xt["A_log"], xt["dt_bias"], xt["norm_w"]),
                        xt["qkv"], xt["z"], xt["alpha"], xt["beta_raw"], torch.from_numpy(par).to("cuda"),
                        xt["state"], xt["conv_state"], ot["cap_state"], cap_conv_t, ot["out"], status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    rt = oracle.verify_tree(shape, inp.as_f64(), par, n_threads=8)
    assert_act_close(to_f64(ot["out"]), rt["out"], shape.act, f"{what} tree out")
    assert_f32_close(to_f64(ot["cap_state"]), rt["cap_state"], f"{what} tree cap_state")
    assert np.array_equal(to_f64(cap_conv_t), rt["cap_conv"]), f"{what} tree cap_conv"


N_PREFILL = 8


def _draw_prefill(i):
    rng = np.random.default_rng(5000 + i)
    hk = int(rng.integers(1, 5))
    r = int(rng.choice([1, 2, 3, 4, 6, 8]))
    while hk * r > 24:
        hk -= 1
    return Shape(f"fuzz_prefill{i}", n_slots=int(rng.integers(1, 4)), n_qk_heads=hk, n_v_heads=hk * r, d_k=128,
                 d_v=128, n_tokens=int(rng.integers(1, 400)), act=str(rng.choice(["bf16", "f32"])), seed=6000 + i)


@pytest.mark.parametrize("i", range(N_PREFILL))
def test_random_shape_prefill(i):
    # the chunkwise prefill (d_k = d_v = 128) on random slot and head counts, ratios and prompt lengths (partial
    # last chunks, prompts shorter than the conv window) against the sequential oracle
    from tests.test_prefill_gpu import run_prefill
    shape = _draw_prefill(i)
    inp = make_inputs(shape)
    gpu = run_prefill(shape, upload(inp))
    ref = oracle.verify(shape, inp.as_f64(), capture=False, n_threads=8)
    what = f"{shape.name} B{shape.n_slots} Hk{shape.n_qk_heads} Hv{shape.n_v_heads} L{shape.n_tokens} {shape.act}"
    assert_f32_close(gpu["state"], ref["state"], f"{what} state")
    assert_act_close(gpu["out"], ref["out"], shape.act, f"{what} out")
    assert np.array_equal(gpu["conv_state"], ref["conv_state"]), what


N_LAYER = 4


def _draw_layer(i):
    rng = np.random.default_rng(7000 + i)
    while True:
        hk = int(rng.integers(1, 4))
        r = int(rng.choice([1, 2, 4, 8]))
        hv = hk * r
        dk = int(rng.choice([32, 64, 128]))
        dv = int(8 * rng.integers(1, 17))
        if hv % 8 == 0 and verify_parts(r, dv):           # the layer step wants H_v a multiple of 8
            break
    return Shape(f"fuzz_layer{i}", n_slots=int(rng.integers(1, 4)), n_qk_heads=hk, n_v_heads=hv, d_k=dk, d_v=dv,
                 n_tokens=int(rng.integers(1, 17)), act="bf16", seed=8000 + i, n_embd=int(8 * rng.integers(1, 97)))


@pytest.mark.parametrize("i", range(N_LAYER))
def test_random_shape_layer_step(i):
    # the layer with its projections (hidden size, heads, d_k, d_v, slots, tokens drawn): each stage on its own
    # GPU input within the verify's bar, as for the fixed layer shapes
    from tests.test_layer_gpu import _check_act, _run_layer, _upload_proj
    from workloads.synth import bf16_bits_to_f64, make_proj
    shape = _draw_layer(i)
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
    what = f"{shape.name} B{shape.n_slots} Hk{shape.n_qk_heads} Hv{H} dk{shape.d_k} dv{shape.d_v} T{shape.n_tokens} " \
           f"E{shape.n_embd}"
    assert_act_close(to_f64(out), ref["out"], "bf16", f"{what} block output")
    assert_f32_close(to_f64(x["state"]), ref["state"], f"{what} state")
    M = shape.n_slots * shape.n_tokens
    o64 = to_f64(out).reshape(M, -1)
    y_ref = oracle.project(o64, w_out)
    bound = 2.0 ** -8 * np.abs(y_ref) + V * 2.0 ** -23 * (np.abs(o64) @ np.abs(w_out).T)
    assert np.all(np.abs(to_f64(y).reshape(M, -1) - y_ref) <= bound), f"{what} y"
