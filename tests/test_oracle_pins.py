"""Pins for the fp64 oracle: each test checks it against something other than
itself -- closed forms, invariants of the gated delta rule, library routines
(numpy / scipy), finite differences, index tables evaluated from the pages'
printed formulas, and a second algorithm (the chunkwise form).  A plausible
mistake (a dropped term, a wrong sign, a transposed operand, an off-by-one in
the rollback index or conv window) fails at least one of them.
"""
import math
import os

import numpy as np
import pytest
import scipy.linalg
import scipy.special

import oracle
from workloads.synth import WORKLOADS, Shape, make_inputs

HERE = os.path.dirname(os.path.abspath(__file__))
rng = np.random.default_rng(12345)


def small_shape(**kw):
    base = dict(name="pin", n_slots=2, n_qk_heads=2, n_v_heads=6, d_k=8, d_v=6, n_tokens=5, act="f32")
    base.update(kw)
    return Shape(**base)


# --------------------------------------------------------------------------
# gates (closed values)
# --------------------------------------------------------------------------

def test_gate_closed_values():
    # A_log = 0 and alpha + dt_bias = 0: g = exp(-1 * ln 2) = 1/2; beta_raw = 0: beta = 1/2
    g, b = oracle.gates(0.0, 0.0, 0.0, 0.0)
    assert g == pytest.approx(0.5, rel=1e-15) and b == 0.5
    g, _ = oracle.gates(0.0, 0.7, -0.7, 0.0)
    assert g == pytest.approx(0.5, rel=1e-15)
    # softplus(x) = 1 at x = ln(e - 1): g = exp(-exp(A_log)) ; with A_log = ln 3, g = e^-3
    g, _ = oracle.gates(math.log(3.0), 0.0, math.log(math.e - 1.0), 0.0)
    assert g == pytest.approx(math.exp(-3.0), rel=1e-14)
    # beta = sigmoid: sigmoid(x) + sigmoid(-x) = 1, sigmoid(ln 3) = 3/4
    _, b = oracle.gates(0.0, 0.0, 0.0, math.log(3.0))
    assert b == pytest.approx(0.75, rel=1e-15)
    # A_log -> -inf: no decay; alpha -> -inf: no decay
    assert oracle.gates(-80.0, 0.0, 3.0, 0.0)[0] == pytest.approx(1.0, abs=1e-30)
    assert oracle.gates(1.0, 0.0, -60.0, 0.0)[0] == pytest.approx(1.0, abs=1e-24)


def test_softplus_identities():
    for x in [-40.0, -3.0, -0.5, 0.0, 0.25, 2.0, 29.0, 31.0, 60.0]:
        # softplus(x) - softplus(-x) = x for every x
        assert oracle.softplus(x) - oracle.softplus(-x) == pytest.approx(x, abs=1e-13)
        # library: logaddexp(0, x) = log(1 + e^x)
        assert oracle.softplus(x) == pytest.approx(np.logaddexp(0.0, x), rel=1e-14)
    assert oracle.softplus(0.0) == pytest.approx(math.log(2.0), rel=1e-16)


# --------------------------------------------------------------------------
# conv + SiLU (library correlate), L2 norm (defining properties)
# --------------------------------------------------------------------------

def test_conv_matches_library_correlate():
    W, T, C = 4, 7, 5
    w = rng.normal(size=(W, C))
    win = rng.normal(size=(W - 1 + T, C))
    y = oracle.conv_silu(w, win)
    for c in range(C):
        pre = np.correlate(win[:, c], w[:, c], mode="valid")          # tap j meets row t+j
        assert np.allclose(y[:, c], pre * scipy.special.expit(pre), rtol=1e-14, atol=1e-15)


def test_conv_last_tap_is_current_token():
    W, T, C = 4, 6, 3
    w = np.zeros((W, C)); w[W - 1] = 1.0
    win = rng.normal(size=(W - 1 + T, C))
    y = oracle.conv_silu(w, win)
    x = win[W - 1:]
    assert np.allclose(y, x * scipy.special.expit(x), rtol=1e-15)
    w = np.zeros((W, C)); w[0] = 1.0                                  # first tap: 3 steps back
    y = oracle.conv_silu(w, win)
    assert np.allclose(y, win[:T] * scipy.special.expit(win[:T]), rtol=1e-15)


def test_l2norm_properties():
    x = rng.normal(size=37)
    eps = 1e-6
    xh = oracle.l2norm(x, eps)
    n = np.linalg.norm(x)
    assert np.linalg.norm(xh) == pytest.approx(n / math.sqrt(n * n + eps), rel=1e-14)
    assert np.dot(xh, x) / (np.linalg.norm(xh) * n) == pytest.approx(1.0, abs=1e-14)
    assert np.all(np.sign(xh) == np.sign(x))
    assert np.all(oracle.l2norm(np.zeros(5), eps) == 0.0)


# --------------------------------------------------------------------------
# one delta-rule step
# --------------------------------------------------------------------------

def _unit(n):
    v = rng.normal(size=n)
    return v / np.linalg.norm(v)


def test_delta_step_identity():
    dk, dv = 8, 6
    S = rng.normal(size=(dk, dv)); k = _unit(dk); q = rng.normal(size=dk); v = rng.normal(size=dv)
    S1, o = oracle.delta_step(S, k, v, q, g=1.0, beta=0.0, q_scale=0.37)
    assert np.array_equal(S1, S)
    assert np.allclose(o, 0.37 * (S.T @ q), rtol=1e-14)


def test_delta_step_pure_decay():
    dk, dv = 8, 6
    S = rng.normal(size=(dk, dv)); k = _unit(dk); q = rng.normal(size=dk); v = rng.normal(size=dv)
    S1, _ = oracle.delta_step(S, k, v, q, g=0.3, beta=0.0)
    assert np.allclose(S1, 0.3 * S, rtol=1e-15)


@pytest.mark.parametrize("g,beta", [(1.0, 1.0), (0.6, 1.0), (0.8, 0.3), (0.05, 0.9)])
def test_delta_step_write_invariant(g, beta):
    # for unit k: S_new^T k = (1 - beta) (g S)^T k + beta v ; with beta = 1 the association of k is v
    dk, dv = 8, 6
    S = rng.normal(size=(dk, dv)); k = _unit(dk); q = rng.normal(size=dk); v = rng.normal(size=dv)
    S1, o = oracle.delta_step(S, k, v, q, g=g, beta=beta)
    assert np.allclose(S1.T @ k, (1 - beta) * g * (S.T @ k) + beta * v, rtol=1e-12, atol=1e-13)
    assert np.allclose(o, S1.T @ q, rtol=1e-13)


def test_delta_step_is_lms_gradient_step():
    # g = 1: one Widrow-Hoff step on L(S) = 1/2 |S^T k - v|^2 with rate beta;
    # the gradient is taken by central finite differences, not by formula
    dk, dv = 5, 4
    S = rng.normal(size=(dk, dv)); k = rng.normal(size=dk); v = rng.normal(size=dv); q = rng.normal(size=dk)
    beta = 0.37
    S1, _ = oracle.delta_step(S, k, v, q, g=1.0, beta=beta)

    def loss(M):
        r = M.T @ k - v
        return 0.5 * float(r @ r)
    grad = np.zeros_like(S)
    h = 1e-6
    for i in range(dk):
        for j in range(dv):
            E = np.zeros_like(S); E[i, j] = h
            grad[i, j] = (loss(S + E) - loss(S - E)) / (2 * h)
    assert np.allclose(S1, S - beta * grad, rtol=1e-7, atol=1e-8)


def test_delta_step_update_is_rank_one_along_k():
    # S_new - g S is an outer product k w^T: rank one, left factor along k (not v)
    dk, dv = 8, 6
    S = rng.normal(size=(dk, dv)); k = _unit(dk); q = rng.normal(size=dk); v = rng.normal(size=dv)
    S1, _ = oracle.delta_step(S, k, v, q, g=0.7, beta=0.4)
    U_, sv, Vt = np.linalg.svd(S1 - 0.7 * S)
    assert sv[1] < 1e-12 * sv[0]
    assert abs(abs(U_[:, 0] @ k) - 1.0) < 1e-12


# --------------------------------------------------------------------------
# gated RMSNorm
# --------------------------------------------------------------------------

def test_rmsnorm_gate_properties():
    dv = 16
    o = rng.normal(size=dv)
    w = np.ones(dv)
    z = np.full(dv, 45.0)                     # SiLU(45) = 45 to 1e-19
    out = oracle.rmsnorm_gate(o, z, w, eps=0.0)
    assert np.mean((out / 45.0) ** 2) == pytest.approx(1.0, rel=1e-14)
    assert np.allclose(oracle.rmsnorm_gate(3.5 * o, z, w, eps=0.0), out, rtol=1e-14)
    # gating: SiLU(z) = z * expit(z) (library sigmoid), norm weight multiplies elementwise
    z2 = rng.normal(size=dv); w2 = rng.uniform(0.5, 1.5, size=dv)
    out2 = oracle.rmsnorm_gate(o, z2, w2, eps=0.0)
    assert np.allclose(out2 / (w2 * z2 * scipy.special.expit(z2)), out / 45.0, rtol=1e-12)
    # eps enters under the root of the mean square
    ms = float(np.mean(o * o))
    out3 = oracle.rmsnorm_gate(o, z, w, eps=ms)
    assert np.allclose(out3, out / math.sqrt(2.0), rtol=1e-14)


# --------------------------------------------------------------------------
# composite verify: closed form via a library triangular solve
# --------------------------------------------------------------------------

def test_verify_matches_closed_form_triangular_solve():
    """The unrolled recurrence S_T = Gamma_T S_0 + sum_s (Gamma_T/Gamma_s) k_s u_s^T with
    (I + A) U = diag(beta)(V - diag(Gamma) K S_0), solved by scipy's triangular solver,
    against the oracle's step-by-step composite (one slot, one value head)."""
    s = small_shape(n_slots=1, n_qk_heads=1, n_v_heads=1, d_k=6, d_v=5, n_tokens=6)
    x = make_inputs(s, seed=77).as_f64()
    # make the conv a pass-through of the current token so q, k, v are known up front
    x["conv_w"][:] = 0.0
    x["conv_w"][3] = 1.0
    res = oracle.verify(s, x)
    silu = lambda a: a * scipy.special.expit(a)
    y = silu(x["qkv"][0])                                   # [T, C]
    dk, dv, T = s.d_k, s.d_v, s.n_tokens
    nrm = lambda a: a / np.sqrt((a * a).sum(-1, keepdims=True) + 1e-6)
    Q, K, V = nrm(y[:, :dk]), nrm(y[:, dk:2 * dk]), y[:, 2 * dk:]
    logg = -np.exp(x["A_log"][0]) * np.logaddexp(0.0, x["alpha"][0, :, 0] + x["dt_bias"][0])
    beta = scipy.special.expit(x["beta_raw"][0, :, 0])
    G = np.exp(np.cumsum(logg))
    S0 = x["state"][0, 0].T                                 # logical [d_k][d_v]
    A = np.tril(beta[:, None] * (G[:, None] / G[None, :]) * (K @ K.T), -1)
    U = scipy.linalg.solve_triangular(np.eye(T) + A, beta[:, None] * (V - G[:, None] * (K @ S0)),
                                      lower=True)
    ST = G[-1] * S0 + sum((G[-1] / G[r]) * np.outer(K[r], U[r]) for r in range(T))
    assert np.allclose(res["state"][0, 0].T, ST, rtol=1e-11, atol=1e-12)
    for t in range(T):
        St = G[t] * S0 + sum((G[t] / G[r]) * np.outer(K[r], U[r]) for r in range(t + 1))
        assert np.allclose(res["cap_state"][0, t, 0].T, St, rtol=1e-11, atol=1e-12)


def test_verify_head_mapping_and_channel_order():
    """beta = 1 makes S_t^T k^_t = v_t exactly (unit k); with a pass-through conv this
    identifies the key slice of key head floor(h/r) and the value slice of head h."""
    s = small_shape(n_slots=1, n_qk_heads=2, n_v_heads=6, d_k=8, d_v=6, n_tokens=3)
    x = make_inputs(s, seed=5).as_f64()
    x["conv_w"][:] = 0.0
    x["conv_w"][3] = 1.0
    x["beta_raw"][:] = 40.0                                # sigmoid(40) = 1 in fp64
    res = oracle.verify(s, x)
    silu = lambda a: a * scipy.special.expit(a)
    y = silu(x["qkv"][0])
    dk, dv, Hk, r = s.d_k, s.d_v, s.n_qk_heads, s.n_v_heads // s.n_qk_heads
    for h in range(s.n_v_heads):
        kh = h // r
        for t in range(s.n_tokens):
            k = y[t, Hk * dk + kh * dk: Hk * dk + (kh + 1) * dk]
            k = k / np.sqrt(k @ k + 1e-6)
            n2 = k @ k                                     # 1 - O(eps)
            v = y[t, 2 * Hk * dk + h * dv: 2 * Hk * dk + (h + 1) * dv]
            St = res["cap_state"][0, t, h].T
            Sp = (res["cap_state"][0, t - 1, h] if t > 0 else x["state"][0, h]).T
            g, _ = oracle.gates(x["A_log"][h], x["dt_bias"][h], x["alpha"][0, t, h], 0.0)
            # beta = 1: S_t^T k = (1 - |k|^2) g S_{t-1}^T k + |k|^2 v
            assert np.allclose(St.T @ k, (1 - n2) * g * (Sp.T @ k) + n2 * v, rtol=1e-12, atol=1e-13)
            assert np.allclose(St.T @ k, v, rtol=1e-3, atol=1e-3)
            # the tiled mapping h mod H_k would use another key head
            kh_alt = h % Hk
            if kh_alt != kh:
                k2 = y[t, Hk * dk + kh_alt * dk: Hk * dk + (kh_alt + 1) * dk]
                k2 = k2 / np.linalg.norm(k2)
                assert not np.allclose(St.T @ k2, v, rtol=1e-3, atol=1e-3)
            # read-out uses q of the same key head; out is RMSNorm(o) * w * SiLU(z)
            q = y[t, kh * dk:(kh + 1) * dk]
            q = q / np.sqrt(q @ q + 1e-6)
            o = St.T @ q
            zt = x["z"][0, t, h * dv:(h + 1) * dv]
            want = oracle.rmsnorm_gate(o, zt, x["norm_w"])
            assert np.allclose(res["out"][0, t, h * dv:(h + 1) * dv], want, rtol=1e-12, atol=1e-13)


def test_verify_capture_and_conv_window():
    s = small_shape()
    inp = make_inputs(s, seed=9)
    x = inp.as_f64()
    res = oracle.verify(s, x)
    # capture element T-1 is the final state, bit for bit
    assert np.array_equal(res["cap_state"][:, -1], res["state"])
    # the conv capture is concat(old conv state, new tokens); new conv state = last W-1 rows
    win = np.concatenate([x["conv_state"], x["qkv"]], axis=1)
    assert np.array_equal(res["cap_conv"], win)
    assert np.array_equal(res["conv_state"], win[:, -3:])


def test_verify_short_batch_keeps_old_conv_rows():
    # T = 2 < W - 1: the new conv state still holds one row of the old one
    s = small_shape(n_tokens=2)
    x = make_inputs(s, seed=10).as_f64()
    res = oracle.verify(s, x)
    assert np.array_equal(res["conv_state"][:, 0], x["conv_state"][:, 2])
    assert np.array_equal(res["conv_state"][:, 1:], x["qkv"][:, :2])


def test_slot_isolation():
    s = small_shape(n_slots=3)
    x = make_inputs(s, seed=11).as_f64()
    res = oracle.verify(s, x)
    for b in range(3):
        xb = {k: (v[b:b + 1] if k in ("qkv", "z", "alpha", "beta_raw", "state", "conv_state", "trim") else v)
              for k, v in x.items()}
        rb = oracle.verify(s.with_(n_slots=1), xb)
        for key in ("state", "conv_state", "out", "cap_state", "cap_conv"):
            assert np.array_equal(rb[key][0], res[key][b]), key


def test_head_mask_computes_only_selected_heads():
    s = small_shape()
    x = make_inputs(s, seed=12).as_f64()
    full = oracle.verify(s, x)
    part = oracle.verify(s, x, head_mask=[1, 4])
    for h in (1, 4):
        assert np.array_equal(part["state"][:, h], full["state"][:, h])
        assert np.array_equal(part["cap_state"][:, :, h], full["cap_state"][:, :, h])
    assert np.array_equal(part["state"][:, 0], x["state"][:, 0])
    assert np.array_equal(part["conv_state"], full["conv_state"])


def test_threads_do_not_change_results():
    s = small_shape(n_slots=3)
    x = make_inputs(s, seed=13).as_f64()
    a = oracle.verify(s, x, n_threads=1)
    b = oracle.verify(s, x, n_threads=5)
    for key in a:
        assert np.array_equal(a[key], b[key])


# --------------------------------------------------------------------------
# rollback: the pages' index table, the prefix invariant, refusal
# --------------------------------------------------------------------------

def _golden_rows():
    rows = []
    with open(os.path.join(HERE, "golden", "rollback_index_T16.txt")) as f:
        for line in f:
            if line.strip() and not line.startswith("#"):
                rows.append([int(v) for v in line.split()])
    return rows


def test_rollback_index_table_from_pages():
    # one slot, S_v = 128, H = 48, kernel 4, T = 16, as in the table's source
    s = Shape("idx", 1, 16, 48, 128, 128, 16, "f32")
    T, C, per = 16, 8, 48 * 128 * 128
    cap_state = np.repeat(np.arange(T, dtype=np.float64), per).reshape(1, T, 48, 128, 128)
    cap_conv = np.repeat(np.arange(3 + T, dtype=np.float64), C).reshape(1, 3 + T, C)
    s_conv = s.with_(n_qk_heads=1, n_v_heads=1, d_k=1, d_v=6)     # 2*1*1 + 6 = 8 conv channels
    rows = _golden_rows()
    assert len(rows) == 15
    for trim, acc, commit_n, byte_off, first, last in rows:
        Cf = s.conv_channels
        st, _, status = oracle.rollback(s, [trim], np.full((1, 48, 128, 128), -1.0),
                                        np.zeros((1, 3, Cf)), cap_state, np.zeros((1, 3 + T, Cf)))
        assert status[0] == 0
        assert np.all(st == acc)                                  # state <- capture[accepted_idx]
        assert acc * per * 4 == byte_off                          # the page's byte offset
        _, cs, _ = oracle.rollback(s_conv, [trim], np.zeros((1, 1, 6, 1)), np.zeros((1, 3, C)),
                                   np.zeros((1, T, 1, 6, 1)), cap_conv)
        assert list(cs[0, :, 0]) == list(range(first, last + 1))  # conv rows commit_n..commit_n+2
        assert commit_n == acc + 1


def test_rollback_trim_zero_and_out_of_range():
    s = small_shape(n_slots=4)
    x = make_inputs(s, seed=14).as_f64()
    res = oracle.verify(s, x)
    trim = [0, s.n_tokens, -1, 2]
    st, cs, status = oracle.rollback(s, trim, res["state"], res["conv_state"], res["cap_state"], res["cap_conv"])
    assert list(status) == [0, 1, 1, 0]
    for b in (0, 1, 2):                                           # untouched
        assert np.array_equal(st[b], res["state"][b]) and np.array_equal(cs[b], res["conv_state"][b])
    assert np.array_equal(st[3], res["cap_state"][3, s.n_tokens - 1 - 2])


@pytest.mark.parametrize("name", ["tiny", "pin"])
def test_rollback_equals_prefix_rerun(name):
    """Rolling back `trim` positions equals running only the accepted prefix from the
    pre-verify state (state and conv state), for every trim."""
    s = WORKLOADS["tiny"] if name == "tiny" else small_shape(n_tokens=6)
    inp = make_inputs(s, seed=21)
    x = inp.as_f64()
    res = oracle.verify(s, x)
    T = s.n_tokens
    for trim in range(T):
        st, cs, status = oracle.rollback(s, [trim] * s.n_slots, res["state"], res["conv_state"],
                                         res["cap_state"], res["cap_conv"])
        assert np.all(status == 0)
        pre = oracle.verify(s, x, capture=False, n_tokens=T - trim)
        assert np.allclose(st, pre["state"], rtol=1e-12, atol=1e-14)
        assert np.array_equal(cs, pre["conv_state"])
        assert np.allclose(res["out"][:, :T - trim], pre["out"], rtol=1e-12, atol=1e-14)


def test_lazy_commit_equals_capture_rollback():
    """Lazy capture keeps only the pre-batch state and re-runs the accepted prefix; it
    must land on the state the per-position capture holds for the same trim (the
    state after token t does not depend on the tokens after it), slot by slot."""
    s = small_shape(n_slots=5, n_tokens=6)
    x = make_inputs(s, seed=23).as_f64()
    res = oracle.verify(s, x)
    trim = [0, 5, 2, 6, -1]                                    # last two are refused
    st, cs, status = oracle.commit_lazy(s, x, trim)
    rst, rcs, rstatus = oracle.rollback(s, trim, res["state"], res["conv_state"], res["cap_state"],
                                        res["cap_conv"])
    np.testing.assert_array_equal(status, [0, 0, 0, 1, 1])
    np.testing.assert_array_equal(status, rstatus)
    for b in range(3):
        np.testing.assert_allclose(st[b], rst[b], rtol=1e-12, atol=1e-14)
        np.testing.assert_array_equal(cs[b], rcs[b])
    for b in (3, 4):                                           # refused: the pre-batch state
        np.testing.assert_array_equal(st[b], x["state"][b])
        np.testing.assert_array_equal(cs[b], x["conv_state"][b])


# --------------------------------------------------------------------------
# chunkwise form vs sequential form (two algorithms)
# --------------------------------------------------------------------------

@pytest.mark.parametrize("T,chunk", [(9, 1), (9, 4), (10, 3), (16, 8), (37, 64), (70, 16)])
def test_chunked_form_matches_sequential(T, chunk):
    s = small_shape(n_slots=2, n_tokens=T)
    x = make_inputs(s, seed=31).as_f64()
    seq = oracle.verify(s, x, capture=False)
    chk = oracle.prefill_chunked(s, x, chunk)
    scale = np.abs(seq["state"]).max()
    assert np.abs(chk["state"] - seq["state"]).max() <= 1e-10 * scale
    assert np.abs(chk["out"] - seq["out"]).max() <= 1e-10 * np.abs(seq["out"]).max()
    assert np.array_equal(chk["conv_state"], seq["conv_state"])


def test_chunked_form_long_sequence_realistic_dims():
    s = small_shape(n_slots=1, n_qk_heads=1, n_v_heads=2, d_k=32, d_v=32, n_tokens=300)
    x = make_inputs(s, seed=32).as_f64()
    seq = oracle.verify(s, x, capture=False)
    chk = oracle.prefill_chunked(s, x, 64)
    assert np.abs(chk["state"] - seq["state"]).max() <= 1e-10 * np.abs(seq["state"]).max()
    assert np.abs(chk["out"] - seq["out"]).max() <= 1e-10 * np.abs(seq["out"]).max()


# ---------------------------------------------------------------------------
# tree (DDTree) verify: token t runs from its parent's state; pinned to the
# chain verify (itself pinned above) through root-to-node paths
# ---------------------------------------------------------------------------

from workloads.synth import make_parents, tree_accept  # noqa: E402


def _path(par, t):
    """Nodes on the path root -> t (token indices, in order)."""
    p = []
    while t >= 0:
        p.append(t)
        t = par[t]
    return p[::-1]


def _tokens(x, s, nodes):
    """The chain-verify inputs of slot s whose tokens are `nodes`, in that order."""
    y = dict(x)
    for k in ("qkv", "z", "alpha", "beta_raw"):
        y[k] = x[k][s:s + 1, nodes]
    y["state"] = x["state"][s:s + 1]
    y["conv_state"] = x["conv_state"][s:s + 1]
    return y


def test_tree_with_chain_parents_is_the_chain_verify():
    s = small_shape(n_slots=2, n_tokens=6)
    x = make_inputs(s).as_f64()
    par = make_parents(s, "chain")
    tr = oracle.verify_tree(s, x, par)
    ch = oracle.verify(s, x, capture=True)
    np.testing.assert_array_equal(tr["cap_state"], ch["cap_state"])
    np.testing.assert_array_equal(tr["out"], ch["out"])
    for t in range(s.n_tokens):            # conv state after t = window rows t+1 .. t+3
        np.testing.assert_array_equal(tr["cap_conv"][:, t], ch["cap_conv"][:, t + 1:t + 4])


@pytest.mark.parametrize("kind", ["random", "star", "spine"])
def test_tree_node_equals_chain_verify_of_its_root_path(kind):
    # every node's capture, conv state and output equal a chain verify run over the tokens
    # on its path from the root: parent state, ancestor conv window and the continuation of
    # the window into the old conv state past the root all enter this check
    s = small_shape(n_slots=2, n_tokens=9, seed=7)
    x = make_inputs(s).as_f64()
    par = make_parents(s, kind, seed=8)
    tr = oracle.verify_tree(s, x, par)
    for b in range(s.n_slots):
        for t in range(s.n_tokens):
            nodes = _path(par[b], t)
            one = s.with_(n_slots=1, n_tokens=len(nodes))
            ref = oracle.verify(one, _tokens(x, b, nodes), capture=False)
            np.testing.assert_allclose(tr["cap_state"][b, t], ref["state"][0], rtol=1e-12, atol=1e-12)
            np.testing.assert_allclose(tr["cap_conv"][b, t], ref["conv_state"][0], rtol=0, atol=0)
            np.testing.assert_allclose(tr["out"][b, t], ref["out"][0, -1], rtol=1e-12, atol=1e-12)


def test_tree_leaves_state_and_conv_state_alone():
    s = small_shape(n_slots=1, n_tokens=5)
    x = make_inputs(s).as_f64()
    st0, cs0 = x["state"].copy(), x["conv_state"].copy()
    oracle.verify_tree(s, x, make_parents(s, "random", seed=3))
    np.testing.assert_array_equal(x["state"], st0)
    np.testing.assert_array_equal(x["conv_state"], cs0)


def test_tree_rejects_parents_out_of_token_order():
    s = small_shape(n_slots=1, n_tokens=4)
    x = make_inputs(s).as_f64()
    for bad in ([-1, 1, 0, 1], [-1, 0, -2, 1], [0, 0, 1, 2]):
        with pytest.raises(ValueError):
            oracle.verify_tree(s, x, np.array([bad], dtype=np.int32))


def test_tree_rollback_moves_to_the_accepted_node():
    s = small_shape(n_slots=4, n_tokens=6, seed=9)
    x = make_inputs(s).as_f64()
    par = make_parents(s, "random", seed=10)
    tr = oracle.verify_tree(s, x, par)
    accept = np.array([-1, 0, 5, 6], dtype=np.int32)            # none, first, last, out of range
    st, cs, status = oracle.rollback_tree(s, accept, x["state"], x["conv_state"], tr["cap_state"], tr["cap_conv"])
    np.testing.assert_array_equal(status, [0, 0, 0, 1])
    np.testing.assert_array_equal(st[0], x["state"][0])
    np.testing.assert_array_equal(cs[0], x["conv_state"][0])
    np.testing.assert_array_equal(st[1], tr["cap_state"][1, 0])
    np.testing.assert_array_equal(cs[2], tr["cap_conv"][2, 5])
    np.testing.assert_array_equal(st[3], x["state"][3])          # refused: untouched
    # the accepted node's state is the chain verify of its root path
    nodes = _path(par[2], 5)
    ref = oracle.verify(s.with_(n_slots=1, n_tokens=len(nodes)), _tokens(x, 2, nodes), capture=False)
    np.testing.assert_allclose(st[2], ref["state"][0], rtol=1e-12, atol=1e-12)
    np.testing.assert_array_equal(cs[2], ref["conv_state"][0])
    assert tree_accept(s, par).shape == (s.n_slots,)


# --------------------------------------------------------------------------
# projections around the block
# --------------------------------------------------------------------------

def test_projection_is_the_row_dot_product_by_brute_force():
    """project(a, w)[m, n] = sum_k a[m, k] w[n, k]: explicit loops on a tiny
    non-square case catch a transposed operand."""
    rng = np.random.default_rng(3)
    a, w = rng.normal(size=(3, 5)), rng.normal(size=(4, 5))
    got = oracle.project(a, w)
    assert got.shape == (3, 4)
    for m in range(3):
        for n in range(4):
            assert abs(got[m, n] - sum(a[m, k] * w[n, k] for k in range(5))) < 1e-12


def test_layer_with_identity_projections_is_the_block():
    """With n_embd = C + H_v d_v + 2 H_v and w_in = I, the hidden input is the
    activation matrix itself: the layer must equal ``verify`` on its column
    blocks taken in the order qkv | z | alpha | beta_raw; with w_out = I
    (n_embd' = H_v d_v) y is the block's output."""
    s = small_shape(n_tokens=4)
    x = make_inputs(s, seed=41).as_f64()
    N = s.conv_channels + s.value_dim + 2 * s.n_v_heads
    hidden = np.concatenate([x["qkv"], x["z"], x["alpha"], x["beta_raw"]], axis=-1)
    assert hidden.shape[-1] == N
    r = oracle.layer_verify(s, x, hidden, np.eye(N), np.eye(s.value_dim), store_bf16=False)
    ref = oracle.verify(s, x)
    np.testing.assert_array_equal(r["act"], hidden)
    for k in ("out", "state", "conv_state", "cap_state"):
        np.testing.assert_array_equal(r[k], ref[k])
    np.testing.assert_array_equal(r["y"], ref["out"])
    # a swapped block order (z before qkv) is a different layer
    sw = np.concatenate([x["z"], x["qkv"], x["alpha"], x["beta_raw"]], axis=-1)
    assert not np.allclose(oracle.layer_verify(s, x, sw, np.eye(N), np.eye(s.value_dim), store_bf16=False)["out"],
                           ref["out"])


def test_bf16_rounding_matches_the_bit_rounding_of_the_generator():
    """round_bf16 (frexp / rint) against the generator's independent f32 -> bf16
    bit rounding on fp32 values (where rounding fp64 directly and rounding the
    same fp32 value agree), including exact ties, which go to the even
    neighbour: 1 + 2^-8 -> 1, 1 + 3 2^-8 -> 1 + 2^-6."""
    from workloads.synth import bf16_bits_to_f64, to_bf16_bits
    rng = np.random.default_rng(5)
    v = np.concatenate([rng.normal(size=20000) * 10.0 ** rng.integers(-6, 6, size=20000),
                        [1 + 2 ** -8, 1 + 3 * 2 ** -8, -(1 + 2 ** -8), 2.0 ** -100, 0.0, 3.0]]).astype(np.float32)
    np.testing.assert_array_equal(oracle.round_bf16(v.astype(np.float64)), bf16_bits_to_f64(to_bf16_bits(v)))
    assert oracle.round_bf16(np.array([1 + 2 ** -8]))[0] == 1.0
    assert oracle.round_bf16(np.array([1 + 3 * 2 ** -8]))[0] == 1 + 2 ** -6
