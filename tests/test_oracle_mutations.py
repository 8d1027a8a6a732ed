"""The pins are strong enough: plant a plausible mistake in a copy of the C
oracle (on the CPU), build it, and check that at least one pin fails.  The
real oracle is untouched; the mutated library only replaces it for the
duration of one test."""
import ctypes
import os
import shutil
import subprocess

import pytest

import oracle
from tests import test_oracle_pins as pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "gdn_oracle.c")
HDR = os.path.join(os.path.dirname(oracle.__file__), "gdn_oracle.h")

# (name, original text, planted mistake)
MUTATIONS = [
    ("drop_decay", "for (int j = 0; j < dv; ++j) S[(size_t)i * dv + j] *= g;",
     "for (int j = 0; j < dv; ++j) S[(size_t)i * dv + j] *= 1.0;"),
    ("update_sign", "S[(size_t)i * dv + j] += beta * k[i] * (v[j] - u[j]);",
     "S[(size_t)i * dv + j] -= beta * k[i] * (v[j] - u[j]);"),
    ("read_with_q", "for (int i = 0; i < dk; ++i) acc += S[(size_t)i * dv + j] * k[i];",
     "for (int i = 0; i < dk; ++i) acc += S[(size_t)i * dv + j] * q[i];"),
    ("state_read_transposed", "for (int i = 0; i < dk; ++i) acc += S[(size_t)i * dv + j] * k[i];",
     "for (int i = 0; i < dk; ++i) acc += S[(size_t)j * dk + i] * k[i];"),
    ("conv_taps_reversed", "acc += conv_w[(size_t)j * C + c] * win[(size_t)(t + j) * C + c];",
     "acc += conv_w[(size_t)(W - 1 - j) * C + c] * win[(size_t)(t + j) * C + c];"),
    ("no_silu_after_conv", "y[(size_t)t * C + c] = silu(acc);", "y[(size_t)t * C + c] = acc;"),
    ("rollback_off_by_one", "const int accepted_idx = T - 1 - trim[s];",
     "const int accepted_idx = T - trim[s] - (trim[s] == 1);"),
    ("conv_rows_off_by_one", "const int commit_n = accepted_idx + 1;", "const int commit_n = accepted_idx;"),
    ("tiled_head_map", "const int r = d->n_v_heads / d->n_qk_heads, kh = h / r;",
     "const int r = d->n_v_heads / d->n_qk_heads, kh = h % d->n_qk_heads; (void)r;"),
    ("no_l2_norm", "double inv = 1.0 / sqrt(ss + eps);\n    for (int i = 0; i < n; ++i) xhat[i] = x[i] * inv;",
     "double inv = 1.0 + 0.0 * ss * eps;\n    for (int i = 0; i < n; ++i) xhat[i] = x[i] * inv;"),
    ("rms_eps_outside_root", "double inv = 1.0 / sqrt(ss / dv + eps);", "double inv = 1.0 / (sqrt(ss / dv) + eps);"),
    ("gate_sign", "return -exp(A_log) * gdno_softplus(alpha + dt_bias);",
     "return exp(A_log) * gdno_softplus(alpha + dt_bias) * 1e-3;"),
    ("softplus_without_log1p", "return log1p(exp(x));", "return exp(x);"),
    ("beta_sign", "*beta = sigmoid(beta_raw);", "*beta = sigmoid(-beta_raw);"),
    ("q_scale_ignored", "o[j] = q_scale * acc;", "o[j] = acc;"),
    ("capture_before_update", "gdno_delta_step(dk, dv, S, kn, v, qn, g, beta, d->q_scale, o);\n        if (J->cap_state)\n            store_state(d, J->cap_state + (st * Hv + h) * dv * dk, S);",
     "if (J->cap_state)\n            store_state(d, J->cap_state + (st * Hv + h) * dv * dk, S);\n        gdno_delta_step(dk, dv, S, kn, v, qn, g, beta, d->q_scale, o);"),
    ("chunk_decay_ratio_inverted", "intra += qk * exp(logG[r] - logG[m]) * U[(size_t)m * dv + j];",
     "intra += qk * exp(logG[m] - logG[r]) * U[(size_t)m * dv + j];"),
    ("tree_ignores_parent_state", "if (p < 0) load_state(d, J->state, s, h, S);",
     "if (p < 0 || p >= 0) load_state(d, J->state, s, h, S);"),
    ("tree_window_stops_at_root", "anc = anc >= 0 ? parent[(size_t)s * T + anc] : anc - 1;",
     "anc = anc >= 0 ? parent[(size_t)s * T + anc] : -1;"),
    ("tree_window_follows_token_order", "anc = anc >= 0 ? parent[(size_t)s * T + anc] : anc - 1;",
     "anc = anc - 1;"),
]


def _pin_calls():
    """Every pin of test_oracle_pins, with its parametrisations expanded."""
    calls = []
    for name in dir(pins):
        if not name.startswith("test_"):
            continue
        fn = getattr(pins, name)
        marks = [m for m in getattr(fn, "pytestmark", []) if m.name == "parametrize"]
        if not marks:
            calls.append((name, fn, {}))
            continue
        argnames, values = marks[0].args[0], marks[0].args[1]
        argnames = [a.strip() for a in argnames.split(",")] if isinstance(argnames, str) else list(argnames)
        for v in values:
            v = v if isinstance(v, (tuple, list)) else (v,)
            calls.append((name, fn, dict(zip(argnames, v))))
    return calls


@pytest.mark.parametrize("name,old,new", MUTATIONS, ids=[m[0] for m in MUTATIONS])
def test_pins_catch_planted_mistake(name, old, new, tmp_path):
    src = open(SRC).read()
    assert old in src, f"mutation site for {name} not found"
    (tmp_path / "gdn_oracle.c").write_text(src.replace(old, new, 1))
    shutil.copy(HDR, tmp_path / "gdn_oracle.h")
    so = tmp_path / "libmut.so"
    subprocess.run(["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-shared", "-fPIC", "-pthread", "-o", str(so),
                    str(tmp_path / "gdn_oracle.c"), "-lm"], check=True)
    mutated = oracle.configure(ctypes.CDLL(str(so)))
    saved = oracle.lib()
    oracle._lib = mutated
    failed = []
    try:
        for pname, fn, kw in _pin_calls():
            try:
                fn(**kw)
            except AssertionError:
                failed.append(pname)
            except Exception:          # a crash of the mutated oracle's arithmetic also counts as caught
                failed.append(pname)
    finally:
        oracle._lib = saved
    assert failed, f"no pin caught the planted mistake {name}"
