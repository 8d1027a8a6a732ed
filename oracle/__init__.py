"""Python access to the fp64 CPU oracle (``gdn_oracle.c``).

TEST INFRASTRUCTURE ONLY: the tests, the smoke check and the bench's CPU
baseline / reference arm use this module; the CUDA library and its binding
never import it.  All arrays crossing into C are contiguous float64 (int32 for
trims); the layouts are those documented in ``gdn_oracle.h``.
"""
from __future__ import annotations

import ctypes
import os
import platform
import subprocess
from typing import Dict, Optional

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gdn_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")

_lib = None


def _foreign() -> bool:
    """True if the existing library was built for another host architecture."""
    marker = _LIB + ".machine"
    return not os.path.exists(marker) or open(marker).read().strip() != platform.machine()


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (plain C11, IEEE fp64, no FMA contraction)."""
    if force or _foreign() or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < max(
            os.path.getmtime(_SRC), os.path.getmtime(os.path.join(_HERE, "gdn_oracle.h"))):
        tmp = _LIB + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-shared", "-fPIC",
               "-pthread", "-o", tmp, _SRC, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB)
        with open(_LIB + ".machine", "w") as fh:
            fh.write(platform.machine() + "\n")
    return _LIB


class _Dims(ctypes.Structure):
    _fields_ = [("n_slots", ctypes.c_int), ("n_qk_heads", ctypes.c_int), ("n_v_heads", ctypes.c_int),
                ("d_k", ctypes.c_int), ("d_v", ctypes.c_int), ("conv_width", ctypes.c_int),
                ("n_tokens", ctypes.c_int), ("rms_eps", ctypes.c_double), ("l2_eps", ctypes.c_double),
                ("q_scale", ctypes.c_double)]


_D = ctypes.POINTER(ctypes.c_double)


def configure(L: ctypes.CDLL) -> ctypes.CDLL:
    """Declare the C signatures on a loaded oracle library."""
    L.gdno_softplus.restype = ctypes.c_double
    L.gdno_softplus.argtypes = [ctypes.c_double]
    L.gdno_gates.argtypes = [ctypes.c_double] * 4 + [_D, _D]
    L.gdno_l2norm.argtypes = [ctypes.c_int, _D, ctypes.c_double, _D]
    L.gdno_conv_silu.argtypes = [ctypes.c_int] * 3 + [_D, _D, _D]
    L.gdno_delta_step.argtypes = [ctypes.c_int, ctypes.c_int, _D, _D, _D, _D,
                                         ctypes.c_double, ctypes.c_double, ctypes.c_double, _D]
    L.gdno_rmsnorm_gate.argtypes = [ctypes.c_int, _D, _D, _D, ctypes.c_double, _D]
    L.gdno_verify.argtypes = [ctypes.POINTER(_Dims)] + [_D] * 13 + [ctypes.c_void_p, ctypes.c_int]
    L.gdno_prefill_chunked.argtypes = ([ctypes.POINTER(_Dims), ctypes.c_int] + [_D] * 11 +
                                              [ctypes.c_void_p, ctypes.c_int])
    L.gdno_rollback.argtypes = [ctypes.POINTER(_Dims), ctypes.c_void_p] + [_D] * 4 + [ctypes.c_void_p]
    L.gdno_verify_tree.argtypes = ([ctypes.POINTER(_Dims), ctypes.c_void_p] + [_D] * 13 +
                                   [ctypes.c_void_p, ctypes.c_int])
    L.gdno_rollback_tree.argtypes = [ctypes.POINTER(_Dims), ctypes.c_void_p] + [_D] * 4 + [ctypes.c_void_p]
    return L


def lib():
    global _lib
    if _lib is None:
        _lib = configure(ctypes.CDLL(build()))
    return _lib


def _p(a: Optional[np.ndarray]):
    if a is None:
        return None
    assert a.dtype == np.float64 and a.flags["C_CONTIGUOUS"], (a.dtype, a.flags)
    return a.ctypes.data_as(_D)


def _f64(a) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=np.float64)


def dims(shape, n_tokens: Optional[int] = None, rms_eps=1e-6, l2_eps=1e-6, q_scale=1.0) -> _Dims:
    return _Dims(shape.n_slots, shape.n_qk_heads, shape.n_v_heads, shape.d_k, shape.d_v,
                 shape.conv_width, shape.n_tokens if n_tokens is None else n_tokens,
                 rms_eps, l2_eps, q_scale)


# ---- stages ---------------------------------------------------------------

def softplus(x: float) -> float:
    return lib().gdno_softplus(float(x))


def gates(A_log, dt_bias, alpha, beta_raw):
    g, b = ctypes.c_double(), ctypes.c_double()
    lib().gdno_gates(float(A_log), float(dt_bias), float(alpha), float(beta_raw),
                     ctypes.byref(g), ctypes.byref(b))
    return g.value, b.value


def l2norm(x, eps=1e-6):
    x = _f64(x)
    out = np.empty_like(x)
    lib().gdno_l2norm(x.size, _p(x), eps, _p(out))
    return out


def conv_silu(conv_w, win):
    conv_w, win = _f64(conv_w), _f64(win)
    W, C = conv_w.shape
    T = win.shape[0] - (W - 1)
    y = np.empty((T, C))
    lib().gdno_conv_silu(W, T, C, _p(conv_w), _p(win), _p(y))
    return y


def delta_step(S, k, v, q, g, beta, q_scale=1.0):
    """S is logical [d_k][d_v]; returns (S_new, o)."""
    S = _f64(S).copy()
    dk, dv = S.shape
    o = np.empty(dv)
    lib().gdno_delta_step(dk, dv, _p(S), _p(_f64(k)), _p(_f64(v)), _p(_f64(q)),
                          float(g), float(beta), float(q_scale), _p(o))
    return S, o


def rmsnorm_gate(o, z, w, eps=1e-6):
    o, z, w = _f64(o), _f64(z), _f64(w)
    out = np.empty_like(o)
    lib().gdno_rmsnorm_gate(o.size, _p(o), _p(z), _p(w), eps, _p(out))
    return out


# ---- composites -----------------------------------------------------------

def _mask(head_mask, n_v_heads):
    if head_mask is None:
        return None, None
    m = np.zeros(n_v_heads, dtype=np.uint8)
    m[np.asarray(head_mask)] = 1
    return m, m.ctypes.data_as(ctypes.c_void_p)


def verify(shape, x: Dict[str, np.ndarray], capture: bool = True, n_tokens: Optional[int] = None,
           head_mask=None, n_threads: int = 1, q_scale: float = 1.0,
           rms_eps: float = 1e-6, l2_eps: float = 1e-6) -> Dict[str, np.ndarray]:
    """Run the verify forward on fp64 copies of ``x`` (the dict of
    ``Inputs.as_f64()``).  ``n_tokens`` < shape.n_tokens runs only the first
    tokens (the prefix re-run).  Returns state, conv_state, out and, with
    ``capture``, cap_state / cap_conv."""
    s = shape
    T = s.n_tokens if n_tokens is None else n_tokens
    d = dims(s, T, rms_eps, l2_eps, q_scale)
    B, C, Hv, dk, dv, W = s.n_slots, s.conv_channels, s.n_v_heads, s.d_k, s.d_v, s.conv_width
    assert x["qkv"].shape[:1] == (B,) and x["qkv"].shape[2] == C and x["qkv"].shape[1] >= T
    assert x["z"].shape[2] == Hv * dv and x["alpha"].shape[2] == Hv and x["beta_raw"].shape[2] == Hv
    assert x["state"].shape == (B, Hv, dv, dk) and x["conv_state"].shape == (B, W - 1, C)
    assert x["conv_w"].shape == (W, C) and x["A_log"].shape == (Hv,) and x["norm_w"].shape == (dv,)
    qkv = _f64(x["qkv"][:, :T])
    z = _f64(x["z"][:, :T])
    alpha = _f64(x["alpha"][:, :T])
    beta_raw = _f64(x["beta_raw"][:, :T])
    state = _f64(x["state"]).copy()
    conv_state = _f64(x["conv_state"]).copy()
    out = np.zeros((B, T, Hv * dv))
    cap_state = np.zeros((B, T, Hv, dv, dk)) if capture else None
    cap_conv = np.zeros((B, W - 1 + T, C)) if capture else None
    m, mp = _mask(head_mask, Hv)
    rc = lib().gdno_verify(ctypes.byref(d), _p(_f64(x["conv_w"])), _p(_f64(x["A_log"])),
                           _p(_f64(x["dt_bias"])), _p(_f64(x["norm_w"])), _p(qkv), _p(z),
                           _p(alpha), _p(beta_raw), _p(state), _p(conv_state), _p(cap_state),
                           _p(cap_conv), _p(out), mp, int(n_threads))
    assert rc == 0
    res = {"state": state, "conv_state": conv_state, "out": out}
    if capture:
        res["cap_state"], res["cap_conv"] = cap_state, cap_conv
    return res


def rollback(shape, trim, state, conv_state, cap_state, cap_conv, n_tokens: Optional[int] = None):
    """Returns (state, conv_state, slot_status) after rolling back copies."""
    T = shape.n_tokens if n_tokens is None else n_tokens
    d = dims(shape, T)
    s = shape
    B, C = s.n_slots, s.conv_channels
    assert np.shape(state) == (B, s.n_v_heads, s.d_v, s.d_k)
    assert np.shape(conv_state) == (B, s.conv_width - 1, C)
    assert np.shape(cap_state) == (B, T, s.n_v_heads, s.d_v, s.d_k)
    assert np.shape(cap_conv) == (B, s.conv_width - 1 + T, C)
    assert np.size(trim) == B
    st, cs = _f64(state).copy(), _f64(conv_state).copy()
    tr = np.ascontiguousarray(trim, dtype=np.int32)
    status = np.zeros(shape.n_slots, dtype=np.int32)
    lib().gdno_rollback(ctypes.byref(d), tr.ctypes.data_as(ctypes.c_void_p), _p(st), _p(cs),
                        _p(_f64(cap_state)), _p(_f64(cap_conv)), status.ctypes.data_as(ctypes.c_void_p))
    return st, cs, status


def commit_lazy(shape, x: Dict[str, np.ndarray], trim, head_mask=None, n_threads: int = 1,
                q_scale: float = 1.0, rms_eps: float = 1e-6, l2_eps: float = 1e-6):
    """Lazy capture's commit (the byte-saving alternative to per-position capture,
    after the single-snapshot rollback of the lucebox-hub page internal.h,
    "Target cache"): the verify kept only the state before the batch, so each
    slot s re-runs its accepted tokens 0 .. T-1-trim[s] from it.  No arithmetic
    of its own: the state after a token is defined by the recurrence over the
    tokens up to it, so this is ``verify`` of one slot over that prefix.  A trim
    outside [0, T-1] leaves the slot as it was with status 1 (as ``rollback``).
    Returns (state, conv_state, slot_status)."""
    s = shape
    T, B = s.n_tokens, s.n_slots
    tr = np.asarray(trim).reshape(-1)
    assert tr.shape == (B,)
    state, conv_state = _f64(x["state"]).copy(), _f64(x["conv_state"]).copy()
    status = np.zeros(B, dtype=np.int32)
    one = s.with_(n_slots=1)
    per_slot = ("qkv", "z", "alpha", "beta_raw", "state", "conv_state")
    for b in range(B):
        if not 0 <= int(tr[b]) < T:
            status[b] = 1
            continue
        xb = {k: (v[b:b + 1] if k in per_slot else v) for k, v in x.items()}
        r = verify(one, xb, capture=False, n_tokens=T - int(tr[b]), head_mask=head_mask, n_threads=n_threads,
                   q_scale=q_scale, rms_eps=rms_eps, l2_eps=l2_eps)
        state[b], conv_state[b] = r["state"][0], r["conv_state"][0]
    return state, conv_state, status


def project(a, w):
    """One projection of the block's neighbours (internal.h, Target weights: the
    TargetLayer GDN projections wqkv, wqkv_gate, ssm_alpha, ssm_beta, ssm_out):
    a [..., K] times the weight w [N, K] (output rows, K contiguous), in fp64:
    result[..., n] = sum_k a[..., k] w[n, k]."""
    a, w = _f64(a), _f64(w)
    assert a.shape[-1] == w.shape[1]
    return np.matmul(a, w.T)


def split_projected(shape, act):
    """The input projection's columns, in the order of its weight rows: qkv
    (C channels [q | k | v]), z (H_v*d_v), alpha (H_v), beta_raw (H_v)."""
    C, V, H = shape.conv_channels, shape.n_v_heads * shape.d_v, shape.n_v_heads
    assert act.shape[-1] == C + V + 2 * H
    return {"qkv": act[..., :C], "z": act[..., C:C + V], "alpha": act[..., C + V:C + V + H],
            "beta_raw": act[..., C + V + H:]}


def round_bf16(a):
    """Round fp64 values to the nearest bf16 (8 significant bits), ties to even,
    returned as fp64: with a = m 2^e, 1/2 <= |m| < 1, the result is
    rint(m 2^8) 2^(e-8) (numpy's rint rounds half to even).  Normal range only
    (bf16 shares fp32's exponent range; no overflow or subnormals occur here)."""
    m, e = np.frexp(_f64(a))
    return np.ldexp(np.rint(m * 256.0), e - 8)


def layer_verify(shape, x: Dict[str, np.ndarray], hidden, w_in, w_out, n_threads: int = 1,
                 store_bf16: bool = True, **kw):
    """The block with its projections: act = hidden @ w_in^T, split into qkv, z,
    alpha, beta_raw; ``verify`` (with capture) on them from x's parameters and
    states; y = out @ w_out^T.  All arithmetic in fp64; with ``store_bf16`` the
    two matrices the layer stores between its steps (act and the block's out,
    held in the activation dtype) are rounded to bf16 there.  Returns verify's
    dict (out unrounded) plus act (unrounded) and y."""
    act = project(hidden, w_in)
    stored = round_bf16(act) if store_bf16 else act
    xin = dict(x)
    xin.update({k: np.ascontiguousarray(v) for k, v in split_projected(shape, stored).items()})
    r = verify(shape, xin, n_threads=n_threads, **kw)
    r["act"] = act
    r["y"] = project(round_bf16(r["out"]) if store_bf16 else r["out"], w_out)
    return r


def verify_tree(shape, x: Dict[str, np.ndarray], parent, head_mask=None, n_threads: int = 1,
                q_scale: float = 1.0, rms_eps: float = 1e-6, l2_eps: float = 1e-6) -> Dict[str, np.ndarray]:
    """Tree (DDTree) verify of shape.n_tokens tokens per slot; parent is [B][T] int
    (parent[s][t] in [-1, t-1]).  state / conv_state are not changed; returns
    out, cap_state [B][T][H_v][d_v][d_k] and cap_conv [B][T][W-1][C]."""
    s = shape
    T = s.n_tokens
    d = dims(s, T, rms_eps, l2_eps, q_scale)
    B, C, Hv, dk, dv, W = s.n_slots, s.conv_channels, s.n_v_heads, s.d_k, s.d_v, s.conv_width
    par = np.ascontiguousarray(parent, dtype=np.int32)
    assert par.shape == (B, T)
    assert x["state"].shape == (B, Hv, dv, dk) and x["conv_state"].shape == (B, W - 1, C)
    out = np.zeros((B, T, Hv * dv))
    cap_state = np.zeros((B, T, Hv, dv, dk))
    cap_conv = np.zeros((B, T, W - 1, C))
    m, mp = _mask(head_mask, Hv)
    rc = lib().gdno_verify_tree(ctypes.byref(d), par.ctypes.data_as(ctypes.c_void_p), _p(_f64(x["conv_w"])),
                                _p(_f64(x["A_log"])), _p(_f64(x["dt_bias"])), _p(_f64(x["norm_w"])),
                                _p(_f64(x["qkv"][:, :T])), _p(_f64(x["z"][:, :T])), _p(_f64(x["alpha"][:, :T])),
                                _p(_f64(x["beta_raw"][:, :T])), _p(_f64(x["state"])), _p(_f64(x["conv_state"])),
                                _p(cap_state), _p(cap_conv), _p(out), mp, int(n_threads))
    if rc == -2:
        raise ValueError("parent is not a tree in token order")
    assert rc == 0
    return {"out": out, "cap_state": cap_state, "cap_conv": cap_conv}


def rollback_tree(shape, accept, state, conv_state, cap_state, cap_conv):
    """Returns (state, conv_state, slot_status) after moving copies to the accepted nodes."""
    s = shape
    T = s.n_tokens
    d = dims(s, T)
    B, C = s.n_slots, s.conv_channels
    assert np.shape(cap_state) == (B, T, s.n_v_heads, s.d_v, s.d_k)
    assert np.shape(cap_conv) == (B, T, s.conv_width - 1, C)
    st, cs = _f64(state).copy(), _f64(conv_state).copy()
    acc = np.ascontiguousarray(accept, dtype=np.int32)
    assert acc.shape == (B,)
    status = np.zeros(B, dtype=np.int32)
    lib().gdno_rollback_tree(ctypes.byref(d), acc.ctypes.data_as(ctypes.c_void_p), _p(st), _p(cs),
                             _p(_f64(cap_state)), _p(_f64(cap_conv)), status.ctypes.data_as(ctypes.c_void_p))
    return st, cs, status


def prefill_chunked(shape, x: Dict[str, np.ndarray], chunk: int, n_tokens: Optional[int] = None,
                    head_mask=None, n_threads: int = 1, q_scale: float = 1.0,
                    rms_eps: float = 1e-6, l2_eps: float = 1e-6) -> Dict[str, np.ndarray]:
    s = shape
    T = s.n_tokens if n_tokens is None else n_tokens
    d = dims(s, T, rms_eps, l2_eps, q_scale)
    state = _f64(x["state"]).copy()
    conv_state = _f64(x["conv_state"]).copy()
    out = np.zeros((s.n_slots, T, s.n_v_heads * s.d_v))
    m, mp = _mask(head_mask, s.n_v_heads)
    rc = lib().gdno_prefill_chunked(ctypes.byref(d), int(chunk), _p(_f64(x["conv_w"])),
                                    _p(_f64(x["A_log"])), _p(_f64(x["dt_bias"])),
                                    _p(_f64(x["norm_w"])), _p(_f64(x["qkv"][:, :T])),
                                    _p(_f64(x["z"][:, :T])), _p(_f64(x["alpha"][:, :T])),
                                    _p(_f64(x["beta_raw"][:, :T])), _p(state), _p(conv_state),
                                    _p(out), mp, int(n_threads))
    assert rc == 0
    return {"state": state, "conv_state": conv_state, "out": out}
