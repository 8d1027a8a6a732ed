"""Python binding of the GB300 Gated DeltaNet verify library (C ABI in
``include/gdn_verify.h``).

Argument marshalling only: every step runs in the CUDA kernels of
``libgdn_verify.so``.  Buffers are passed as torch tensors (their
``data_ptr()``) or raw integer device addresses; the stream defaults to
torch's current stream.  If the library has not been built the import of
``lib()`` raises -- there is no CPU fallback.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libgdn_verify.so")

GDN_OK = 0
GDN_ERR_ARG = 1
GDN_ERR_SHAPE = 2
GDN_ERR_ALIGN = 3
GDN_ERR_DTYPE = 4
GDN_ERR_TRIM_RANGE = 5
GDN_ERR_NO_CAPTURE = 6
GDN_ERR_LAUNCH = 7
GDN_ERR_TIMEOUT = 8
GDN_ERR_WORKSPACE = 9
GDN_ERR_TREE = 10
GDN_ERR_BOUNDS = 11
STATUS_NAMES = {0: "GDN_OK", 1: "GDN_ERR_ARG", 2: "GDN_ERR_SHAPE", 3: "GDN_ERR_ALIGN", 4: "GDN_ERR_DTYPE",
                5: "GDN_ERR_TRIM_RANGE", 6: "GDN_ERR_NO_CAPTURE", 7: "GDN_ERR_LAUNCH", 8: "GDN_ERR_TIMEOUT",
                9: "GDN_ERR_WORKSPACE", 10: "GDN_ERR_TREE",
                11: "GDN_ERR_BOUNDS"}

GDN_F32 = 0
GDN_BF16 = 1

EXPORTED_SYMBOLS = ("gdn_verify_forward", "gdn_verify_tree", "gdn_rollback", "gdn_rollback_tree",
                    "gdn_rollback_layers", "gdn_rollback_tree_layers", "gdn_verify_after_rollback", "gdn_verify_lazy", "gdn_commit_lazy", "gdn_step_io_layout",
                    "gdn_verify_step_host", "gdn_proj_in_ld", "gdn_layer_workspace_bytes",
                    "gdn_project_in", "gdn_project_out", "gdn_layer_verify", "gdn_prefill_workspace_bytes",
                    "gdn_prefill_chunked", "gdn_prefill_chunked_static", "gdn_prefill_static_scratch_bytes",
                    "gdn_last_error", "gdn_version")


class GdnError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{STATUS_NAMES.get(status, status)}: {message}")
        self.status = status


class Dims(ctypes.Structure):
    _fields_ = [("n_slots", ctypes.c_int), ("n_qk_heads", ctypes.c_int), ("n_v_heads", ctypes.c_int),
                ("d_k", ctypes.c_int), ("d_v", ctypes.c_int), ("conv_width", ctypes.c_int),
                ("n_tokens", ctypes.c_int), ("act_dtype", ctypes.c_int), ("rms_eps", ctypes.c_float),
                ("l2_eps", ctypes.c_float), ("q_scale", ctypes.c_float)]


class LayerParams(ctypes.Structure):
    _fields_ = [("conv_w", ctypes.c_void_p), ("A_log", ctypes.c_void_p), ("dt_bias", ctypes.c_void_p),
                ("norm_w", ctypes.c_void_p)]


class StepIO(ctypes.Structure):
    _fields_ = [("qkv", ctypes.c_size_t), ("z", ctypes.c_size_t), ("alpha", ctypes.c_size_t),
                ("beta_raw", ctypes.c_size_t), ("trim", ctypes.c_size_t), ("in_bytes", ctypes.c_size_t),
                ("out_bytes", ctypes.c_size_t)]


class ProjWeights(ctypes.Structure):
    _fields_ = [("n_embd", ctypes.c_int), ("w_in", ctypes.c_void_p), ("w_out", ctypes.c_void_p)]


def make_dims(n_slots: int, n_qk_heads: int, n_v_heads: int, d_k: int, d_v: int, n_tokens: int,
              act_dtype: int = GDN_BF16, conv_width: int = 4, rms_eps: float = 1e-6,
              l2_eps: float = 1e-6, q_scale: float = 1.0) -> Dims:
    return Dims(n_slots, n_qk_heads, n_v_heads, d_k, d_v, conv_width, n_tokens, act_dtype,
                rms_eps, l2_eps, q_scale)


_lib = None


def lib() -> ctypes.CDLL:
    """The loaded CUDA library; raises if it was not built (no fallback)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it with "
                               "`python -c 'import __graft_entry__ as g; g.build()'`")
        L = ctypes.CDLL(LIB_PATH)
        vp, ip = ctypes.c_void_p, ctypes.c_int
        L.gdn_verify_forward.argtypes = [ctypes.POINTER(Dims), ctypes.POINTER(LayerParams)] + [vp] * 11
        L.gdn_verify_forward.restype = ip
        L.gdn_rollback.argtypes = [ctypes.POINTER(Dims)] + [vp] * 7
        L.gdn_rollback.restype = ip
        L.gdn_verify_tree.argtypes = [ctypes.POINTER(Dims), ctypes.POINTER(LayerParams)] + [vp] * 12
        L.gdn_verify_tree.restype = ip
        L.gdn_rollback_tree.argtypes = [ctypes.POINTER(Dims)] + [vp] * 7
        L.gdn_rollback_tree.restype = ip
        L.gdn_rollback_layers.argtypes = [ctypes.POINTER(Dims), ctypes.c_int] + [vp] * 7
        L.gdn_rollback_layers.restype = ip
        L.gdn_rollback_tree_layers.argtypes = [ctypes.POINTER(Dims), ctypes.c_int] + [vp] * 7
        L.gdn_rollback_tree_layers.restype = ip
        L.gdn_verify_after_rollback.argtypes = [ctypes.POINTER(Dims), ctypes.POINTER(LayerParams)] + [vp] * 12
        L.gdn_verify_after_rollback.restype = ip
        L.gdn_step_io_layout.argtypes = [ctypes.POINTER(Dims), ctypes.POINTER(StepIO)]
        L.gdn_step_io_layout.restype = ip
        L.gdn_verify_step_host.argtypes = ([ctypes.POINTER(Dims), ctypes.POINTER(LayerParams), ip] + [vp] * 3 +
                                           [ctypes.c_size_t] + [vp] * 6)
        L.gdn_verify_step_host.restype = ip
        L.gdn_verify_lazy.argtypes = [ctypes.POINTER(Dims), ctypes.POINTER(LayerParams)] + [vp] * 13
        L.gdn_verify_lazy.restype = ip
        L.gdn_commit_lazy.argtypes = [ctypes.POINTER(Dims), ctypes.POINTER(LayerParams)] + [vp] * 8
        L.gdn_commit_lazy.restype = ip
        L.gdn_proj_in_ld.argtypes = [ctypes.POINTER(Dims)]
        L.gdn_proj_in_ld.restype = ctypes.c_longlong
        L.gdn_layer_workspace_bytes.argtypes = [ctypes.POINTER(Dims), ip]
        L.gdn_layer_workspace_bytes.restype = ctypes.c_size_t
        for fn in (L.gdn_project_in, L.gdn_project_out):
            fn.argtypes = [ctypes.POINTER(Dims), ctypes.POINTER(ProjWeights), vp, vp, vp, ctypes.c_size_t, vp]
            fn.restype = ip
        L.gdn_layer_verify.argtypes = ([ctypes.POINTER(Dims), ctypes.POINTER(LayerParams),
                                        ctypes.POINTER(ProjWeights)] + [vp] * 7 + [ctypes.c_size_t, vp, vp])
        L.gdn_layer_verify.restype = ip
        L.gdn_prefill_workspace_bytes.argtypes = [ctypes.POINTER(Dims)]
        L.gdn_prefill_workspace_bytes.restype = ctypes.c_size_t
        L.gdn_prefill_chunked.argtypes = ([ctypes.POINTER(Dims), ctypes.POINTER(LayerParams)] + [vp] * 8 +
                                          [ctypes.c_size_t, vp, vp])
        L.gdn_prefill_chunked.restype = ip
        L.gdn_prefill_chunked_static.argtypes = [ctypes.POINTER(Dims), ctypes.POINTER(LayerParams)] + [vp] * 9
        L.gdn_prefill_chunked_static.restype = ip
        L.gdn_prefill_static_scratch_bytes.argtypes = []
        L.gdn_prefill_static_scratch_bytes.restype = ctypes.c_size_t
        L.gdn_last_error.restype = ctypes.c_char_p
        L.gdn_version.restype = ctypes.c_char_p
        _lib = L
    return _lib


def _ptr(x) -> Optional[int]:
    if x is None:
        return None
    if isinstance(x, int):
        return x
    return x.data_ptr()


def _stream(stream) -> Optional[int]:
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check(rc: int) -> None:
    if rc != GDN_OK:
        raise GdnError(rc, gdn_last_error())


def layer_params(conv_w, A_log, dt_bias, norm_w) -> LayerParams:
    return LayerParams(_ptr(conv_w), _ptr(A_log), _ptr(dt_bias), _ptr(norm_w))


def gdn_last_error() -> str:
    return lib().gdn_last_error().decode()


def gdn_version() -> str:
    return lib().gdn_version().decode()


def gdn_verify_forward(dims: Dims, params: LayerParams, qkv, z, alpha, beta_raw, state, conv_state,
                       cap_state=None, cap_conv=None, out=None, d_status=None, stream=None) -> None:
    _check(lib().gdn_verify_forward(ctypes.byref(dims), ctypes.byref(params), _ptr(qkv), _ptr(z),
                                    _ptr(alpha), _ptr(beta_raw), _ptr(state), _ptr(conv_state),
                                    _ptr(cap_state), _ptr(cap_conv), _ptr(out), _ptr(d_status),
                                    _stream(stream)))


def gdn_rollback(dims: Dims, d_trim, state, conv_state, cap_state, cap_conv, d_status=None,
                 stream=None) -> None:
    _check(lib().gdn_rollback(ctypes.byref(dims), _ptr(d_trim), _ptr(state), _ptr(conv_state),
                              _ptr(cap_state), _ptr(cap_conv), _ptr(d_status), _stream(stream)))


def pointer_table(tensors, device="cuda"):
    """A DEVICE int64 array of the tensors' data pointers (the tables gdn_rollback_layers reads)."""
    import torch
    return torch.tensor([t.data_ptr() for t in tensors], dtype=torch.int64, device=device)


def gdn_rollback_layers(dims: Dims, n_layers: int, d_trim, tab_state, tab_conv_state, tab_cap_state, tab_cap_conv,
                        d_status=None, stream=None) -> None:
    """gdn_rollback of n_layers layers in one launch; the tab_* are device pointer tables (pointer_table)."""
    _check(lib().gdn_rollback_layers(ctypes.byref(dims), int(n_layers), _ptr(d_trim), _ptr(tab_state),
                                     _ptr(tab_conv_state), _ptr(tab_cap_state), _ptr(tab_cap_conv), _ptr(d_status),
                                     _stream(stream)))


def gdn_rollback_tree_layers(dims: Dims, n_layers: int, d_accept, tab_state, tab_conv_state, tab_cap_state,
                             tab_cap_conv, d_status=None, stream=None) -> None:
    """gdn_rollback_tree of n_layers layers in one launch; the tab_* are device pointer tables (pointer_table)."""
    _check(lib().gdn_rollback_tree_layers(ctypes.byref(dims), int(n_layers), _ptr(d_accept), _ptr(tab_state),
                                          _ptr(tab_conv_state), _ptr(tab_cap_state), _ptr(tab_cap_conv),
                                          _ptr(d_status), _stream(stream)))


def gdn_verify_tree(dims: Dims, params: LayerParams, qkv, z, alpha, beta_raw, d_parent, state, conv_state,
                    cap_state, cap_conv, out, d_status=None, stream=None) -> None:
    _check(lib().gdn_verify_tree(ctypes.byref(dims), ctypes.byref(params), _ptr(qkv), _ptr(z), _ptr(alpha),
                                 _ptr(beta_raw), _ptr(d_parent), _ptr(state), _ptr(conv_state), _ptr(cap_state),
                                 _ptr(cap_conv), _ptr(out), _ptr(d_status), _stream(stream)))


def gdn_rollback_tree(dims: Dims, d_accept, state, conv_state, cap_state, cap_conv, d_status=None,
                      stream=None) -> None:
    _check(lib().gdn_rollback_tree(ctypes.byref(dims), _ptr(d_accept), _ptr(state), _ptr(conv_state),
                                   _ptr(cap_state), _ptr(cap_conv), _ptr(d_status), _stream(stream)))


def gdn_verify_after_rollback(dims: Dims, params: LayerParams, d_prev_trim, qkv, z, alpha, beta_raw, state,
                              conv_state, cap_state, cap_conv, out, d_status=None, stream=None) -> None:
    """Verify starting from what gdn_rollback(d_prev_trim) would leave, read from the
    previous batch's captures (which this call overwrites)."""
    _check(lib().gdn_verify_after_rollback(ctypes.byref(dims), ctypes.byref(params), _ptr(d_prev_trim), _ptr(qkv),
                                           _ptr(z), _ptr(alpha), _ptr(beta_raw), _ptr(state), _ptr(conv_state),
                                           _ptr(cap_state), _ptr(cap_conv), _ptr(out), _ptr(d_status),
                                           _stream(stream)))


def gdn_step_io_layout(dims: Dims) -> StepIO:
    io = StepIO()
    _check(lib().gdn_step_io_layout(ctypes.byref(dims), ctypes.byref(io)))
    return io


def gdn_verify_step_host(dims: Dims, params: LayerParams, rollback_first: int, h_in, h_out, d_io, d_io_bytes: int,
                         state, conv_state, cap_state, cap_conv, d_status=None, stream=None) -> None:
    """One verify step from host memory (packed pinned input block, output block)."""
    _check(lib().gdn_verify_step_host(ctypes.byref(dims), ctypes.byref(params), int(rollback_first), _ptr(h_in),
                                      _ptr(h_out), _ptr(d_io), int(d_io_bytes), _ptr(state), _ptr(conv_state),
                                      _ptr(cap_state), _ptr(cap_conv), _ptr(d_status), _stream(stream)))


def gdn_verify_lazy(dims: Dims, params: LayerParams, qkv, z, alpha, beta_raw, state, conv_state, out,
                    d_status=None, stream=None, prev_trim=None, prev_qkv=None, prev_alpha=None,
                    prev_beta_raw=None) -> None:
    """Outputs-only verify; with prev_trim (device int32[B]) it first commits the
    pending batch (prev_qkv, prev_alpha, prev_beta_raw) into state / conv_state."""
    _check(lib().gdn_verify_lazy(ctypes.byref(dims), ctypes.byref(params), _ptr(prev_trim), _ptr(prev_qkv),
                                 _ptr(prev_alpha), _ptr(prev_beta_raw), _ptr(qkv), _ptr(z), _ptr(alpha),
                                 _ptr(beta_raw), _ptr(state), _ptr(conv_state), _ptr(out), _ptr(d_status),
                                 _stream(stream)))


def gdn_commit_lazy(dims: Dims, params: LayerParams, d_trim, qkv, alpha, beta_raw, state, conv_state,
                    d_status=None, stream=None) -> None:
    _check(lib().gdn_commit_lazy(ctypes.byref(dims), ctypes.byref(params), _ptr(d_trim), _ptr(qkv),
                                 _ptr(alpha), _ptr(beta_raw), _ptr(state), _ptr(conv_state), _ptr(d_status),
                                 _stream(stream)))


def proj_weights(n_embd: int, w_in, w_out) -> "ProjWeights":
    """The projection weights of one layer (device tensors or pointers): w_in
    [C + H_v*d_v + 2*H_v][n_embd] (wqkv, wqkv_gate, ssm_alpha, ssm_beta rows),
    w_out [n_embd][H_v*d_v]; both bf16."""
    return ProjWeights(int(n_embd), _ptr(w_in), _ptr(w_out))


def gdn_proj_in_ld(dims: Dims) -> int:
    return int(lib().gdn_proj_in_ld(ctypes.byref(dims)))


def gdn_layer_workspace_bytes(dims: Dims, n_embd: int) -> int:
    return int(lib().gdn_layer_workspace_bytes(ctypes.byref(dims), int(n_embd)))


def gdn_project_in(dims: Dims, w: "ProjWeights", x, act, workspace, ws_bytes: int, stream=None) -> None:
    _check(lib().gdn_project_in(ctypes.byref(dims), ctypes.byref(w), _ptr(x), _ptr(act), _ptr(workspace),
                                int(ws_bytes), _stream(stream)))


def gdn_project_out(dims: Dims, w: "ProjWeights", out, y, workspace, ws_bytes: int, stream=None) -> None:
    _check(lib().gdn_project_out(ctypes.byref(dims), ctypes.byref(w), _ptr(out), _ptr(y), _ptr(workspace),
                                 int(ws_bytes), _stream(stream)))


def gdn_layer_verify(dims: Dims, params: LayerParams, w: "ProjWeights", x, state, conv_state, cap_state, cap_conv,
                     y, workspace, ws_bytes: int, d_status=None, stream=None) -> None:
    _check(lib().gdn_layer_verify(ctypes.byref(dims), ctypes.byref(params), ctypes.byref(w), _ptr(x), _ptr(state),
                                  _ptr(conv_state), _ptr(cap_state), _ptr(cap_conv), _ptr(y), _ptr(workspace),
                                  int(ws_bytes), _ptr(d_status), _stream(stream)))


def gdn_prefill_workspace_bytes(dims: Dims) -> int:
    return int(lib().gdn_prefill_workspace_bytes(ctypes.byref(dims)))


def gdn_prefill_chunked(dims: Dims, params: LayerParams, qkv, z, alpha, beta_raw, state, conv_state, out,
                        workspace=None, ws_bytes: int = 0, d_status=None, stream=None) -> None:
    _check(lib().gdn_prefill_chunked(ctypes.byref(dims), ctypes.byref(params), _ptr(qkv), _ptr(z),
                                     _ptr(alpha), _ptr(beta_raw), _ptr(state), _ptr(conv_state), _ptr(out),
                                     _ptr(workspace), ctypes.c_size_t(ws_bytes), _ptr(d_status),
                                     _stream(stream)))


def prefill_static_scratch_bytes() -> int:
    """Size of the library's built-in prefill scratch (GDN_PREFILL_STATIC_SCRATCH_BYTES), read from the library."""
    return int(lib().gdn_prefill_static_scratch_bytes())


def gdn_prefill_chunked_static(dims: Dims, params: LayerParams, qkv, z, alpha, beta_raw, state, conv_state, out,
                               d_status=None, stream=None) -> None:
    """gdn_prefill_chunked with the library's built-in scratch instead of a workspace."""
    _check(lib().gdn_prefill_chunked_static(ctypes.byref(dims), ctypes.byref(params), _ptr(qkv), _ptr(z),
                                            _ptr(alpha), _ptr(beta_raw), _ptr(state), _ptr(conv_state),
                                            _ptr(out), _ptr(d_status), _stream(stream)))
