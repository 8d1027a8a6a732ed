"""The C-ABI library: loads, exports every symbol the header declares, and
rejects bad arguments on the host before any CUDA call (no GPU needed)."""
import ctypes
import os
import re

import pytest

import gated_deltanet_verify_gb300 as gdn

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared_functions():
    names = set()
    inc = os.path.join(ROOT, "include")
    for f in os.listdir(inc):
        if not f.endswith(".h"):
            continue
        text = open(os.path.join(inc, f)).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        for m in re.finditer(r"^\s*(?:const\s+)?[A-Za-z_][\w\s\*]*?\b(gdn_\w+)\s*\(", text, flags=re.M):
            names.add(m.group(1))
    return names


@pytest.fixture(scope="module")
def lib():
    import __graft_entry__
    __graft_entry__.build_library()
    return gdn.lib()


def test_header_declares_the_boundary():
    names = _declared_functions()
    for n in ("gdn_verify_forward", "gdn_rollback", "gdn_prefill_chunked", "gdn_prefill_workspace_bytes",
              "gdn_last_error"):
        assert n in names
    assert set(names) <= set(gdn.EXPORTED_SYMBOLS)


def _doc_block(name):
    """The comment block that documents a declaration: the last /* ... */ before it with nothing but
    other declarations in between."""
    text = open(os.path.join(ROOT, "include", "gdn_verify.h")).read()
    m = re.search(r"^(?![ \t]*(?:/\*|\*))[^\n]*\b" + name + r"\s*\(", text, flags=re.M)
    assert m, name
    before = text[:m.start()]
    i = before.rfind("/*")
    return before[i:before.index("*/", i) + 2]


# the calls of the boundary, each with the page and the section (or the function on it) that defines it
BOUNDARY = {
    "gdn_verify_forward": ("internal.h", "ssm_intermediate"),
    "gdn_rollback": ("qwen35_target.rs", "rollback_kv"),
    "gdn_prefill_chunked": ("internal.h", "create_target_cache"),
    "gdn_prefill_workspace_bytes": ("internal.h", "create_target_cache"),
    "gdn_last_error": ("internal.h", "set_last_error"),
}


@pytest.mark.parametrize("name", sorted(BOUNDARY))
def test_boundary_calls_cite_their_passage(name):
    page, section = BOUNDARY[name]
    doc = _doc_block(name)
    assert page in doc and section in doc, (name, doc)


def test_static_scratch_size_matches_the_header(lib):
    text = open(os.path.join(ROOT, "include", "gdn_verify.h")).read()
    m = re.search(r"#define\s+GDN_PREFILL_STATIC_SCRATCH_BYTES\s+\(\(size_t\)(\d+)\s*<<\s*(\d+)\)", text)
    assert m
    assert gdn.prefill_static_scratch_bytes() == int(m.group(1)) << int(m.group(2))


def test_library_exports_every_declared_symbol(lib):
    for n in _declared_functions():
        assert hasattr(lib, n), n
    assert "sm_103a" in gdn.gdn_version()


def _dims(**kw):
    base = dict(n_slots=1, n_qk_heads=2, n_v_heads=4, d_k=32, d_v=32, n_tokens=4, act_dtype=gdn.GDN_F32)
    base.update(kw)
    return gdn.make_dims(**base)


A = 0x10000          # fake, 16-byte aligned device addresses: never dereferenced (validation fails first)


def _params(**kw):
    p = dict(conv_w=A, A_log=A, dt_bias=A, norm_w=A)
    p.update(kw)
    return gdn.layer_params(**p)


def _call_verify(d, p=None, **kw):
    bufs = dict(qkv=A, z=A, alpha=A, beta_raw=A, state=A, conv_state=A, cap_state=None, cap_conv=None, out=A)
    bufs.update(kw)
    return gdn.lib().gdn_verify_forward(ctypes.byref(d), ctypes.byref(p or _params()), bufs["qkv"], bufs["z"],
                                        bufs["alpha"], bufs["beta_raw"], bufs["state"], bufs["conv_state"],
                                        bufs["cap_state"], bufs["cap_conv"], bufs["out"], None, None)


@pytest.mark.parametrize("kw,code", [
    (dict(conv_width=3), gdn.GDN_ERR_SHAPE),
    (dict(n_v_heads=5), gdn.GDN_ERR_SHAPE),
    (dict(d_k=48), gdn.GDN_ERR_SHAPE),
    (dict(d_v=12), gdn.GDN_ERR_SHAPE),
    (dict(n_tokens=0), gdn.GDN_ERR_SHAPE),
    (dict(n_tokens=65), gdn.GDN_ERR_SHAPE),
    (dict(n_slots=0), gdn.GDN_ERR_SHAPE),
    (dict(act_dtype=7), gdn.GDN_ERR_DTYPE),
    (dict(n_qk_heads=1, n_v_heads=32), gdn.GDN_ERR_SHAPE),     # 32 value heads per key head: no cluster fits
])
def test_verify_rejects_bad_dims(lib, kw, code):
    assert _call_verify(_dims(**kw)) == code
    assert gdn.gdn_last_error() != ""


def test_verify_rejects_null_and_misaligned(lib):
    assert _call_verify(_dims(), qkv=None) == gdn.GDN_ERR_ARG
    assert _call_verify(_dims(), p=_params(A_log=None)) == gdn.GDN_ERR_ARG
    assert _call_verify(_dims(), state=A + 4) == gdn.GDN_ERR_ALIGN
    assert _call_verify(_dims(), cap_state=A + 8) == gdn.GDN_ERR_ALIGN
    assert _call_verify(_dims(), p=_params(norm_w=A + 4)) == gdn.GDN_ERR_ALIGN
    assert "aligned" in gdn.gdn_last_error()
    assert gdn.lib().gdn_verify_forward(None, ctypes.byref(_params()), *([A] * 6), None, None, A, None,
                                        None) == gdn.GDN_ERR_ARG


def test_rollback_host_validation(lib):
    d = _dims()
    L = gdn.lib()
    assert L.gdn_rollback(ctypes.byref(d), A, A, A, None, A, None, None) == gdn.GDN_ERR_NO_CAPTURE
    assert L.gdn_rollback(ctypes.byref(d), A, A, A, A, None, None, None) == gdn.GDN_ERR_NO_CAPTURE
    assert L.gdn_rollback(ctypes.byref(d), None, A, A, A, A, None, None) == gdn.GDN_ERR_ARG
    assert L.gdn_rollback(ctypes.byref(d), A, A + 4, A, A, A, None, None) == gdn.GDN_ERR_ALIGN
    assert L.gdn_rollback(ctypes.byref(_dims(conv_width=2)), A, A, A, A, A, None, None) == gdn.GDN_ERR_SHAPE


def test_prefill_host_validation(lib):
    d = _dims(n_tokens=300)
    L = gdn.lib()
    ws = gdn.gdn_prefill_workspace_bytes(d)
    assert gdn.gdn_prefill_workspace_bytes(_dims(conv_width=5)) == 0
    args = [A] * 7
    rc = L.gdn_prefill_chunked(ctypes.byref(_dims(d_k=40)), ctypes.byref(_params()), *args, None, 0, None, None)
    assert rc == gdn.GDN_ERR_SHAPE
    if ws > 0:
        rc = L.gdn_prefill_chunked(ctypes.byref(d), ctypes.byref(_params()), *args, None, 0, None, None)
        assert rc == gdn.GDN_ERR_WORKSPACE
        rc = L.gdn_prefill_chunked(ctypes.byref(d), ctypes.byref(_params()), *args, A + 16, ws, None, None)
        assert rc == gdn.GDN_ERR_ALIGN


def test_binding_raises_on_error(lib):
    with pytest.raises(gdn.GdnError) as ei:
        gdn.gdn_rollback(_dims(), A, A, A, None, A, stream=0)
    assert ei.value.status == gdn.GDN_ERR_NO_CAPTURE


def test_step_io_layout(lib):
    d = _dims(n_slots=3, n_tokens=5, act_dtype=gdn.GDN_BF16)
    io = gdn.gdn_step_io_layout(d)
    C, V, H, M = 2 * 2 * 32 + 4 * 32, 4 * 32, 4, 15
    up = lambda n: -(-n // 256) * 256
    assert (io.qkv, io.z) == (0, up(M * C * 2))
    assert io.alpha == io.z + up(M * V * 2) and io.beta_raw == io.alpha + up(M * H * 2)
    assert io.trim == io.beta_raw + up(M * H * 2) and io.in_bytes == io.trim + up(3 * 4)
    assert io.out_bytes == up(M * V * 2)
    assert all(v % 256 == 0 for v in (io.qkv, io.z, io.alpha, io.beta_raw, io.trim, io.in_bytes))


def test_step_host_validation(lib):
    d = _dims()
    io = gdn.gdn_step_io_layout(d)
    L = gdn.lib()

    def call(rf=0, h_in=A, d_io=A, n=None):
        return L.gdn_verify_step_host(ctypes.byref(d), ctypes.byref(_params()), rf, h_in, A, d_io,
                                      io.in_bytes + io.out_bytes if n is None else n, A, A, A, A, None, None)

    assert call(h_in=None) == gdn.GDN_ERR_ARG
    assert call(n=io.in_bytes) == gdn.GDN_ERR_WORKSPACE
    assert call(d_io=A + 16) == gdn.GDN_ERR_ALIGN
    assert call(rf=2) == gdn.GDN_ERR_ARG


def test_lazy_and_rolled_host_validation(lib):
    d = _dims()
    L = gdn.lib()
    p = ctypes.byref(_params())
    # commit without trims; lazy verify with a pending batch but no pending activations
    assert L.gdn_commit_lazy(ctypes.byref(d), p, None, A, A, A, A, A, None, None) == gdn.GDN_ERR_ARG
    assert L.gdn_verify_lazy(ctypes.byref(d), p, A, None, A, A, A, A, A, A, A, A, A, None, None) == gdn.GDN_ERR_ARG
    # the rolled verify needs the previous captures and trims
    assert L.gdn_verify_after_rollback(ctypes.byref(d), p, A, A, A, A, A, A, A, None, A, A, None,
                                       None) == gdn.GDN_ERR_NO_CAPTURE
    assert L.gdn_verify_after_rollback(ctypes.byref(d), p, None, A, A, A, A, A, A, A, A, A, None,
                                       None) == gdn.GDN_ERR_ARG


def test_projection_host_validation(lib):
    L = gdn.lib()
    bf = _dims(n_v_heads=8, act_dtype=gdn.GDN_BF16)
    w = gdn.ProjWeights(64, A, A)
    need = gdn.gdn_layer_workspace_bytes(bf, 64)
    M, ld = 4, gdn.gdn_proj_in_ld(bf)
    assert ld % 8 == 0 and ld >= 2 * 2 * 32 + 8 * 32 + 8 * 32 + 16
    assert need >= M * ld * 2 + M * 8 * 32 * 2

    def call(d=bf, ww=w, n=need, ws=A):
        return L.gdn_layer_verify(ctypes.byref(d), ctypes.byref(_params()), ctypes.byref(ww), A, A, A, None, None,
                                  A, ws, n, None, None)

    assert call(d=_dims(n_v_heads=8)) == gdn.GDN_ERR_DTYPE                          # f32 activations
    assert call(ww=gdn.ProjWeights(60, A, A)) == gdn.GDN_ERR_SHAPE                  # n_embd not a multiple of 8
    assert call(d=_dims(n_v_heads=4, act_dtype=gdn.GDN_BF16)) == gdn.GDN_ERR_SHAPE  # H_v not a multiple of 8
    assert call(n=need - 1) == gdn.GDN_ERR_WORKSPACE
    assert call(ws=A + 16) == gdn.GDN_ERR_ALIGN
    assert call(ww=gdn.ProjWeights(64, None, A)) == gdn.GDN_ERR_ARG
