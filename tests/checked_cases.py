"""Cases run through both the ordinary and the bounds-checked library (see
test_checked_gpu.py): every verify mode, the rollbacks and the layer step on
small seeded shapes.  ``python -m tests.checked_cases OUT.npz [all|lost_chunk|scratch_contexts]``
runs them on the checked library -- the test build, which also carries the
test hooks (the prefill's host-side fault injection, the static-scratch
address lookup) -- and saves the results and status words."""
import os
import sys

import numpy as np
import torch

import gated_deltanet_verify_gb300 as gdn
from tests.gpu_util import dims_of, params_of, upload
from workloads.device import act_host, empty_outputs, to_f64
from workloads.synth import Shape, make_inputs, make_parents, make_proj


def _shape(**kw):
    base = dict(name="chk", n_slots=3, n_qk_heads=2, n_v_heads=6, d_k=128, d_v=128, n_tokens=7, act="bf16", seed=71)
    base.update(kw)
    return Shape(**base)


def run_all() -> dict:
    torch.cuda.set_device(0)
    res = {}
    status = torch.zeros(1, dtype=torch.int32, device="cuda")

    def keep(prefix, **tensors):
        for k, v in tensors.items():
            res[f"{prefix}.{k}"] = to_f64(v)

    from tests.test_fuzz_shapes_gpu import supported_draws
    shapes = [("chain", _shape()), ("f32_dk32", _shape(d_k=32, d_v=32, act="f32", n_tokens=4)),
              ("dk64_r4", _shape(d_k=64, d_v=64, n_qk_heads=2, n_v_heads=8, n_tokens=5)),
              ("dv72_unequal", _shape(d_k=64, d_v=72, n_qk_heads=2, n_v_heads=4, n_tokens=6)),
              ("dv16_T40_one_warp", _shape(d_v=16, n_qk_heads=2, n_v_heads=8, n_tokens=40, act="f32"))]
    shapes += [(s.name, s) for s in supported_draws(4, 500)]      # random shapes the verify accepts
    for name, shape in shapes:
        x = upload(make_inputs(shape))
        o = empty_outputs(shape, "cuda")
        d = dims_of(shape)
        gdn.gdn_verify_forward(d, params_of(x), x["qkv"], x["z"], x["alpha"], x["beta_raw"], x["state"],
                               x["conv_state"], o["cap_state"], o["cap_conv"], o["out"], status)
        T = shape.n_tokens
        trims = torch.tensor([[0, min(2, T - 1), T - 1][b % 3] for b in range(shape.n_slots)], dtype=torch.int32,
                             device="cuda")
        gdn.gdn_rollback(d, trims, x["state"], x["conv_state"], o["cap_state"], o["cap_conv"], status)
        # the rolled verify from those captures, then a lazy verify committing that batch, then a commit
        y = upload(make_inputs(shape, seed=72))
        gdn.gdn_verify_after_rollback(d, params_of(x), trims, y["qkv"], y["z"], y["alpha"], y["beta_raw"],
                                      x["state"], x["conv_state"], o["cap_state"], o["cap_conv"], o["out"], status)
        keep(name, out=o["out"], cap_state=o["cap_state"], cap_conv=o["cap_conv"], state=x["state"],
             conv_state=x["conv_state"])
        lz = upload(make_inputs(shape, seed=73))
        out2 = empty_outputs(shape, "cuda", capture=False)["out"]
        gdn.gdn_verify_lazy(d, params_of(x), lz["qkv"], lz["z"], lz["alpha"], lz["beta_raw"], x["state"],
                            x["conv_state"], out2, status, prev_trim=trims, prev_qkv=y["qkv"], prev_alpha=y["alpha"],
                            prev_beta_raw=y["beta_raw"])
        gdn.gdn_commit_lazy(d, params_of(x), trims, lz["qkv"], lz["alpha"], lz["beta_raw"], x["state"],
                            x["conv_state"], status)
        keep(name + ".lazy", out=out2, state=x["state"], conv_state=x["conv_state"])
        # tree verify and the rollback to the accepted node
        xt = upload(make_inputs(shape, seed=74))
        ot = empty_outputs(shape, "cuda")
        cap_conv_t = torch.empty((shape.n_slots, shape.n_tokens, 3, shape.conv_channels), dtype=torch.float32,
                                 device="cuda")
        par = torch.from_numpy(make_parents(shape, "random", seed=75).astype(np.int32)).to("cuda")
        gdn.gdn_verify_tree(d, params_of(xt), xt["qkv"], xt["z"], xt["alpha"], xt["beta_raw"], par, xt["state"],
                            xt["conv_state"], ot["cap_state"], cap_conv_t, ot["out"], status)
        acc = torch.tensor([[-1, 0, T - 1][b % 3] for b in range(shape.n_slots)], dtype=torch.int32, device="cuda")
        gdn.gdn_rollback_tree(d, acc, xt["state"], xt["conv_state"], ot["cap_state"], cap_conv_t, status)
        keep(name + ".tree", out=ot["out"], cap_state=ot["cap_state"], cap_conv=cap_conv_t, state=xt["state"],
             conv_state=xt["conv_state"])
        # two layers verified, then rolled back in one launch from device pointer tables
        lay = []
        for li in range(2):
            xl = upload(make_inputs(shape, layer=li + 1))
            ol = empty_outputs(shape, "cuda")
            gdn.gdn_verify_forward(d, params_of(xl), xl["qkv"], xl["z"], xl["alpha"], xl["beta_raw"], xl["state"],
                                   xl["conv_state"], ol["cap_state"], ol["cap_conv"], ol["out"], status)
            lay.append((xl, ol))
        tabs = [gdn.pointer_table([xl["state"] for xl, _ in lay]), gdn.pointer_table([xl["conv_state"] for xl, _ in lay]),
                gdn.pointer_table([ol["cap_state"] for _, ol in lay]), gdn.pointer_table([ol["cap_conv"] for _, ol in lay])]
        gdn.gdn_rollback_layers(d, 2, trims, *tabs, status)
        for li, (xl, _) in enumerate(lay):
            keep(f"{name}.layers{li}", state=xl["state"], conv_state=xl["conv_state"])

    # the layer step with its projections
    shape = _shape(n_v_heads=8, d_k=64, d_v=64, n_embd=256)
    x = upload(make_inputs(shape))
    p = {k: act_host(v, shape).to("cuda") for k, v in make_proj(shape).items()}
    d = dims_of(shape)
    w = gdn.proj_weights(shape.n_embd, p["w_in"], p["w_out"])
    o = empty_outputs(shape, "cuda")
    ws_bytes = gdn.gdn_layer_workspace_bytes(d, shape.n_embd)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device="cuda")
    yv = torch.empty((shape.n_slots, shape.n_tokens, shape.n_embd), dtype=torch.bfloat16, device="cuda")
    gdn.gdn_layer_verify(d, params_of(x), w, p["x"], x["state"], x["conv_state"], o["cap_state"], o["cap_conv"], yv,
                         ws, ws_bytes, status)
    keep("layer", y=yv, cap_state=o["cap_state"], state=x["state"])
    torch.cuda.synchronize()
    res["status"] = np.array([int(status.item())])
    return res


LOST_CHUNK_SHAPE = Shape("prefill_small", n_slots=1, n_qk_heads=2, n_v_heads=6, d_k=128, d_v=128, n_tokens=300,
                         act="bf16", seed=46)


def _prefill(shape, x, status):
    d = dims_of(shape)
    ws_bytes = gdn.gdn_prefill_workspace_bytes(d)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device="cuda")
    out = torch.empty((shape.n_slots, shape.n_tokens, shape.n_v_heads * shape.d_v), dtype=torch.bfloat16,
                      device="cuda")
    gdn.gdn_prefill_chunked(d, params_of(x), x["qkv"], x["z"], x["alpha"], x["beta_raw"], x["state"],
                            x["conv_state"], out, ws, ws_bytes, status)
    torch.cuda.synchronize()
    return out


def run_lost_chunk() -> dict:
    """A fault injected on the host (test build only): with GDN_FAULT_DROP_CHUNK=2 the prefill never
    publishes chunk 2, the state CTA's bounded wait gives up and the call reports GDN_ERR_TIMEOUT; then a
    clean call on the same device."""
    torch.cuda.set_device(0)
    inp = make_inputs(LOST_CHUNK_SHAPE)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    os.environ["GDN_FAULT_DROP_CHUNK"] = "2"
    _prefill(LOST_CHUNK_SHAPE, upload(inp), status)
    first = int(status.item())
    del os.environ["GDN_FAULT_DROP_CHUNK"]
    status.zero_()
    x = upload(inp)
    out = _prefill(LOST_CHUNK_SHAPE, x, status)
    return {"status_dropped": np.array([first]), "status_clean": np.array([int(status.item())]),
            "state": to_f64(x["state"]), "out": to_f64(out)}


def run_scratch_contexts() -> dict:
    """The static-scratch address the library uses in the primary context, in a second context made
    current on the same device, and in the primary context again.  Only the address lookup runs in the
    second context (no kernel is launched there)."""
    import ctypes
    torch.cuda.set_device(0)
    torch.zeros(1, device="cuda")                      # the primary context is current
    L = gdn.lib()
    f = L.gdn_test_static_scratch_address
    f.restype = ctypes.c_void_p
    f.argtypes = []
    cu = ctypes.CDLL("libcuda.so.1")
    a0, a1 = f(), f()
    dev = ctypes.c_int()
    assert cu.cuCtxGetDevice(ctypes.byref(dev)) == 0
    ctx = ctypes.c_void_p()
    assert cu.cuCtxCreate_v2(ctypes.byref(ctx), 0, dev) == 0     # pushed: current on this thread
    b0, b1 = f(), f()
    popped = ctypes.c_void_p()
    assert cu.cuCtxPopCurrent_v2(ctypes.byref(popped)) == 0
    a2 = f()
    assert cu.cuCtxDestroy_v2(ctx) == 0
    return {"addr": np.array([a0 or 0, a1 or 0, b0 or 0, b1 or 0, a2 or 0], dtype=np.uint64)}


if __name__ == "__main__":
    from gated_deltanet_verify_gb300 import _build
    gdn.LIB_PATH = _build.CHECKED_LIB
    case = sys.argv[2] if len(sys.argv) > 2 else "all"
    r = {"all": run_all, "lost_chunk": run_lost_chunk, "scratch_contexts": run_scratch_contexts}[case]()
    r["version"] = np.frombuffer(gdn.gdn_version().encode(), dtype=np.uint8)
    np.savez(sys.argv[1], **r)
