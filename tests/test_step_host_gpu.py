"""gdn_verify_step_host (one verify step from a packed host block): the same
bits as the device-buffer calls it stands for, in both modes."""
import numpy as np
import pytest
import torch

import gated_deltanet_verify_gb300 as gdn
from tests.gpu_util import dims_of, params_of, run_verify, upload
from workloads.device import act_host, empty_outputs
from workloads.synth import Shape, make_inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()
    torch.cuda.set_device(0)


def _shape(**kw):
    base = dict(name="host_step", n_slots=3, n_qk_heads=2, n_v_heads=6, d_k=128, d_v=128, n_tokens=8, act="bf16",
                seed=91)
    base.update(kw)
    return Shape(**base)


def _packed(shape, inp, trims):
    io = gdn.gdn_step_io_layout(dims_of(shape))
    h = torch.zeros(io.in_bytes, dtype=torch.uint8).pin_memory()
    for off, t in ((io.qkv, act_host(inp.qkv, shape)), (io.z, act_host(inp.z, shape)),
                   (io.alpha, act_host(inp.alpha, shape)), (io.beta_raw, act_host(inp.beta_raw, shape)),
                   (io.trim, torch.tensor(trims, dtype=torch.int32))):
        b = t.contiguous().view(torch.uint8).reshape(-1)
        h[off:off + b.numel()].copy_(b)
    return io, h


def _random_shapes():
    from tests.test_fuzz_shapes_gpu import supported_draws
    return {s.name: s for s in supported_draws(3, 600)}


@pytest.mark.parametrize("act", ["bf16", "f32"] + list(_random_shapes()))
def test_host_step_equals_verify_then_rollback(act):
    # the fixed shape in both activation dtypes, and random shapes the verify accepts (the packed block's
    # section offsets then fall on odd sizes)
    shape = _random_shapes()[act] if act.startswith("fuzz") else _shape(act=act)
    inp = make_inputs(shape)
    trims = [[0, min(3, shape.n_tokens - 1), shape.n_tokens - 1][b % 3] for b in range(shape.n_slots)]
    # device-buffer calls
    xa = upload(inp)
    oa = run_verify(shape, xa)
    gdn.gdn_rollback(dims_of(shape), torch.tensor(trims, dtype=torch.int32, device="cuda"), xa["state"],
                     xa["conv_state"], oa["cap_state"], oa["cap_conv"])
    # the host step
    xb = upload(inp)
    ob = empty_outputs(shape, "cuda")
    io, h_in = _packed(shape, inp, trims)
    h_out = torch.empty(io.out_bytes, dtype=torch.uint8).pin_memory()
    d_io = torch.empty(io.in_bytes + io.out_bytes, dtype=torch.uint8, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    gdn.gdn_verify_step_host(dims_of(shape), params_of(xb), 0, h_in, h_out, d_io, d_io.numel(), xb["state"],
                             xb["conv_state"], ob["cap_state"], ob["cap_conv"], status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    nb = oa["out"].numel() * oa["out"].element_size()
    assert torch.equal(h_out[:nb].view(oa["out"].dtype).view(oa["out"].shape), oa["out"].cpu())
    for k in ("cap_state", "cap_conv"):
        assert torch.equal(oa[k], ob[k]), k
    assert torch.equal(xa["state"], xb["state"]) and torch.equal(xa["conv_state"], xb["conv_state"])


def test_host_step_rolled_equals_verify_after_rollback():
    shape = _shape()
    inp = make_inputs(shape)
    xa, xb = upload(inp), upload(inp)
    oa, ob = run_verify(shape, xa), run_verify(shape, xb)         # captures of a first batch
    nxt = make_inputs(shape, seed=92)
    trims = [5, 0, 2]
    ya = upload(nxt)
    gdn.gdn_verify_after_rollback(dims_of(shape), params_of(xa), torch.tensor(trims, dtype=torch.int32, device="cuda"),
                                  ya["qkv"], ya["z"], ya["alpha"], ya["beta_raw"], xa["state"], xa["conv_state"],
                                  oa["cap_state"], oa["cap_conv"], oa["out"])
    io, h_in = _packed(shape, nxt, trims)
    h_out = torch.empty(io.out_bytes, dtype=torch.uint8).pin_memory()
    d_io = torch.empty(io.in_bytes + io.out_bytes, dtype=torch.uint8, device="cuda")
    gdn.gdn_verify_step_host(dims_of(shape), params_of(xb), 1, h_in, h_out, d_io, d_io.numel(), xb["state"],
                             xb["conv_state"], ob["cap_state"], ob["cap_conv"])
    torch.cuda.synchronize()
    nb = oa["out"].numel() * oa["out"].element_size()
    assert torch.equal(h_out[:nb].view(oa["out"].dtype).view(oa["out"].shape), oa["out"].cpu())
    assert torch.equal(oa["cap_state"], ob["cap_state"])
    assert torch.equal(xa["state"], xb["state"]) and torch.equal(xa["conv_state"], xb["conv_state"])


def test_host_step_checks_the_staging_size():
    shape = _shape()
    inp = make_inputs(shape)
    x = upload(inp)
    o = empty_outputs(shape, "cuda")
    io, h_in = _packed(shape, inp, [0, 0, 0])
    h_out = torch.empty(io.out_bytes, dtype=torch.uint8).pin_memory()
    d_io = torch.empty(io.in_bytes + io.out_bytes, dtype=torch.uint8, device="cuda")
    with pytest.raises(gdn.GdnError) as ei:
        gdn.gdn_verify_step_host(dims_of(shape), params_of(x), 0, h_in, h_out, d_io, io.in_bytes, x["state"],
                                 x["conv_state"], o["cap_state"], o["cap_conv"])
    assert ei.value.status == gdn.GDN_ERR_WORKSPACE
