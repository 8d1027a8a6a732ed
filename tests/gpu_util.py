"""Helpers for the GPU tests: run the CUDA path through the C ABI on seeded
inputs and read the results back as fp64 numpy arrays."""
import os
import subprocess
import sys
from typing import Dict, Optional

import numpy as np
import torch

import gated_deltanet_verify_gb300 as gdn
from workloads.device import empty_outputs, to_device, to_f64
from workloads.synth import Inputs, Shape


def dims_of(shape: Shape, n_tokens: Optional[int] = None, q_scale: float = 1.0) -> gdn.Dims:
    return gdn.make_dims(shape.n_slots, shape.n_qk_heads, shape.n_v_heads, shape.d_k, shape.d_v,
                         shape.n_tokens if n_tokens is None else n_tokens,
                         gdn.GDN_BF16 if shape.act == "bf16" else gdn.GDN_F32, q_scale=q_scale)


def params_of(x: Dict[str, torch.Tensor]) -> gdn.LayerParams:
    return gdn.layer_params(x["conv_w"], x["A_log"], x["dt_bias"], x["norm_w"])


def prefix(x: Dict[str, torch.Tensor], n_tokens: int) -> Dict[str, torch.Tensor]:
    """The first n_tokens positions of every slot's activations (contiguous copies)."""
    y = dict(x)
    for k in ("qkv", "z", "alpha", "beta_raw"):
        y[k] = x[k][:, :n_tokens].clone(memory_format=torch.contiguous_format)
    y["state"] = x["state"].clone()
    y["conv_state"] = x["conv_state"].clone()
    return y


def run_verify(shape: Shape, x: Dict[str, torch.Tensor], capture: bool = True, n_tokens: Optional[int] = None,
               q_scale: float = 1.0, status: Optional[torch.Tensor] = None) -> Dict[str, torch.Tensor]:
    """Verify forward on device tensors x (state / conv_state updated in place)."""
    T = shape.n_tokens if n_tokens is None else n_tokens
    o = empty_outputs(shape, x["qkv"].device, capture=capture, n_tokens=T)
    gdn.gdn_verify_forward(dims_of(shape, T, q_scale), params_of(x), x["qkv"], x["z"], x["alpha"], x["beta_raw"],
                           x["state"], x["conv_state"], o.get("cap_state"), o.get("cap_conv"), o["out"], status)
    torch.cuda.synchronize()
    o["state"] = x["state"]
    o["conv_state"] = x["conv_state"]
    return o


def as_f64(d: Dict[str, torch.Tensor]) -> Dict[str, np.ndarray]:
    return {k: to_f64(v) for k, v in d.items()}


def upload(inp: Inputs, device="cuda") -> Dict[str, torch.Tensor]:
    return to_device(inp, device)


ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def run_test_build(tmp_path, case: str) -> dict:
    """Run one case of tests/checked_cases.py in a child process on the test build."""
    import __graft_entry__
    __graft_entry__.build()
    from gated_deltanet_verify_gb300 import _build
    _build.build(checked=True)
    out = tmp_path / f"{case}.npz"
    r = subprocess.run([sys.executable, "-m", "tests.checked_cases", str(out), case], cwd=ROOT,
                       capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stdout + r.stderr
    return dict(np.load(out))
