"""Upload seeded inputs (``workloads.synth.Inputs``) to a CUDA device as torch
tensors in the layouts of ``include/gdn_verify.h``.  Plumbing only: no
arithmetic of the method happens here."""
from __future__ import annotations

from typing import Dict

import numpy as np
import torch

from .synth import Inputs, Shape


def act_torch_dtype(shape: Shape) -> torch.dtype:
    return torch.bfloat16 if shape.act == "bf16" else torch.float32


def act_host(a: np.ndarray, shape: Shape) -> torch.Tensor:
    t = torch.from_numpy(np.ascontiguousarray(a))
    return t.view(torch.bfloat16) if shape.act == "bf16" else t


def to_device(inp: Inputs, device="cuda", pin: bool = False) -> Dict[str, torch.Tensor]:
    s = inp.shape

    def put(t: torch.Tensor) -> torch.Tensor:
        if device == "cpu":
            return t.pin_memory() if pin else t.clone()
        return t.to(device)

    d = {
        "qkv": put(act_host(inp.qkv, s)),
        "z": put(act_host(inp.z, s)),
        "alpha": put(act_host(inp.alpha, s)),
        "beta_raw": put(act_host(inp.beta_raw, s)),
        "conv_w": put(torch.from_numpy(inp.conv_w)),
        "A_log": put(torch.from_numpy(inp.A_log)),
        "dt_bias": put(torch.from_numpy(inp.dt_bias)),
        "norm_w": put(torch.from_numpy(inp.norm_w)),
        "state": put(torch.from_numpy(inp.state)),
        "conv_state": put(torch.from_numpy(inp.conv_state)),
        "trim": put(torch.from_numpy(inp.trim.astype(np.int32))),
    }
    return d


def empty_outputs(shape: Shape, device="cuda", capture: bool = True, n_tokens: int = None) -> Dict[str, torch.Tensor]:
    s = shape
    T = s.n_tokens if n_tokens is None else n_tokens
    out = {"out": torch.empty((s.n_slots, T, s.n_v_heads * s.d_v), dtype=act_torch_dtype(s), device=device)}
    if capture:
        out["cap_state"] = torch.empty((s.n_slots, T, s.n_v_heads, s.d_v, s.d_k), dtype=torch.float32, device=device)
        out["cap_conv"] = torch.empty((s.n_slots, s.conv_width - 1 + T, s.conv_channels), dtype=torch.float32,
                                      device=device)
    return out


def to_f64(t: torch.Tensor) -> np.ndarray:
    return t.detach().to("cpu").to(torch.float64).numpy()
