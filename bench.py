#!/usr/bin/env python3
"""Benchmark of the GDN verify hot path on GB300.

Default (the largest single-GPU configuration): a 48-layer x 8-slot stack of
the GDN block of a 64-layer hybrid target (16 QK / 48 V heads, d_k = d_v =
128, K+1 = 16 verify tokens, bf16 activations, fp32 state); one step = one
verify forward (conv + SiLU, q/k L2 norm, gates, gated delta-rule recurrence
with per-position state capture, gated RMSNorm, conv-state advance) followed
by one rollback, for every layer, over seeded synthetic inputs already
resident in HBM.  The same JSON line carries per-config entries for one layer
at 1 slot and at 32 slots, the 8192-token chunked prefill and the layer with
its projections.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl gdn|reference]
                    [--workload layer_verify|multislot_verify|stack_verify|prefill|tree_verify|
                                rolled_verify|rolled_multislot_verify|rolled_stack_verify|
                                lazy_verify|lazy_multislot_verify|lazy_stack_verify|proj_verify]
                    [--no-per-config] [--no-e2e] [--no-cpu-baseline]

The tree_verify workload verifies a draft tree and rolls back to the accepted
node; the rolled_* workloads fold each step's rollback into the next verify
(one launch per step); the lazy_* workloads run lazy capture on the same
inputs as their capture counterparts: one launch per step commits the pending
batch (re-runs its accepted tokens) and writes the new batch's outputs,
nothing captured.  proj_verify adds the projections around the block
(hidden 5120; the library's own tcgen05 GEMM).

Prints one JSON line.  ``value`` = verified tokens/s over all ranks (device
time, CUDA events, steps replayed from CUDA graphs over rotating buffer sets:
each set is evicted from L2 by the others before it comes round again).  A
token counts once it has been through every layer of the workload.
``roofline`` is for the dominant kernel (verify): algorithmic bytes per launch
/ its average launch duration.
``e2e`` = the same metric through the public API with pinned host buffers,
host->device copies of each step's activations and a device->host read of
its output inside the timed region.  ``cpu_baseline`` = the fp64 oracle on
the host cores on a bounded sample.  ``--impl reference`` times the oracle
alone (the reference arm).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

from workloads.synth import make_parents, make_proj, proj_in_rows, WORKLOADS, make_inputs, randint  # noqa: E402

METRIC = "GDN verify tokens/sec at 1 GB300; achieved HBM GB/s vs roofline"
FALLBACK_BF16_TFLOPS = 1900.0
FALLBACK_HBM_GBS = 6800.0


# ---------------------------------------------------------------------------
# algorithmic bytes (compulsory traffic) per launch
# ---------------------------------------------------------------------------

def verify_bytes(s, capture=True) -> int:
    a = 2 if s.act == "bf16" else 4
    B, T, C, Hv, dk, dv, W = s.n_slots, s.n_tokens, s.conv_channels, s.n_v_heads, s.d_k, s.d_v, s.conv_width
    st = B * Hv * dv * dk * 4
    n = st * 2                                            # state read once, final state written once
    if capture:
        n += T * st                                       # one captured state per position
        n += B * (W - 1 + T) * C * 4                      # conv window capture
    n += B * T * C * a + B * T * Hv * dv * a * 2          # qkv in, z in, out
    n += 2 * B * T * Hv * a                               # alpha, beta_raw
    n += 2 * B * (W - 1) * C * 4                          # conv state read + write
    n += W * C * 4 + 2 * Hv * 4 + dv * 4                  # parameters
    return n


def tree_verify_bytes(s) -> int:
    """Compulsory bytes of a tree verify: the state read once, a captured state and a
    per-node conv state (3 rows) for every node, activations, the old conv state,
    parent ids and parameters.  Parent states re-read from the capture (L2) are not
    counted, and a tree verify writes neither the state nor the conv state."""
    a = 2 if s.act == "bf16" else 4
    B, T, C, Hv, dk, dv, W = s.n_slots, s.n_tokens, s.conv_channels, s.n_v_heads, s.d_k, s.d_v, s.conv_width
    st = B * Hv * dv * dk * 4
    n = st + T * st + B * T * (W - 1) * C * 4
    n += B * T * C * a + B * T * Hv * dv * a * 2 + 2 * B * T * Hv * a
    n += B * (W - 1) * C * 4 + B * T * 4
    n += W * C * 4 + 2 * Hv * 4 + dv * 4
    return n


def lazy_verify_bytes(s) -> int:
    """Compulsory bytes of an outputs-only verify: the state and conv state read once,
    activations in and out, parameters; nothing else is written."""
    st = s.n_slots * s.n_v_heads * s.d_v * s.d_k * 4
    return verify_bytes(s, capture=False) - st - s.n_slots * (s.conv_width - 1) * s.conv_channels * 4


def lazy_step_bytes(s, trims) -> int:
    """Compulsory bytes of a lazy verify with a pending batch: the outputs-only verify
    plus, per slot, the committed state and conv state written and the pending
    batch's accepted tokens (qkv, alpha, beta_raw) read."""
    a = 2 if s.act == "bf16" else 4
    st = s.n_v_heads * s.d_v * s.d_k * 4
    n = lazy_verify_bytes(s) + 4 * s.n_slots
    for tr in np.asarray(trims).reshape(-1):
        keep = s.n_tokens - int(tr)
        n += st + (s.conv_width - 1) * s.conv_channels * 4 + keep * (s.conv_channels + 2 * s.n_v_heads) * a
    return n


def commit_bytes(s, trims) -> int:
    """Compulsory bytes of the lazy commit: per slot with a valid trim, the state read and
    written, the conv state read and written, and the accepted tokens' qkv, alpha and
    beta_raw read again; the parameters once."""
    a = 2 if s.act == "bf16" else 4
    st = s.n_v_heads * s.d_v * s.d_k * 4
    n = 0
    for tr in np.asarray(trims).reshape(-1):
        if 0 <= tr < s.n_tokens:
            keep = s.n_tokens - int(tr)
            n += 2 * st + 2 * (s.conv_width - 1) * s.conv_channels * 4
            n += keep * (s.conv_channels + 2 * s.n_v_heads) * a
    n += 4 * s.n_slots + s.conv_width * s.conv_channels * 4 + 2 * s.n_v_heads * 4
    return n


def proj_in_bytes(s) -> int:
    """Compulsory bytes of the fused input projection: x and w_in read, the
    activation matrix (row stride rounded up to 8 columns) written."""
    M = s.n_slots * s.n_tokens
    ld = -(-proj_in_rows(s) // 8) * 8
    return 2 * (M * s.n_embd + proj_in_rows(s) * s.n_embd + M * ld)


def proj_out_bytes(s) -> int:
    M = s.n_slots * s.n_tokens
    return 2 * (M * s.value_dim + s.n_embd * s.value_dim + M * s.n_embd)


def rollback_bytes(s, trims) -> int:
    per_slot = 2 * (s.n_v_heads * s.d_v * s.d_k * 4 + (s.conv_width - 1) * s.conv_channels * 4)
    return int(np.count_nonzero(np.asarray(trims))) * per_slot + 4 * s.n_slots


def resident_bytes(s) -> int:
    """Bytes of one layer's buffers that stay in L2 between steps: the state, conv state, conv window,
    activations, outputs and parameters -- every buffer but the captured states, which the kernels
    stream out evict-first."""
    a = 2 if s.act == "bf16" else 4
    B, T, C, Hv, dk, dv, W = s.n_slots, s.n_tokens, s.conv_channels, s.n_v_heads, s.d_k, s.d_v, s.conv_width
    n = B * Hv * dv * dk * 4 + B * (W - 1) * C * 4 + B * (W - 1 + T) * C * 4
    n += B * T * C * a + 2 * B * T * Hv * dv * a + 2 * B * T * Hv * a
    return n + W * C * 4 + 2 * Hv * 4 + dv * 4


def prefill_bytes(s) -> int:
    return verify_bytes(s, capture=False)


# dense products of one (slot, value head, 64-token chunk) in the chunkwise form,
# 2 flops per multiply-add: G = [K;Q]K^T, W and U~ (T times two 64x128
# operands), U -= W S, O = (Gamma Q) S, O += P U, S += (Gamma_C/Gamma K)^T U
PREFILL_FLOPS_PER_CHUNK = 2 * (128 * 64 * 128 + 2 * 128 * 64 * 64 + 128 * 64 * 128 + 128 * 64 * 128
                               + 128 * 64 * 64 + 128 * 128 * 64)
TF32_PER_BF16 = 1.1 / 2.25      # nominal dense tf32 / bf16 tensor rate of the part
HBM_NOMINAL_GBS = 7900.0        # the part's nominal HBM3e rate (the measured copy rate is the roofline's peak)


def prefill_flops(s) -> int:
    return s.n_slots * s.n_v_heads * (-(-s.n_tokens // s.chunk)) * PREFILL_FLOPS_PER_CHUNK


def tf32_peak():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            return float(json.load(f)["bf16_tflops"]) * TF32_PER_BF16, "measured"
    return FALLBACK_BF16_TFLOPS * TF32_PER_BF16, "fallback"


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    return FALLBACK_HBM_GBS, "fallback"


def kernel_source_sha(names) -> str:
    h = hashlib.sha256()
    for n in names:
        with open(os.path.join(ROOT, "gated_deltanet_verify_gb300", "csrc", n), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def recorded_step_traffic(workload: str, sha: str):
    """DRAM bytes per step over a long range of steps (ncu range capture: the captured states' write-backs
    included), if taken on this exact source; else None."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        e = json.load(f).get("step", {}).get(workload)
    if not e or e.get("source_sha") != sha:
        return None
    return e.get("dram_bytes_per_step")


def recorded_traffic(kernel: str, sha: str, workload: str):
    """DRAM bytes per launch from a committed ncu summary, if it was taken on
    this exact kernel source and workload; else None."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        d = json.load(f)
    e = d.get(kernel, {}).get(workload)
    if not e or e.get("source_sha") != sha:
        return None
    return e.get("dram_bytes_per_launch")


# ---------------------------------------------------------------------------
# clocks
# ---------------------------------------------------------------------------

class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap,clocks.mem,clocks.max.mem,temperature.memory")

    def __init__(self, gpu_index: int):
        self.idx = gpu_index
        self.samples = []
        self.proc = None
        self.thread = None

    def _parse(self, line):
        parts = [p.strip() for p in line.split(",")]
        if len(parts) < 8:
            return None
        try:
            s = {"sm": float(parts[0]), "max": float(parts[1]), "hw": parts[4], "hw_thermal": parts[5],
                 "sw_thermal": parts[6], "sw_power": parts[7], "t": time.time()}
            for key, i in (("mem", 8), ("mem_max", 9), ("mem_temp", 10)):     # context: HBM clock, temperature
                try:
                    s[key] = float(parts[i])
                except (IndexError, ValueError):
                    pass
            return s
        except ValueError:
            return None

    def once(self):
        try:
            r = subprocess.run(["nvidia-smi", f"--id={self.idx}", f"--query-gpu={self.FIELDS}",
                                "--format=csv,noheader,nounits"], capture_output=True, text=True, timeout=20)
            s = self._parse(r.stdout.strip().splitlines()[0]) if r.stdout.strip() else None
            if s:
                self.samples.append(s)
        except Exception:
            pass

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.idx}", f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
            return

        def reader():
            for line in self.proc.stdout:
                s = self._parse(line)
                if s:
                    self.samples.append(s)
        self.thread = threading.Thread(target=reader, daemon=True)
        self.thread.start()

    def stop(self):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
        if self.thread:
            self.thread.join(timeout=5)

    def summary(self, t0, t1):
        inside = [s for s in self.samples if t0 <= s["t"] <= t1] or self.samples
        if not inside:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        reasons = set()
        for s in inside:
            for key, name in (("hw", "hw_slowdown"), ("hw_thermal", "hw_thermal_slowdown"),
                              ("sw_thermal", "sw_thermal_slowdown"), ("sw_power", "sw_power_cap")):
                if s[key].lower().startswith("active"):
                    reasons.add(name)
        res = {"sm_mhz": float(np.median([s["sm"] for s in inside])),
               "sm_max_mhz": float(max(s["max"] for s in inside)), "reasons": sorted(reasons),
               "samples": len(inside)}
        for key, name in (("mem", "mem_mhz"), ("mem_max", "mem_max_mhz"), ("mem_temp", "mem_temp_c")):
            vals = [s[key] for s in inside if key in s]
            if vals:
                res[name] = float(np.median(vals)) if key != "mem_max" else float(max(vals))
        return res


# ---------------------------------------------------------------------------
# the CUDA arm
# ---------------------------------------------------------------------------

def _dist():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def max_over_ranks(value: float, device=None) -> float:
    """The slowest rank's time: replicas run the same work, so the job's clock
    is the maximum over ranks.  No-op without an initialised process group."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(value)
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(units_per_rank_step: float, steps: int, world: int, seconds: float) -> float:
    """Whole-job throughput: every rank processes its own units (weak scaling)."""
    return units_per_rank_step * steps * world / seconds


class VerifyWorkload:
    """Rotating buffer sets of one verify+rollback workload (one or more layers)."""

    def __init__(self, shape, device, l2_bytes):
        import torch
        import gated_deltanet_verify_gb300 as gdn
        from workloads.device import empty_outputs, to_device
        self.gdn, self.torch = gdn, torch
        self.shape = s = shape
        self.layers = s.n_layers
        self.tree = s.name.startswith("tree")          # draft-tree verify + rollback to the accepted node
        # lazy capture: one launch per step commits the pending batch (this buffer set's previous
        # one, with its trims) and verifies the new one, outputs only
        self.lazy = s.name.startswith("lazy")
        # the layer with its projections: x -> GEMM -> verify (strided activations) -> GEMM -> y
        self.proj = s.n_embd > 0
        # the rollback of each step folded into the next verify: one launch per step
        self.rolled = s.name.startswith("rolled")
        # the rotation is sized on what a step leaves in L2: everything but the captured states (streamed
        # out with evict-first stores), so that each step reads its state and activations from DRAM
        per_set = resident_bytes(s) * self.layers
        if self.proj:
            per_set += (proj_in_bytes(s) + proj_out_bytes(s)) * self.layers
        self.n_sets = 1 if per_set > 3 * l2_bytes else int(min(128, -(-3 * l2_bytes // per_set) + 1))
        self.resident_per_set = per_set
        self.dims = gdn.make_dims(s.n_slots, s.n_qk_heads, s.n_v_heads, s.d_k, s.d_v, s.n_tokens,
                                  gdn.GDN_BF16 if s.act == "bf16" else gdn.GDN_F32)
        self.sets = []
        self.host_inputs = []
        n_layer_inputs = self.layers if self.layers > 1 else 1
        for li in range(n_layer_inputs):
            inp = make_inputs(s, layer=li)
            self.host_inputs.append(inp)
        # a slot's trim is decided once per step (after every layer has verified) and rolls back every layer
        trims = np.repeat(randint(s.seed, 12, self.n_sets * s.n_slots, s.n_tokens).reshape(self.n_sets, 1, s.n_slots),
                          self.layers, axis=1)
        if self.tree:                                # accepted node per slot, -1 .. T-1
            trims = trims.astype(np.int64) - 1
        self.trims = trims
        self.parents = make_parents(s, "spine")
        for k in range(self.n_sets):
            layers = []
            for li in range(self.layers):
                x = to_device(self.host_inputs[li if self.layers > 1 else 0], device)
                x["trim"] = torch.from_numpy(trims[k, li].astype(np.int32)).to(device)
                x.update(empty_outputs(s, device, capture=not self.lazy))
                if self.tree:
                    x["parent"] = torch.from_numpy(self.parents).to(device)
                    x["cap_conv"] = torch.empty((s.n_slots, s.n_tokens, s.conv_width - 1, s.conv_channels),
                                                dtype=torch.float32, device=device)
                x["status"] = torch.zeros(1, dtype=torch.int32, device=device)
                x["params"] = gdn.layer_params(x["conv_w"], x["A_log"], x["dt_bias"], x["norm_w"])
                if self.proj:                   # every buffer set has its own weights, so they rotate too
                    if not hasattr(self, "host_proj"):
                        self.host_proj = make_proj(s)
                    for key, v in self.host_proj.items():
                        x[key] = torch.from_numpy(v).view(torch.bfloat16).to(device)
                    x["w"] = gdn.proj_weights(s.n_embd, x["w_in"], x["w_out"])
                    x["ws_bytes"] = gdn.gdn_layer_workspace_bytes(self.dims, s.n_embd)
                    x["ws"] = torch.empty(x["ws_bytes"], dtype=torch.uint8, device=device)
                    x["y"] = torch.empty((s.n_slots, s.n_tokens, s.n_embd), dtype=torch.bfloat16, device=device)
                    M = s.n_slots * s.n_tokens
                    act_b = M * gdn.gdn_proj_in_ld(self.dims) * 2
                    out_off = -(-act_b // 256) * 256
                    x["lt_off"] = out_off + -(-(M * s.value_dim * 2) // 256) * 256
                    x["act"] = x["ws"][:act_b]
                    x["act_out"] = x["ws"][out_off:out_off + M * s.value_dim * 2]
                layers.append(x)
            self.sets.append(layers)
        if self.rolled:                 # every set's captures start out valid
            for layers in self.sets:
                for li, x in enumerate(layers):
                    gdn.gdn_verify_forward(self.dims, x["params"], x["qkv"], x["z"], x["alpha"], x["beta_raw"],
                                           x["state"], x["conv_state"], x["cap_state"], x["cap_conv"], x["out"])
        self.tokens_per_step = s.n_slots * s.n_tokens
        self.kernels_per_step = (1 if self.lazy or self.rolled else 2) * self.layers
        # a multi-layer chain step rolls every layer back in one launch (gdn_rollback_layers, device pointer
        # tables of each set's layers)
        self.tabs = None
        if self.layers > 1 and not (self.lazy or self.rolled or self.tree or self.proj):
            self.tabs = [[gdn.pointer_table([x[key] for x in layers], device)
                          for key in ("state", "conv_state", "cap_state", "cap_conv")] for layers in self.sets]
            self.kernels_per_step = self.layers + 1

    def verify(self, k, li, stream, x=None):
        x = self.sets[k][li] if x is None else x
        if self.tree:
            self.gdn.gdn_verify_tree(self.dims, x["params"], x["qkv"], x["z"], x["alpha"], x["beta_raw"],
                                     x["parent"], x["state"], x["conv_state"], x["cap_state"], x["cap_conv"],
                                     x["out"], x["status"], stream)
            return
        if self.proj:
            self.gdn.gdn_layer_verify(self.dims, x["params"], x["w"], x["x"], x["state"], x["conv_state"],
                                      x["cap_state"], x["cap_conv"], x["y"], x["ws"], x["ws_bytes"], x["status"],
                                      stream)
            return
        if self.rolled:
            self.gdn.gdn_verify_after_rollback(self.dims, x["params"], x["trim"], x["qkv"], x["z"], x["alpha"],
                                               x["beta_raw"], x["state"], x["conv_state"], x["cap_state"],
                                               x["cap_conv"], x["out"], x["status"], stream)
            return
        if self.lazy:
            self.gdn.gdn_verify_lazy(self.dims, x["params"], x["qkv"], x["z"], x["alpha"], x["beta_raw"],
                                     x["state"], x["conv_state"], x["out"], x["status"], stream,
                                     prev_trim=x["trim"], prev_qkv=x["qkv"], prev_alpha=x["alpha"],
                                     prev_beta_raw=x["beta_raw"])
            return
        self.gdn.gdn_verify_forward(self.dims, x["params"], x["qkv"], x["z"], x["alpha"], x["beta_raw"], x["state"],
                                    x["conv_state"], x["cap_state"], x["cap_conv"], x["out"], x["status"], stream)

    def gemm_in(self, k, li, stream):
        x = self.sets[k][li]
        lt = x["ws"][x["lt_off"]:]
        self.gdn.gdn_project_in(self.dims, x["w"], x["x"], x["act"], lt, lt.numel(), stream)

    def gemm_out(self, k, li, stream):
        x = self.sets[k][li]
        lt = x["ws"][x["lt_off"]:]
        self.gdn.gdn_project_out(self.dims, x["w"], x["act_out"], x["y"], lt, lt.numel(), stream)

    def rollback(self, k, li, stream, x=None):
        x = self.sets[k][li] if x is None else x
        if self.lazy or self.rolled:    # the commit / rollback rides in the next verify
            return
        fn = self.gdn.gdn_rollback_tree if self.tree else self.gdn.gdn_rollback
        fn(self.dims, x["trim"], x["state"], x["conv_state"], x["cap_state"], x["cap_conv"], x["status"], stream)

    def rollback_all(self, k, li, stream, tabs=None, trim=None):
        """Every layer of set k rolled back in one launch (li unused: the signature of the per-kernel timer)."""
        x = self.sets[k][0]
        self.gdn.gdn_rollback_layers(self.dims, self.layers, x["trim"] if trim is None else trim,
                                     *(self.tabs[k] if tabs is None else tabs), x["status"], stream)

    def step(self, k, stream):
        # the verify pass through every layer, then (the accepted lengths known) the rollback of every layer
        for li in range(self.layers):
            self.verify(k, li, stream)
        if self.tabs is not None:
            self.rollback_all(k, 0, stream)
            return
        for li in range(self.layers):
            self.rollback(k, li, stream)

    def step_bytes(self, k):
        if self.lazy:
            return sum(lazy_step_bytes(self.shape, self.trims[k][li]) for li in range(self.layers))
        if self.rolled:                 # the captured state replaces the state as the verify's input
            return verify_bytes(self.shape) * self.layers
        if self.proj:
            s = self.shape
            return sum(verify_bytes(s) + proj_in_bytes(s) + proj_out_bytes(s) + rollback_bytes(s, self.trims[k][li])
                       for li in range(self.layers))
        vb = tree_verify_bytes(self.shape) if self.tree else verify_bytes(self.shape)
        moved = (self.trims[k] >= 0) if self.tree else self.trims[k]     # slots whose rollback copies
        return sum(vb + rollback_bytes(self.shape, moved[li]) for li in range(self.layers))

    def e2e_step_host(self, steps, device):
        """One C-ABI call per step with host buffers (gdn_verify_step_host): the
        packed pinned input block goes to the device in one copy, the verify and
        the rollback (or the rolled verify) run, the outputs come back in one copy;
        one host wait per step.  The ctypes arguments are marshalled once."""
        import ctypes
        torch, gdn = self.torch, self.gdn
        from workloads.device import act_host
        s = self.shape
        io = gdn.gdn_step_io_layout(self.dims)
        inp = self.host_inputs[0]
        host_in = torch.zeros(io.in_bytes, dtype=torch.uint8).pin_memory()
        for off, t in ((io.qkv, act_host(inp.qkv, s)), (io.z, act_host(inp.z, s)), (io.alpha, act_host(inp.alpha, s)),
                       (io.beta_raw, act_host(inp.beta_raw, s)),
                       (io.trim, torch.from_numpy(self.trims[0, 0].astype(np.int32)))):
            b = t.contiguous().view(torch.uint8).reshape(-1)
            host_in[off:off + b.numel()].copy_(b)
        host_out = torch.empty(io.out_bytes, dtype=torch.uint8).pin_memory()
        d_io = torch.empty(io.in_bytes + io.out_bytes, dtype=torch.uint8, device=device)
        x = self.sets[0][0]
        stream = torch.cuda.current_stream()
        fn = gdn.lib().gdn_verify_step_host
        args = (ctypes.byref(self.dims), ctypes.byref(x["params"]), 1 if self.rolled else 0, host_in.data_ptr(),
                host_out.data_ptr(), d_io.data_ptr(), d_io.numel(), x["state"].data_ptr(), x["conv_state"].data_ptr(),
                x["cap_state"].data_ptr(), x["cap_conv"].data_ptr(), x["status"].data_ptr(), stream.cuda_stream)

        def one(k):
            rc = fn(*args)
            if rc != 0:
                raise RuntimeError(f"gdn_verify_step_host: {rc} {gdn.gdn_last_error()}")
            stream.synchronize()

        for k in range(10):
            one(k)
        t0 = time.perf_counter()
        for k in range(steps):
            one(k)
        dt = time.perf_counter() - t0
        return dt, io.in_bytes, io.out_bytes

    def e2e(self, steps, device):
        if self.layers == 1 and not (self.tree or self.lazy or self.proj):
            return self.e2e_step_host(steps, device)
        return self.e2e_staged(steps, device)

    def e2e_staged(self, steps, device):
        """Public-API loop with host buffers: every step copies all its inputs (every
        layer's activations, trims, parent ids or hidden state) host -> device as one
        pinned buffer, runs verify + rollback per layer through the C ABI, copies all
        outputs device -> host as one buffer, and synchronises the host once.  The
        device tensors the calls read and write are views into the two staging
        buffers (each view 256-byte aligned).  (Replaying the step from a CUDA
        graph instead measured slower at one slot: 352K against 387K tokens/s.)
        A multi-layer chain step runs as a serving step would: the verify of every
        layer, the outputs back to the host and a host synchronisation (the accepted
        lengths are decided there), then the trims host -> device and the rollback
        of every layer.  With several layers the copies are pipelined on a second
        stream: layer l's inputs go host -> device while the layers before it run,
        and its outputs come back while the layers after it run."""
        torch = self.torch
        from workloads.device import act_host
        s = self.shape
        out_key = "y" if self.proj else "out"
        split_rollback = self.layers > 1 and not (self.lazy or self.rolled or self.tree or self.proj)
        hosts = []
        for li in range(self.layers):
            inp = self.host_inputs[li if self.layers > 1 else 0]
            if self.proj:                   # the layer's input is the hidden state x
                h = {"x": act_host(self.host_proj["x"], s)}
            else:
                h = {"qkv": act_host(inp.qkv, s), "z": act_host(inp.z, s), "alpha": act_host(inp.alpha, s),
                     "beta_raw": act_host(inp.beta_raw, s)}
            if not split_rollback:
                h["trim"] = torch.from_numpy(self.trims[0, li].astype(np.int32))
            if self.tree:
                h["parent"] = torch.from_numpy(self.parents)
            hosts.append(h)

        def layout(tensors):
            offs, n = [], 0
            for t in tensors:
                offs.append(n)
                n += -(-t.numel() * t.element_size() // 256) * 256
            return offs, n

        ins = [(li, k, t) for li, h in enumerate(hosts) for k, t in h.items()]
        in_offs, in_bytes = layout([t for _, _, t in ins])
        outs_ref = [self.sets[0][li][out_key] for li in range(self.layers)]
        out_offs, out_bytes = layout(outs_ref)
        host_in = torch.empty(in_bytes, dtype=torch.uint8).pin_memory()
        dev_in = torch.empty(in_bytes, dtype=torch.uint8, device=device)
        host_out = torch.empty(out_bytes, dtype=torch.uint8).pin_memory()
        dev_out = torch.empty(out_bytes, dtype=torch.uint8, device=device)
        xs = [dict(self.sets[0][li]) for li in range(self.layers)]
        for (li, k, t), off in zip(ins, in_offs):
            nb = t.numel() * t.element_size()
            host_in[off:off + nb].copy_(t.contiguous().view(torch.uint8).reshape(-1))
            xs[li][k] = dev_in[off:off + nb].view(t.dtype).view(t.shape)
        for li, (ref, off) in enumerate(zip(outs_ref, out_offs)):
            nb = ref.numel() * ref.element_size()
            xs[li][out_key] = dev_out[off:off + nb].view(ref.dtype).view(ref.shape)
        stream = torch.cuda.current_stream()
        sp = stream.cuda_stream
        host_trim = torch.from_numpy(self.trims[0, 0].astype(np.int32)).pin_memory()
        dev_trim = torch.empty_like(host_trim, device=device)
        if split_rollback:
            for li in range(self.layers):
                xs[li]["trim"] = dev_trim

        # per-layer byte ranges of the staging buffers (the inputs are laid out layer by layer)
        in_rng = []
        for li in range(self.layers):
            offs = [(off, t.numel() * t.element_size()) for (l2, _, t), off in zip(ins, in_offs) if l2 == li]
            in_rng.append((min(o for o, _ in offs), max(o + n for o, n in offs)))
        out_rng = [(off, off + ref.numel() * ref.element_size()) for ref, off in zip(outs_ref, out_offs)]
        copy_stream = torch.cuda.Stream()
        ev_in = [torch.cuda.Event() for _ in range(self.layers)]
        ev_done = [torch.cuda.Event() for _ in range(self.layers)]

        def one_pipelined(k):
            with torch.cuda.stream(copy_stream):
                for li, (a, b) in enumerate(in_rng):
                    dev_in[a:b].copy_(host_in[a:b], non_blocking=True)
                    ev_in[li].record(copy_stream)
            for li in range(self.layers):
                stream.wait_event(ev_in[li])
                self.verify(0, li, sp, xs[li])
                if not split_rollback:
                    self.rollback(0, li, sp, xs[li])
                ev_done[li].record(stream)
                copy_stream.wait_event(ev_done[li])
                with torch.cuda.stream(copy_stream):
                    a, b = out_rng[li]
                    host_out[a:b].copy_(dev_out[a:b], non_blocking=True)
            copy_stream.synchronize()
            if split_rollback:
                dev_trim.copy_(host_trim, non_blocking=True)
                self.rollback_all(0, 0, sp, trim=dev_trim)

        def one(k):
            if self.layers > 1:
                one_pipelined(k)
                return
            dev_in.copy_(host_in, non_blocking=True)
            if split_rollback:
                for li in range(self.layers):
                    self.verify(0, li, sp, xs[li])
                host_out.copy_(dev_out, non_blocking=True)
                stream.synchronize()
                dev_trim.copy_(host_trim, non_blocking=True)
                self.rollback_all(0, 0, sp, trim=dev_trim)
                return
            for li in range(self.layers):
                self.verify(0, li, sp, xs[li])
                self.rollback(0, li, sp, xs[li])
            host_out.copy_(dev_out, non_blocking=True)
            stream.synchronize()

        for k in range(10):
            one(k)
        stream.synchronize()
        t0 = time.perf_counter()
        for k in range(steps):
            one(k)
        stream.synchronize()
        dt = time.perf_counter() - t0
        return dt, in_bytes + (host_trim.numel() * 4 if split_rollback else 0), out_bytes


class PrefillWorkload:
    def __init__(self, shape, device, l2_bytes):
        import torch
        import gated_deltanet_verify_gb300 as gdn
        from workloads.device import act_torch_dtype, to_device
        self.gdn, self.torch = gdn, torch
        self.shape = s = shape
        self.layers = 1
        self.dims = gdn.make_dims(s.n_slots, s.n_qk_heads, s.n_v_heads, s.d_k, s.d_v, s.n_tokens,
                                  gdn.GDN_BF16 if s.act == "bf16" else gdn.GDN_F32)
        per_set = prefill_bytes(s)
        self.n_sets = 1 if per_set > 3 * l2_bytes else int(-(-3 * l2_bytes // per_set) + 1)
        self.resident_per_set = per_set
        inp = make_inputs(s)
        self.host_inputs = [inp]
        self.ws_bytes = gdn.gdn_prefill_workspace_bytes(self.dims)
        self.sets = []
        for _ in range(self.n_sets):
            x = to_device(inp, device)
            x["out"] = torch.empty((s.n_slots, s.n_tokens, s.n_v_heads * s.d_v), dtype=act_torch_dtype(s),
                                   device=device)
            x["ws"] = torch.empty(max(self.ws_bytes, 256), dtype=torch.uint8, device=device)
            x["status"] = torch.zeros(1, dtype=torch.int32, device=device)
            x["params"] = gdn.layer_params(x["conv_w"], x["A_log"], x["dt_bias"], x["norm_w"])
            self.sets.append([x])
        self.tokens_per_step = s.n_slots * s.n_tokens
        # the chunkwise kernel (one cooperative launch per group of (slot, head) pairs) + the conv-state kernel
        self.kernels_per_step = 2 if s.n_slots * s.n_v_heads * 3 <= 152 else None

    def prefill(self, k, li, stream):
        x = self.sets[k][0]
        self.gdn.gdn_prefill_chunked(self.dims, x["params"], x["qkv"], x["z"], x["alpha"], x["beta_raw"],
                                     x["state"], x["conv_state"], x["out"], x["ws"], self.ws_bytes, x["status"],
                                     stream)

    def step(self, k, stream):
        self.prefill(k, 0, stream)

    def step_bytes(self, k):
        return prefill_bytes(self.shape)

    def e2e(self, steps, device):
        """Public-API loop with host buffers: H2D of the prompt's activations,
        prefill, D2H of out; one host sync per step."""
        torch = self.torch
        from workloads.device import act_host
        s = self.shape
        inp = self.host_inputs[0]
        host = {"qkv": act_host(inp.qkv, s).pin_memory(), "z": act_host(inp.z, s).pin_memory(),
                "alpha": act_host(inp.alpha, s).pin_memory(), "beta_raw": act_host(inp.beta_raw, s).pin_memory()}
        out_host = torch.empty(self.sets[0][0]["out"].shape, dtype=self.sets[0][0]["out"].dtype).pin_memory()
        h2d = sum(t.numel() * t.element_size() for t in host.values())
        d2h = out_host.numel() * out_host.element_size()
        stream = torch.cuda.current_stream()
        sp = stream.cuda_stream

        def one(k):
            x = self.sets[k % self.n_sets][0]
            for key, t in host.items():
                x[key].copy_(t, non_blocking=True)
            self.prefill(k % self.n_sets, 0, sp)
            out_host.copy_(x["out"], non_blocking=True)
            stream.synchronize()

        for k in range(3):
            one(k)
        t0 = time.perf_counter()
        for k in range(steps):
            one(k)
        return time.perf_counter() - t0, h2d, d2h


def capture_graph(torch, fn_list):
    g = torch.cuda.CUDAGraph()
    cs = torch.cuda.Stream()
    cs.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(cs):
        sp = cs.cuda_stream
        for f in fn_list:          # one eager pass on the capture stream first (lazy init, attributes)
            f(sp)
    torch.cuda.synchronize()
    with torch.cuda.graph(g, stream=cs):
        sp = torch.cuda.current_stream().cuda_stream
        for f in fn_list:
            f(sp)
    torch.cuda.synchronize()
    return g


def time_graph_steps(torch, wl, steps, graph_len, first=0):
    """Graphs of `graph_len` steps over rotating buffer sets (starting at set `first`) covering exactly
    `steps` steps."""
    n_full, rem = divmod(steps, graph_len)
    fns = [lambda sp, k=k: wl.step((first + k) % wl.n_sets, sp) for k in range(graph_len)]
    g_full = capture_graph(torch, fns) if n_full else None
    g_rem = capture_graph(torch, fns[:rem]) if rem else None
    return g_full, n_full, g_rem


def kernel_duration(torch, wl, which, n_launch, flush=None):
    """Duration of one kernel kind: CUDA events around each of five replays of a graph of n_launch
    back-to-back launches cycling over the buffer sets and layers (each set's data evicted from L2 by
    the others before it comes round again); the median replay, per launch."""
    fns = []
    for k in range(n_launch):
        kk, li = k % wl.n_sets, (k // wl.n_sets) % wl.layers
        fns.append(lambda sp, kk=kk, li=li: getattr(wl, which)(kk, li, sp))
    g = capture_graph(torch, fns)
    for _ in range(3):
        g.replay()
    if flush is not None:
        flush()
    torch.cuda.synchronize()
    reps = 5
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(reps + 1)]
    ev[0].record()
    for i in range(reps):
        g.replay()
        ev[i + 1].record()
    ev[-1].synchronize()
    per = sorted(ev[i].elapsed_time(ev[i + 1]) for i in range(reps))
    return per[reps // 2] / 1e3 / n_launch


def eager_step_duration(torch, wl, n):
    """Launch-to-launch time of a step issued eagerly (no graph): n steps back to back on one stream,
    cycling over the buffer sets, each step one or two C-ABI calls from Python; CUDA events around the
    burst.  Against the graph replays this shows what the host's launch path costs a short step."""
    sp = torch.cuda.current_stream().cuda_stream
    for k in range(3):
        wl.step(k % wl.n_sets, sp)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for k in range(n):
        wl.step(k % wl.n_sets, sp)
    e1.record()
    e1.synchronize()
    return e0.elapsed_time(e1) / 1e3 / n


def describe(shape) -> str:
    return (f"{shape.name}: {shape.n_layers} layer(s) x {shape.n_slots} slot(s), {shape.n_qk_heads} QK / "
            f"{shape.n_v_heads} V heads, d_k=d_v={shape.d_k}, {shape.n_tokens} tokens")


# steps a per-config entry times at least (about 10 ms of device work or more)
MIN_STEPS = {"layer_verify": 1000, "multislot_verify": 64, "prefill": 20, "proj_verify": 500, "tree_verify": 1000,
             "rolled_verify": 1000, "lazy_verify": 1000}
HEADLINE = "stack_verify"                                   # 48 layers x 8 slots: the largest configuration
# one layer at one slot, 32 slots, the 8192-token prefill, the layer with its projections around the block
# (hidden 5120, the library's GEMM), and at one slot the draft-tree verify, the verify with the previous
# step's rollback folded in, and the lazy-capture verify
PER_CONFIG = ("layer_verify", "multislot_verify", "prefill", "proj_verify", "tree_verify", "rolled_verify",
              "lazy_verify")


def measure(name, steps, warmup, device, world, l2, clocks, with_e2e, graph_len_max=64):
    """Time `steps` steps of one workload (after `warmup` untimed ones) and its kernels; returns the
    fields of a bench line (without the CPU baseline)."""
    import torch
    import torch.distributed as dist
    shape = WORKLOADS[name]
    wl = PrefillWorkload(shape, device, l2) if name == "prefill" else VerifyWorkload(shape, device, l2)
    torch.cuda.synchronize()
    # a step graph covers at most one rotation of the buffer sets, so no set comes round twice in a graph
    graph_len = max(1, min(graph_len_max, steps, wl.n_sets))
    if wl.layers > 1 or name == "prefill":
        graph_len = 1
    g_full, n_full, g_rem = time_graph_steps(torch, wl, steps, graph_len)
    g_warm, nw_full, g_wrem = time_graph_steps(torch, wl, warmup, max(1, min(graph_len, warmup)),
                                               first=wl.n_sets // 2)
    # a buffer larger than L2, written between the warm-up and the timed steps
    flush_buf = torch.empty(int(3 * l2), dtype=torch.uint8, device=device)
    flush = lambda: flush_buf.fill_(1)
    for _ in range(nw_full):
        g_warm.replay()
    if g_wrem:
        g_wrem.replay()
    flush()
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t_wall0 = time.time()
    torch.cuda.synchronize()
    e0.record()
    for _ in range(n_full):
        g_full.replay()
    if g_rem:
        g_rem.replay()
    e1.record()
    torch.cuda.synchronize()
    t_wall1 = time.time()
    if world > 1:
        dist.barrier()
    dt = e0.elapsed_time(e1) / 1e3
    bad = [int(x["status"].item()) for layers in wl.sets for x in layers if int(x["status"].item()) != 0]

    # per-kernel durations (own timed regions, graphs of back-to-back launches over every set and layer)
    n_launch = max(8, min(256, wl.n_sets * wl.layers))
    if name == "prefill":
        kdur = {"prefill": kernel_duration(torch, wl, "prefill", max(2, wl.n_sets), flush)}
    elif wl.lazy:
        kdur = {"lazy_verify": kernel_duration(torch, wl, "verify", n_launch, flush)}
    elif wl.rolled:
        kdur = {"verify": kernel_duration(torch, wl, "verify", n_launch, flush)}
    elif wl.proj:
        # the layer call is GEMM + verify + GEMM; what it takes beyond the two GEMMs timed alone is the
        # verify plus the launch gaps between the library's kernels and it
        kdur = {"layer": kernel_duration(torch, wl, "verify", n_launch, flush),
                "gemm_in": kernel_duration(torch, wl, "gemm_in", n_launch, flush),
                "gemm_out": kernel_duration(torch, wl, "gemm_out", n_launch, flush),
                "rollback": kernel_duration(torch, wl, "rollback", n_launch, flush)}
        kdur["verify_and_launch_gaps"] = max(0.0, kdur["layer"] - kdur["gemm_in"] - kdur["gemm_out"])
    else:
        kdur = {"verify": kernel_duration(torch, wl, "verify", n_launch, flush),
                "rollback": kernel_duration(torch, wl, "rollback", n_launch, flush)}
        if wl.tabs is not None:     # the step's one rollback launch over every layer
            kdur["rollback_all_layers"] = kernel_duration(torch, wl, "rollback_all", max(2, wl.n_sets), flush)
    t_wall2 = time.time()

    dt = max_over_ranks(dt, device)
    value = job_throughput(wl.tokens_per_step, steps, world, dt)
    hbm, peak_kind = peaks()
    if name == "prefill":
        dom, dom_bytes, dom_src = "prefill", prefill_bytes(shape), ["prefill.cu", "internal.cuh"]
    elif wl.proj:
        dom, dom_bytes, dom_src = "gemm_in", proj_in_bytes(shape), ["proj.cu"]
    elif wl.lazy:
        dom = "lazy_verify"
        dom_bytes = float(np.mean([lazy_step_bytes(shape, t) for t in wl.trims.reshape(-1, shape.n_slots)]))
        dom_src = ["verify.cu", "internal.cuh"]
    else:
        dom, dom_bytes, dom_src = "verify", (tree_verify_bytes(shape) if getattr(wl, "tree", False)
                                             else verify_bytes(shape)), ["verify.cu", "internal.cuh"]
    # The verify's launch time is its share of the timed step: the step time minus the step's other kernels
    # (the rollbacks) timed alone, per layer.  Timed alone, back to back, a 1-slot verify was measured
    # slower on some GB300s than inside the step (19.9 + 4.5 us of verify and rollback against a 20.9 us
    # step): back-to-back launches of the write-heavy verify never occur in the workload.  The alone figure
    # stays in kernels_us and as launch_us_alone.
    t_launch, how = kdur[dom], "timed alone: CUDA events around graph replays of back-to-back launches"
    if name != "prefill" and not wl.proj:
        others = (kdur["rollback_all_layers"] if wl.tabs is not None
                  else 0.0 if (wl.lazy or wl.rolled) else kdur["rollback"] * wl.layers)
        in_step = (dt / steps - others) / wl.layers
        if in_step > 0:
            t_launch = in_step
            how = ("its share of the timed step: CUDA events around the step replays, minus the step's "
                   "rollback launches timed alone, per layer")
    achieved = dom_bytes / t_launch / 1e9
    sha = kernel_source_sha(dom_src)
    traffic = recorded_traffic(dom, sha, name)
    roof = {"bound": "hbm", "achieved": achieved, "peak": hbm, "unit": "GB/s", "frac": achieved / hbm,
            "traffic": traffic, "kernel": dom, "bytes_per_launch": dom_bytes, "launch_us": t_launch * 1e6,
            "launch_us_alone": kdur[dom] * 1e6, "launch_time": how,
            "frac_of_nominal": achieved / HBM_NOMINAL_GBS, "nominal_gbs": HBM_NOMINAL_GBS,
            "peak_source": f"{peak_kind} hbm_gbs" + (" (MEASURED_PEAKS.json)" if peak_kind == "measured"
                                                     else " (recipe fallback)")}
    if traffic:
        # the same launch judged on the DRAM bytes ncu counted for it (L2 hits excluded)
        roof["dram_gbs"] = traffic / t_launch / 1e9
        roof["dram_frac"] = roof["dram_gbs"] / hbm
        roof["traffic_over_algorithmic"] = traffic / dom_bytes
    if name == "prefill":
        # the chunkwise products at the tf32 tensor rate take longer than the algorithmic bytes at the
        # copy rate: the prefill is tensor-bound
        flops = prefill_flops(shape)
        tpk, tkind = tf32_peak()
        t_ach = flops / kdur[dom] / 1e12
        roof = {"bound": "tensor", "achieved": t_ach, "peak": tpk, "unit": "TFLOP/s", "frac": t_ach / tpk,
                "traffic": traffic, "kernel": dom, "flops_per_launch": flops, "bytes_per_launch": dom_bytes,
                "launch_us": kdur[dom] * 1e6, "hbm_gbs": achieved, "hbm_frac": achieved / hbm,
                "peak_source": (f"{tkind} bf16_tflops x nominal tf32/bf16 ratio 1.1/2.25"
                                + (" (MEASURED_PEAKS.json)" if tkind == "measured" else " (recipe fallback)")),
                "note": "operands run as 3xTF32 (three tf32 products per fp32 product); flops counted once"}
        if traffic:
            roof["traffic_over_algorithmic"] = traffic / dom_bytes
    step = ("chunked prefill" if name == "prefill" else
            "layer: input projection GEMM + verify + output projection GEMM, then rollback" if wl.proj else
            "verify with the previous step's rollback folded in (one launch)" if wl.rolled else
            "lazy verify: commit of the pending batch (accepted-prefix re-run) + outputs of the new one"
            if wl.lazy else ("the verify of every layer, then the rollback of every layer (one trim per slot)"
                             if wl.layers > 1 else "verify+rollback"))
    res = {
        "value": value, "unit": "tokens/s", "steps": steps, "warmup": warmup,
        "ms_per_step": dt / steps * 1e3,
        "config": {
            "workload": describe(shape), "act_dtype": shape.act, "state_dtype": "f32", "step": step,
            "l2": (f"{wl.n_sets} rotating buffer set(s), {wl.resident_per_set / 1e6:.0f} MB left in L2 per set "
                   f"(state, conv state and window, activations; captures stream out evict-first); every set "
                   f"is evicted by the others before it comes round again (> 3x L2 {l2 / 2**20:.0f} MiB), "
                   f"and a {3 * l2 / 2**20:.0f} MiB buffer is written between the warm-up and the timed steps"),
            "timing": f"CUDA events around CUDA-graph replays of {graph_len} step(s)",
        },
        "roofline": roof,
        "kernels_us": {k: v * 1e6 for k, v in kdur.items()},
        "step_bytes": wl.step_bytes(0),
        "step_gbs": wl.step_bytes(0) * steps / dt / 1e9,
        "gpu_launches": (wl.kernels_per_step if wl.kernels_per_step is not None
                         else 1 + -(-shape.n_slots * shape.n_v_heads * 3 // 152)) * steps,
        "clocks": clocks.summary(t_wall0 - 0.5, t_wall1 + 0.5),
        "kernel_clocks": clocks.summary(t_wall1, t_wall2 + 0.5),
    }
    st = recorded_step_traffic(name, kernel_source_sha(["verify.cu", "internal.cuh", "rollback.cu"]))
    if st and name != "prefill":
        sb = wl.step_bytes(0)
        res["step_traffic"] = {"dram_bytes_per_step": st, "over_algorithmic": st / sb,
                               "dram_gbs": st * steps / dt / 1e9, "dram_frac": st * steps / dt / 1e9 / hbm,
                               "how": "ncu range capture over many steps (profiles/traffic.json, key step)"}
    if wl.layers > 1:
        res["config"]["units"] = (f"tokens/s = slots x {shape.n_tokens} verify tokens through all "
                                  f"{shape.n_layers} layers per step")
    if name != "prefill" and not wl.tree:
        # accepted tokens: per slot T - trim of the step's rollback (averaged over the sets and layers)
        frac = float(np.mean(shape.n_tokens - wl.trims)) / shape.n_tokens
        res["accepted"] = {"value": value * frac, "unit": "accepted tokens/s",
                           "fraction": frac, "note": "the trims are drawn U{0..T-1} per slot, set and layer"}
    if name != "prefill" and wl.layers == 1 and not wl.proj:
        n_eager = 200
        res["eager"] = {"us_per_step": eager_step_duration(torch, wl, n_eager) * 1e6, "steps": n_eager,
                        "timing": "the same step launched eagerly from Python (no CUDA graph), back to back; "
                                  "ms_per_step above is the graph-amortised figure"}
    if bad:
        res["device_status_errors"] = bad
    if with_e2e:
        e_steps = max(20, min(steps, 500)) if name != "prefill" else max(5, min(steps, 50))
        if wl.layers > 1:
            e_steps = max(5, min(steps, 50))
        edt, h2d, d2h = wl.e2e(e_steps, device)
        edt = max_over_ranks(edt, device)
        res["e2e"] = {"value": wl.tokens_per_step * e_steps * world / edt, "unit": "tokens/s",
                      "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": e_steps,
                      "timing": ("wall clock, host sync per step; one H2D copy of all the step's inputs "
                                 "and one D2H copy of its outputs" if name != "prefill"
                                 else "wall clock, host sync per step"),
                      "api": ("gdn_verify_step_host (one C-ABI call per step with host buffers)"
                              if name != "prefill" and wl.layers == 1
                              and not (wl.tree or wl.lazy or wl.proj) else "the C-ABI calls of the step")}
    del wl
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    return res


def run_cuda(args):
    import torch
    import torch.distributed as dist

    world, rank, local = _dist()
    if world > 1:
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    import __graft_entry__
    if rank == 0 or world == 1:
        __graft_entry__.build()
    if world > 1:
        dist.barrier()
    import gated_deltanet_verify_gb300 as gdn
    gdn.lib()

    shape = WORKLOADS[args.workload]
    props = torch.cuda.get_device_properties(local)
    l2 = getattr(props, "L2_cache_size", 126 * 2 ** 20) or 126 * 2 ** 20
    if args.profile:
        # profiling mode (for ncu): eager steps over the rotating sets on the current stream, no timing
        if args.slots:
            shape = shape.with_(n_slots=args.slots)
        wl = (PrefillWorkload(shape, device, l2) if args.workload == "prefill"
              else VerifyWorkload(shape, device, l2))
        torch.cuda.synchronize()
        sp = torch.cuda.current_stream().cuda_stream
        if args.profile_range:
            # one rotation first (every set touched, L2 in its steady state), then the K steps inside one
            # cudaProfilerStart/Stop range, so that a range capture sees the captures' write-backs too
            for k in range(wl.n_sets):
                wl.step(k, sp)
            torch.cuda.synchronize()
            torch.cuda.profiler.start()
        for k in range(args.profile):
            wl.step(k % wl.n_sets, sp)
        torch.cuda.synchronize()
        if args.profile_range:
            torch.cuda.profiler.stop()
        return

    vis = [v for v in os.environ.get("CUDA_VISIBLE_DEVICES", "").split(",") if v.strip()]
    clocks = ClockSampler(int(vis[local]) if len(vis) > local and vis[local].strip().isdigit() else local)
    clocks.start()
    glm = max(args.graph_len, 128)
    head = measure(args.workload, args.steps, args.warmup, device, world, l2, clocks, not args.no_e2e, glm)
    per_config = {}
    if args.workload == HEADLINE and not args.no_per_config:
        for name in PER_CONFIG:
            k = max(args.steps, MIN_STEPS[name])
            per_config[name] = measure(name, k, max(args.warmup, 3), device, world, l2, clocks, False, glm)
    clocks.stop()

    res = {"metric": METRIC, "value": head.pop("value"), "unit": "tokens/s", "n_gpus": world,
           "steps": args.steps, "warmup": args.warmup, "ms_per_step": head.pop("ms_per_step"),
           "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
           "data": "synthetic (seeded splitmix64/Box-Muller)"}
    head.pop("steps")
    head.pop("warmup")
    res.update(head)
    res["config"]["parallelism"] = f"replicas x{world}"
    res["gpu_launches"] = head["gpu_launches"]
    if per_config:
        res["per_config"] = per_config
    if rank == 0 and not args.no_cpu_baseline:
        res["cpu_baseline"] = cpu_baseline(shape, args.cpu_seconds)
    if world > 1:
        dist.barrier()
        dist.destroy_process_group()
    if rank == 0:
        print(json.dumps(res))


# ---------------------------------------------------------------------------
# the oracle on the host cores
# ---------------------------------------------------------------------------

_PROJ_CACHE = {}


def _oracle_pass(shape, x, heads, n_threads, trims):
    import oracle
    if shape.n_embd:
        if shape.name not in _PROJ_CACHE:
            from workloads.synth import bf16_bits_to_f64
            _PROJ_CACHE[shape.name] = {k: bf16_bits_to_f64(v) for k, v in make_proj(shape).items()}
        p = _PROJ_CACHE[shape.name]
        r = oracle.layer_verify(shape, x, p["x"], p["w_in"], p["w_out"], head_mask=heads, n_threads=n_threads)
        oracle.rollback(shape, trims, r["state"], r["conv_state"], r["cap_state"], r["cap_conv"])
        return
    if shape.name == "prefill":
        oracle.verify(shape, x, capture=False, head_mask=heads, n_threads=n_threads)
        return
    if shape.name.startswith("rolled"):         # the same work as verify + rollback
        r = oracle.verify(shape, x, head_mask=heads, n_threads=n_threads)
        oracle.rollback(shape, trims, r["state"], r["conv_state"], r["cap_state"], r["cap_conv"])
        return
    if shape.name.startswith("lazy"):
        oracle.verify(shape, x, capture=False, head_mask=heads, n_threads=n_threads)
        oracle.commit_lazy(shape, x, trims, head_mask=heads, n_threads=n_threads)
        return
    if shape.name.startswith("tree"):
        r = oracle.verify_tree(shape, x, make_parents(shape, "spine"), head_mask=heads, n_threads=n_threads)
        oracle.rollback_tree(shape, np.asarray(trims, dtype=np.int32) - 1, x["state"], x["conv_state"],
                             r["cap_state"], r["cap_conv"])
        return
    r = oracle.verify(shape, x, head_mask=heads, n_threads=n_threads)
    oracle.rollback(shape, trims, r["state"], r["conv_state"], r["cap_state"], r["cap_conv"])


def _layer_inputs(shape, n):
    """Inputs of the first n layers of a workload (one layer: the workload's own)."""
    one = shape.with_(n_layers=1)
    return one, [make_inputs(one, layer=li) for li in range(max(1, min(n, shape.n_layers)))]


def _oracle_layers(one, layers, n_passes, cores):
    """n_passes whole passes of the step (every slot and every head) over the given layers in turn."""
    for k in range(n_passes):
        inp = layers[k % len(layers)]
        _oracle_pass(one, inp.as_f64(), None, cores, inp.trim)


def cpu_baseline(shape, seconds):
    """The fp64 oracle as it stands on all host cores: whole passes of the step over every slot and
    head of one layer, repeated (over the workload's layers in turn) for about `seconds`; tokens/s
    counts a token once it has been through every layer of the workload."""
    import oracle
    oracle.build()
    cores = os.cpu_count() or 1
    one, layers = _layer_inputs(shape, 4)
    t0 = time.perf_counter()
    _oracle_layers(one, layers, 1, cores)
    t_pass = time.perf_counter() - t0
    reps = max(1, int(seconds / max(t_pass, 1e-3)))
    t0 = time.perf_counter()
    _oracle_layers(one, layers, reps, cores)
    dt = time.perf_counter() - t0
    tok = one.n_slots * one.n_tokens * reps / shape.n_layers
    # one whole pass on a single thread as well, when it is expected to take under half a minute
    single = None
    if t_pass * cores < 30.0:
        t0 = time.perf_counter()
        _oracle_layers(one, layers, 1, 1)
        t1 = time.perf_counter() - t0
        single = {"value": one.n_slots * one.n_tokens / shape.n_layers / t1, "unit": "tokens/s",
                  "seconds": t1, "sample": "one whole pass of the step, 1 thread"}
    return {"value": tok / dt, "unit": "tokens/s", "cores": cores, "kind": "oracle",
            "single_thread": single,
            "sample": (f"{reps} whole pass(es) of the step (verify+rollback, or the prefill) over all "
                       f"{one.n_slots} slot(s) and {shape.n_v_heads} value heads of one layer, "
                       f"{one.n_tokens} tokens, fp64, {cores} threads, {dt:.1f} s; a token counts once it has "
                       f"been through all {shape.n_layers} layer(s)")}


def run_reference(args):
    world, rank, _ = _dist()
    if rank != 0:
        return
    import oracle
    oracle.build()
    shape = WORKLOADS[args.workload]
    cores = os.cpu_count() or 1
    one, layers = _layer_inputs(shape, 4)
    # each step: whole layer passes of the workload, as many as keep the run within about two minutes
    budget = 120.0 / max(1, args.steps + args.warmup)
    t0 = time.perf_counter()
    _oracle_layers(one, layers, 1, cores)
    t_pass = time.perf_counter() - t0
    per_step = int(max(1, min(shape.n_layers, budget / max(t_pass, 1e-4))))
    for _ in range(args.warmup):
        _oracle_layers(one, layers, per_step, cores)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        _oracle_layers(one, layers, per_step, cores)
    dt = time.perf_counter() - t0
    tok = one.n_slots * one.n_tokens * per_step * args.steps / shape.n_layers
    value = tok / dt
    sample = (f"each step: {per_step} whole pass(es) of the step over all {one.n_slots} slot(s) and "
              f"{shape.n_v_heads} value heads of one layer of {shape.name} (fp64 oracle, {cores} threads); "
              f"a token counts once it has been through all {shape.n_layers} layer(s)")
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt / args.steps * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded splitmix64/Box-Muller)",
        "config": {"workload": describe(shape), "act_dtype": shape.act, "parallelism": "host cores"},
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": cores, "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }))


def main():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["gdn", "reference"], default="gdn")
    ap.add_argument("--workload", choices=list(WORKLOADS), default=HEADLINE)
    ap.add_argument("--graph-len", type=int, default=64)
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-per-config", action="store_true",
                    help="time only the chosen workload (by default the headline also times one slot, 32 slots, "
                         "the prefill and the layer with its projections)")
    ap.add_argument("--slots", type=int, default=0, help="override the workload's slot count (profiling cases)")
    ap.add_argument("--profile", type=int, default=0, metavar="K",
                    help="run K untimed eager steps and exit (for ncu captures)")
    ap.add_argument("--profile-range", action="store_true",
                    help="with --profile: the K steps inside one profiler start/stop range (ncu range capture)")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.workload == "tiny":
        ap.error("the tiny workload is a parity case, not a bench workload")
    if args.impl == "reference":
        run_reference(args)
    else:
        run_cuda(args)


if __name__ == "__main__":
    main()
