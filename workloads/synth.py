"""Seeded synthetic inputs for the Gated DeltaNet verify / rollback / prefill path.

This module is the only code shared by the CUDA path's harness (tests, bench)
and the fp64 oracle.  It holds none of the method's arithmetic: it draws
random numbers, rounds them to the storage dtypes the kernels consume, and
names the workload shapes.  Both sides receive the *rounded* values, so any
difference between them is arithmetic, never input.

Generator: splitmix64 (Steele, Lea & Flood, "Fast splittable pseudorandom
number generators", OOPSLA 2014) in counter mode -- element i of a stream is
``mix(key + (i + 1) * GOLDEN)`` -- followed by the Box-Muller transform (cosine
branch, two uniforms per normal).  Everything is vectorised numpy uint64/fp64
and gives identical values on x86-64 and aarch64.

Workload shapes follow the GDN dims of the Qwen3.5 target in the lucebox-hub
``server/src/internal.h`` page (struct TargetWeights metadata: ssm_d_conv=4,
ssm_d_inner=6144, ssm_d_state=128, ssm_dt_rank=48, ssm_n_group=16), which give
16 QK heads x 128, 48 V heads x 128 and 2*16*128 + 48*128 = 10240 conv channels.
"""
from __future__ import annotations

import dataclasses
from typing import Dict, Optional

import numpy as np

GOLDEN = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)


def _mix(z: np.ndarray) -> np.ndarray:
    z = (z ^ (z >> np.uint64(30))) * _M1
    z = (z ^ (z >> np.uint64(27))) * _M2
    return z ^ (z >> np.uint64(31))


_CHUNK = 1 << 14


def _key(seed: int, tag: int) -> np.uint64:
    return _mix(np.array([(seed * 0x100000001B3 + tag) & 0xFFFFFFFFFFFFFFFF], dtype=np.uint64))[0]


def stream_u64(seed: int, tag: int, n: int, offset: int = 0) -> np.ndarray:
    """n uint64 draws of the stream (seed, tag), starting at element ``offset``."""
    with np.errstate(over="ignore"):
        ctr = np.arange(offset + 1, offset + n + 1, dtype=np.uint64)
        return _mix(_key(seed, tag) + ctr * GOLDEN)


def _draws(seed: int, tag: int, n: int, per_value: int, fn, out_dtype) -> np.ndarray:
    """Apply ``fn`` to consecutive blocks of uniforms in (0,1] (``per_value``
    uniforms per output value) without materialising the whole stream."""
    out = np.empty(n, dtype=out_dtype)
    key = _key(seed, tag)
    scale = 2.0 ** -53
    for lo in range(0, n, _CHUNK):
        hi = min(n, lo + _CHUNK)
        with np.errstate(over="ignore"):
            ctr = np.arange(per_value * lo + 1, per_value * hi + 1, dtype=np.uint64)
            u = _mix(key + ctr * GOLDEN)
        f = ((u >> np.uint64(11)).astype(np.float64) + 1.0) * scale
        out[lo:hi] = fn(f.reshape(hi - lo, per_value))
    return out


def uniform01(seed: int, tag: int, n: int) -> np.ndarray:
    """Uniforms in (0, 1]: the top 53 bits plus one, times 2^-53."""
    return _draws(seed, tag, n, 1, lambda f: f[:, 0], np.float64)


def normal(seed: int, tag: int, n: int, std: float = 1.0) -> np.ndarray:
    """Box-Muller normals N(0, std) (second argument is the standard deviation)."""
    return _draws(seed, tag, n, 2,
                  lambda f: std * np.sqrt(-2.0 * np.log(f[:, 0])) * np.cos(2.0 * np.pi * f[:, 1]),
                  np.float64)


def _box_muller(f: np.ndarray, std: float) -> np.ndarray:
    return std * np.sqrt(-2.0 * np.log(f[:, 0])) * np.cos(2.0 * np.pi * f[:, 1])


def normal_f32(seed: int, tag: int, n: int, std: float = 1.0) -> np.ndarray:
    """``normal`` rounded to float32 block by block (same values, less memory)."""
    return _draws(seed, tag, n, 2, lambda f: _box_muller(f, std), np.float32)


def normal_bf16_bits(seed: int, tag: int, n: int, std: float = 1.0) -> np.ndarray:
    """``normal`` rounded to bf16 (as ``to_bf16_bits``) block by block."""
    return _draws(seed, tag, n, 2, lambda f: to_bf16_bits(_box_muller(f, std)), np.uint16)


def uniform(seed: int, tag: int, n: int, lo: float, hi: float) -> np.ndarray:
    return lo + (hi - lo) * (uniform01(seed, tag, n) - 2.0 ** -53)


def randint(seed: int, tag: int, n: int, hi_exclusive: int) -> np.ndarray:
    """Integers uniform in {0 .. hi_exclusive-1} (floor of a [0,1) uniform)."""
    u = uniform01(seed, tag, n) - 2.0 ** -53
    return np.minimum((u * hi_exclusive).astype(np.int64), hi_exclusive - 1).astype(np.int32)


# ---------------------------------------------------------------------------
# storage rounding (round-to-nearest-even), done in integer arithmetic
# ---------------------------------------------------------------------------

def to_f32(x: np.ndarray) -> np.ndarray:
    return np.asarray(x, dtype=np.float64).astype(np.float32)


def to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """fp64 -> fp32 (RNE) -> bf16 (RNE) bit patterns as uint16."""
    f = to_f32(x)
    b = f.view(np.uint32).astype(np.uint64)
    rounding = np.uint64(0x7FFF) + ((b >> np.uint64(16)) & np.uint64(1))
    return ((b + rounding) >> np.uint64(16)).astype(np.uint16)


def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    return (bits.astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)


# ---------------------------------------------------------------------------
# workloads
# ---------------------------------------------------------------------------

@dataclasses.dataclass(frozen=True)
class Shape:
    name: str
    n_slots: int
    n_qk_heads: int
    n_v_heads: int
    d_k: int
    d_v: int
    n_tokens: int
    act: str            # "f32" or "bf16": dtype of qkv, z, alpha, beta_raw and out
    conv_width: int = 4
    n_layers: int = 1
    seed: int = 0
    chunk: int = 64     # prefill chunk length (prefill workloads only)
    n_embd: int = 0     # hidden size of the projections around the block (0: the block alone)

    @property
    def conv_channels(self) -> int:
        return 2 * self.n_qk_heads * self.d_k + self.n_v_heads * self.d_v

    @property
    def value_dim(self) -> int:
        return self.n_v_heads * self.d_v

    def with_(self, **kw) -> "Shape":
        return dataclasses.replace(self, **kw)


WORKLOADS: Dict[str, Shape] = {
    # 1 slot, 2 QK heads, 4 V heads (2 V per K), d=32, K+1=4, fp32 everything
    "tiny": Shape("tiny", 1, 2, 4, 32, 32, 4, "f32", seed=0),
    # one GDN layer of a 64-layer hybrid target, one verify slot, K+1=16
    "layer_verify": Shape("layer_verify", 1, 16, 48, 128, 128, 16, "bf16", seed=1),
    # 32 independent slots, same layer shape
    "multislot_verify": Shape("multislot_verify", 32, 16, 48, 128, 128, 16, "bf16", seed=2),
    # 48 GDN layers x 8 slots (every 4th layer of the 64 is full attention)
    "stack_verify": Shape("stack_verify", 8, 16, 48, 128, 128, 16, "bf16", n_layers=48, seed=3),
    # chunked prefill, 8192 tokens in chunks of 64
    "prefill": Shape("prefill", 1, 16, 48, 128, 128, 8192, "bf16", seed=4, chunk=64),
    # tree (DDTree) verify of a 16-node draft tree, one slot of the layer shape
    "tree_verify": Shape("tree_verify", 1, 16, 48, 128, 128, 16, "bf16", seed=5),
    # lazy capture on the layer shape (same inputs): outputs-only verify, then the accepted prefix re-run
    "lazy_verify": Shape("lazy_verify", 1, 16, 48, 128, 128, 16, "bf16", seed=1),
    "lazy_multislot_verify": Shape("lazy_multislot_verify", 32, 16, 48, 128, 128, 16, "bf16", seed=2),
    "lazy_stack_verify": Shape("lazy_stack_verify", 8, 16, 48, 128, 128, 16, "bf16", n_layers=48, seed=3),
    # the layer shape with each step's rollback folded into the next verify (one launch per step)
    "rolled_verify": Shape("rolled_verify", 1, 16, 48, 128, 128, 16, "bf16", seed=1),
    "rolled_multislot_verify": Shape("rolled_multislot_verify", 32, 16, 48, 128, 128, 16, "bf16", seed=2),
    "rolled_stack_verify": Shape("rolled_stack_verify", 8, 16, 48, 128, 128, 16, "bf16", n_layers=48, seed=3),
    # the layer with its projections (hidden 5120): x -> [qkv | z | alpha | beta] -> verify -> y
    "proj_verify": Shape("proj_verify", 1, 16, 48, 128, 128, 16, "bf16", seed=1, n_embd=5120),
}

# stream tags (one independent stream per tensor and layer)
_TAGS = {"qkv": 1, "z": 2, "alpha": 3, "beta_raw": 4, "A_log": 5, "dt_bias": 6,
         "conv_w": 7, "norm_w": 8, "state": 9, "conv_state": 10, "trim": 11, "parent": 13, "accept": 14,
         "x": 15, "w_in": 16, "w_out": 17}


def _tag(name: str, layer: int) -> int:
    return _TAGS[name] + 64 * layer


@dataclasses.dataclass
class Inputs:
    """Inputs for one layer, as the kernels store them.

    Activations are ``uint16`` bf16 bit patterns when ``shape.act == 'bf16'``
    and ``float32`` otherwise; parameters and states are ``float32``.
    ``as_f64()`` gives the exact fp64 values of those stored numbers, which is
    what the oracle consumes.
    """
    shape: Shape
    qkv: np.ndarray          # [B, T, C]
    z: np.ndarray            # [B, T, H_v*d_v]
    alpha: np.ndarray        # [B, T, H_v]
    beta_raw: np.ndarray     # [B, T, H_v]
    conv_w: np.ndarray       # [W, C] f32
    A_log: np.ndarray        # [H_v] f32
    dt_bias: np.ndarray      # [H_v] f32
    norm_w: np.ndarray       # [d_v] f32
    state: np.ndarray        # [B, H_v, d_v, d_k] f32
    conv_state: np.ndarray   # [B, W-1, C] f32
    trim: np.ndarray         # [B] int32

    def act_to_f64(self, a: np.ndarray) -> np.ndarray:
        if self.shape.act == "bf16":
            return bf16_bits_to_f64(a)
        return a.astype(np.float64)

    def as_f64(self) -> Dict[str, np.ndarray]:
        return {
            "qkv": self.act_to_f64(self.qkv), "z": self.act_to_f64(self.z),
            "alpha": self.act_to_f64(self.alpha), "beta_raw": self.act_to_f64(self.beta_raw),
            "conv_w": self.conv_w.astype(np.float64), "A_log": self.A_log.astype(np.float64),
            "dt_bias": self.dt_bias.astype(np.float64), "norm_w": self.norm_w.astype(np.float64),
            "state": self.state.astype(np.float64), "conv_state": self.conv_state.astype(np.float64),
            "trim": self.trim.copy(),
        }


def make_inputs(shape: Shape, layer: int = 0, seed: Optional[int] = None) -> Inputs:
    """Draw one layer's inputs for ``shape``.

    Distributions: qkv, z, alpha, beta_raw ~ N(0,1); A_log ~ U(0,2);
    dt_bias ~ N(0,0.5); conv w ~ N(0,0.5); norm w ~ U(0.5,1.5);
    state ~ N(0,0.1); conv_state ~ N(0,1) (it holds past raw qkv inputs);
    trim ~ U{0..T-1} per slot.
    """
    s = shape
    seed = s.seed if seed is None else seed
    B, T, C, Hv, dk, dv, W = s.n_slots, s.n_tokens, s.conv_channels, s.n_v_heads, s.d_k, s.d_v, s.conv_width
    rnd = s.act == "bf16"

    def act(name, shp):
        gen = normal_bf16_bits if rnd else normal_f32
        return gen(seed, _tag(name, layer), int(np.prod(shp))).reshape(shp)

    return Inputs(
        shape=s,
        qkv=act("qkv", (B, T, C)),
        z=act("z", (B, T, Hv * dv)),
        alpha=act("alpha", (B, T, Hv)),
        beta_raw=act("beta_raw", (B, T, Hv)),
        conv_w=to_f32(normal(seed, _tag("conv_w", layer), W * C, 0.5)).reshape(W, C),
        A_log=to_f32(uniform(seed, _tag("A_log", layer), Hv, 0.0, 2.0)),
        dt_bias=to_f32(normal(seed, _tag("dt_bias", layer), Hv, 0.5)),
        norm_w=to_f32(uniform(seed, _tag("norm_w", layer), dv, 0.5, 1.5)),
        state=normal_f32(seed, _tag("state", layer), B * Hv * dv * dk, 0.1).reshape(B, Hv, dv, dk),
        conv_state=normal_f32(seed, _tag("conv_state", layer), B * (W - 1) * C).reshape(B, W - 1, C),
        trim=randint(seed, _tag("trim", layer), B, T),
    )


def make_parents(shape: Shape, kind: str = "random", seed: Optional[int] = None, layer: int = 0) -> np.ndarray:
    """Draft-tree parents for a tree verify, [B][T] int32, parent[s][t] in [-1, t-1]
    (-1: the committed state before the batch).

    kind: "chain" (t-1: the linear verify), "star" (every token hangs off the
    root), "random" (each parent uniform over -1 .. t-1), "spine" (a DDTree-like
    shape: a main chain through every other token, each remaining token a
    one-token branch off the chain node before it).
    """
    s = shape
    seed = s.seed if seed is None else seed
    B, T = s.n_slots, s.n_tokens
    t = np.arange(T)
    if kind == "chain":
        par = np.tile(t - 1, (B, 1))
    elif kind == "star":
        par = np.full((B, T), -1)
    elif kind == "random":
        u = uniform01(seed, _tag("parent", layer), B * T).reshape(B, T) - 2.0 ** -53
        par = np.floor(u * (t + 1)).astype(np.int64) - 1          # uniform over -1 .. t-1
        par = np.minimum(par, t - 1)
    elif kind == "spine":
        par = np.empty((B, T), dtype=np.int64)
        for b in range(B):
            last = -1
            for i in range(T):
                if i % 2 == 0:                 # chain node
                    par[b, i] = last
                    last = i
                else:                          # branch off the previous chain node
                    par[b, i] = i - 1
    else:
        raise ValueError(kind)
    return par.astype(np.int32)


def tree_accept(shape: Shape, parents: np.ndarray, seed: Optional[int] = None, layer: int = 0) -> np.ndarray:
    """An accepted node per slot, uniform over -1 .. T-1 (-1: nothing accepted)."""
    s = shape
    seed = s.seed if seed is None else seed
    return (randint(seed, _tag("accept", layer), s.n_slots, s.n_tokens + 1) - 1).astype(np.int32)


def proj_in_rows(shape: Shape) -> int:
    """Output rows of the fused input projection: qkv channels, z, alpha, beta_raw."""
    return shape.conv_channels + shape.value_dim + 2 * shape.n_v_heads


def make_proj(shape: Shape, layer: int = 0, seed: Optional[int] = None) -> Dict[str, np.ndarray]:
    """Hidden input and random projection weights of one layer, as bf16 bit patterns
    (uint16): x [B, T, n_embd] ~ N(0, 1); w_in [C + H_v*d_v + 2*H_v, n_embd] and
    w_out [n_embd, H_v*d_v] ~ N(0, 1/fan_in), so the projected activations are
    ~N(0, 1) like the block's own inputs."""
    s = shape
    assert s.n_embd > 0
    seed = s.seed if seed is None else seed
    E, V = s.n_embd, s.value_dim
    return {
        "x": normal_bf16_bits(seed, _tag("x", layer), s.n_slots * s.n_tokens * E).reshape(s.n_slots, s.n_tokens, E),
        "w_in": normal_bf16_bits(seed, _tag("w_in", layer), proj_in_rows(s) * E, E ** -0.5).reshape(
            proj_in_rows(s), E),
        "w_out": normal_bf16_bits(seed, _tag("w_out", layer), E * V, V ** -0.5).reshape(E, V),
    }
