"""Seeded synthetic inputs for the gated-delta SSM layer step.

This module only draws random numbers and lays them out in memory. It holds
none of the layer's arithmetic, so both the CUDA path and the CPU oracle can
consume its output without sharing any computation.

Every draw comes from ``numpy.random.default_rng(seed)`` in float32, in the
fixed order listed in ``_DRAW_ORDER``. Activations that the workload stores as
bf16 are rounded once, round-to-nearest-even, and both sides consume the same
bits (the oracle widens them to float64).

Distributions (per workload description of the Qwen3-Next style GDN layer):
  q/k/v pre-conv inputs  N(0, 1)
  conv weights           N(0, 0.5^2), no bias
  alpha                  N(0, 1)
  dt                     U(-1, 1)
  A_log                  U(0, ln 16)
  beta logits            N(0, 1)
  z                      N(0, 1)
  norm weight            1 + N(0, 0.1^2)
  initial state          zero, or N(0, 0.1^2) for the "warm" workloads
  conv history           zero, or N(0, 1) for the "warm" workloads
  accept counts          1 or 2, each with probability 0.5
"""
from __future__ import annotations

import dataclasses
import math

import numpy as np

_DRAW_ORDER = (
    "conv_w", "dt", "A_log", "norm_w", "state", "hist",
    "x", "z", "alpha", "beta_logit", "accept",
)


@dataclasses.dataclass(frozen=True)
class Shape:
    """Sizes and memory layout of one layer-step workload.

    ``x`` rows hold the token's projected [Q | K | V] stream in their first
    ``conv_dim`` elements and are ``x_stride`` elements apart. When
    ``z_in_x`` is set, the z gate lives inside the same row at element offset
    ``conv_dim`` (a fused qkvz projection row); otherwise z has its own dense
    ``[B][T][Hv*d]`` array.
    """
    B: int                 # sequences
    T: int                 # tokens per sequence in one call
    Hq: int                # QK heads
    Hv: int                # V heads (multiple of Hq)
    d: int = 128           # head_dim = d_k = d_v
    W: int = 4             # conv taps (d_conv)
    act_dtype: str = "bf16"  # "bf16" or "f32" for x, z, alpha, beta_logit
    x_stride: int = 0      # 0 -> conv_dim
    z_in_x: bool = False
    warm: bool = False     # random initial state / history instead of zeros
    chunk: int = 64

    @property
    def conv_dim(self) -> int:
        return (2 * self.Hq + self.Hv) * self.d

    @property
    def r(self) -> int:
        return self.Hv // self.Hq

    @property
    def xs(self) -> int:
        return self.x_stride or self.conv_dim

    @property
    def state_bytes(self) -> int:
        return self.B * self.Hv * self.d * self.d * 4


# The five workloads the layer is specified on (sizes from the workload list;
# Hq for the batched decode follows from conv_dim = (2 Hq + Hv) d).
WORKLOADS = {
    "tiny_seq": Shape(B=1, T=16, Hq=4, Hv=4, act_dtype="f32"),
    "decode_b1": Shape(B=1, T=1, Hq=16, Hv=32, warm=True),
    "decode_b64": Shape(B=64, T=1, Hq=16, Hv=48, x_stride=2 * 10240,
                        z_in_x=True, warm=True),
    "verify_k2": Shape(B=32, T=2, Hq=16, Hv=32, warm=True),
    "prefill": Shape(B=4, T=8192, Hq=16, Hv=32),
}


def bf16_round(a: np.ndarray) -> np.ndarray:
    """Round float32 values to bf16 (round to nearest, ties to even).

    Returns the 16-bit patterns as uint16. Inputs are finite.
    """
    u = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32)
    bias = ((u >> 16) & 1) + np.uint32(0x7FFF)
    return ((u + bias) >> 16).astype(np.uint16)


def bf16_to_f32(b: np.ndarray) -> np.ndarray:
    """Widen bf16 bit patterns (uint16) to float32, exactly."""
    return (b.astype(np.uint32) << 16).view(np.float32)


def _act(a: np.ndarray, dtype: str) -> np.ndarray:
    return bf16_round(a) if dtype == "bf16" else a.astype(np.float32)


def make_inputs(shape: Shape, seed: int, T: int | None = None) -> dict:
    """Draw one workload's inputs.

    Returns a dict of numpy arrays in the C-ABI layouts:
      x          [B][T][x_stride]   act dtype (uint16 bf16 bits or float32)
      z          [B][T][Hv*d]       act dtype (a strided view into x if z_in_x)
      alpha      [B][T][Hv]         act dtype
      beta_logit [B][T][Hv]         act dtype
      conv_w     [conv_dim][W]      float32
      dt, A_log  [Hv]               float32
      norm_w     [d]                float32
      state      [B][Hv][d][d]      float32, row j (v index) contiguous over i (k index)
      hist       [B][conv_dim][W-1] float32, oldest first
      accept     [B]                int32 in {1, 2}
    ``T`` overrides the shape's token count (e.g. to draw a shorter prefix).
    """
    T = shape.T if T is None else T
    rng = np.random.default_rng(seed)
    B, Hv, d, W, cd = shape.B, shape.Hv, shape.d, shape.W, shape.conv_dim
    f32 = np.float32
    out = {}
    out["conv_w"] = (rng.standard_normal((cd, W), dtype=f32) * f32(0.5))
    out["dt"] = rng.uniform(-1.0, 1.0, Hv).astype(f32)
    out["A_log"] = rng.uniform(0.0, math.log(16.0), Hv).astype(f32)
    out["norm_w"] = (f32(1.0) + rng.standard_normal(d, dtype=f32) * f32(0.1))
    if shape.warm:
        out["state"] = rng.standard_normal((B, Hv, d, d), dtype=f32) * f32(0.1)
        out["hist"] = rng.standard_normal((B, cd, W - 1), dtype=f32)
    else:
        out["state"] = np.zeros((B, Hv, d, d), f32)
        out["hist"] = np.zeros((B, cd, W - 1), f32)
    xs = shape.xs
    qkv = rng.standard_normal((B, T, cd), dtype=f32)
    z = rng.standard_normal((B, T, Hv * d), dtype=f32)
    if shape.z_in_x:
        assert xs >= cd + Hv * d
        row = np.zeros((B, T, xs), f32)
        row[..., :cd] = qkv
        row[..., cd:cd + Hv * d] = z
        out["x"] = _act(row, shape.act_dtype).reshape(B, T, xs)
        out["z"] = out["x"][..., cd:cd + Hv * d]
    else:
        if xs == cd:
            out["x"] = _act(qkv, shape.act_dtype).reshape(B, T, cd)
        else:
            row = np.zeros((B, T, xs), f32)
            row[..., :cd] = qkv
            out["x"] = _act(row, shape.act_dtype).reshape(B, T, xs)
        out["z"] = _act(z, shape.act_dtype).reshape(B, T, Hv * d)
    del qkv, z
    out["alpha"] = _act(rng.standard_normal((B, T, Hv), dtype=f32), shape.act_dtype).reshape(B, T, Hv)
    out["beta_logit"] = _act(rng.standard_normal((B, T, Hv), dtype=f32), shape.act_dtype).reshape(B, T, Hv)
    out["accept"] = (1 + (rng.random(B) < 0.5)).astype(np.int32)
    return out


def widen(a: np.ndarray, dtype: str) -> np.ndarray:
    """Activation array (bf16 bits or float32) -> float64, value-exact."""
    if dtype == "bf16":
        return bf16_to_f32(np.ascontiguousarray(a)).astype(np.float64)
    return np.asarray(a, dtype=np.float64)
