"""Seeded synthetic inputs for the GDN sublayer (shared by the tests, the benchmark and the oracle).

This module only draws random tensors; it holds none of the method's arithmetic.  Shapes and
distributions follow the workloads the GDN pages describe (pegainfer PR #1152 "Reference golden
for the GDN sublayer", Summary: hidden size 2560, 16 K heads and 48 V heads of width 128, a
four-tap conv, a sigmoid output gate):

  x (conv input)  [T, C]        bf16  ~ N(0, 1)           C = 2*Hk*Dk + Hv*Dv = 10240
  conv weight     [C, W]        bf16  ~ 0.5 * N(0, 1)
  g (log decay)   [T, Hv]       fp32  = -U(0.001, 2)
  beta            [T, Hv]       fp32  = sigmoid(N(0, 1))
  z (gate input)  [T, Hv, Dv]   bf16  ~ N(0, 1)
  norm weight     [Dv]          bf16  = 1 + 0.1 * N(0, 1)
  state           [N, Hv, Dv, Dk] fp32 ~ 0.1 * N(0, 1)  (or zeros)
  conv state      [N, C, W-1]   bf16  ~ N(0, 1)           (or zeros)

All tensors are generated on the CPU from one ``torch.Generator`` seeded with ``seed``, in a
fixed order, so that the same seed gives the same bytes on every machine.
"""
from __future__ import annotations

import math
from dataclasses import dataclass

import torch


@dataclass(frozen=True)
class Geometry:
    num_k_heads: int = 16
    num_v_heads: int = 48
    head_k_dim: int = 128
    head_v_dim: int = 128
    conv_width: int = 4

    @property
    def conv_dim(self) -> int:
        return 2 * self.num_k_heads * self.head_k_dim + self.num_v_heads * self.head_v_dim

    @property
    def q_scale(self) -> float:
        return 1.0 / math.sqrt(self.head_k_dim)


QWEN_GDN = Geometry()

# the lengths of the five workloads (prefill sequences or decode batch)
CHUNK_BOUNDARY_LENGTHS = (63, 64, 65, 80, 128)
BATCHED_LENGTHS = (4096, 4096, 4096, 4096)
VARLEN_LENGTHS = (1, 17, 63, 64, 65, 1000, 8191, 22334)
DECODE_BATCH = 256
DECODE_STEPS = 64


def cu_seqlens_of(lengths) -> torch.Tensor:
    cu = [0]
    for L in lengths:
        cu.append(cu[-1] + int(L))
    return torch.tensor(cu, dtype=torch.int32)


def _normal(gen, shape, std=1.0, mean=0.0):
    t = torch.randn(shape, generator=gen, dtype=torch.float32)
    if std != 1.0:
        t.mul_(std)
    if mean != 0.0:
        t.add_(mean)
    return t


def prefill_inputs(lengths, seed: int, geo: Geometry = QWEN_GDN, zero_state: bool = False,
                   random_conv_state: bool = False) -> dict:
    """Inputs of one packed (varlen) prefill call over sequences of the given lengths."""
    gen = torch.Generator().manual_seed(int(seed))
    lengths = [int(L) for L in lengths]
    N, T, C = len(lengths), sum(lengths), geo.conv_dim
    hv, dv, dk, W = geo.num_v_heads, geo.head_v_dim, geo.head_k_dim, geo.conv_width
    x = _normal(gen, (T, C)).to(torch.bfloat16)
    conv_w = _normal(gen, (C, W), std=0.5).to(torch.bfloat16)
    g = -(torch.rand((T, hv), generator=gen, dtype=torch.float32) * (2.0 - 0.001) + 0.001)
    beta = torch.sigmoid(_normal(gen, (T, hv)))
    z = _normal(gen, (T, hv, dv)).to(torch.bfloat16)
    norm_w = _normal(gen, (dv,), std=0.1, mean=1.0).to(torch.bfloat16)
    if zero_state:
        state0 = torch.zeros((N, hv, dv, dk), dtype=torch.float32)
    else:
        state0 = _normal(gen, (N, hv, dv, dk), std=0.1)
    if random_conv_state:
        conv_state0 = _normal(gen, (N, C, W - 1)).to(torch.bfloat16)
    else:
        conv_state0 = torch.zeros((N, C, W - 1), dtype=torch.bfloat16)
    return {
        "lengths": lengths, "cu_seqlens": cu_seqlens_of(lengths), "x": x, "conv_w": conv_w,
        "g": g, "beta": beta, "z": z, "norm_w": norm_w, "state0": state0,
        "conv_state0": conv_state0, "geo": geo, "q_scale": geo.q_scale,
    }


def decode_inputs(batch: int, steps: int, seed: int, geo: Geometry = QWEN_GDN) -> dict:
    """Inputs of `steps` consecutive decode steps over `batch` independent sequences."""
    gen = torch.Generator().manual_seed(int(seed))
    B, C = int(batch), geo.conv_dim
    hv, dv, dk, W = geo.num_v_heads, geo.head_v_dim, geo.head_k_dim, geo.conv_width
    conv_w = _normal(gen, (C, W), std=0.5).to(torch.bfloat16)
    norm_w = _normal(gen, (dv,), std=0.1, mean=1.0).to(torch.bfloat16)
    state0 = _normal(gen, (B, hv, dv, dk), std=0.1)
    conv_state0 = _normal(gen, (B, C, W - 1)).to(torch.bfloat16)
    x = _normal(gen, (steps, B, C)).to(torch.bfloat16)
    g = -(torch.rand((steps, B, hv), generator=gen, dtype=torch.float32) * (2.0 - 0.001) + 0.001)
    beta = torch.sigmoid(_normal(gen, (steps, B, hv)))
    z = _normal(gen, (steps, B, hv, dv)).to(torch.bfloat16)
    return {
        "batch": B, "steps": int(steps), "x": x, "conv_w": conv_w, "g": g, "beta": beta, "z": z,
        "norm_w": norm_w, "state0": state0, "conv_state0": conv_state0, "geo": geo,
        "q_scale": geo.q_scale,
    }


def gate_inputs(rows: int, seed: int, geo: Geometry = QWEN_GDN) -> dict:
    """Projection outputs and parameters of the gates for `rows` rows (tokens or sequences).

    a, b ~ N(0, 1) -> bf16 [rows, Hv]; A_log ~ U(-1, 0.5) and dt_bias ~ 0.5 N(0, 1) fp32 [Hv] (no
    checkpoint is available; these put g mostly in (-4, 0), near the -U(0.001, 2) of the g
    workloads, with a tail of stronger decays).
    """
    gen = torch.Generator().manual_seed(int(seed))
    hv = geo.num_v_heads
    return {
        "a": _normal(gen, (rows, hv)).to(torch.bfloat16),
        "b": _normal(gen, (rows, hv)).to(torch.bfloat16),
        "A_log": torch.rand((hv,), generator=gen, dtype=torch.float32) * 1.5 - 1.0,
        "dt_bias": _normal(gen, (hv,), std=0.5),
    }


# The KDA layer's geometry on the pages: q, k and v of 64 heads of 128 (a 3 x 64 x 128 conv),
# one V head per K head.
KDA_GEO = Geometry(num_k_heads=64, num_v_heads=64, head_k_dim=128, head_v_dim=128, conv_width=4)


def kda_decode_inputs(batch: int, steps: int, seed: int, geo: Geometry = KDA_GEO) -> dict:
    """decode_inputs with a per-key-channel log decay g = -U(0.001, 2) [steps, batch, Hv, Dk]."""
    d = decode_inputs(batch, steps, seed, geo)
    gen = torch.Generator().manual_seed(int(seed) + 1)
    d["g"] = -(torch.rand((steps, batch, geo.num_v_heads, geo.head_k_dim), generator=gen,
                          dtype=torch.float32) * (2.0 - 0.001) + 0.001)
    return d


def kda_prefill_inputs(lengths, seed: int, geo: Geometry = KDA_GEO, **kw) -> dict:
    """prefill_inputs with a per-key-channel log decay g = -U(0.001, 2) [T, Hv, Dk]."""
    d = prefill_inputs(lengths, seed, geo, **kw)
    gen = torch.Generator().manual_seed(int(seed) + 1)
    T = sum(int(L) for L in lengths)
    d["g"] = -(torch.rand((T, geo.num_v_heads, geo.head_k_dim), generator=gen,
                          dtype=torch.float32) * (2.0 - 0.001) + 0.001)
    return d
