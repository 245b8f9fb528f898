"""Seeded synthetic inputs for the attention-backward workloads.

This module only draws random tensors: it holds none of the backward
arithmetic, so both the CUDA path and the float64 oracle can be fed from it.
Every tensor is drawn on the CPU from a ``torch.Generator`` seeded per
workload, in a fixed order, and then cast to the dtype the workload states.
The same host tensors are what the oracle reads (upcast to float64) and what
is copied to the GPU.

Shapes follow the workloads of the Hesper LoRA fine-tuning run (Hesper pull
request #1, commit log: a 30-layer model with 20 query heads and 5 KV heads,
head dim 128, hidden 2560) and the single-head specs of the Hesper
``VerifiedBackward`` API page.

Layouts (row-major):
  decode : q, dout, dq ``[B][Hq][D]``; K/V cache ``[B][S][Hkv][D]``
  causal : q, o, dout, dq ``[B][T][Hq][D]``; k, v, dk, dv ``[B][T][Hkv][D]``;
           lse ``[B][Hq][T]``
  rows   : x, dy, dx ``[rows][n]``; gamma ``[n]``
"""
from __future__ import annotations

import math
from dataclasses import dataclass

import torch

SEED_BASE = 1000


def _gen(seed: int) -> torch.Generator:
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed))
    return g


def _randn(g, *shape, std=1.0):
    t = torch.randn(*shape, generator=g, dtype=torch.float32)
    return t * std if std != 1.0 else t


# --------------------------------------------------------------------------
# Workload descriptions
# --------------------------------------------------------------------------
@dataclass(frozen=True)
class DecodeShape:
    B: int
    Hq: int
    Hkv: int
    S: int
    D: int
    kv_dtype: torch.dtype = torch.bfloat16
    rope_base: float = 500000.0
    q_pos: int = -1          # -1: no RoPE on dq

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.D)


@dataclass(frozen=True)
class CausalShape:
    B: int
    T: int
    Hq: int
    Hkv: int
    D: int
    rope_base: float = 10000.0   # <= 0: no RoPE on dq / dk
    pos0: int = 0
    qk_mult: float = 1.0         # Q and K multiplied by this after drawing

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.D)


# Decode-style batched backward with GQA (64 sequences, one query each).
DECODE_GQA = DecodeShape(B=64, Hq=20, Hkv=5, S=1024, D=128,
                         kv_dtype=torch.bfloat16, rope_base=500000.0, q_pos=1023)
RMSNORM_DECODE = (64, 2560)            # rows, hidden

# Causal training backward, T = 2048.
CAUSAL_2K = CausalShape(B=4, T=2048, Hq=20, Hkv=20, D=128, rope_base=10000.0)
# Long-context causal backward with Q, K pushed into softmax saturation.
CAUSAL_8K = CausalShape(B=1, T=8192, Hq=32, Hkv=32, D=128, rope_base=0.0, qk_mult=4.0)
# One layer of the 30-layer LoRA-shaped chain (GQA 20/5).
CHAIN_LAYER = CausalShape(B=2, T=512, Hq=20, Hkv=5, D=128, rope_base=500000.0)
CHAIN_LAYERS = 30
CHAIN_HIDDEN = 2560
CHAIN_DOUT_STD = 0.01


# --------------------------------------------------------------------------
# Single-head / tiny workload
# --------------------------------------------------------------------------
def tiny_inputs(seed: int = SEED_BASE + 1) -> dict:
    """Single-head single-query attention (D=8, 16 keys), a length-16
    softmax row, four RoPE pairs with angles in (-pi, pi), and an n=8
    RMSNorm row.  All fp32."""
    g = _gen(seed)
    out = {
        "q": _randn(g, 8),
        "k": _randn(g, 16, 8),
        "v": _randn(g, 16, 8),
        "dout": _randn(g, 8),
        # softmax: logits and an upstream gradient
        "soft_x": _randn(g, 16),
        "soft_dy": _randn(g, 16),
        # RoPE pairs
        "rope_x0": _randn(g, 4),
        "rope_x1": _randn(g, 4),
        "rope_theta": (torch.rand(4, generator=g) * 2.0 - 1.0) * math.pi,
        # RMSNorm row
        "rms_x": _randn(g, 8),
        "rms_gamma": 1.0 + 0.1 * _randn(g, 8),
        "rms_dy": _randn(g, 8),
        "scale": 1.0 / math.sqrt(8.0),
        "eps": 1e-6,
    }
    return out


# --------------------------------------------------------------------------
# Decode
# --------------------------------------------------------------------------
def decode_inputs(shape: DecodeShape = DECODE_GQA, seed: int = SEED_BASE + 2) -> dict:
    """q, dout fp32 N(0,1); K, V in ``shape.kv_dtype`` (N(0,1) then cast)."""
    g = _gen(seed)
    B, Hq, Hkv, S, D = shape.B, shape.Hq, shape.Hkv, shape.S, shape.D
    q = _randn(g, B, Hq, D)
    k = _randn(g, B, S, Hkv, D).to(shape.kv_dtype)
    v = _randn(g, B, S, Hkv, D).to(shape.kv_dtype)
    dout = _randn(g, B, Hq, D)
    return {"q": q, "k": k, "v": v, "dout": dout}


def rmsnorm_inputs(rows: int, n: int, seed: int, x_dtype=torch.float32,
                   dy_std: float = 1.0) -> dict:
    """x ~ N(0,1) (cast to ``x_dtype``), gamma = 1 + 0.1 N(0,1), dy ~ N(0, dy_std^2)."""
    g = _gen(seed)
    x = _randn(g, rows, n).to(x_dtype)
    gamma = 1.0 + 0.1 * _randn(g, n)
    dy = _randn(g, rows, n, std=dy_std)
    return {"x": x, "gamma": gamma, "dy": dy, "eps": 1e-6}


def softmax_rows_inputs(rows: int, n: int, seed: int) -> dict:
    """Logits x ~ N(0,1) and an upstream gradient dy ~ N(0,1)."""
    g = _gen(seed)
    return {"x": _randn(g, rows, n), "dy": _randn(g, rows, n)}


def rope_inputs(B: int, T: int, H: int, D: int, seed: int, explicit_theta: bool = False) -> dict:
    """dy ~ N(0,1) of shape [B][T][H][D]; optional explicit angles U(-pi, pi)
    of shape [B*T][D/2]."""
    g = _gen(seed)
    out = {"dy": _randn(g, B, T, H, D)}
    if explicit_theta:
        out["theta"] = (torch.rand(B * T, D // 2, generator=g) * 2.0 - 1.0) * math.pi
    return out


# --------------------------------------------------------------------------
# Causal
# --------------------------------------------------------------------------
def causal_inputs(shape: CausalShape, seed: int, dout_std: float = 1.0) -> dict:
    """Q, K, V, dOut bf16: N(0,1) draws (Q and K multiplied by
    ``shape.qk_mult`` before the cast; x4 is exact in bf16)."""
    g = _gen(seed)
    B, T, Hq, Hkv, D = shape.B, shape.T, shape.Hq, shape.Hkv, shape.D
    q = _randn(g, B, T, Hq, D) * shape.qk_mult
    k = _randn(g, B, T, Hkv, D) * shape.qk_mult
    v = _randn(g, B, T, Hkv, D)
    dout = _randn(g, B, T, Hq, D, std=dout_std)
    return {"q": q.to(torch.bfloat16), "k": k.to(torch.bfloat16),
            "v": v.to(torch.bfloat16), "dout": dout.to(torch.bfloat16)}


def chain_layer_inputs(layer: int, shape: CausalShape = CHAIN_LAYER,
                       hidden: int = CHAIN_HIDDEN, cfg: int = 5) -> dict:
    """Saved activations of one layer of the chain: the normed input x
    (N(0,1), bf16), gamma, and the layer's Q, K, V (bf16 N(0,1))."""
    g = _gen(100000 * cfg + layer)
    B, T, Hq, Hkv, D = shape.B, shape.T, shape.Hq, shape.Hkv, shape.D
    x = _randn(g, B * T, hidden).to(torch.bfloat16)
    gamma = 1.0 + 0.1 * _randn(g, hidden)
    q = _randn(g, B, T, Hq, D).to(torch.bfloat16)
    k = _randn(g, B, T, Hkv, D).to(torch.bfloat16)
    v = _randn(g, B, T, Hkv, D).to(torch.bfloat16)
    return {"x": x, "gamma": gamma, "q": q, "k": k, "v": v, "eps": 1e-6}


def chain_dhidden(shape: CausalShape = CHAIN_LAYER, hidden: int = CHAIN_HIDDEN,
                  cfg: int = 5) -> torch.Tensor:
    """The residual-stream gradient dHidden ~ N(0, 0.01^2), fp32, one draw;
    the residual connection hands it unchanged to every layer."""
    g = _gen(SEED_BASE + cfg)
    return _randn(g, shape.B * shape.T, hidden, std=CHAIN_DOUT_STD)
