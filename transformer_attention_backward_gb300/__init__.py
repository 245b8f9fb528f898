"""Attention backward chain for NVIDIA GB300 (sm_103a).

A thin PyTorch-facing binding of the C ABI in ``include/attn_bwd.h``: each
function checks dtypes, shapes and contiguity, allocates missing outputs with
torch (device memory only), and passes device pointers plus the current CUDA
stream to the library.  Every arithmetic step runs in the library's CUDA
kernels; nothing here computes, and there is no fallback path.

Functions (same names as the C ABI):
  softmax_bwd, rope_bwd, rmsnorm_bwd, rmsnorm_bwd_dgamma, relu2_mul_bwd,
  lora_bwd, attn_bwd_decode, attn_fwd_causal, attn_bwd_causal,
  attn_bwd_causal_saved_p, attn_bwd_causal_workspace_bytes, device_check
"""
from __future__ import annotations

import ctypes
import math

import torch

from . import _binding as _b

__all__ = ["softmax_bwd", "rope_bwd", "rmsnorm_bwd", "rmsnorm_bwd_dgamma", "relu2_mul_bwd", "lora_bwd",
           "attn_bwd_decode", "attn_fwd_causal", "attn_bwd_causal", "attn_bwd_causal_saved_p",
           "attn_bwd_causal_workspace_bytes", "device_check", "AbwError", "library"]

AbwError = _b.AbwError

_DT = {torch.float32: _b.F32, torch.bfloat16: _b.BF16}


def library():
    """The loaded ctypes library (built for sm_103a on first use)."""
    return _b.load()


def _p(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _s(stream):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _req(t, name, dtypes, shape=None):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype not in dtypes:
        raise TypeError(f"{name} dtype {t.dtype} not in {dtypes}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} shape {tuple(t.shape)} != {tuple(shape)}")


def device_check(stream=None) -> None:
    """Synchronize and raise if a kernel's bounded wait ran out."""
    _b.check(library().abw_device_check(_s(stream)), "abw_device_check")


def softmax_bwd(s, dy, dx=None, stream=None):
    """dx = s * (dy - sum(s * dy)) over the last axis; s, dy fp32."""
    _req(s, "s", (torch.float32,))
    _req(dy, "dy", (torch.float32,), s.shape)
    n = s.shape[-1] if s.dim() else 1
    rows = s.numel() // max(n, 1)
    if dx is None:
        dx = torch.empty_like(s)
    _req(dx, "dx", (torch.float32,), s.shape)
    _b.check(library().softmax_bwd(_p(s), _p(dy), _p(dx), rows, n, _s(stream)), "softmax_bwd")
    return dx


def rope_bwd(dy, theta=None, pos0=0, base=10000.0, interleaved=True, dx=None, stream=None):
    """R(-theta) on the rotary pairs of dy [B][T][H][D] fp32; theta [B*T][D/2]
    fp32 or None (then theta = (pos0 + t) base^(-2i/D)).  dx may be dy."""
    _req(dy, "dy", (torch.float32,))
    if dy.dim() != 4:
        raise ValueError("dy must be [B][T][H][D]")
    B, T, H, D = dy.shape
    if theta is not None:
        _req(theta, "theta", (torch.float32,), (B * T, D // 2))
    if dx is None:
        dx = torch.empty_like(dy)
    _req(dx, "dx", (torch.float32,), dy.shape)
    _b.check(library().rope_bwd(_p(dy), _p(dx), B, T, H, D, _p(theta), int(pos0), float(base),
                                1 if interleaved else 0, _s(stream)), "rope_bwd")
    return dx


def rmsnorm_bwd(x, gamma, dy, eps=1e-6, dx=None, dx_dtype=torch.float32, stream=None):
    """RMSNorm backward per row: x [rows][n] fp32/bf16, gamma [n] fp32,
    dy [rows][n] fp32 -> dx [rows][n] (fp32 or bf16)."""
    _req(x, "x", (torch.float32, torch.bfloat16))
    n = x.shape[-1]
    rows = x.numel() // n
    _req(gamma, "gamma", (torch.float32,), (n,))
    _req(dy, "dy", (torch.float32,), x.shape)
    if dx is None:
        dx = torch.empty(x.shape, dtype=dx_dtype, device=x.device)
    _req(dx, "dx", (torch.float32, torch.bfloat16), x.shape)
    _b.check(library().rmsnorm_bwd(_p(x), _DT[x.dtype], _p(gamma), _p(dy), _p(dx), _DT[dx.dtype], rows, n,
                                   float(eps), _s(stream)), "rmsnorm_bwd")
    return dx


def rmsnorm_bwd_dgamma(x, gamma, dy, eps=1e-6, dx=None, dgamma=None, dx_dtype=torch.float32, want_dx=True,
                       stream=None):
    """RMSNorm backward with the scale gradient.  x [rows][n] fp32/bf16,
    gamma [n] fp32, dy [rows][n] fp32.  Returns (dx or None, dgamma [n] fp32)."""
    _req(x, "x", (torch.float32, torch.bfloat16))
    n = x.shape[-1]
    rows = x.numel() // n
    _req(dy, "dy", (torch.float32,), x.shape)
    if want_dx:
        _req(gamma, "gamma", (torch.float32,), (n,))
        if dx is None:
            dx = torch.empty(x.shape, dtype=dx_dtype, device=x.device)
        _req(dx, "dx", (torch.float32, torch.bfloat16), x.shape)
    else:
        dx = None
    if dgamma is None:
        dgamma = torch.empty(n, dtype=torch.float32, device=x.device)
    _req(dgamma, "dgamma", (torch.float32,), (n,))
    _b.check(library().rmsnorm_bwd_dgamma(_p(x), _DT[x.dtype], _p(gamma) if want_dx else None, _p(dy), _p(dx),
                                          _DT[dx.dtype] if dx is not None else _b.F32, _p(dgamma), rows, n,
                                          float(eps), _s(stream)), "rmsnorm_bwd_dgamma")
    return dx, dgamma


def relu2_mul_bwd(gate, up, dh, dgate=None, dup=None, stream=None):
    """Backward of hidden = ReLU(gate)^2 * up: gate, up fp32/bf16 (same
    dtype), dh fp32, all the same shape.  Returns (dgate, dup) fp32."""
    _req(gate, "gate", (torch.float32, torch.bfloat16))
    _req(up, "up", (gate.dtype,), gate.shape)
    _req(dh, "dh", (torch.float32,), gate.shape)
    dgate = torch.empty(gate.shape, dtype=torch.float32, device=gate.device) if dgate is None else dgate
    dup = torch.empty(gate.shape, dtype=torch.float32, device=gate.device) if dup is None else dup
    _req(dgate, "dgate", (torch.float32,), gate.shape)
    _req(dup, "dup", (torch.float32,), gate.shape)
    _b.check(library().relu2_mul_bwd(_p(gate), _p(up), _DT[gate.dtype], _p(dh), _p(dgate), _p(dup), gate.numel(),
                                     _s(stream)), "relu2_mul_bwd")
    return dgate, dup


def lora_bwd_workspace_bytes(rows, r) -> int:
    return int(library().lora_bwd_workspace_bytes(rows, r))


def lora_bwd(x, dy, A, B, scale, dA=None, dB=None, workspace=None, stream=None):
    """LoRA adapter gradients of y = scale * B (A x): x [rows][n_in]
    fp32/bf16, dy [rows][n_out] fp32, A [r][n_in], B [n_out][r] fp32.
    Returns (dA, dB) fp32."""
    _req(x, "x", (torch.float32, torch.bfloat16))
    _req(A, "A", (torch.float32,))
    r, n_in = A.shape
    rows = x.numel() // n_in
    _req(x, "x", (x.dtype,), (rows, n_in))
    _req(B, "B", (torch.float32,))
    n_out = B.shape[0]
    _req(B, "B", (torch.float32,), (n_out, r))
    _req(dy, "dy", (torch.float32,), (rows, n_out))
    dA = torch.empty_like(A) if dA is None else dA
    dB = torch.empty_like(B) if dB is None else dB
    _req(dA, "dA", (torch.float32,), A.shape)
    _req(dB, "dB", (torch.float32,), B.shape)
    need = lora_bwd_workspace_bytes(rows, r)
    if workspace is None:
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=x.device)
    _req(workspace, "workspace", (torch.uint8,))
    _b.check(library().lora_bwd(_p(x), _DT[x.dtype], _p(dy), _p(A), _p(B), _p(dA), _p(dB), rows, n_in, n_out, r,
                                float(scale), _p(workspace), workspace.numel(), _s(stream)), "lora_bwd")
    return dA, dB


def attn_bwd_decode(q, k, v, dout, scale=None, rope_base=0.0, q_pos=-1, dq=None, dk=None, dv=None,
                    stream=None):
    """One query per sequence over a KV cache with grouped KV heads.
    q, dout [B][Hq][D] fp32; k, v [B][S][Hkv][D] fp32/bf16.
    Returns (dq [B][Hq][D], dk, dv [B][S][Hkv][D]) fp32."""
    _req(q, "q", (torch.float32,))
    B, Hq, D = q.shape
    _req(k, "k", (torch.float32, torch.bfloat16))
    _, S, Hkv, _ = k.shape
    _req(k, "k", (k.dtype,), (B, S, Hkv, D))
    _req(v, "v", (k.dtype,), (B, S, Hkv, D))
    _req(dout, "dout", (torch.float32,), (B, Hq, D))
    scale = 1.0 / math.sqrt(D) if scale is None else scale
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty(k.shape, dtype=torch.float32, device=k.device) if dk is None else dk
    dv = torch.empty(v.shape, dtype=torch.float32, device=v.device) if dv is None else dv
    _req(dq, "dq", (torch.float32,), q.shape)
    _req(dk, "dk", (torch.float32,), k.shape)
    _req(dv, "dv", (torch.float32,), v.shape)
    _b.check(library().attn_bwd_decode(_p(q), _p(k), _p(v), _p(dout), _p(dq), _p(dk), _p(dv), B, Hq, Hkv, S, D,
                                       _DT[k.dtype], float(scale), float(rope_base), int(q_pos), _s(stream)),
             "attn_bwd_decode")
    return dq, dk, dv


def attn_fwd_causal(q, k, v, scale=None, o=None, lse=None, stream=None):
    """Causal attention forward: q [B][T][Hq][D], k, v [B][T][Hkv][D] bf16.
    Returns (o [B][T][Hq][D] bf16, lse [B][Hq][T] fp32), the activations
    attn_bwd_causal consumes."""
    bf = (torch.bfloat16,)
    _req(q, "q", bf)
    B, T, Hq, D = q.shape
    _req(k, "k", bf)
    Hkv = k.shape[2]
    _req(k, "k", bf, (B, T, Hkv, D))
    _req(v, "v", bf, (B, T, Hkv, D))
    scale = 1.0 / math.sqrt(D) if scale is None else scale
    o = torch.empty_like(q) if o is None else o
    lse = torch.empty(B, Hq, T, dtype=torch.float32, device=q.device) if lse is None else lse
    _req(o, "o", bf, q.shape)
    _req(lse, "lse", (torch.float32,), (B, Hq, T))
    _b.check(library().attn_fwd_causal(_p(q), _p(k), _p(v), _p(o), _p(lse), B, T, Hq, Hkv, D, float(scale),
                                       _s(stream)), "attn_fwd_causal")
    return o, lse


def attn_bwd_causal_workspace_bytes(B, T, Hq, D) -> int:
    return int(library().attn_bwd_causal_workspace_bytes(B, T, Hq, D))


def attn_bwd_causal(q, k, v, o, dout, lse, scale=None, rope_base=0.0, pos0=0, dq=None, dk=None, dv=None,
                    workspace=None, stream=None):
    """Causal attention backward.  q, o, dout [B][T][Hq][D] bf16; k, v
    [B][T][Hkv][D] bf16; lse [B][Hq][T] fp32.  Returns fp32 (dq, dk, dv)."""
    bf = (torch.bfloat16,)
    _req(q, "q", bf)
    B, T, Hq, D = q.shape
    _req(k, "k", bf)
    Hkv = k.shape[2]
    _req(k, "k", bf, (B, T, Hkv, D))
    _req(v, "v", bf, (B, T, Hkv, D))
    _req(o, "o", bf, q.shape)
    _req(dout, "dout", bf, q.shape)
    _req(lse, "lse", (torch.float32,), (B, Hq, T))
    scale = 1.0 / math.sqrt(D) if scale is None else scale
    dq = torch.empty(q.shape, dtype=torch.float32, device=q.device) if dq is None else dq
    dk = torch.empty(k.shape, dtype=torch.float32, device=k.device) if dk is None else dk
    dv = torch.empty(v.shape, dtype=torch.float32, device=v.device) if dv is None else dv
    _req(dq, "dq", (torch.float32,), q.shape)
    _req(dk, "dk", (torch.float32,), k.shape)
    _req(dv, "dv", (torch.float32,), v.shape)
    need = attn_bwd_causal_workspace_bytes(B, T, Hq, D)
    if workspace is None:
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=q.device)
    _req(workspace, "workspace", (torch.uint8,))
    _b.check(library().attn_bwd_causal(_p(q), _p(k), _p(v), _p(o), _p(dout), _p(lse), _p(dq), _p(dk), _p(dv),
                                       B, T, Hq, Hkv, D, float(scale), float(rope_base), int(pos0),
                                       _p(workspace), workspace.numel(), _s(stream)),
             "attn_bwd_causal")
    return dq, dk, dv


def attn_bwd_causal_saved_p(q, k, v, p_attn, o, dout, scale=None, rope_base=0.0, pos0=0, dq=None, dk=None, dv=None,
                            workspace=None, stream=None):
    """Causal attention backward from the saved attention weights p_attn
    [B][Hq][T][T] bf16 (row = query) instead of the log-sum-exp.  q, o, dout
    [B][T][Hq][D] bf16; k, v [B][T][Hkv][D] bf16.  Returns fp32 (dq, dk, dv)."""
    bf = (torch.bfloat16,)
    _req(q, "q", bf)
    B, T, Hq, D = q.shape
    _req(k, "k", bf)
    Hkv = k.shape[2]
    _req(k, "k", bf, (B, T, Hkv, D))
    _req(v, "v", bf, (B, T, Hkv, D))
    _req(p_attn, "p_attn", bf, (B, Hq, T, T))
    _req(o, "o", bf, q.shape)
    _req(dout, "dout", bf, q.shape)
    scale = 1.0 / math.sqrt(D) if scale is None else scale
    dq = torch.empty(q.shape, dtype=torch.float32, device=q.device) if dq is None else dq
    dk = torch.empty(k.shape, dtype=torch.float32, device=k.device) if dk is None else dk
    dv = torch.empty(v.shape, dtype=torch.float32, device=v.device) if dv is None else dv
    _req(dq, "dq", (torch.float32,), q.shape)
    _req(dk, "dk", (torch.float32,), k.shape)
    _req(dv, "dv", (torch.float32,), v.shape)
    need = attn_bwd_causal_workspace_bytes(B, T, Hq, D)
    if workspace is None:
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=q.device)
    _req(workspace, "workspace", (torch.uint8,))
    _b.check(library().attn_bwd_causal_saved_p(_p(q), _p(k), _p(v), _p(p_attn), _p(o), _p(dout), _p(dq), _p(dk),
                                               _p(dv), B, T, Hq, Hkv, D, float(scale), float(rope_base), int(pos0),
                                               _p(workspace), workspace.numel(), _s(stream)),
             "attn_bwd_causal_saved_p")
    return dq, dk, dv
