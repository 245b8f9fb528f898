"""Forward-pass activations that the causal backward consumes (O and lse).

The backward path starts from the tensors a training forward pass saves: the
attention output O (bf16) and the log-sum-exp of the scaled scores (fp32).
This module produces them for synthetic inputs, in fp32 arithmetic on the
GPU with torch, outside any timed region.  It is input preparation, like
drawing the random tensors; it is not part of the backward path, which runs
entirely in the library's kernels.
"""
from __future__ import annotations

import torch


@torch.no_grad()
def causal_forward(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, scale: float):
    """q [B][T][Hq][D], k, v [B][T][Hkv][D] (bf16, on the GPU).
    Returns (o [B][T][Hq][D] bf16, lse [B][Hq][T] fp32)."""
    B, T, Hq, D = q.shape
    Hkv = k.shape[2]
    G = Hq // Hkv
    o = torch.empty_like(q)
    lse = torch.empty(B, Hq, T, dtype=torch.float32, device=q.device)
    mask = torch.ones(T, T, dtype=torch.bool, device=q.device).triu_(1)
    # keep one [heads][T][T] fp32 score block under ~2 GiB
    hstep = max(1, min(Hq, (2 << 30) // max(1, T * T * 4)))
    for b in range(B):
        for h0 in range(0, Hq, hstep):
            h1 = min(Hq, h0 + hstep)
            qh = q[b, :, h0:h1].float().transpose(0, 1)                        # [h][T][D]
            kh = k[b, :, [h // G for h in range(h0, h1)]].float().transpose(0, 1)
            vh = v[b, :, [h // G for h in range(h0, h1)]].float().transpose(0, 1)
            s = torch.matmul(qh, kh.transpose(1, 2)) * scale
            s.masked_fill_(mask, float("-inf"))
            l = torch.logsumexp(s, dim=-1)                                      # [h][T]
            p = torch.exp(s - l[..., None])
            o[b, :, h0:h1] = torch.matmul(p, vh).transpose(0, 1).to(torch.bfloat16)
            lse[b, h0:h1] = l
            del s, p
    return o, lse
