"""Float64 CPU oracle for the attention backward chain.

TEST INFRASTRUCTURE.  Only the tests, the package's ``smoke()`` check and
the benchmark's CPU-baseline leg may import this package.  It shares no code
with the CUDA path and imports nothing from it: every function here takes
plain numpy arrays (any float dtype; they are upcast to float64 on entry)
and returns float64 arrays.

Each function is the plain definition of one step, written from these pages:

  * "Hesper.Training.VerifiedBackward" API documentation (sections Softmax,
    RoPE, RMSNorm, Scaled Dot-Product, Attention (full single-head),
    Numerical Gradient Verification) -- the CPU specs of the backward ops;
  * Hesper pull request #1, commit log ("Attention backward GPU kernels",
    "RMSNorm backward in attention chain", the 30-layer reverse iteration,
    "Tests/WrongBackwardTest.lean", the FFN-backward commit with the
    ReLU^2 x Mul backward, the LoRA backward at the end of the chain, the
    FlashAttention commits' online-softmax forward) -- the order of the chain,
    the negative controls and the steps around the attention backward;
  * DaisyChain-Train ``web/public/transformer.js`` (causal softmax in
    ``forward``, the batched attention block of ``backward``) -- the causal
    mask and the dK = dS^T Q / dV = A^T dctx products.

A library matmul serves as a step where the definition is a matrix product;
there is no blocking, fusion or reordering beyond the definitions.

Pins (see ``tests/test_oracle_pins.py``): central-difference VJPs, the
softmax sum-to-zero invariant, the RoPE round trip and closed forms, the
RMSNorm scale-invariance identity, adjoint (transpose) identities of every
contraction, brute-force VJPs of the whole attention on tiny shapes, the
decode = last-causal-row identity, GQA = repeated-KV MHA, and the negative
controls (zero / identity / negated backward and wrong RoPE sign must fail).
No function here is parity-unpinned.
"""
from __future__ import annotations

import math

import numpy as np

__all__ = [
    "softmax_forward", "softmax_backward", "softmax_backward_from_logits",
    "softmax_backward_sums_to_zero",
    "rope_forward_pair", "rope_backward_pair", "rope_roundtrip_check",
    "rope_angles", "rope_forward", "rope_backward",
    "rmsnorm_forward", "rmsnorm_backward", "rmsnorm_backward_gamma",
    "dot_product", "scaled_dot_forward", "scaled_dot_backward_q",
    "scaled_dot_backward_k",
    "attention_forward_single", "attention_backward_single",
    "attention_head_forward", "attention_head_backward", "attention_head_backward_saved_p",
    "decode_backward", "causal_forward", "causal_backward",
    "chain_layer_backward",
    "relu2_mul_forward", "relu2_mul_backward",
    "lora_forward", "lora_backward",
    "numerical_grad", "check_gradient",
]


def _f64(a):
    return np.asarray(a, dtype=np.float64)


# ==========================================================================
# Softmax  (VerifiedBackward, section "Softmax")
# ==========================================================================
def softmax_forward(x):
    """s_i = exp(x_i - max x) / sum_j exp(x_j - max x) along the last axis.

    softmaxForward; the max subtraction follows the causal softmax of
    transformer.js ``forward``."""
    x = _f64(x)
    m = np.max(x, axis=-1, keepdims=True)
    e = np.exp(x - m)
    return e / np.sum(e, axis=-1, keepdims=True)


def softmax_backward(s, dy):
    """dx_i = s_i * (dy_i - sum_j s_j * dy_j), given the probabilities s.

    softmaxBackward states this formula; Hesper's GPU path evaluates it on the
    probabilities it saved during the forward pass (pull request #1, the
    softmax-backward fix)."""
    s = _f64(s)
    dy = _f64(dy)
    inner = np.sum(s * dy, axis=-1, keepdims=True)
    return s * (dy - inner)


def softmax_backward_from_logits(x, dy):
    """softmaxBackward in the page's own signature (logits x, gradient dy)."""
    return softmax_backward(softmax_forward(x), dy)


def softmax_backward_sums_to_zero(x, dy):
    """softmaxBackwardSumsToZero: the sum of the backward output (must be 0)."""
    return np.sum(softmax_backward_from_logits(x, dy), axis=-1)


# ==========================================================================
# RoPE  (VerifiedBackward, section "RoPE (Rotary Position Embedding)")
# ==========================================================================
def rope_forward_pair(x0, x1, theta):
    """ropeForward: (x0 cos t - x1 sin t, x0 sin t + x1 cos t)."""
    x0, x1, theta = _f64(x0), _f64(x1), _f64(theta)
    c, s = np.cos(theta), np.sin(theta)
    return x0 * c - x1 * s, x0 * s + x1 * c


def rope_backward_pair(dy0, dy1, theta):
    """ropeBackward = rotation by -theta:
    (dy0 cos t + dy1 sin t, -dy0 sin t + dy1 cos t)."""
    dy0, dy1, theta = _f64(dy0), _f64(dy1), _f64(theta)
    c, s = np.cos(theta), np.sin(theta)
    return dy0 * c + dy1 * s, -dy0 * s + dy1 * c


def rope_roundtrip_check(x0, x1, theta, tol=1e-6):
    """ropeRoundtripCheck: R(-t) R(t) x == x within ``tol``."""
    y0, y1 = rope_forward_pair(x0, x1, theta)
    z0, z1 = rope_backward_pair(y0, y1, theta)
    return bool(np.all(np.abs(z0 - _f64(x0)) <= tol) and np.all(np.abs(z1 - _f64(x1)) <= tol))


def rope_angles(positions, D, base):
    """theta[p, i] = p * base^(-2i/D) for i in [0, D/2).

    The pages never state the frequency schedule; this is the standard
    rotary schedule, with ``base`` from the workload."""
    positions = _f64(positions)
    i = np.arange(D // 2, dtype=np.float64)
    inv_freq = np.power(float(base), -2.0 * i / float(D))
    return positions[..., None] * inv_freq


def _pair_views(x, interleaved):
    D = x.shape[-1]
    if interleaved:
        return x[..., 0::2], x[..., 1::2]
    return x[..., : D // 2], x[..., D // 2:]


def _assemble(a, b, interleaved):
    out = np.empty(a.shape[:-1] + (2 * a.shape[-1],), dtype=np.float64)
    if interleaved:
        out[..., 0::2] = a
        out[..., 1::2] = b
    else:
        h = a.shape[-1]
        out[..., :h] = a
        out[..., h:] = b
    return out


def rope_forward(x, theta, interleaved=True):
    """Rotate every pair of ``x [B][T][H][D]`` by theta ``[B][T][D/2]``
    (broadcast over heads).  Pairs are (2i, 2i+1) when ``interleaved``,
    else (i, i + D/2)."""
    x = _f64(x)
    th = _f64(theta)[:, :, None, :]
    a, b = _pair_views(x, interleaved)
    y0, y1 = rope_forward_pair(a, b, th)
    return _assemble(y0, y1, interleaved)


def rope_backward(dy, theta, interleaved=True):
    """Inverse rotation R(-theta) of every pair of ``dy [B][T][H][D]``."""
    dy = _f64(dy)
    th = _f64(theta)[:, :, None, :]
    a, b = _pair_views(dy, interleaved)
    z0, z1 = rope_backward_pair(a, b, th)
    return _assemble(z0, z1, interleaved)


# ==========================================================================
# RMSNorm  (VerifiedBackward, section "RMSNorm")
# ==========================================================================
def rmsnorm_forward(x, gamma, eps=1e-6):
    """y_i = gamma_i * x_i / rms, rms = sqrt(sum_j x_j^2 / n + eps), per row.

    The page does not render rmsNormForward's body; this is the standard
    RMSNorm consistent with the backward formula it does state."""
    x = _f64(x)
    gamma = _f64(gamma)
    n = x.shape[-1]
    rms = np.sqrt(np.sum(x * x, axis=-1, keepdims=True) / n + eps)
    return gamma * x / rms


def rmsnorm_backward(x, gamma, dy, eps=1e-6):
    """rmsNormBackward:
    dx_i = (1/rms) * (dy_i g_i - x_i * sum_j(dy_j g_j x_j) / (n rms^2))."""
    x = _f64(x)
    gamma = _f64(gamma)
    dy = _f64(dy)
    n = x.shape[-1]
    rms = np.sqrt(np.sum(x * x, axis=-1, keepdims=True) / n + eps)
    c = np.sum(dy * gamma * x, axis=-1, keepdims=True)
    return (dy * gamma - x * c / (n * rms * rms)) / rms


def rmsnorm_backward_gamma(x, dy, eps=1e-6):
    """Gradient of the RMSNorm scale, summed over rows:
    dgamma_i = sum over rows of dy_i x_i / rms.

    The page states only dx; the forward y_i = gamma_i x_i / rms is linear in
    gamma, so this is its plain derivative (the norm's other gradient)."""
    x = _f64(x)
    dy = _f64(dy)
    n = x.shape[-1]
    rms = np.sqrt(np.sum(x * x, axis=-1, keepdims=True) / n + eps)
    return np.sum((dy * x / rms).reshape(-1, n), axis=0)


# ==========================================================================
# Scaled dot product  (VerifiedBackward, section "Scaled Dot-Product")
# ==========================================================================
def dot_product(a, b):
    return float(np.sum(_f64(a) * _f64(b)))


def scaled_dot_forward(q, k, scale):
    """score = scale * q . k"""
    return scale * dot_product(q, k)


def scaled_dot_backward_q(k, scale, dscore):
    """dq = scale * dScore * k"""
    return _f64(k) * scale * dscore


def scaled_dot_backward_k(q, scale, dscore):
    """dk = scale * dScore * q"""
    return _f64(q) * scale * dscore


# ==========================================================================
# Attention, single head single query  (section "Attention (full single-head)")
# ==========================================================================
def attention_forward_single(q, K, V, scale):
    """output[d] = sum_s softmax(scale * q . K[s])_s * V[s][d]."""
    K, V = _f64(K), _f64(V)
    scores = np.array([scaled_dot_forward(q, K[s], scale) for s in range(K.shape[0])])
    attn = softmax_forward(scores)
    return attn @ V


def attention_backward_single(q, K, V, scale, dout):
    """attentionBackwardQ / attentionBackwardV, plus dK from scaledDotBackwardK.

    1. dAttn[s] = sum_d dOut[d] V[s][d]
    2. dScores = softmax_backward(scores, dAttn)
    3. dQ[d] = scale * sum_s dScores[s] K[s][d]
       dK[s] = scale * dScores[s] * q;  dV[s][d] = attn[s] * dOut[d]."""
    q, K, V, dout = _f64(q), _f64(K), _f64(V), _f64(dout)
    S = K.shape[0]
    scores = np.array([scaled_dot_forward(q, K[s], scale) for s in range(S)])
    attn = softmax_forward(scores)
    d_attn = np.array([dot_product(dout, V[s]) for s in range(S)])
    d_scores = softmax_backward(attn, d_attn)
    dq = np.zeros_like(q)
    for s in range(S):
        dq += scaled_dot_backward_q(K[s], scale, d_scores[s])
    dK = np.stack([scaled_dot_backward_k(q, scale, d_scores[s]) for s in range(S)])
    dV = np.outer(attn, dout)
    return dq, dK, dV


# ==========================================================================
# Attention, one head, many queries (matrix form of the same definitions)
# ==========================================================================
def _mask(Tq, S, causal, q_offset):
    """allowed[i, j]: query i (at absolute position q_offset + i) sees key j."""
    if not causal:
        return np.ones((Tq, S), dtype=bool)
    qi = np.arange(Tq)[:, None] + q_offset
    kj = np.arange(S)[None, :]
    return kj <= qi


def attention_head_forward(Q, K, V, scale, causal, q_offset=0):
    """Scores, masked softmax, output and log-sum-exp for one head.

    Returns (O [Tq][D], lse [Tq], P [Tq][S]); lse_i = log sum_j exp(s_ij)
    over the keys query i sees (natural log, of the scaled scores)."""
    Q, K, V = _f64(Q), _f64(K), _f64(V)
    s = scale * (Q @ K.T)
    allowed = _mask(Q.shape[0], K.shape[0], causal, q_offset)
    s = np.where(allowed, s, -np.inf)
    m = np.max(s, axis=-1, keepdims=True)
    e = np.exp(s - m)
    z = np.sum(e, axis=-1, keepdims=True)
    P = e / z
    lse = (m + np.log(z))[:, 0]
    return P @ V, lse, P


def attention_head_backward(Q, K, V, dO, scale, causal, q_offset=0):
    """dQ, dK, dV of one head (matrix form of the single-query steps):

    dP = dO V^T;  delta_i = sum_j P_ij dP_ij;  dS = P * (dP - delta);
    dQ = scale dS K;  dK = scale dS^T Q;  dV = P^T dO."""
    Q, K, V, dO = _f64(Q), _f64(K), _f64(V), _f64(dO)
    _, _, P = attention_head_forward(Q, K, V, scale, causal, q_offset)
    dP = dO @ V.T
    dS = softmax_backward(P, dP)
    dQ = scale * (dS @ K)
    dK = scale * (dS.T @ Q)
    dV = P.T @ dO
    return dQ, dK, dV


def attention_head_backward_saved_p(P, Q, K, V, dO, scale):
    """dQ, dK, dV of one head from a saved probability matrix P [Tq][S]
    (the attention weights the forward kept, masked entries 0) instead of
    recomputing it -- the form of transformer.js backward(), which reads the
    cached attention A: dV = A^T dctx, dA = dctx V^T,
    dS = A (dA - sum_j A dA), dQ = scale dS K, dK = scale dS^T Q."""
    P, Q, K, V, dO = _f64(P), _f64(Q), _f64(K), _f64(V), _f64(dO)
    dP = dO @ V.T
    dS = softmax_backward(P, dP)
    return scale * (dS @ K), scale * (dS.T @ Q), P.T @ dO


# ==========================================================================
# Decode-style batched backward with GQA
# ==========================================================================
def decode_backward(q, k, v, dout, scale, rope_base=0.0, q_pos=-1, interleaved=True):
    """One query per sequence over a KV cache.

    q, dout [B][Hq][D]; k, v [B][S][Hkv][D].  Query head h reads KV head
    h // (Hq/Hkv); dK, dV of a KV head sum over the query heads that share it.
    When ``q_pos >= 0`` and ``rope_base > 0`` the inverse rotation
    R(-theta(q_pos)) is applied to dq (RoPE backward on dQ)."""
    q, k, v, dout = _f64(q), _f64(k), _f64(v), _f64(dout)
    B, Hq, D = q.shape
    S, Hkv = k.shape[1], k.shape[2]
    G = Hq // Hkv
    dq = np.zeros_like(q)
    dk = np.zeros_like(k)
    dv = np.zeros_like(v)
    for b in range(B):
        for h in range(Hq):
            kv = h // G
            dQ, dK, dV = attention_head_backward(q[b, h][None, :], k[b, :, kv], v[b, :, kv],
                                                 dout[b, h][None, :], scale, causal=False)
            dq[b, h] = dQ[0]
            dk[b, :, kv] += dK
            dv[b, :, kv] += dV
    if q_pos >= 0 and rope_base > 0:
        theta = rope_angles(np.full((B, 1), q_pos), D, rope_base)      # [B][1][D/2]
        dq = rope_backward(dq[:, None], theta, interleaved)[:, 0]
    return dq, dk, dv


# ==========================================================================
# Causal multi-query backward
# ==========================================================================
def causal_forward(q, k, v, scale, heads=None):
    """O [B][T][Hq][D] and lse [B][Hq][T] of causal attention (keys j <= i).

    ``heads``: optional list of (b, h) to compute; the rest stay NaN."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    B, T, Hq, D = q.shape
    G = Hq // k.shape[2]
    o = np.full(q.shape, np.nan)
    lse = np.full((B, Hq, T), np.nan)
    for b, h in (heads if heads is not None else [(b, h) for b in range(B) for h in range(Hq)]):
        O, L, _ = attention_head_forward(q[b, :, h], k[b, :, h // G], v[b, :, h // G], scale, True)
        o[b, :, h] = O
        lse[b, h] = L
    return o, lse


def causal_backward(q, k, v, dout, scale, rope_base=0.0, pos0=0, kv_heads=None,
                    interleaved=True):
    """dq [B][T][Hq][D], dk, dv [B][T][Hkv][D] of causal attention.

    dK, dV of a KV head sum over its query heads.  When ``rope_base > 0``
    the RoPE backward R(-theta(pos0 + t)) is applied to dq and dk.
    ``kv_heads``: optional list of (b, kv_head) to compute (all query heads of
    the group are included); entries outside it stay NaN."""
    q, k, v, dout = _f64(q), _f64(k), _f64(v), _f64(dout)
    B, T, Hq, D = q.shape
    Hkv = k.shape[2]
    G = Hq // Hkv
    dq = np.full(q.shape, np.nan)
    dk = np.full(k.shape, np.nan)
    dv = np.full(v.shape, np.nan)
    units = kv_heads if kv_heads is not None else [(b, j) for b in range(B) for j in range(Hkv)]
    for b, kv in units:
        dk[b, :, kv] = 0.0
        dv[b, :, kv] = 0.0
        for h in range(kv * G, (kv + 1) * G):
            dQ, dK, dV = attention_head_backward(q[b, :, h], k[b, :, kv], v[b, :, kv],
                                                 dout[b, :, h], scale, causal=True)
            dq[b, :, h] = dQ
            dk[b, :, kv] += dK
            dv[b, :, kv] += dV
    if rope_base > 0:
        pos = np.broadcast_to(np.arange(T) + pos0, (B, T))
        theta = rope_angles(pos, D, rope_base)
        dq = rope_backward(dq, theta, interleaved)
        dk = rope_backward(dk, theta, interleaved)
    return dq, dk, dv


# ==========================================================================
# One layer of the backward chain (Hesper pull request #1, the commit that
# completes the attention backward chain: the sub-norm RMSNorm backward runs
# first, then the attention steps -- apply, softmax, score -- and RoPE last)
# ==========================================================================
def chain_layer_backward(x, gamma, dhidden, q, k, v, eps, scale, rope_base,
                         kv_heads=None):
    """RMSNorm backward of the saved normed input, its output reshaped to
    attention's dOut [B][T][Hq][D], then causal attention backward with RoPE
    backward on dq and dk.  Returns (dx, dq, dk, dv)."""
    B, T, Hq, D = q.shape
    dx = rmsnorm_backward(x, gamma, dhidden, eps)                 # [B*T][Hq*D]
    dout = dx.reshape(B, T, Hq, D)
    dq, dk, dv = causal_backward(q, k, v, dout, scale, rope_base, 0, kv_heads)
    return dx, dq, dk, dv


# ==========================================================================
# FFN gate (Hesper pull request #1, the FFN-backward commit: "ReLU^2 x Mul
# backward", the gated activation between the FFN's gate/up projections and
# its down projection)
# ==========================================================================
def relu2_mul_forward(gate, up):
    """hidden = ReLU(gate)^2 * up, element by element."""
    gate, up = _f64(gate), _f64(up)
    r = np.maximum(gate, 0.0)
    return r * r * up


def relu2_mul_backward(gate, up, dh):
    """The page's two formulas, element by element:
    dGate = dH * up * 2 ReLU(gate),  dUp = dH * ReLU(gate)^2."""
    gate, up, dh = _f64(gate), _f64(up), _f64(dh)
    r = np.maximum(gate, 0.0)
    return dh * up * 2.0 * r, dh * r * r


# ==========================================================================
# LoRA adapter gradients (Hesper pull request #1: "LoRA gradients use
# per-layer saved normedBuf", the chain that ends "RoPE backward -> dQ ->
# LoRA backward", and the residual fix: LoRA's input gradient feeds only the
# adapter's own parameter gradients dA, dB)
# ==========================================================================
def lora_forward(x, A, B, scale):
    """The adapter's added output y = scale * B (A x) per row: x [rows][n_in],
    A [r][n_in], B [n_out][r]; returns [rows][n_out].  The pages name the
    adapter (rank 8 on the Q and V projections) but print no formula; this is
    the standard low-rank update, with `scale` its alpha / r factor."""
    x, A, B = _f64(x), _f64(A), _f64(B)
    return scale * ((x @ A.T) @ B.T)


def lora_backward(x, A, B, dy, scale):
    """Parameter gradients of lora_forward, summed over rows:
    h = x A^T;  dB = scale dy^T h;  dh = scale dy B;  dA = dh^T x.
    Returns (dA [r][n_in], dB [n_out][r])."""
    x, A, B, dy = _f64(x), _f64(A), _f64(B), _f64(dy)
    h = x @ A.T
    dB = scale * (dy.T @ h)
    dh = scale * (dy @ B)
    dA = dh.T @ x
    return dA, dB


# ==========================================================================
# Numerical gradient verification (section "Numerical Gradient Verification")
# ==========================================================================
def numerical_grad(f, x, eps=1e-4):
    """Central differences (f(x + eps e_i) - f(x - eps e_i)) / (2 eps) of a
    scalar function, for every entry of x."""
    x = _f64(x).copy()
    g = np.zeros_like(x)
    flat = x.reshape(-1)
    gf = g.reshape(-1)
    for i in range(flat.size):
        old = flat[i]
        flat[i] = old + eps
        fp = f(x)
        flat[i] = old - eps
        fm = f(x)
        flat[i] = old
        gf[i] = (fp - fm) / (2.0 * eps)
    return g


def check_gradient(analytical, numerical, tol=1e-3):
    """|a - n| <= tol * max(1, |n|) for every entry (the page does not render
    whether checkGradient's tolerance is absolute or relative; this mixed
    form is absolute for small gradients and relative for large ones)."""
    a = _f64(analytical)
    n = _f64(numerical)
    if a.shape != n.shape:
        return False
    if not (np.all(np.isfinite(a)) and np.all(np.isfinite(n))):
        return False
    return bool(np.all(np.abs(a - n) <= tol * np.maximum(1.0, np.abs(n))))
