"""GPU parity of the row kernels (softmax_bwd, rope_bwd, rmsnorm_bwd) against
the float64 oracle, through the C ABI.  fp32 inputs: max relative error
<= 1e-4; bf16 in/out: 2e-2."""
import math

import numpy as np
import pytest
import torch

import oracle as O
from tests.helpers import TOL_BF16, TOL_F32, max_rel_err, to_np
from transformer_attention_backward_gb300 import workloads as W

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def abw():
    import transformer_attention_backward_gb300 as m
    m.library()
    return m


def dev(t):
    return t.to("cuda")


# ------------------------------------------------------------------ softmax
def test_softmax_tiny(abw):
    t = W.tiny_inputs()
    s = torch.from_numpy(O.softmax_forward(t["soft_x"].numpy())).float()
    dx = abw.softmax_bwd(dev(s[None]), dev(t["soft_dy"][None]))
    ref = O.softmax_backward(to_np(s), to_np(t["soft_dy"]))
    assert max_rel_err(to_np(dx)[0], ref) <= TOL_F32
    assert abs(float(dx.double().sum())) < 1e-6


@pytest.mark.parametrize("rows,n", [(1, 1), (3, 5), (7, 1023), (129, 256), (5, 4096), (2048, 128), (300, 1000)])
def test_softmax_shapes(abw, rows, n):
    inp = W.softmax_rows_inputs(rows, n, seed=10 + rows + n)
    s = torch.from_numpy(O.softmax_forward(inp["x"].numpy())).float()
    dx = abw.softmax_bwd(dev(s), dev(inp["dy"]))
    ref = O.softmax_backward(to_np(s), to_np(inp["dy"]))
    assert max_rel_err(to_np(dx), ref) <= TOL_F32
    # sum over each row vanishes (up to fp32 rounding of the inputs)
    assert float(dx.double().sum(-1).abs().max()) < 1e-5 * max(1.0, float(dx.abs().max()))


# ------------------------------------------------------------------ RoPE
def test_rope_tiny_pairs(abw):
    t = W.tiny_inputs()
    dy = torch.stack([t["rope_x0"], t["rope_x1"]], -1).reshape(1, 4, 1, 2).contiguous()
    theta = t["rope_theta"].reshape(4, 1).contiguous()
    dx = abw.rope_bwd(dev(dy), theta=dev(theta))
    z0, z1 = O.rope_backward_pair(to_np(t["rope_x0"]), to_np(t["rope_x1"]), to_np(t["rope_theta"]))
    got = to_np(dx).reshape(4, 2)
    assert max_rel_err(got, np.stack([z0, z1], -1)) <= TOL_F32


@pytest.mark.parametrize("B,T,H,D,pos0,base,inter", [
    (2, 17, 3, 8, 0, 10000.0, True),
    (1, 33, 2, 6, 5, 10000.0, True),        # D % 4 != 0: scalar path
    (2, 9, 4, 16, 100, 500000.0, False),    # half-split pairs
    (1, 64, 32, 128, 8128, 10000.0, True),  # positions up to 8191
    (4, 2048, 20, 128, 0, 10000.0, True),   # the T = 2048 dq shape
])
def test_rope_positions(abw, B, T, H, D, pos0, base, inter):
    inp = W.rope_inputs(B, T, H, D, seed=B * T + H + D)
    dx = abw.rope_bwd(dev(inp["dy"]), pos0=pos0, base=base, interleaved=inter)
    pos = np.broadcast_to(np.arange(T) + pos0, (B, T))
    ref = O.rope_backward(to_np(inp["dy"]), O.rope_angles(pos, D, base), inter)
    assert max_rel_err(to_np(dx), ref) <= TOL_F32


def test_rope_explicit_theta_in_place(abw):
    inp = W.rope_inputs(3, 11, 5, 64, seed=77, explicit_theta=True)
    y = dev(inp["dy"]).clone()
    out = abw.rope_bwd(y, theta=dev(inp["theta"]), dx=y)
    assert out.data_ptr() == y.data_ptr()
    ref = O.rope_backward(to_np(inp["dy"]), to_np(inp["theta"]).reshape(3, 11, 32))
    assert max_rel_err(to_np(y), ref) <= TOL_F32


def test_rope_roundtrip_norm_on_gpu(abw):
    """R(-theta) preserves every pair's norm (RoPE section, Tier 1)."""
    inp = W.rope_inputs(2, 100, 4, 128, seed=5)
    dx = abw.rope_bwd(dev(inp["dy"]), base=10000.0)
    a = inp["dy"].double().reshape(-1, 2).norm(dim=-1)
    b = dx.double().cpu().reshape(-1, 2).norm(dim=-1)
    assert float((a - b).abs().max()) < 1e-5


# ------------------------------------------------------------------ RMSNorm
def test_rmsnorm_single_element_rows(abw):
    """n = 1: dx = dy g eps / ((x^2 + eps) rms) is a cancellation of two terms of
    size |dy g| / rms; fp32 error is bounded relative to those terms, not to
    the (tiny) result."""
    inp = W.rmsnorm_inputs(64, 1, seed=1)
    dx = abw.rmsnorm_bwd(dev(inp["x"]), dev(inp["gamma"]), dev(inp["dy"]), eps=inp["eps"])
    x, g, dy = to_np(inp["x"]), to_np(inp["gamma"]), to_np(inp["dy"])
    ref = O.rmsnorm_backward(x, g, dy, inp["eps"])
    scale = np.abs(dy * g) / np.sqrt(x * x + inp["eps"])
    assert np.all(np.abs(to_np(dx) - ref) <= 1e-5 * scale + 1e-30)


def test_rmsnorm_tiny(abw):
    t = W.tiny_inputs()
    dx = abw.rmsnorm_bwd(dev(t["rms_x"][None]), dev(t["rms_gamma"]), dev(t["rms_dy"][None]), eps=t["eps"])
    ref = O.rmsnorm_backward(to_np(t["rms_x"]), to_np(t["rms_gamma"]), to_np(t["rms_dy"]), t["eps"])
    assert max_rel_err(to_np(dx)[0], ref) <= TOL_F32


@pytest.mark.parametrize("rows,n,xdt,dxdt", [
    (64, 2560, torch.float32, torch.float32),     # decode-batch rows
    (1024, 2560, torch.bfloat16, torch.bfloat16),  # one chain layer, bf16 out
    (1024, 2560, torch.bfloat16, torch.float32),
    (3, 1001, torch.float32, torch.float32),       # n % 4 != 0
    (2, 10000, torch.float32, torch.bfloat16),     # n > 8192: two-pass path
    (5, 4, torch.float32, torch.float32),
])
def test_rmsnorm_shapes(abw, rows, n, xdt, dxdt):
    inp = W.rmsnorm_inputs(rows, n, seed=rows + n, x_dtype=xdt)
    dx = abw.rmsnorm_bwd(dev(inp["x"]), dev(inp["gamma"]), dev(inp["dy"]), eps=inp["eps"], dx_dtype=dxdt)
    ref = O.rmsnorm_backward(to_np(inp["x"]), to_np(inp["gamma"]), to_np(inp["dy"]), inp["eps"])
    tol = TOL_BF16 if dxdt == torch.bfloat16 else TOL_F32
    assert max_rel_err(to_np(dx), ref) <= tol
