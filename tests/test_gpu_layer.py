"""GPU parity of the steps around the attention backward -- the RMSNorm scale
gradient, the FFN's ReLU^2 x Mul backward and the LoRA adapter gradients --
against the float64 oracle, through the C ABI.  fp32 arithmetic on values
the oracle reads exactly (bf16 inputs are upcast from their bits): max
relative error <= 1e-4 per output tensor."""
import numpy as np
import pytest
import torch

import oracle as O
from tests.helpers import TOL_BF16, TOL_F32, checked, to_np
from transformer_attention_backward_gb300 import workloads as W

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def abw():
    import transformer_attention_backward_gb300 as m
    m.library()
    return m


# ------------------------------------------------------------------ RMSNorm dgamma
@pytest.mark.parametrize("rows,n,xdt,dxdt", [
    (1, 8, torch.float32, torch.float32),          # the single-row spec size
    (3, 5, torch.float32, torch.float32),          # n % 4 != 0: per-element path
    (64, 2560, torch.float32, torch.float32),      # decode hidden rows
    (1024, 2560, torch.bfloat16, torch.bfloat16),  # one chain layer's rows
    (700, 2560, torch.bfloat16, torch.float32),    # more rows than blocks: rows strided per block
    (7, 10000, torch.float32, torch.float32),      # row longer than the register path
])
def test_rmsnorm_dgamma(abw, rows, n, xdt, dxdt):
    inp = W.rmsnorm_inputs(rows, n, seed=rows + n, x_dtype=xdt)
    x, g, dy = inp["x"].cuda(), inp["gamma"].cuda(), inp["dy"].cuda()
    dx, dg = abw.rmsnorm_bwd_dgamma(x, g, dy, eps=inp["eps"], dx_dtype=dxdt)
    abw.device_check()
    xs, gs, dys = to_np(inp["x"]), to_np(inp["gamma"]), to_np(inp["dy"])
    tag = f"rmsnorm_dgamma {rows}x{n} {str(xdt)[6:]}"
    assert checked("dgamma", to_np(dg), O.rmsnorm_backward_gamma(xs, dys, inp["eps"]), tag) <= TOL_F32
    tol = TOL_BF16 if dxdt == torch.bfloat16 else TOL_F32
    assert checked("dx", to_np(dx), O.rmsnorm_backward(xs, gs, dys, inp["eps"]), tag) <= tol


def test_rmsnorm_dgamma_only_and_twice(abw):
    """dx = NULL gives dgamma alone; a second call overwrites (the output is
    zeroed by the call, not accumulated into)."""
    inp = W.rmsnorm_inputs(300, 2560, seed=5, x_dtype=torch.bfloat16)
    x, dy = inp["x"].cuda(), inp["dy"].cuda()
    dg = torch.full((2560,), 7.0, device="cuda")
    for _ in range(2):
        dx, dg = abw.rmsnorm_bwd_dgamma(x, None, dy, eps=inp["eps"], dgamma=dg, want_dx=False)
        assert dx is None
    abw.device_check()
    ref = O.rmsnorm_backward_gamma(to_np(inp["x"]), to_np(inp["dy"]), inp["eps"])
    assert checked("dgamma", to_np(dg), ref, "rmsnorm_dgamma only") <= TOL_F32


# ------------------------------------------------------------------ ReLU^2 x Mul
@pytest.mark.parametrize("shape,dt", [
    ((4,), torch.float32),                 # the hand-derived closed-form size
    ((7,), torch.float32),                 # tail only
    ((1023,), torch.bfloat16),             # vector body + 3-element tail
    ((1024, 6912), torch.bfloat16),        # one chain layer's FFN activations
    ((333, 777), torch.float32),
])
def test_relu2_mul_bwd(abw, shape, dt):
    g = torch.Generator().manual_seed(int(np.prod(shape)))
    gate = torch.randn(*shape, generator=g).to(dt)
    up = torch.randn(*shape, generator=g).to(dt)
    dh = torch.randn(*shape, generator=g)
    dg, du = abw.relu2_mul_bwd(gate.cuda(), up.cuda(), dh.cuda())
    abw.device_check()
    rg, ru = O.relu2_mul_backward(to_np(gate), to_np(up), to_np(dh))
    tag = f"relu2_mul {shape} {str(dt)[6:]}"
    assert checked("dgate", to_np(dg), rg, tag) <= TOL_F32
    assert checked("dup", to_np(du), ru, tag) <= TOL_F32
    # ReLU: no gradient reaches either input where the gate is not positive
    off = (gate <= 0).cuda()
    assert float(dg[off].abs().max() if off.any() else 0.0) == 0.0
    assert float(du[off].abs().max() if off.any() else 0.0) == 0.0


def test_relu2_mul_bwd_golden(abw):
    import json
    import os
    with open(os.path.join(os.path.dirname(__file__), "golden", "closed_forms.json")) as f:
        gd = json.load(f)["relu2_mul"]
    t = lambda k: torch.tensor(gd[k], dtype=torch.float32).cuda()
    dg, du = abw.relu2_mul_bwd(t("gate"), t("up"), t("dh"))
    assert dg.cpu().tolist() == gd["dgate"] and du.cpu().tolist() == gd["dup"]


# ------------------------------------------------------------------ LoRA
@pytest.mark.parametrize("rows,n_in,n_out,r,xdt", [
    (1024, 2560, 2560, 8, torch.bfloat16),    # Q adapter of one chain layer
    (1024, 2560, 640, 8, torch.bfloat16),     # V adapter (5 KV heads x 128)
    (3, 16, 8, 5, torch.float32),             # rank not a multiple of 4
    (77, 256, 132, 16, torch.float32),        # largest rank, ragged row chunk
    (130, 4100, 1028, 8, torch.bfloat16),     # column parts of unequal width, ragged row tiles
    (33, 8, 4, 3, torch.float32),             # fewer 4-column groups than column parts
    (1, 4, 4, 1, torch.float32),
])
def test_lora_bwd(abw, rows, n_in, n_out, r, xdt):
    g = torch.Generator().manual_seed(rows * 7 + r)
    x = torch.randn(rows, n_in, generator=g).to(xdt)
    dy = torch.randn(rows, n_out, generator=g) * 0.01
    A = torch.randn(r, n_in, generator=g) * 0.02
    B = torch.randn(n_out, r, generator=g) * 0.02
    scale = 2.0
    dA, dB = abw.lora_bwd(x.cuda(), dy.cuda(), A.cuda(), B.cuda(), scale)
    abw.device_check()
    rA, rB = O.lora_backward(to_np(x), to_np(A), to_np(B), to_np(dy), scale)
    tag = f"lora {rows}x{n_in}->{n_out} r{r}"
    assert checked("dA", to_np(dA), rA, tag) <= TOL_F32
    assert checked("dB", to_np(dB), rB, tag) <= TOL_F32


def test_lora_bwd_no_rows_gives_zero(abw):
    x = torch.empty(0, 8, device="cuda")
    dy = torch.empty(0, 4, device="cuda")
    A, B = torch.ones(2, 8, device="cuda"), torch.ones(4, 2, device="cuda")
    dA = torch.full_like(A, 3.0)
    dB = torch.full_like(B, 3.0)
    abw.lora_bwd(x, dy, A, B, 1.0, dA=dA, dB=dB)
    abw.device_check()
    assert float(dA.abs().max()) == 0.0 and float(dB.abs().max()) == 0.0
