"""GPU parity of attn_fwd_causal (the forward whose O and log-sum-exp the
causal backward consumes) against the float64 oracle, through the C ABI.
O is bf16 (max relative error <= 2e-2); the log-sum-exp is fp32 arithmetic
on exact inputs (<= 1e-4).  Q and K x4 push the softmax into saturation, so
the running max moves by large steps and the lazy rescale of the output
accumulator runs."""
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


def compare(abw, shape, seed, heads=None):
    inp = W.causal_inputs(shape, seed=seed)
    g = {k: v.cuda() for k, v in inp.items()}
    o, lse = abw.attn_fwd_causal(g["q"], g["k"], g["v"], shape.scale)
    abw.device_check()
    heads = heads or [(b, h) for b in range(shape.B) for h in range(shape.Hq)]
    ro, rl = O.causal_forward(to_np(inp["q"]), to_np(inp["k"]), to_np(inp["v"]), shape.scale, heads=heads)
    tag = f"fwd B{shape.B} T{shape.T} Hq{shape.Hq}/{shape.Hkv} x{shape.qk_mult:g}"
    errs = []
    for b, h in heads:
        errs.append(checked("o", to_np(o[b, :, h]), ro[b, :, h], tag) / TOL_BF16)
        errs.append(checked("lse", to_np(lse[b, h]), rl[b, h], tag) / TOL_F32)
    assert max(errs) <= 1.0, errs
    return o, lse


@pytest.mark.parametrize("shape", [
    W.CausalShape(B=1, T=1, Hq=1, Hkv=1, D=128),
    W.CausalShape(B=2, T=130, Hq=4, Hkv=2, D=128),                # ragged tail, GQA
    W.CausalShape(B=1, T=256, Hq=2, Hkv=2, D=128),
    W.CausalShape(B=1, T=300, Hq=3, Hkv=1, D=128),                # G = 3
    W.CausalShape(B=1, T=257, Hq=2, Hkv=1, D=128, qk_mult=4.0),   # saturated, 1-row tail block
    W.CausalShape(B=1, T=1000, Hq=2, Hkv=2, D=128, qk_mult=4.0),  # many rescales
])
def test_forward_small(abw, shape):
    compare(abw, shape, seed=shape.T + 17)


def test_forward_t2048_sampled(abw):
    compare(abw, W.CAUSAL_2K, W.SEED_BASE + 3, heads=[(0, 0), (3, 19), (1, 7)])


def test_forward_t8192_saturated_sampled(abw):
    o, lse = compare(abw, W.CAUSAL_8K, W.SEED_BASE + 4, heads=[(0, 0), (0, 31)])
    assert bool(torch.isfinite(lse).all()) and bool(torch.isfinite(o.float()).all())
