"""GPU parity of attn_bwd_decode against the float64 oracle, through the C ABI.

bf16 K/V with fp32 q/dout: the bound is 2e-2, but bf16 values are consumed
exactly and all arithmetic is fp32, so 1e-4 is asserted as well."""
import math

import numpy as np
import pytest
import torch

import oracle as O
from tests.helpers import TOL_F32, checked, max_rel_err, to_np
from transformer_attention_backward_gb300 import workloads as W

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def abw():
    import transformer_attention_backward_gb300 as m
    m.library()
    return m


def run_and_compare(abw, shape, seed, units=None, tol=TOL_F32):
    inp = W.decode_inputs(shape, seed=seed)
    g = {k: v.cuda() for k, v in inp.items()}
    dq, dk, dv = abw.attn_bwd_decode(g["q"], g["k"], g["v"], g["dout"], shape.scale, shape.rope_base, shape.q_pos)
    abw.device_check()
    q, k, v, do = (to_np(inp[n]) for n in ("q", "k", "v", "dout"))
    G = shape.Hq // shape.Hkv
    if units is None:
        rq, rk, rv = O.decode_backward(q, k, v, do, shape.scale, shape.rope_base, shape.q_pos)
        got = (to_np(dq), to_np(dk), to_np(dv))
        ref = (rq, rk, rv)
    else:
        got, ref = [[], [], []], [[], [], []]
        for b, j in units:
            hs = slice(j * G, (j + 1) * G)
            rq, rk, rv = O.decode_backward(q[b:b + 1, hs], k[b:b + 1, :, j:j + 1], v[b:b + 1, :, j:j + 1],
                                           do[b:b + 1, hs], shape.scale, shape.rope_base, shape.q_pos)
            for lst, x in zip(ref, (rq, rk, rv)):
                lst.append(x)
            got[0].append(to_np(dq[b:b + 1, hs]))
            got[1].append(to_np(dk[b:b + 1, :, j:j + 1]))
            got[2].append(to_np(dv[b:b + 1, :, j:j + 1]))
        got = [np.concatenate(x) for x in got]
        ref = [np.concatenate(x) for x in ref]
    tag = f"decode B{shape.B} Hq{shape.Hq}/{shape.Hkv} S{shape.S} D{shape.D} pos{shape.q_pos}"
    errs = [checked(n, a, r, tag) for n, a, r in zip(("dq", "dk", "dv"), got, ref)]
    assert max(errs) <= tol, errs
    return dq, dk, dv, inp


def test_decode_tiny_single_head(abw):
    """D = 8, 16 keys, one head, fp32 (the single-head spec shape)."""
    t = W.tiny_inputs()
    q = t["q"].reshape(1, 1, 8).cuda()
    k = t["k"].reshape(1, 16, 1, 8).cuda()
    v = t["v"].reshape(1, 16, 1, 8).cuda()
    do = t["dout"].reshape(1, 1, 8).cuda()
    dq, dk, dv = abw.attn_bwd_decode(q, k, v, do, t["scale"])
    rq, rk, rv = O.attention_backward_single(to_np(t["q"]), to_np(t["k"]), to_np(t["v"]), t["scale"], to_np(t["dout"]))
    assert max_rel_err(to_np(dq)[0, 0], rq) <= TOL_F32
    assert max_rel_err(to_np(dk)[0, :, 0], rk) <= TOL_F32
    assert max_rel_err(to_np(dv)[0, :, 0], rv) <= TOL_F32


@pytest.mark.parametrize("shape", [
    W.DecodeShape(B=2, Hq=8, Hkv=2, S=200, D=128, rope_base=500000.0, q_pos=199),   # ragged last tile
    W.DecodeShape(B=3, Hq=4, Hkv=4, S=65, D=64, kv_dtype=torch.float32),            # fp32 cache, 2 CTAs
    W.DecodeShape(B=1, Hq=8, Hkv=1, S=2000, D=128, rope_base=10000.0, q_pos=5),     # G = 8, 4 tiles per CTA
    W.DecodeShape(B=2, Hq=6, Hkv=2, S=513, D=32),                                   # G = 3, 5-CTA cluster
    W.DecodeShape(B=1, Hq=2, Hkv=1, S=1, D=16),                                     # one key
    W.DecodeShape(B=2, Hq=4, Hkv=2, S=77, D=256),                                   # 512-byte rows
    W.DecodeShape(B=1, Hq=2, Hkv=2, S=33, D=8, kv_dtype=torch.float32),             # 32-byte rows
    W.DecodeShape(B=2, Hq=16, Hkv=2, S=128, D=64, rope_base=10000.0, q_pos=127),    # swizzled D=64, G=8
    W.DecodeShape(B=1, Hq=2, Hkv=1, S=1024, D=64),                                  # swizzled D=64, G=2
    W.DecodeShape(B=1, Hq=8, Hkv=8, S=3000, D=64, kv_dtype=torch.float32),          # fp32 streaming, G=1
])
def test_decode_shapes(abw, shape):
    run_and_compare(abw, shape, seed=shape.S + shape.D)


# Shapes that take the tensor-core path: bf16 cache, D = 128 and 513 <= S <=
# 1024, so each CTA of the cluster owns one 128-key chunk (the last one
# possibly ragged).  The score and dP products then run as M=128 x N=16
# tcgen05 chains whose B operands hold 2G rows (each head's vector split into
# bf16 high and low parts), so every group size G = 1..8 is a different
# operand layout.
@pytest.mark.parametrize("shape", [
    W.DecodeShape(B=4, Hq=5, Hkv=5, S=1024, D=128, rope_base=500000.0, q_pos=1023),     # G = 1
    W.DecodeShape(B=4, Hq=10, Hkv=5, S=1024, D=128, rope_base=500000.0, q_pos=1023),    # G = 2
    W.DecodeShape(B=2, Hq=16, Hkv=2, S=1024, D=128, rope_base=500000.0, q_pos=1023),    # G = 8, N = 16 full
    W.DecodeShape(B=3, Hq=20, Hkv=5, S=1000, D=128, rope_base=500000.0, q_pos=999),     # ragged last chunk
    W.DecodeShape(B=3, Hq=20, Hkv=5, S=1024, D=128, rope_base=500000.0, q_pos=-1),      # RoPE off
    W.DecodeShape(B=2, Hq=12, Hkv=4, S=600, D=128, rope_base=10000.0, q_pos=17),        # G = 3, 5-CTA cluster
    W.DecodeShape(B=1, Hq=7, Hkv=1, S=513, D=128, rope_base=0.0, q_pos=-1),             # G = 7, 1-key tail
])
def test_decode_tensor_core_shapes(abw, shape):
    run_and_compare(abw, shape, seed=shape.S + shape.Hq)


def test_decode_one_key_closed_form(abw):
    shape = W.DecodeShape(B=2, Hq=4, Hkv=2, S=1, D=64, kv_dtype=torch.float32)
    dq, dk, dv, inp = run_and_compare(abw, shape, seed=3)
    # dS = P (dP - delta) is exactly 0; dq = scale (A - delta B) / L cancels to
    # fp32 rounding of one product (|dP K| ~ 10)
    assert float(dk.abs().max()) == 0.0
    assert float(dq.abs().max()) < 1e-5
    dsum = inp["dout"].reshape(2, 2, 2, 64).sum(2)   # sum over the group's heads
    assert torch.allclose(dv.cpu()[:, 0], dsum, atol=1e-6)


def test_decode_full_gqa(abw):
    """B = 64, 20 query heads over 5 KV heads, D = 128, S = 1024, bf16 cache,
    RoPE base 5e5 at position 1023 -- every output against the oracle."""
    dq, dk, dv, inp = run_and_compare(abw, W.DECODE_GQA, seed=W.SEED_BASE + 2)
    # invariants at full size: sum_j dK_j = 0 and sum_j dV_j = sum of the group's dout
    G = 4
    sk = dk.double().sum(1)
    assert float(sk.abs().max()) < 1e-4 * float(dk.abs().max()) * math.sqrt(1024)
    sv = dv.double().sum(1)
    ds = inp["dout"].double().reshape(64, 5, G, 128).sum(2).cuda()
    assert float((sv - ds).abs().max()) < 1e-4 * float(ds.abs().max())
