"""attn_bwd_causal_noalloc: the causal backward for callers that cannot
allocate device memory (inside a stream capture or an allocator callback, or
with device memory owned by another framework's pool).  Its scratch is the
library's fixed 32 MiB device array instead of a caller workspace.

Checked through the C ABI: two calls in a row (different shapes, so the
second call must not see the first call's leftovers in the shared array)
against attn_bwd_causal with a caller workspace, and the size limit.  This
file is collected last so that, in a run that stops at the first failure,
every other test has already run."""
import ctypes

import pytest
import torch

from tests.helpers import TOL_F32, max_rel_err, to_np
from transformer_attention_backward_gb300 import _binding as B
from transformer_attention_backward_gb300 import workloads as W

pytestmark = pytest.mark.gpu


def _p(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else None


def _run(lib, shape, seed, noalloc):
    g = {k: v.cuda() for k, v in W.causal_inputs(shape, seed=seed).items()}
    import transformer_attention_backward_gb300 as m
    o, lse = m.attn_fwd_causal(g["q"], g["k"], g["v"], shape.scale)
    dq = torch.empty(g["q"].shape, dtype=torch.float32, device="cuda")
    dk = torch.empty(g["k"].shape, dtype=torch.float32, device="cuda")
    dv = torch.empty_like(dk)
    st = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    args = [_p(g["q"]), _p(g["k"]), _p(g["v"]), _p(o), _p(g["dout"]), _p(lse), _p(dq), _p(dk), _p(dv),
            shape.B, shape.T, shape.Hq, shape.Hkv, shape.D, shape.scale, shape.rope_base, shape.pos0]
    if noalloc:
        status = lib.attn_bwd_causal_noalloc(*args, st)
    else:
        need = lib.attn_bwd_causal_workspace_bytes(shape.B, shape.T, shape.Hq, shape.D)
        ws = torch.empty(need, dtype=torch.uint8, device="cuda")
        status = lib.attn_bwd_causal(*args, _p(ws), need, st)
    assert status == B.OK, B.last_error()
    assert lib.abw_device_check(st) == B.OK
    return dq, dk, dv


def test_noalloc_matches_workspace_version_twice():
    lib = B.load()
    shapes = [
        (W.CausalShape(B=2, T=512, Hq=20, Hkv=5, D=128, rope_base=500000.0), 5),   # one chain layer
        (W.CausalShape(B=1, T=130, Hq=4, Hkv=2, D=128, rope_base=10000.0), 6),     # ragged, after a larger call
    ]
    for shape, seed in shapes:
        ref = _run(lib, shape, seed, noalloc=False)
        got = _run(lib, shape, seed, noalloc=True)
        for a, r in zip(got, ref):
            assert max_rel_err(to_np(a), to_np(r)) <= TOL_F32


def test_noalloc_rejects_sizes_beyond_the_scratch():
    lib = B.load()
    # B=4, T=2048, Hq=20 needs ~360 MB of scratch (mostly the bf16 dS tiles
    # of the causal half): refused before any launch
    assert lib.attn_bwd_causal_workspace_bytes(4, 2048, 20, 128) > 32 << 20
    status = lib.attn_bwd_causal_noalloc(None, None, None, None, None, None, None, None, None,
                                         4, 2048, 20, 20, 128, 0.088, 0.0, 0, None)
    assert status == B.EWORKSPACE
    assert "built-in" in B.last_error()
