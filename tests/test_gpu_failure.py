"""Failure detection on the GPU without faulting it: a bounded wait on a
barrier nothing arrives at runs out, the kernel records the timeout and
returns, the host reads ABW_ETIMEOUT, and the context stays usable."""
import pytest
import torch

from transformer_attention_backward_gb300 import _binding as B
from transformer_attention_backward_gb300 import workloads as W

pytestmark = pytest.mark.gpu


def test_wait_timeout_reported_and_context_usable():
    import transformer_attention_backward_gb300 as m
    lib = m.library()
    st = torch.cuda.current_stream()
    assert lib.abw_device_check(st.cuda_stream) == B.OK          # clean to start with
    assert lib.abw_selftest_wait_timeout(2_000_000, st.cuda_stream) == B.OK   # 2 ms limit
    assert lib.abw_device_check(st.cuda_stream) == B.ETIMEOUT
    assert "bounded wait" in B.last_error()
    assert lib.abw_device_check(st.cuda_stream) == B.OK          # the word was cleared
    # the context still works
    x = torch.randn(4, 64, device="cuda")
    s = torch.softmax(x, -1)
    dx = m.softmax_bwd(s, torch.ones_like(s))
    m.device_check()
    assert float(dx.abs().max()) < 1e-5                          # dy constant -> dx = 0


def test_zero_wait_limit_still_completes():
    """With a zero limit every TMA wait in the decode kernel may time out; the
    kernel flags it, drains its copies with a second bounded wait, and the
    results are still right."""
    import transformer_attention_backward_gb300 as m
    lib = m.library()
    shape = W.DecodeShape(B=2, Hq=4, Hkv=2, S=256, D=128)
    g = {k: v.cuda() for k, v in W.decode_inputs(shape, seed=9).items()}
    ref = m.attn_bwd_decode(g["q"], g["k"], g["v"], g["dout"])
    m.device_check()
    lib.abw_set_wait_limit_ns(0)
    try:
        got = m.attn_bwd_decode(g["q"], g["k"], g["v"], g["dout"])
        status = lib.abw_device_check(torch.cuda.current_stream().cuda_stream)
    finally:
        lib.abw_set_wait_limit_ns(2_000_000_000)
    assert status in (B.OK, B.ETIMEOUT)
    for a, b in zip(got, ref):
        assert torch.equal(a, b)
