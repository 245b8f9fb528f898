"""Host-side checks of the C ABI that need no GPU: the library builds and
loads, exports every function ``include/attn_bwd.h`` declares, and rejects
invalid arguments with the documented status before touching the device."""
import ctypes
import os
import re

import numpy as np
import pytest

from transformer_attention_backward_gb300 import _binding as B

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "attn_bwd.h")


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"^\s*(?:const\s+)?[A-Za-z_][A-Za-z0-9_]*\s*\*?\s*([a-z_][a-z0-9_]*)\s*\(", text, flags=re.M)
    return sorted(set(names))


@pytest.fixture(scope="module")
def lib():
    return B.load()


def test_header_declares_the_five_operations():
    names = declared_functions()
    for op in ("softmax_bwd", "rope_bwd", "rmsnorm_bwd", "attn_bwd_decode", "attn_bwd_causal"):
        assert op in names


def test_every_declared_symbol_is_exported(lib):
    names = declared_functions()
    assert len(names) >= 10
    for n in names:
        assert hasattr(lib, n), n
        assert n in B.SIGNATURES, f"binding lacks {n}"
    assert lib.abw_version() == 100


def _ptr(a):
    return ctypes.c_void_p(a.ctypes.data)


def test_softmax_validation(lib):
    assert lib.softmax_bwd(None, None, None, 4, 0, None) == B.EINVAL
    assert lib.softmax_bwd(None, None, None, -1, 8, None) == B.EINVAL
    assert lib.softmax_bwd(None, None, None, 2, 8, None) == B.EINVAL        # null pointers
    assert "NULL" in B.last_error()
    assert lib.softmax_bwd(None, None, None, 0, 8, None) == B.OK            # nothing to do
    buf = np.zeros(64, dtype=np.float32)
    p = buf.ctypes.data
    # output overlapping an input
    assert lib.softmax_bwd(ctypes.c_void_p(p), ctypes.c_void_p(p + 128), ctypes.c_void_p(p + 32), 1, 16, None) == B.EINVAL
    assert "overlaps" in B.last_error()
    # misaligned pointer
    assert lib.softmax_bwd(ctypes.c_void_p(p + 4), ctypes.c_void_p(p + 4 + 256), ctypes.c_void_p(p + 4 + 512),
                           1, 1, None) == B.EINVAL


def test_rope_validation(lib):
    assert lib.rope_bwd(None, None, 1, 1, 1, 3, None, 0, 10000.0, 1, None) == B.EINVAL   # odd D
    assert lib.rope_bwd(None, None, 1, 1, 1, 1024, None, 0, 10000.0, 1, None) == B.ENOTSUP
    assert lib.rope_bwd(None, None, 1, 1, 1, 8, None, 0, 0.0, 1, None) == B.EINVAL       # base <= 0
    assert lib.rope_bwd(None, None, 1, 1, 1, 8, None, -1, 100.0, 1, None) == B.EINVAL    # pos0 < 0
    assert lib.rope_bwd(None, None, 0, 4, 2, 8, None, 0, 100.0, 1, None) == B.OK         # empty


def test_rmsnorm_validation(lib):
    assert lib.rmsnorm_bwd(None, 0, None, None, None, 0, 4, 0, 1e-6, None) == B.EINVAL
    assert lib.rmsnorm_bwd(None, 7, None, None, None, 0, 4, 8, 1e-6, None) == B.EINVAL    # dtype
    assert lib.rmsnorm_bwd(None, 0, None, None, None, 0, 4, 8, -1.0, None) == B.EINVAL    # eps
    assert lib.rmsnorm_bwd(None, 0, None, None, None, 0, 0, 8, 1e-6, None) == B.OK


def test_decode_validation(lib):
    call = lambda B_, Hq, Hkv, S, D, dt=1: lib.attn_bwd_decode(None, None, None, None, None, None, None,
                                                               B_, Hq, Hkv, S, D, dt, 0.1, 0.0, -1, None)
    assert call(1, 4, 3, 8, 128) == B.EINVAL          # Hq % Hkv
    assert call(1, 4, 0, 8, 128) == B.EINVAL
    assert call(1, 32, 2, 8, 128) == B.ENOTSUP        # group of 16
    assert call(1, 4, 2, 0, 128) == B.EINVAL          # no keys
    assert call(1, 4, 2, 8, 12) == B.ENOTSUP          # 24 bytes per bf16 row
    assert call(1, 4, 2, 8, 512) == B.ENOTSUP         # 1 KiB rows
    assert call(1, 4, 2, 8, 128, dt=0) == B.EINVAL    # f32 rows of 512 B are fine -> null pointers
    assert call(1, 4, 2, 8, 256, dt=0) == B.ENOTSUP   # f32 rows of 1 KiB
    assert call(0, 4, 2, 8, 128) == B.OK              # empty batch


def test_causal_validation(lib):
    def call(D=128, ws=None, wsb=0, Hq=4, Hkv=2, T=16):
        return lib.attn_bwd_causal(None, None, None, None, None, None, None, None, None, 1, T, Hq, Hkv, D,
                                   0.1, 0.0, 0, ws, wsb, None)
    assert call(D=64) == B.ENOTSUP
    assert call(Hq=4, Hkv=3) == B.EINVAL
    assert call() == B.EWORKSPACE
    need = lib.attn_bwd_causal_workspace_bytes(1, 16, 4, 128)
    # delta and lse*log2(e) over T rounded up to 64, and the [T][D/2] (cos, sin) table
    assert need >= 2 * 4 * 64 * 4 + 16 * 64 * 8
    assert call(ws=ctypes.c_void_p(256), wsb=need - 1) == B.EWORKSPACE
    assert call(T=0) == B.OK
    assert lib.attn_bwd_causal_workspace_bytes(-1, 1, 1, 128) == 0


def test_comparator_negative_control():
    """The parity metric must fail a correct output with one element's sign
    flipped (and pass the output itself)."""
    import oracle
    from tests.helpers import max_rel_err, TOL_BF16
    r = np.random.default_rng(3)
    q, k, v, do = r.normal(size=(1, 6, 2, 4)), r.normal(size=(1, 6, 1, 4)), r.normal(size=(1, 6, 1, 4)), r.normal(size=(1, 6, 2, 4))
    dq, _, _ = oracle.causal_backward(q, k, v, do, 0.5)
    bad = dq.copy()
    i = np.unravel_index(np.argmax(np.abs(bad)), bad.shape)
    bad[i] = -bad[i]
    assert max_rel_err(dq, dq) == 0.0
    assert max_rel_err(bad, dq) > TOL_BF16
    nan = dq.copy()
    nan[0, 0, 0, 0] = np.nan
    assert max_rel_err(nan, dq) == float("inf")
