"""Pins for the float64 oracle: each test checks it against something other
than itself -- hand-derived closed forms (tests/golden), central-difference
VJPs of the forward definitions, algebraic invariants, and brute force on
tiny shapes.  The negative controls of Hesper's WrongBackwardTest (zero,
identity, negated backward, wrong RoPE sign) must FAIL the same checks, and so
must mistakes planted in copies of the oracle's functions.

Pages: "Hesper.Training.VerifiedBackward" API documentation (Verification
Strategy: Tier 1 algebraic identities, Tier 2 finite differences with
eps 1e-4, tol 1e-3) and Hesper pull request #1 ("Tests/WrongBackwardTest.lean").
"""
import json
import math
import os

import numpy as np
import pytest

import oracle as O

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "closed_forms.json")


@pytest.fixture(scope="module")
def golden():
    with open(GOLDEN) as f:
        return json.load(f)


def rng(seed):
    return np.random.default_rng(seed)


# --------------------------------------------------------------------------
# Closed forms (tests/golden)
# --------------------------------------------------------------------------
def test_golden_softmax(golden):
    g = golden["softmax_forward"]
    np.testing.assert_allclose(O.softmax_forward(g["x"]), g["s"], rtol=0, atol=1e-15)
    g = golden["softmax_backward_2"]
    np.testing.assert_allclose(O.softmax_backward_from_logits(g["x"], g["dy"]), g["dx"], atol=1e-15)


def test_golden_rope(golden):
    g = golden["rope_quarter_turn"]
    t = g["theta"]
    np.testing.assert_allclose(O.rope_forward_pair(*g["forward_in"], t), g["forward_out"], atol=1e-15)
    np.testing.assert_allclose(O.rope_backward_pair(*g["backward_in_a"], t), g["backward_out_a"], atol=1e-15)
    np.testing.assert_allclose(O.rope_backward_pair(*g["backward_in_b"], t), g["backward_out_b"], atol=1e-15)
    g = golden["rope_angles"]
    np.testing.assert_allclose(O.rope_angles(np.array(g["positions"]), g["D"], g["base"]), g["theta"],
                               rtol=1e-14, atol=0)


def test_golden_rmsnorm(golden):
    g = golden["rmsnorm_backward_eps0"]
    np.testing.assert_allclose(O.rmsnorm_backward(g["x"], g["gamma"], g["dy"], g["eps"]), g["dx"],
                               rtol=1e-14)


def test_golden_attention(golden):
    g = golden["attention_two_keys"]
    dq, dK, dV = O.attention_backward_single(g["q"], g["K"], g["V"], g["scale"], g["dout"])
    np.testing.assert_allclose(dq, g["dq"], rtol=1e-14)
    np.testing.assert_allclose(dK, g["dK"], rtol=1e-14)
    np.testing.assert_allclose(dV, g["dV"], rtol=1e-14)
    g = golden["attention_single_key"]
    dq, dK, dV = O.attention_backward_single(g["q"], g["K"], g["V"], g["scale"], g["dout"])
    assert np.all(dq == 0) and np.all(dK == 0)
    np.testing.assert_allclose(dV[0], g["dout"], rtol=0, atol=0)


# --------------------------------------------------------------------------
# Softmax: VJP, sum to zero
# --------------------------------------------------------------------------
@pytest.mark.parametrize("n,seed", [(1, 0), (2, 1), (5, 2), (16, 3)])
def test_softmax_backward_vjp(n, seed):
    r = rng(seed)
    x, dy = r.normal(size=n), r.normal(size=n)
    num = O.numerical_grad(lambda z: float(np.dot(dy, O.softmax_forward(z))), x)
    assert O.check_gradient(O.softmax_backward_from_logits(x, dy), num)
    # and more tightly than the page's tolerance
    np.testing.assert_allclose(O.softmax_backward_from_logits(x, dy), num, atol=1e-8)


def test_softmax_sums_to_zero():
    r = rng(7)
    for n in (1, 3, 16, 1000):
        x, dy = r.normal(size=n) * 3, r.normal(size=n)
        assert abs(O.softmax_backward_sums_to_zero(x, dy)) < 1e-12
    # shift invariance of the forward and the rowwise (batched) form
    x = r.normal(size=(4, 9))
    np.testing.assert_allclose(O.softmax_forward(x + 5.0), O.softmax_forward(x), atol=1e-15)
    np.testing.assert_allclose(O.softmax_forward(x).sum(-1), 1.0, atol=1e-15)
    dy = r.normal(size=(4, 9))
    rows = np.stack([O.softmax_backward_from_logits(x[i], dy[i]) for i in range(4)])
    np.testing.assert_allclose(O.softmax_backward_from_logits(x, dy), rows, atol=1e-15)


# --------------------------------------------------------------------------
# RoPE: VJP, round trip, norm, closed forms, tensor layouts
# --------------------------------------------------------------------------
def test_rope_pair_vjp_and_roundtrip():
    r = rng(11)
    for _ in range(20):
        x = r.normal(size=2)
        theta = r.uniform(-math.pi, math.pi)
        dy = r.normal(size=2)
        f = lambda z: float(np.dot(dy, O.rope_forward_pair(z[0], z[1], theta)))
        num = O.numerical_grad(f, x)
        assert O.check_gradient(np.array(O.rope_backward_pair(dy[0], dy[1], theta)), num)
        assert O.rope_roundtrip_check(x[0], x[1], theta, tol=1e-6)
        # rotation preserves the pair norm
        y = O.rope_forward_pair(x[0], x[1], theta)
        assert abs(math.hypot(*y) - math.hypot(*x)) < 1e-13
        z = O.rope_backward_pair(dy[0], dy[1], theta)
        assert abs(math.hypot(*z) - math.hypot(*dy)) < 1e-13
    # theta = 0 is the identity; theta = pi/2 maps (dy0, dy1) to (dy1, -dy0)
    assert O.rope_backward_pair(0.3, -0.7, 0.0) == (0.3, -0.7)
    z0, z1 = O.rope_backward_pair(0.3, -0.7, math.pi / 2)
    assert abs(z0 - (-0.7)) < 1e-15 and abs(z1 - (-0.3)) < 1e-15
    # and the forward rotation the other way: (x0, x1) -> (-x1, x0)
    y0, y1 = O.rope_forward_pair(0.3, -0.7, math.pi / 2)
    assert abs(y0 - 0.7) < 1e-15 and abs(y1 - 0.3) < 1e-15


def test_rope_roundtrip_check_rejects_broken_inverses(monkeypatch):
    """ropeRoundtripCheck must return False when the backward is not the
    inverse rotation: planted slips in a copy of the pair backward (wrong
    sign, identity, a perturbation above the 1e-6 tolerance) each fail, and a
    perturbation below it still passes."""
    x0, x1, theta = 0.8, -1.3, 1.1
    assert O.rope_roundtrip_check(x0, x1, theta)
    good = O.rope_backward_pair
    slips = {
        "wrong sign": lambda a, b, t: O.rope_forward_pair(a, b, t),
        "identity": lambda a, b, t: (a, b),
        "perturbed 1e-5": lambda a, b, t: (good(a, b, t)[0] + 1e-5, good(a, b, t)[1]),
    }
    for name, slip in slips.items():
        monkeypatch.setattr(O, "rope_backward_pair", slip)
        assert not O.rope_roundtrip_check(x0, x1, theta), name
    monkeypatch.setattr(O, "rope_backward_pair", lambda a, b, t: (good(a, b, t)[0] + 1e-8, good(a, b, t)[1]))
    assert O.rope_roundtrip_check(x0, x1, theta)


@pytest.mark.parametrize("interleaved", [True, False])
def test_rope_tensor_matches_pairs(interleaved):
    r = rng(12)
    B, T, H, D = 2, 3, 2, 8
    dy = r.normal(size=(B, T, H, D))
    theta = O.rope_angles(np.arange(T)[None, :].repeat(B, 0) + 5, D, 10000.0)
    out = O.rope_backward(dy, theta, interleaved)
    for b in range(B):
        for t in range(T):
            for h in range(H):
                for i in range(D // 2):
                    a, c = (2 * i, 2 * i + 1) if interleaved else (i, i + D // 2)
                    z0, z1 = O.rope_backward_pair(dy[b, t, h, a], dy[b, t, h, c], theta[b, t, i])
                    assert out[b, t, h, a] == z0 and out[b, t, h, c] == z1
    back = O.rope_forward(out, theta, interleaved)
    np.testing.assert_allclose(back, dy, atol=1e-12)


def test_rope_tensor_vjp():
    r = rng(13)
    B, T, H, D = 1, 2, 2, 4
    theta = r.uniform(-3, 3, size=(B, T, D // 2))
    x = r.normal(size=(B, T, H, D))
    dy = r.normal(size=(B, T, H, D))
    for inter in (True, False):
        num = O.numerical_grad(lambda z: float(np.sum(dy * O.rope_forward(z, theta, inter))), x)
        assert O.check_gradient(O.rope_backward(dy, theta, inter), num)


# --------------------------------------------------------------------------
# RMSNorm: VJP, scale-invariance identity
# --------------------------------------------------------------------------
@pytest.mark.parametrize("n,eps,seed", [(1, 1e-6, 0), (8, 1e-6, 1), (33, 1e-6, 2), (8, 0.5, 3)])
def test_rmsnorm_backward_vjp(n, eps, seed):
    r = rng(seed)
    x, dy = r.normal(size=n), r.normal(size=n)
    gamma = 1.0 + 0.1 * r.normal(size=n)
    num = O.numerical_grad(lambda z: float(np.dot(dy, O.rmsnorm_forward(z, gamma, eps))), x)
    assert O.check_gradient(O.rmsnorm_backward(x, gamma, dy, eps), num)
    np.testing.assert_allclose(O.rmsnorm_backward(x, gamma, dy, eps), num, atol=1e-7)


def test_rmsnorm_scale_identity():
    """y(c x) with eps -> the same y: d/dc <dy, y(c x)> at c = 1 equals
    <dx, x>.  With eps, y(c x) = g x / sqrt(ms + eps/c^2), which gives
    <dx, x> = (eps / (ms + eps)) <dy g, x> / rms."""
    r = rng(21)
    for eps in (1e-6, 0.3, 2.0):
        x, dy = r.normal(size=17), r.normal(size=17)
        gamma = 1 + 0.1 * r.normal(size=17)
        ms = np.mean(x * x)
        rms = math.sqrt(ms + eps)
        lhs = float(np.dot(O.rmsnorm_backward(x, gamma, dy, eps), x))
        rhs = eps / (ms + eps) * float(np.dot(dy * gamma, x)) / rms
        assert abs(lhs - rhs) < 1e-12 * max(1.0, abs(rhs))
    # forward: with gamma = 1 and eps = 0 the output has unit mean square
    y = O.rmsnorm_forward(x, np.ones_like(x), 0.0)
    assert abs(np.mean(y * y) - 1.0) < 1e-14


@pytest.mark.parametrize("eps", [1e-6, 0.5])
def test_rmsnorm_gamma_gradient(eps):
    """<dy, y> is linear in gamma, so its central difference is exact up to
    rounding: dgamma summed over the rows must match it tightly."""
    r = rng(22)
    x, dy = r.normal(size=(5, 12)), r.normal(size=(5, 12))
    gamma = 1 + 0.1 * r.normal(size=12)
    num = O.numerical_grad(lambda g: float(np.sum(dy * O.rmsnorm_forward(x, g, eps))), gamma)
    got = O.rmsnorm_backward_gamma(x, dy, eps)
    assert O.check_gradient(got, num)
    np.testing.assert_allclose(got, num, atol=1e-9)
    # one row at a time sums to the same
    rows = sum(O.rmsnorm_backward_gamma(x[i:i + 1], dy[i:i + 1], eps) for i in range(5))
    np.testing.assert_allclose(got, rows, atol=1e-13)


# --------------------------------------------------------------------------
# Scaled dot product and single-query attention
# --------------------------------------------------------------------------
@pytest.mark.parametrize("causal", [False, True])
def test_contraction_adjoints(causal):
    """Each product of the backward is the adjoint of its forward product:
    <dO, P V'> = <dV, V'> for any V' (dV = P^T dO), and with dS = the softmax
    backward of dP = dO V^T, <dS, scale Q' K^T> = <dQ, Q'> and
    <dS, scale Q K'^T> = <dK, K'> for any Q', K'.  A transposed or swapped
    operand in dQ, dK or dV breaks one of these."""
    r = rng(41 + causal)
    Tq, S, D, scale = 5, 7, 4, 0.4
    Q, K, V, dO = r.normal(size=(Tq, D)), r.normal(size=(S, D)), r.normal(size=(S, D)), r.normal(size=(Tq, D))
    off = S - Tq if causal else 0
    _, _, P = O.attention_head_forward(Q, K, V, scale, causal, off)
    dQ, dK, dV = O.attention_head_backward(Q, K, V, dO, scale, causal, off)
    dS = O.softmax_backward(P, dO @ V.T)
    Qp, Kp, Vp = r.normal(size=Q.shape), r.normal(size=K.shape), r.normal(size=V.shape)
    assert abs(np.sum(dO * (P @ Vp)) - np.sum(dV * Vp)) < 1e-12
    assert abs(np.sum(dS * (scale * Qp @ K.T)) - np.sum(dQ * Qp)) < 1e-12
    assert abs(np.sum(dS * (scale * Q @ Kp.T)) - np.sum(dK * Kp)) < 1e-12
    if causal:   # masked pairs carry no gradient
        assert np.all(dS[~(np.arange(S)[None, :] <= np.arange(Tq)[:, None] + off)] == 0.0)


@pytest.mark.parametrize("causal", [False, True])
def test_saved_p_backward_matches_recompute(causal):
    """Given the exact probabilities, the saved-P backward is the recompute
    backward."""
    r = rng(45 + causal)
    Tq, S, D, scale = 4, 6, 3, 0.6
    Q, K, V, dO = r.normal(size=(Tq, D)), r.normal(size=(S, D)), r.normal(size=(S, D)), r.normal(size=(Tq, D))
    off = S - Tq if causal else 0
    _, _, P = O.attention_head_forward(Q, K, V, scale, causal, off)
    for a, b in zip(O.attention_head_backward_saved_p(P, Q, K, V, dO, scale),
                    O.attention_head_backward(Q, K, V, dO, scale, causal, off)):
        np.testing.assert_allclose(a, b, atol=1e-13)


def test_scaled_dot_vjp():
    r = rng(31)
    q, k = r.normal(size=6), r.normal(size=6)
    scale, ds = 0.37, 1.7
    nq = O.numerical_grad(lambda z: ds * O.scaled_dot_forward(z, k, scale), q)
    nk = O.numerical_grad(lambda z: ds * O.scaled_dot_forward(q, z, scale), k)
    assert O.check_gradient(O.scaled_dot_backward_q(k, scale, ds), nq)
    assert O.check_gradient(O.scaled_dot_backward_k(q, scale, ds), nk)


@pytest.mark.parametrize("S,D,seed", [(1, 4, 0), (3, 2, 1), (16, 8, 2)])
def test_attention_single_vjp(S, D, seed):
    """Brute force: numerical gradients of <dOut, attentionForward(q, K, V)>."""
    r = rng(seed)
    q, K, V, dout = r.normal(size=D), r.normal(size=(S, D)), r.normal(size=(S, D)), r.normal(size=D)
    scale = 1 / math.sqrt(D)
    dq, dK, dV = O.attention_backward_single(q, K, V, scale, dout)
    f = lambda q_, K_, V_: float(np.dot(dout, O.attention_forward_single(q_, K_, V_, scale)))
    assert O.check_gradient(dq, O.numerical_grad(lambda z: f(z, K, V), q))
    assert O.check_gradient(dK, O.numerical_grad(lambda z: f(q, z, V), K))
    assert O.check_gradient(dV, O.numerical_grad(lambda z: f(q, K, z), V))


def test_matrix_form_equals_single_query_loop():
    r = rng(41)
    T, S, D = 5, 7, 3
    Q, K, V, dO = r.normal(size=(T, D)), r.normal(size=(S, D)), r.normal(size=(S, D)), r.normal(size=(T, D))
    scale = 0.6
    dQ, dK, dV = O.attention_head_backward(Q, K, V, dO, scale, causal=False)
    sK = np.zeros_like(K)
    sV = np.zeros_like(V)
    for i in range(T):
        dq, dk, dv = O.attention_backward_single(Q[i], K, V, scale, dO[i])
        np.testing.assert_allclose(dQ[i], dq, atol=1e-13)
        sK += dk
        sV += dv
    np.testing.assert_allclose(dK, sK, atol=1e-13)
    np.testing.assert_allclose(dV, sV, atol=1e-13)
    # forward matrix form equals the single-query forward
    Om, _, _ = O.attention_head_forward(Q, K, V, scale, causal=False)
    for i in range(T):
        np.testing.assert_allclose(Om[i], O.attention_forward_single(Q[i], K, V, scale), atol=1e-14)


def test_causal_rows_are_prefix_attention():
    """Causal row i equals full attention over keys 0..i (transformer.js mask)."""
    r = rng(42)
    T, D = 6, 3
    Q, K, V, dO = (r.normal(size=(T, D)) for _ in range(4))
    Om, lse, _ = O.attention_head_forward(Q, K, V, 0.5, causal=True)
    dQ, _, _ = O.attention_head_backward(Q, K, V, dO, 0.5, causal=True)
    for i in range(T):
        np.testing.assert_allclose(Om[i], O.attention_forward_single(Q[i], K[: i + 1], V[: i + 1], 0.5), atol=1e-14)
        dq, _, _ = O.attention_backward_single(Q[i], K[: i + 1], V[: i + 1], 0.5, dO[i])
        np.testing.assert_allclose(dQ[i], dq, atol=1e-13)
        s = 0.5 * (K[: i + 1] @ Q[i])
        assert abs(lse[i] - math.log(np.sum(np.exp(s)))) < 1e-13


# --------------------------------------------------------------------------
# Whole decode / causal paths: brute force VJPs including GQA and RoPE
# --------------------------------------------------------------------------
def _decode_forward(q_pre, k, v, scale, theta_q, G):
    """Decode forward with RoPE on the query: q = R(theta) q_pre."""
    B, Hq, D = q_pre.shape
    q = O.rope_forward(q_pre[:, None], theta_q)[:, 0]
    out = np.zeros_like(q)
    for b in range(B):
        for h in range(Hq):
            out[b, h] = O.attention_forward_single(q[b, h], k[b, :, h // G], v[b, :, h // G], scale)
    return out


def test_decode_backward_vjp_gqa_rope():
    r = rng(51)
    B, Hq, Hkv, S, D = 1, 4, 2, 5, 4
    G = Hq // Hkv
    q_pre = r.normal(size=(B, Hq, D))
    k, v = r.normal(size=(B, S, Hkv, D)), r.normal(size=(B, S, Hkv, D))
    dout = r.normal(size=(B, Hq, D))
    scale, base, pos = 0.5, 10000.0, 3
    theta = O.rope_angles(np.full((B, 1), pos), D, base)
    q = O.rope_forward(q_pre[:, None], theta)[:, 0]
    dq, dk, dv = O.decode_backward(q, k, v, dout, scale, base, pos)
    f = lambda qp, k_, v_: float(np.sum(dout * _decode_forward(qp, k_, v_, scale, theta, G)))
    assert O.check_gradient(dq, O.numerical_grad(lambda z: f(z, k, v), q_pre))
    assert O.check_gradient(dk, O.numerical_grad(lambda z: f(q_pre, z, v), k))
    assert O.check_gradient(dv, O.numerical_grad(lambda z: f(q_pre, k, z), v))


def _causal_forward_rope(q_pre, k_pre, v, scale, theta):
    q = O.rope_forward(q_pre, theta)
    k = O.rope_forward(k_pre, theta)
    o, _ = O.causal_forward(q, k, v, scale)
    return o


def test_causal_backward_vjp_gqa_rope():
    r = rng(52)
    B, T, Hq, Hkv, D = 1, 5, 4, 2, 4
    q_pre, k_pre = r.normal(size=(B, T, Hq, D)), r.normal(size=(B, T, Hkv, D))
    v, dout = r.normal(size=(B, T, Hkv, D)), r.normal(size=(B, T, Hq, D))
    scale, base = 0.5, 100.0
    theta = O.rope_angles(np.arange(T)[None, :], D, base)
    q, k = O.rope_forward(q_pre, theta), O.rope_forward(k_pre, theta)
    dq, dk, dv = O.causal_backward(q, k, v, dout, scale, base, 0)
    f = lambda a, b_, c: float(np.sum(dout * _causal_forward_rope(a, b_, c, scale, theta)))
    assert O.check_gradient(dq, O.numerical_grad(lambda z: f(z, k_pre, v), q_pre))
    assert O.check_gradient(dk, O.numerical_grad(lambda z: f(q_pre, z, v), k_pre))
    assert O.check_gradient(dv, O.numerical_grad(lambda z: f(q_pre, k_pre, z), v))


def test_causal_directional_derivative_medium():
    """At a size too large for entry-by-entry brute force: the derivative of
    <dO, Attn> along random directions equals <grad, direction>."""
    r = rng(53)
    B, T, Hq, Hkv, D = 1, 40, 2, 1, 8
    q, k, v, dout = (r.normal(size=s) for s in [(B, T, Hq, D), (B, T, Hkv, D), (B, T, Hkv, D), (B, T, Hq, D)])
    scale = 1 / math.sqrt(D)
    dq, dk, dv = O.causal_backward(q, k, v, dout, scale)
    f = lambda a, b_, c: float(np.sum(dout * O.causal_forward(a, b_, c, scale)[0]))
    eps = 1e-5
    for grad, which in ((dq, 0), (dk, 1), (dv, 2)):
        u = r.normal(size=grad.shape)
        args_p = [q, k, v]
        args_m = [q, k, v]
        args_p = [a + eps * u if i == which else a for i, a in enumerate(args_p)]
        args_m = [a - eps * u if i == which else a for i, a in enumerate(args_m)]
        num = (f(*args_p) - f(*args_m)) / (2 * eps)
        assert abs(num - float(np.sum(grad * u))) < 1e-6 * max(1.0, abs(num))


def test_chain_layer_vjp():
    """Tiny chain layer with a consistent forward: y = RMSNorm(Attn(R q, R k, v));
    numerical gradients of <dHidden, y> match chain_layer_backward fed with
    x = the attention output."""
    r = rng(54)
    B, T, Hq, Hkv, D = 1, 3, 2, 1, 4
    n = Hq * D
    q_pre, k_pre = r.normal(size=(B, T, Hq, D)), r.normal(size=(B, T, Hkv, D))
    v = r.normal(size=(B, T, Hkv, D))
    gamma = 1 + 0.1 * r.normal(size=n)
    dh = r.normal(size=(B * T, n))
    scale, base, eps = 0.5, 50.0, 1e-6
    theta = O.rope_angles(np.arange(T)[None, :], D, base)
    q, k = O.rope_forward(q_pre, theta), O.rope_forward(k_pre, theta)
    x = O.causal_forward(q, k, v, scale)[0].reshape(B * T, n)
    _, dq, dk, dv = O.chain_layer_backward(x, gamma, dh, q, k, v, eps, scale, base)

    def f(a, b_, c):
        o = _causal_forward_rope(a, b_, c, scale, theta).reshape(B * T, n)
        return float(np.sum(dh * O.rmsnorm_forward(o, gamma, eps)))
    assert O.check_gradient(dq, O.numerical_grad(lambda z: f(z, k_pre, v), q_pre))
    assert O.check_gradient(dk, O.numerical_grad(lambda z: f(q_pre, z, v), k_pre))
    assert O.check_gradient(dv, O.numerical_grad(lambda z: f(q_pre, k_pre, z), v))


# --------------------------------------------------------------------------
# Invariants and special cases
# --------------------------------------------------------------------------
def test_attention_invariants():
    r = rng(61)
    B, T, Hq, Hkv, D = 2, 9, 4, 2, 5
    q, k, v, dout = (r.normal(size=s) for s in [(B, T, Hq, D), (B, T, Hkv, D), (B, T, Hkv, D), (B, T, Hq, D)])
    dq, dk, dv = O.causal_backward(q, k, v, dout, 0.4)
    G = Hq // Hkv
    for b in range(B):
        for j in range(Hkv):
            # sum_j dS_ij = 0 for every row i, so sum over keys of dK vanishes
            np.testing.assert_allclose(dk[b, :, j].sum(0), 0.0, atol=1e-12)
            # every P row sums to 1, so sum over keys of dV equals sum of dO
            np.testing.assert_allclose(dv[b, :, j].sum(0), dout[b, :, j * G:(j + 1) * G].sum((0, 1)), atol=1e-12)
    # delta_i = sum_j P_ij dP_ij equals dO_i . O_i
    Om, _, P = O.attention_head_forward(q[0, :, 0], k[0, :, 0], v[0, :, 0], 0.4, True)
    dP = dout[0, :, 0] @ v[0, :, 0].T
    np.testing.assert_allclose(np.sum(P * dP, -1), np.sum(dout[0, :, 0] * Om, -1), atol=1e-12)


def test_decode_is_last_causal_row():
    r = rng(62)
    B, S, Hq, Hkv, D = 2, 7, 4, 2, 3
    q, k, v, dout = (r.normal(size=s) for s in [(B, S, Hq, D), (B, S, Hkv, D), (B, S, Hkv, D), (B, S, Hq, D)])
    dq_c, _, _ = O.causal_backward(q, k, v, dout, 0.3)
    dq_d, dk_d, dv_d = O.decode_backward(q[:, -1], k, v, dout[:, -1], 0.3)
    np.testing.assert_allclose(dq_d, dq_c[:, -1], atol=1e-13)
    # the decode dK/dV equal the causal ones with only the last query's dO
    dmask = np.zeros_like(dout)
    dmask[:, -1] = dout[:, -1]
    _, dk_c, dv_c = O.causal_backward(q, k, v, dmask, 0.3)
    np.testing.assert_allclose(dk_d, dk_c, atol=1e-13)
    np.testing.assert_allclose(dv_d, dv_c, atol=1e-13)


def test_gqa_equals_repeated_mha():
    r = rng(63)
    B, T, Hq, Hkv, D = 1, 6, 6, 2, 4
    G = Hq // Hkv
    q, k, v, dout = (r.normal(size=s) for s in [(B, T, Hq, D), (B, T, Hkv, D), (B, T, Hkv, D), (B, T, Hq, D)])
    dq, dk, dv = O.causal_backward(q, k, v, dout, 0.5, 1000.0)
    kr, vr = np.repeat(k, G, axis=2), np.repeat(v, G, axis=2)
    dq2, dk2, dv2 = O.causal_backward(q, kr, vr, dout, 0.5, 1000.0)
    np.testing.assert_allclose(dq, dq2, atol=1e-13)
    np.testing.assert_allclose(dk, dk2.reshape(B, T, Hkv, G, D).sum(3), atol=1e-13)
    np.testing.assert_allclose(dv, dv2.reshape(B, T, Hkv, G, D).sum(3), atol=1e-13)


def test_single_key_and_zero_query():
    r = rng(64)
    q, k, v, dout = r.normal(size=(1, 2, 3)), r.normal(size=(1, 1, 1, 3)), r.normal(size=(1, 1, 1, 3)), r.normal(size=(1, 2, 3))
    dq, dk, dv = O.decode_backward(q, k, v, dout, 0.7)
    assert np.all(dq == 0) and np.all(dk == 0)
    np.testing.assert_allclose(dv[0, 0, 0], dout[0].sum(0), atol=1e-15)
    # q = 0: uniform attention, dV[j] = dOut / S
    S = 5
    k, v = r.normal(size=(1, S, 1, 3)), r.normal(size=(1, S, 1, 3))
    _, _, dv = O.decode_backward(np.zeros((1, 1, 3)), k, v, dout[:, :1], 0.7)
    np.testing.assert_allclose(dv[0, :, 0], np.repeat(dout[:, :1] / S, S, 0)[:, 0], atol=1e-15)


# --------------------------------------------------------------------------
# Negative controls (Hesper's WrongBackwardTest) and planted mistakes
# --------------------------------------------------------------------------
def _vjp_cases():
    r = rng(71)
    x, dy = r.normal(size=6), r.normal(size=6)
    gamma = 1 + 0.1 * r.normal(size=6)
    theta = 1.1   # sin(theta) far from 0 so identity and wrong sign differ
    return x, dy, gamma, theta


def test_negative_controls_fail():
    x, dy, gamma, theta = _vjp_cases()
    # softmax
    num = O.numerical_grad(lambda z: float(np.dot(dy, O.softmax_forward(z))), x)
    good = O.softmax_backward_from_logits(x, dy)
    assert O.check_gradient(good, num)
    assert not O.check_gradient(np.zeros_like(good), num)       # zero backward
    assert not O.check_gradient(dy, num)                        # identity backward
    assert not O.check_gradient(-good, num)                     # negated backward
    # RMSNorm
    num = O.numerical_grad(lambda z: float(np.dot(dy, O.rmsnorm_forward(z, gamma))), x)
    good = O.rmsnorm_backward(x, gamma, dy)
    assert O.check_gradient(good, num)
    for bad in (np.zeros_like(good), dy, -good):
        assert not O.check_gradient(bad, num)
    # RoPE, including the wrong rotation sign R(+theta)
    p = x[:2]
    num = O.numerical_grad(lambda z: float(np.dot(dy[:2], O.rope_forward_pair(z[0], z[1], theta))), p)
    good = np.array(O.rope_backward_pair(dy[0], dy[1], theta))
    wrong_sign = np.array(O.rope_forward_pair(dy[0], dy[1], theta))
    assert O.check_gradient(good, num)
    for bad in (np.zeros(2), dy[:2], -good, wrong_sign):
        assert not O.check_gradient(bad, num)
    # attention dQ := dOut is the identity control for a shape-preserving map
    r = rng(72)
    q, K, V, dout = r.normal(size=4), r.normal(size=(6, 4)), r.normal(size=(6, 4)), r.normal(size=4)
    dq, _, _ = O.attention_backward_single(q, K, V, 0.5, dout)
    num = O.numerical_grad(lambda z: float(np.dot(dout, O.attention_forward_single(z, K, V, 0.5))), q)
    assert O.check_gradient(dq, num)
    for bad in (np.zeros(4), dout, -dq):
        assert not O.check_gradient(bad, num)


def test_planted_mistakes_fail():
    """Plausible slips in the oracle's own formulas are caught by the pins."""
    r = rng(73)
    x, dy = r.normal(size=7), r.normal(size=7)
    gamma = 1 + 0.1 * r.normal(size=7)
    s = O.softmax_forward(x)
    num_sm = O.numerical_grad(lambda z: float(np.dot(dy, O.softmax_forward(z))), x)
    assert not O.check_gradient(s * dy, num_sm)                                 # dropped sum term
    assert not O.check_gradient(s * (dy + np.sum(s * dy)), num_sm)              # wrong sign
    num_rn = O.numerical_grad(lambda z: float(np.dot(dy, O.rmsnorm_forward(z, gamma))), x)
    n = x.size
    rms = math.sqrt(np.mean(x * x) + 1e-6)
    c = np.sum(dy * gamma * x)
    assert not O.check_gradient(dy * gamma / rms, num_rn)                       # dropped c term
    assert not O.check_gradient((dy * gamma - x * c / (n * rms)) / rms, num_rn)  # rms instead of rms^2
    # attention: transposed operand in dK (dS Q instead of dS^T Q) and P for dP
    T, D = 5, 5
    Q, K, V, dO = (r.normal(size=(T, D)) for _ in range(4))
    _, _, P = O.attention_head_forward(Q, K, V, 0.5, True)
    dP = dO @ V.T
    dS = O.softmax_backward(P, dP)
    f = lambda kk: float(np.sum(dO * O.attention_head_forward(Q, kk, V, 0.5, True)[0]))
    num_k = O.numerical_grad(f, K)
    assert O.check_gradient(0.5 * dS.T @ Q, num_k)
    assert not O.check_gradient(0.5 * dS @ Q, num_k)
    fv = lambda vv: float(np.sum(dO * O.attention_head_forward(Q, K, vv, 0.5, True)[0]))
    num_v = O.numerical_grad(fv, V)
    assert not O.check_gradient(P @ dO, num_v)
    # RoPE angle with the wrong exponent (-i/D instead of -2i/D) breaks the closed form
    wrong = np.arange(4)[:, None] * np.power(10000.0, -np.arange(2) / 4.0)
    assert not np.allclose(wrong, O.rope_angles(np.arange(4), 4, 10000.0))


# --------------------------------------------------------------------------
# Causal forward (O, lse), FFN gate, LoRA: closed forms, VJPs, planted slips
# --------------------------------------------------------------------------
def test_golden_attention_forward(golden):
    """Two keys, hand-derived: O = 3/2 and lse = ln 4 (the forward's saved
    statistics that the backward consumes)."""
    g = golden["attention_two_keys"]
    O_, lse, P = O.attention_head_forward(np.array([g["q"]]), np.array(g["K"]), np.array(g["V"]), g["scale"],
                                          causal=False)
    np.testing.assert_allclose(O_[0], g["O"], rtol=1e-15)
    np.testing.assert_allclose(lse, g["lse"], rtol=1e-15)
    # the causal form over a single query at the last position is the same
    o, l = O.causal_forward(np.array(g["q"])[None, None, None, :].repeat(2, 1),
                            np.array(g["K"])[None, :, None, :], np.array(g["V"])[None, :, None, :], g["scale"])
    np.testing.assert_allclose(o[0, 1, 0], g["O"], rtol=1e-15)
    np.testing.assert_allclose(l[0, 0, 1], g["lse"], rtol=1e-15)


def test_golden_relu2_mul(golden):
    g = golden["relu2_mul"]
    np.testing.assert_allclose(O.relu2_mul_forward(g["gate"], g["up"]), g["hidden"], rtol=0, atol=0)
    dg, du = O.relu2_mul_backward(g["gate"], g["up"], g["dh"])
    np.testing.assert_allclose(dg, g["dgate"], rtol=0, atol=0)
    np.testing.assert_allclose(du, g["dup"], rtol=0, atol=0)


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_relu2_mul_vjp_and_controls(seed):
    r = rng(400 + seed)
    gate, up, dh = r.normal(size=11), r.normal(size=11), r.normal(size=11)
    dg, du = O.relu2_mul_backward(gate, up, dh)
    num_g = O.numerical_grad(lambda z: float(np.dot(dh, O.relu2_mul_forward(z, up))), gate)
    num_u = O.numerical_grad(lambda z: float(np.dot(dh, O.relu2_mul_forward(gate, z))), up)
    assert O.check_gradient(dg, num_g) and O.check_gradient(du, num_u)
    relu = np.maximum(gate, 0.0)
    for bad in (np.zeros_like(dg), dh, -dg, dh * up * relu):          # zero, identity, negated, dropped 2
        assert not O.check_gradient(bad, num_g)
    for bad in (np.zeros_like(du), dh, -du, dh * relu):                # ..., ReLU for ReLU^2
        assert not O.check_gradient(bad, num_u)


def test_golden_lora(golden):
    g = golden["lora_rank1"]
    np.testing.assert_allclose(O.lora_forward(g["x"], g["A"], g["B"], g["scale"]), g["y"], rtol=0, atol=0)
    dA, dB = O.lora_backward(g["x"], g["A"], g["B"], g["dy"], g["scale"])
    np.testing.assert_allclose(dA, g["dA"], rtol=0, atol=0)
    np.testing.assert_allclose(dB, g["dB"], rtol=0, atol=0)


def test_lora_vjp_and_controls():
    r = rng(410)
    rows, n_in, rank, n_out, s = 5, 7, 3, 6, 0.75
    x, A, B, dy = (r.normal(size=(rows, n_in)), r.normal(size=(rank, n_in)), r.normal(size=(n_out, rank)),
                   r.normal(size=(rows, n_out)))
    dA, dB = O.lora_backward(x, A, B, dy, s)
    num_A = O.numerical_grad(lambda z: float(np.sum(dy * O.lora_forward(x, z, B, s))), A)
    num_B = O.numerical_grad(lambda z: float(np.sum(dy * O.lora_forward(x, A, z, s))), B)
    assert O.check_gradient(dA, num_A) and O.check_gradient(dB, num_B)
    h = x @ A.T
    assert not O.check_gradient(dA / s, num_A)                        # dropped scale
    assert not O.check_gradient(-dA, num_A)                           # negated
    assert not O.check_gradient((dy @ B).T @ x * 0.0, num_A)          # zero
    assert not O.check_gradient(s * (dy.T @ (x @ A.T)) * 0.5, num_B)  # halved
    assert not O.check_gradient(s * (dy.T @ h[:, ::-1]), num_B)       # wrong rank index order
    # rows are independent terms of the sums: the whole equals the row sum
    parts = [O.lora_backward(x[i:i + 1], A, B, dy[i:i + 1], s) for i in range(rows)]
    np.testing.assert_allclose(sum(p[0] for p in parts), dA, rtol=1e-13, atol=1e-13)
    np.testing.assert_allclose(sum(p[1] for p in parts), dB, rtol=1e-13, atol=1e-13)
