"""The gradient oracle (fp64 autograd of the sequential recurrence) checked
against what does not depend on it (CPU only): central finite differences of
the C forward oracle along random directions, and two closed forms --
causal linear attention (b = 0, w = 1, no decay) and pure decay (b = w = 0)."""
import numpy as np
import pytest

import oracle
import pins

NAMES = ("q", "k", "v", "b", "w", "g", "S0")


def loss(args, do, dST):
    o, ST = oracle.forward(*args, nthreads=1)
    return float(np.sum(o * do) + (np.sum(ST * dST) if dST is not None else 0.0))


@pytest.mark.parametrize("with_dst", [True, False])
@pytest.mark.parametrize("shape", [(1, 5, 2, 4, 3), (2, 9, 1, 3, 5)])
def test_backward_matches_finite_differences(shape, with_dst):
    B, T, H, dk, dv = shape
    rng = np.random.default_rng(T * 10 + dk + (1 if with_dst else 0))
    args = list(pins.rand_problem(rng, B=B, T=T, H=H, dk=dk, dv=dv, b_hi=2.0))
    do = rng.standard_normal((B, T, H, dv))
    dST = rng.standard_normal((B, H, dk, dv)) if with_dst else None
    grads = oracle.backward(*args, do, dST)
    eps = 1e-6
    for i, name in enumerate(NAMES):
        d = rng.standard_normal(args[i].shape)
        plus = [a.copy() for a in args]
        minus = [a.copy() for a in args]
        plus[i] = args[i] + eps * d
        minus[i] = args[i] - eps * d
        fd = (loss(plus, do, dST) - loss(minus, do, dST)) / (2 * eps)
        an = float(np.sum(grads[i] * d))
        assert abs(fd - an) <= 1e-6 * max(1.0, abs(fd)), f"d{name}: autograd {an:.10g} vs FD {fd:.10g}"


def test_backward_linear_attention_closed_form():
    # b = 0, w = 1, g = 0: o_t = sum_{i<=t} (q_t . k_i) v_i + S0^T q_t and S_T = S0 + sum_i k_i v_i^T
    rng = np.random.default_rng(3)
    B, T, H, dk, dv = 2, 11, 2, 5, 4
    q, k, v, _, _, _, S0 = pins.rand_problem(rng, B=B, T=T, H=H, dk=dk, dv=dv)
    zeros_k, ones_v = np.zeros((B, T, H, dk)), np.ones((B, T, H, dv))
    do = rng.standard_normal((B, T, H, dv))
    dST = rng.standard_normal((B, H, dk, dv))
    dq, dk_, dv_, _, _, _, dS0 = oracle.backward(q, k, v, zeros_k, ones_v, zeros_k, S0, do, dST)
    mask = np.tril(np.ones((T, T)))               # [t, i]: i <= t
    for bb in range(B):
        for h in range(H):
            Q, K, V, dO = q[bb, :, h], k[bb, :, h], v[bb, :, h], do[bb, :, h]
            A = (Q @ K.T) * mask                    # A[t, i] = q_t . k_i for i <= t
            P = (dO @ V.T) * mask                   # P[t, i] = do_t . v_i for i <= t
            np.testing.assert_allclose(dq[bb, :, h], P @ K + dO @ S0[bb, h].T, rtol=1e-11, atol=1e-11)
            np.testing.assert_allclose(dv_[bb, :, h], A.T @ dO + K @ dST[bb, h], rtol=1e-11, atol=1e-11)
            np.testing.assert_allclose(dk_[bb, :, h], P.T @ Q + V @ dST[bb, h].T, rtol=1e-11, atol=1e-11)
            np.testing.assert_allclose(dS0[bb, h], Q.T @ dO + dST[bb, h], rtol=1e-11, atol=1e-11)


def test_backward_pure_decay_closed_form():
    # b = w = 0: S_t = diag(e^{G_t}) S0 with G_t = sum_{s<=t} g_s, o_t = S_t^T q_t
    rng = np.random.default_rng(4)
    B, T, H, dk, dv = 1, 7, 2, 4, 3
    q, k, v, _, _, g, S0 = pins.rand_problem(rng, B=B, T=T, H=H, dk=dk, dv=dv)
    z_k, z_v = np.zeros((B, T, H, dk)), np.zeros((B, T, H, dv))
    do = rng.standard_normal((B, T, H, dv))
    dST = rng.standard_normal((B, H, dk, dv))
    _, _, _, _, _, dg, dS0 = oracle.backward(q, k, v, z_k, z_v, g, S0, do, dST)
    G = np.cumsum(g, axis=1)                                       # [B, T, H, dk]
    # per token t and channel j: dL/dG_t[j] = e^{G_t[j]} q_t[j] (S0[j] . do_t), plus the final-state term at T
    row = np.einsum("bhjn,bthn->bthj", S0, do)                       # S0[j] . do_t
    dG = np.exp(G) * q * row
    dG[:, -1] += np.exp(G[:, -1]) * np.einsum("bhjn,bhjn->bhj", S0, dST)
    expect_dg = np.flip(np.cumsum(np.flip(dG, axis=1), axis=1), axis=1)   # dg_s = sum_{t>=s} dG_t
    np.testing.assert_allclose(dg, expect_dg, rtol=1e-11, atol=1e-12)
    expect_dS0 = np.einsum("bthj,bthn->bhjn", np.exp(G) * q, do) + np.exp(G[:, -1])[..., None] * dST
    np.testing.assert_allclose(dS0, expect_dS0, rtol=1e-11, atol=1e-12)
