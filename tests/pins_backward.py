"""Pins of the gradient oracle: facts that do not depend on it, each a function
of a backward implementation ``bwd(q, k, v, b, w, g, S0, do, dST)`` returning
(dq, dk, dv, db, dw, dg, dS0) that gives a score (0 for an exact match):

* ``finite_differences``: central differences of the C forward oracle along
  random directions, for every input, with and without a gradient at S_T;
* ``linear_attention``: b = 0, w = 1, no decay gives o_t = sum_{i<=t} (q_t .
  k_i) v_i + S0^T q_t and S_T = S0 + sum_i k_i v_i^T, whose gradients have a
  closed form;
* ``pure_decay``: b = w = 0 gives S_t = diag(e^{G_t}) S0, G_t = sum_{s<=t}
  g_s, whose gradients with respect to g and S0 have a closed form.

Each score is relative: |difference| / max(1, |expected|), the maximum over
the case's entries."""
import numpy as np

import oracle
import pins

NAMES = ("q", "k", "v", "b", "w", "g", "S0")
TOL = {"finite_differences": 1e-6, "linear_attention": 1e-10, "pure_decay": 1e-10}


def _loss(args, do, dST):
    o, ST = oracle.forward(*args, nthreads=1)
    return float(np.sum(o * do) + (np.sum(ST * dST) if dST is not None else 0.0))


def _rel(got, want):
    got, want = np.asarray(got, dtype=np.float64), np.asarray(want, dtype=np.float64)
    if got.shape != want.shape:
        return float("inf")
    return float(np.max(np.abs(got - want)) / max(1.0, float(np.max(np.abs(want)))))


def finite_differences(bwd, shapes=((1, 5, 2, 4, 3), (2, 9, 1, 3, 5))):
    worst = 0.0
    for shape in shapes:
        for with_dst in (True, False):
            B, T, H, dk, dv = shape
            rng = np.random.default_rng(T * 10 + dk + (1 if with_dst else 0))
            args = list(pins.rand_problem(rng, B=B, T=T, H=H, dk=dk, dv=dv, b_hi=2.0))
            do = rng.standard_normal((B, T, H, dv))
            dST = rng.standard_normal((B, H, dk, dv)) if with_dst else None
            grads = bwd(*args, do, dST)
            eps = 1e-6
            for i in range(len(NAMES)):
                d = rng.standard_normal(args[i].shape)
                plus = [a.copy() for a in args]
                minus = [a.copy() for a in args]
                plus[i] = args[i] + eps * d
                minus[i] = args[i] - eps * d
                fd = (_loss(plus, do, dST) - _loss(minus, do, dST)) / (2 * eps)
                an = float(np.sum(grads[i] * d))
                worst = max(worst, abs(fd - an) / max(1.0, abs(fd)))
    return worst


def linear_attention(bwd):
    rng = np.random.default_rng(3)
    B, T, H, dk, dv = 2, 11, 2, 5, 4
    q, k, v, _, _, _, S0 = pins.rand_problem(rng, B=B, T=T, H=H, dk=dk, dv=dv)
    zeros_k, ones_v = np.zeros((B, T, H, dk)), np.ones((B, T, H, dv))
    do = rng.standard_normal((B, T, H, dv))
    dST = rng.standard_normal((B, H, dk, dv))
    dq, dk_, dv_, _, _, _, dS0 = bwd(q, k, v, zeros_k, ones_v, zeros_k, S0, do, dST)
    mask = np.tril(np.ones((T, T)))               # [t, i]: i <= t
    worst = 0.0
    for bb in range(B):
        for h in range(H):
            Q, K, V, dO = q[bb, :, h], k[bb, :, h], v[bb, :, h], do[bb, :, h]
            A = (Q @ K.T) * mask                    # A[t, i] = q_t . k_i for i <= t
            P = (dO @ V.T) * mask                   # P[t, i] = do_t . v_i for i <= t
            worst = max(worst,
                        _rel(dq[bb, :, h], P @ K + dO @ S0[bb, h].T),
                        _rel(dv_[bb, :, h], A.T @ dO + K @ dST[bb, h]),
                        _rel(dk_[bb, :, h], P.T @ Q + V @ dST[bb, h].T),
                        _rel(dS0[bb, h], Q.T @ dO + dST[bb, h]))
    return worst


def pure_decay(bwd):
    rng = np.random.default_rng(4)
    B, T, H, dk, dv = 1, 7, 2, 4, 3
    q, k, v, _, _, g, S0 = pins.rand_problem(rng, B=B, T=T, H=H, dk=dk, dv=dv)
    z_k, z_v = np.zeros((B, T, H, dk)), np.zeros((B, T, H, dv))
    do = rng.standard_normal((B, T, H, dv))
    dST = rng.standard_normal((B, H, dk, dv))
    _, _, _, _, _, dg, dS0 = bwd(q, k, v, z_k, z_v, g, S0, do, dST)
    G = np.cumsum(g, axis=1)                                       # [B, T, H, dk]
    # per token t and channel j: dL/dG_t[j] = e^{G_t[j]} q_t[j] (S0[j] . do_t), plus the final-state term at T
    row = np.einsum("bhjn,bthn->bthj", S0, do)                       # S0[j] . do_t
    dG = np.exp(G) * q * row
    dG[:, -1] += np.exp(G[:, -1]) * np.einsum("bhjn,bhjn->bhj", S0, dST)
    expect_dg = np.flip(np.cumsum(np.flip(dG, axis=1), axis=1), axis=1)   # dg_s = sum_{t>=s} dG_t
    expect_dS0 = np.einsum("bthj,bthn->bhjn", np.exp(G) * q, do) + np.exp(G[:, -1])[..., None] * dST
    return max(_rel(dg, expect_dg), _rel(dS0, expect_dS0))


PINS = {"finite_differences": finite_differences, "linear_attention": linear_attention, "pure_decay": pure_decay}
