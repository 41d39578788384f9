"""The algebra of the one-pass prefill, checked in fp64 on the CPU against the
oracle: for one chunk of C <= 64 tokens with start state S,

    S' = diag(gamma) S + M' S + Y U,      O = P S + X U,

with G_r = sum_{t<=r} g_t, c = b * k, u = w * v,
A_kk[r,i] = sum_j c_r k_i e^{G_r - G_i} (i < r), A_qk[r,i] = the same with q (i <= r),
T = (I + A_kk)^-1, Cb = c e^G, Qb = q e^G, Kb = k e^{G_C - G}, W = T Cb,
M' = -Kb^T W, Y = Kb^T T, P = Qb - A_qk W, X = A_qk T, gamma = e^{G_C}.

These are the maps the preparation kernel writes per (chunk, head) and the chain
kernel applies; the test fixes the derivation (not a kernel) against the plain
recurrence (update equation of the Gated DeltaNet-2 page)."""
import numpy as np
import pytest

import oracle


def _maps(q, k, v, b, w, g):
    C, dk = q.shape
    G = np.cumsum(g, axis=0)
    c = b * k
    diff = G[:, None, :] - G[None, :, :]                      # [r, i, j] = G_r - G_i
    E = np.exp(np.where(np.arange(C)[:, None, None] >= np.arange(C)[None, :, None], diff, -np.inf))
    Akk = np.einsum("rj,ij,rij->ri", c, k, E) * (np.arange(C)[:, None] > np.arange(C)[None, :])
    Aqk = np.einsum("rj,ij,rij->ri", q, k, E)
    Tm = np.linalg.inv(np.eye(C) + Akk)
    Cb, Qb, Kb = c * np.exp(G), q * np.exp(G), k * np.exp(G[-1] - G)
    W = Tm @ Cb
    return dict(M=-Kb.T @ W, Y=Kb.T @ Tm, P=Qb - Aqk @ W, X=Aqk @ Tm, gamma=np.exp(G[-1]), U=w * v)


@pytest.mark.parametrize("C,dk,dv,seed", [(1, 4, 3, 0), (7, 5, 4, 1), (16, 8, 6, 2), (64, 16, 8, 3)])
def test_chunk_is_the_affine_map(C, dk, dv, seed):
    rng = np.random.default_rng(seed)
    unit = lambda x: x / np.linalg.norm(x, axis=-1, keepdims=True)
    q, k = unit(rng.standard_normal((C, dk))), unit(rng.standard_normal((C, dk)))
    v, w = rng.standard_normal((C, dv)), rng.random((C, dv))
    b, g = 2.0 * rng.random((C, dk)), -0.5 * rng.random((C, dk))
    S = rng.standard_normal((dk, dv))
    m = _maps(q, k, v, b, w, g)
    S_next = m["gamma"][:, None] * S + m["M"] @ S + m["Y"] @ m["U"]
    O = m["P"] @ S + m["X"] @ m["U"]
    ro, rS = oracle.forward(*(x[None, :, None, :] for x in (q, k, v, b, w, g)), S[None, None])
    assert np.max(np.abs(O - ro[0, :, 0])) <= 1e-10 * max(1.0, np.max(np.abs(ro)))
    assert np.max(np.abs(S_next - rS[0, 0])) <= 1e-10 * max(1.0, np.max(np.abs(rS)))
