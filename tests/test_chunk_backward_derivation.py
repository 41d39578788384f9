"""The chunk-level backward of the chunked (P-form) prefill, written out in fp64
NumPy and checked against the autograd gradient oracle (CPU only).  It is the
specification a chunked backward kernel follows; the library's own backward is
token-sequential.

Forward of one chunk (rows r, chunk-start state S, G_r = sum_{t<=r} g_t per key
channel, c = b * k, u = w * v):
    Cb = c e^G,  Qb = q e^G,  Kb = k e^{G_C - G},  K^ = k e^{-G}
    A_kk = strict_tril(Cb K^T),  A_qk = tril(Qb K^T),  T = (I + A_kk)^-1
    W = T Cb,  E = T u - W S,  O = Qb S + A_qk E,  S' = diag(e^{G_C}) S + Kb^T E
Backward, with dO the gradient at the chunk's outputs and dS' the one at S':
    dE = A_qk^T dO + Kb dS'               dS = diag(e^{G_C}) dS' + Qb^T dO - W^T dE
    dQb = dO S^T + dA_qk K^,  dA_qk = tril(dO E^T),  dKb = E dS'^T,  dW = -dE S^T
    du = T^T dE,  dT = dE u^T + dW Cb^T,  dA_kk = strict_tril(-T^T dT T^T)
    dCb = T^T dW + dA_kk K^,  dK^ = dA_kk^T Cb + dA_qk^T Qb
    then through the exponential factors, c = b k, u = w v and G's prefix sums.
Only dE and dS run from chunk to chunk; everything else is per chunk."""
import numpy as np
import pytest

import oracle
import pins


def chunk_forward(q, k, v, b, w, g, S):
    G = np.cumsum(g, axis=0)
    GC = G[-1]
    c, u = b * k, w * v
    Cb, Qb, Kb, Kh = c * np.exp(G), q * np.exp(G), k * np.exp(GC - G), k * np.exp(-G)
    Akk = np.tril(Cb @ Kh.T, -1)
    Aqk = np.tril(Qb @ Kh.T, 0)
    T = np.linalg.inv(np.eye(len(q)) + Akk)
    W = T @ Cb
    E = T @ u - W @ S
    O = Qb @ S + Aqk @ E
    Sn = np.exp(GC)[:, None] * S + Kb.T @ E
    return O, Sn, dict(G=G, GC=GC, u=u, Cb=Cb, Qb=Qb, Kb=Kb, Kh=Kh, Aqk=Aqk, T=T, W=W, E=E, S=S)


def chunk_backward(dO, dSn, k, v, b, w, f):
    G, GC, u, Cb, Qb, Kb, Kh = f["G"], f["GC"], f["u"], f["Cb"], f["Qb"], f["Kb"], f["Kh"]
    Aqk, T, W, E, S = f["Aqk"], f["T"], f["W"], f["E"], f["S"]
    dE = Aqk.T @ dO + Kb @ dSn
    dS = np.exp(GC)[:, None] * dSn + Qb.T @ dO - W.T @ dE
    dAqk = np.tril(dO @ E.T, 0)
    dKb = E @ dSn.T
    dW = -dE @ S.T
    du = T.T @ dE
    dT = dE @ u.T + dW @ Cb.T
    dAkk = np.tril(-T.T @ dT @ T.T, -1)
    dCb = T.T @ dW + dAkk @ Kh
    dQb = dO @ S.T + dAqk @ Kh
    dKh = dAkk.T @ Cb + dAqk.T @ Qb
    dc = dCb * np.exp(G)
    dq = dQb * np.exp(G)
    dk = dKb * np.exp(GC - G) + dKh * np.exp(-G) + dc * b
    dG = dCb * Cb + dQb * Qb - dKb * Kb - dKh * Kh
    dG[-1] += (dKb * Kb).sum(axis=0) + np.exp(GC) * (dSn * S).sum(axis=1)
    dg = np.cumsum(dG[::-1], axis=0)[::-1]
    return dq, dk, du * w, dc * k, du * v, dg, dS


@pytest.mark.parametrize("seed,T,chunk,dk,dv", [(0, 29, 8, 5, 4), (1, 40, 16, 6, 3), (2, 7, 8, 3, 5)])
def test_chunk_backward_matches_autograd(seed, T, chunk, dk, dv):
    rng = np.random.default_rng(seed)
    q, k, v, b, w, g, S0 = pins.rand_problem(rng, B=1, T=T, H=1, dk=dk, dv=dv, b_hi=2.0)
    g = 0.3 * g   # the plain e^{+-G} factors of this check stay finite over the chunk
    do = rng.standard_normal((1, T, 1, dv))
    dST = rng.standard_normal((1, 1, dk, dv))
    ref = oracle.backward(q, k, v, b, w, g, S0, do, dST)
    Q, K, V, Bv, Wv, Gv, DO = (a[0, :, 0] for a in (q, k, v, b, w, g, do))
    S = S0[0, 0].copy()
    saved = []
    outs = []
    for t0 in range(0, T, chunk):
        s = slice(t0, min(t0 + chunk, T))
        O, S, f = chunk_forward(Q[s], K[s], V[s], Bv[s], Wv[s], Gv[s], S)
        saved.append((s, f))
        outs.append(O)
    o_ref, S_ref = oracle.forward(q, k, v, b, w, g, S0)
    np.testing.assert_allclose(np.concatenate(outs), o_ref[0, :, 0], rtol=1e-10, atol=1e-10)
    np.testing.assert_allclose(S, S_ref[0, 0], rtol=1e-10, atol=1e-10)
    grads = [np.zeros_like(a) for a in (Q, K, V, Bv, Wv, Gv)]
    dS = dST[0, 0].copy()
    for s, f in reversed(saved):
        *gs, dS = chunk_backward(DO[s], dS, K[s], V[s], Bv[s], Wv[s], f)
        for acc, x in zip(grads, gs):
            acc[s] = x
    for name, got, rf in zip(("dq", "dk", "dv", "db", "dw", "dlog_decay"), grads, ref[:6]):
        rf = rf[0, :, 0]
        assert np.abs(got - rf).max() <= 1e-10 * np.abs(rf).max(), name
    assert np.abs(dS - ref[6][0, 0]).max() <= 1e-10 * np.abs(ref[6]).max()
