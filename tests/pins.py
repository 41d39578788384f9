"""Pins for the CPU oracle: facts the Gated DeltaNet-2 page and plain
mathematics fix, each written independently of the oracle's own loop.

Every pin takes a forward function ``fwd(q, k, v, b, w, g, S0) -> (o, S_T)``
(float64 NumPy in and out, token tensors [B, T, H, d], states [B, H, dk, dv])
and returns the largest relative error it sees.  The oracle must score below
``TOL`` on every pin; ``test_oracle_mutants`` checks that plausible mistakes
(a transposed erase, a dropped gate, a wrong decay placement, ...) push at
least one pin far above it.
"""
from __future__ import annotations

import glob
import json
import os

import numpy as np

TOL = 1e-11
GOLDEN_DIR = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def rel_err(got, ref) -> float:
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    if got.shape != ref.shape:
        return float("inf")
    scale = max(float(np.max(np.abs(ref))), 1e-300)
    d = np.max(np.abs(got - ref)) if ref.size else 0.0
    if not np.isfinite(d):
        return float("inf")
    return float(d) / scale


def unit_rows(x):
    return x / np.linalg.norm(x, axis=-1, keepdims=True)


def rand_problem(rng, B=2, T=6, H=2, dk=5, dv=3, *, s0=True, b_hi=1.0):
    q = unit_rows(rng.standard_normal((B, T, H, dk)))
    k = unit_rows(rng.standard_normal((B, T, H, dk)))
    v = rng.standard_normal((B, T, H, dv))
    b = rng.uniform(0.0, b_hi, (B, T, H, dk))
    w = rng.uniform(0.0, 1.0, (B, T, H, dv))
    g = -rng.uniform(0.0, 1.5, (B, T, H, dk))
    S0 = rng.standard_normal((B, H, dk, dv)) if s0 else None
    return q, k, v, b, w, g, S0


# --------------------------------------------------------------------------
# hand-computed worked examples (tests/golden/*.json)
# --------------------------------------------------------------------------
def golden_cases():
    out = []
    for path in sorted(glob.glob(os.path.join(GOLDEN_DIR, "worked_example_*.json"))):
        with open(path) as f:
            out.append((os.path.basename(path), json.load(f)))
    return out


def pin_golden(fwd) -> float:
    worst = 0.0
    for _, c in golden_cases():
        B, T, H, dk, dv = c["B"], c["T"], c["H"], c["dk"], c["dv"]
        tok = lambda key, d: np.array(c[key], dtype=np.float64).reshape(B, T, H, d)
        S0 = None if c["S0"] is None else np.array(c["S0"]).reshape(B, H, dk, dv)
        o, ST = fwd(tok("q", dk), tok("k", dk), tok("v", dv), tok("b", dk),
                    tok("w", dv), tok("log_decay", dk), S0)
        worst = max(worst, rel_err(o, tok("o", dv)),
                    rel_err(ST, np.array(c["S_T"]).reshape(B, H, dk, dv)))
    return worst


# --------------------------------------------------------------------------
# brute force: S_T as an explicit sum of matrix products (T <= 8)
# --------------------------------------------------------------------------
def brute_force(q, k, v, b, w, g, S0):
    """S_t = A_t ... A_1 S0 + sum_{s<=t} A_t ... A_{s+1} k_s u_s^T with
    A_t = (I - k_t (b_t*k_t)^T) diag(exp g_t), u_s = w_s*v_s; o_t = S_t^T q_t.
    Every S_t is rebuilt from scratch out of explicit products (no recursion)."""
    B, T, H, dk = q.shape
    dv = v.shape[-1]
    o = np.zeros((B, T, H, dv))
    ST = np.zeros((B, H, dk, dv))
    for bi in range(B):
        for h in range(H):
            A = []
            for t in range(T):
                kt = k[bi, t, h]
                erase = np.eye(dk) - np.outer(kt, b[bi, t, h] * kt)
                A.append(erase @ np.diag(np.exp(g[bi, t, h])))

            def chain(lo, hi):  # A_hi ... A_lo  (identity if lo > hi)
                M = np.eye(dk)
                for s in range(lo, hi + 1):
                    M = A[s] @ M
                return M

            s0 = np.zeros((dk, dv)) if S0 is None else S0[bi, h]
            for t in range(T):
                St = chain(0, t) @ s0
                for s in range(t + 1):
                    u = w[bi, s, h] * v[bi, s, h]
                    St = St + chain(s + 1, t) @ np.outer(k[bi, s, h], u)
                o[bi, t, h] = St.T @ q[bi, t, h]
                if t == T - 1:
                    ST[bi, h] = St
            if T == 0:
                ST[bi, h] = s0
    return o, ST


def pin_bruteforce(fwd) -> float:
    rng = np.random.default_rng(101)
    worst = 0.0
    for (dk, dv, T) in ((4, 4, 8), (8, 8, 5), (5, 3, 7), (3, 6, 1)):
        p = rand_problem(rng, B=1, T=T, H=2, dk=dk, dv=dv, b_hi=2.0)
        o, ST = fwd(*p)
        ro, rST = brute_force(*p)
        worst = max(worst, rel_err(o, ro), rel_err(ST, rST))
    return worst


# --------------------------------------------------------------------------
# reductions named on the page: KDA (b = w = one scalar) and Gated DeltaNet
# (additionally a scalar decay)
# --------------------------------------------------------------------------
def kda_recurrence(q, k, v, beta, alpha_log, S0):
    """KDA form: S_t = (I - beta_t k_t k_t^T) diag(exp a_t) S_{t-1} + beta_t k_t v_t^T."""
    B, T, H, dk = q.shape
    dv = v.shape[-1]
    o = np.zeros((B, T, H, dv))
    ST = np.zeros((B, H, dk, dv))
    for bi in range(B):
        for h in range(H):
            S = np.zeros((dk, dv)) if S0 is None else S0[bi, h].copy()
            for t in range(T):
                kt, bt = k[bi, t, h], beta[bi, t, h]
                S = (np.eye(dk) - bt * np.outer(kt, kt)) @ (np.exp(alpha_log[bi, t, h])[:, None] * S)
                S = S + bt * np.outer(kt, v[bi, t, h])
                o[bi, t, h] = S.T @ q[bi, t, h]
            ST[bi, h] = S
    return o, ST


def gdn_recurrence(q, k, v, beta, alpha_log, S0):
    """Gated DeltaNet form with a scalar decay alpha_t = exp(a_t):
    S_t = alpha_t (I - beta_t k_t k_t^T) S_{t-1} + beta_t k_t v_t^T."""
    B, T, H, dk = q.shape
    dv = v.shape[-1]
    o = np.zeros((B, T, H, dv))
    ST = np.zeros((B, H, dk, dv))
    for bi in range(B):
        for h in range(H):
            S = np.zeros((dk, dv)) if S0 is None else S0[bi, h].copy()
            for t in range(T):
                kt, bt = k[bi, t, h], beta[bi, t, h]
                S = np.exp(alpha_log[bi, t, h]) * (S - bt * np.outer(kt, kt @ S)) + bt * np.outer(kt, v[bi, t, h])
                o[bi, t, h] = S.T @ q[bi, t, h]
            ST[bi, h] = S
    return o, ST


def pin_kda(fwd) -> float:
    rng = np.random.default_rng(202)
    q, k, v, _, _, g, S0 = rand_problem(rng, B=2, T=7, H=2, dk=6, dv=4)
    beta = rng.uniform(0, 1, q.shape[:3])
    b = np.repeat(beta[..., None], 6, axis=-1)
    w = np.repeat(beta[..., None], 4, axis=-1)
    o, ST = fwd(q, k, v, b, w, g, S0)
    ro, rST = kda_recurrence(q, k, v, beta, g, S0)
    return max(rel_err(o, ro), rel_err(ST, rST))


def pin_gdn(fwd) -> float:
    rng = np.random.default_rng(303)
    q, k, v, _, _, _, S0 = rand_problem(rng, B=2, T=7, H=2, dk=6, dv=4)
    beta = rng.uniform(0, 1, q.shape[:3])
    a = -rng.uniform(0, 1.0, q.shape[:3])
    b = np.repeat(beta[..., None], 6, axis=-1)
    w = np.repeat(beta[..., None], 4, axis=-1)
    g = np.repeat(a[..., None], 6, axis=-1)
    o, ST = fwd(q, k, v, b, w, g, S0)
    ro, rST = gdn_recurrence(q, k, v, beta, a, S0)
    return max(rel_err(o, ro), rel_err(ST, rST))


# --------------------------------------------------------------------------
# invariants and closed forms
# --------------------------------------------------------------------------
def pin_exact_recall(fwd) -> float:
    """||k_t|| = 1, b = w = 1, D = I  =>  S_t^T k_t = v_t (read with q_t = k_t)."""
    rng = np.random.default_rng(404)
    q, k, v, b, w, g, S0 = rand_problem(rng, B=2, T=9, H=2, dk=6, dv=5)
    b[:] = 1.0
    w[:] = 1.0
    g[:] = 0.0
    o, _ = fwd(k.copy(), k, v, b, w, g, S0)
    return rel_err(o, v)


def pin_general_recall(fwd) -> float:
    """||k_t|| = 1, b_t = 1, any D_t  =>  S_t^T k_t = w_t * v_t."""
    rng = np.random.default_rng(505)
    q, k, v, b, w, g, S0 = rand_problem(rng, B=2, T=9, H=2, dk=6, dv=5)
    b[:] = 1.0
    o, _ = fwd(k.copy(), k, v, b, w, g, S0)
    return rel_err(o, w * v)


def pin_noop(fwd) -> float:
    """b = w = 0 and D = I leave S unchanged: S_T = S0, o_t = S0^T q_t."""
    rng = np.random.default_rng(606)
    q, k, v, b, w, g, S0 = rand_problem(rng, B=2, T=5, H=2, dk=4, dv=6)
    b[:] = 0.0
    w[:] = 0.0
    g[:] = 0.0
    o, ST = fwd(q, k, v, b, w, g, S0)
    ro = np.einsum("bhij,bthi->bthj", S0, q)
    return max(rel_err(ST, S0), rel_err(o, ro))


def pin_pure_decay(fwd) -> float:
    """b = w = 0: S_t = diag(exp(sum_{s<=t} g_s)) S0."""
    rng = np.random.default_rng(707)
    q, k, v, b, w, g, S0 = rand_problem(rng, B=2, T=6, H=2, dk=4, dv=3)
    b[:] = 0.0
    w[:] = 0.0
    o, ST = fwd(q, k, v, b, w, g, S0)
    G = np.cumsum(g, axis=1)                                   # [B, T, H, dk]
    St = np.exp(G)[..., :, None] * S0[:, None]                 # [B, T, H, dk, dv]
    ro = np.einsum("bthij,bthi->bthj", St, q)
    return max(rel_err(ST, St[:, -1]), rel_err(o, ro))


def pin_linear_attention(fwd) -> float:
    """b = 0, w = 1, D = I: causal linear attention O = tril(Q K^T) V + Q S0."""
    rng = np.random.default_rng(808)
    q, k, v, b, w, g, S0 = rand_problem(rng, B=2, T=8, H=2, dk=5, dv=4)
    b[:] = 0.0
    w[:] = 1.0
    g[:] = 0.0
    o, ST = fwd(q, k, v, b, w, g, S0)
    qh = q.transpose(0, 2, 1, 3)
    kh = k.transpose(0, 2, 1, 3)
    vh = v.transpose(0, 2, 1, 3)
    scores = np.tril(qh @ kh.transpose(0, 1, 3, 2))
    ro = (scores @ vh + qh @ S0).transpose(0, 2, 1, 3)
    rST = S0 + kh.transpose(0, 1, 3, 2) @ vh
    return max(rel_err(o, ro), rel_err(ST, rST))


def pin_gla(fwd) -> float:
    """b = 0, w = 1, any D: gated linear attention,
    o_t = sum_{i<=t} (sum_j q_t[j] k_i[j] e^{G_t[j]-G_i[j]}) v_i + S0^T (q_t * e^{G_t})
    with G_t = sum_{s<=t} g_s."""
    rng = np.random.default_rng(909)
    q, k, v, b, w, g, S0 = rand_problem(rng, B=1, T=7, H=2, dk=5, dv=4)
    b[:] = 0.0
    w[:] = 1.0
    o, ST = fwd(q, k, v, b, w, g, S0)
    G = np.cumsum(g, axis=1)
    B, T, H, dk = q.shape
    ro = np.zeros_like(o)
    rST = np.zeros_like(ST)
    for bi in range(B):
        for h in range(H):
            for t in range(T):
                acc = S0[bi, h].T @ (q[bi, t, h] * np.exp(G[bi, t, h]))
                for i in range(t + 1):
                    s = np.sum(q[bi, t, h] * k[bi, i, h] * np.exp(G[bi, t, h] - G[bi, i, h]))
                    acc = acc + s * v[bi, i, h]
                ro[bi, t, h] = acc
            rST[bi, h] = np.exp(G[bi, -1, h])[:, None] * S0[bi, h] + sum(
                np.outer(k[bi, i, h] * np.exp(G[bi, -1, h] - G[bi, i, h]), v[bi, i, h])
                for i in range(T))
    return max(rel_err(o, ro), rel_err(ST, rST))


def pin_linearity(fwd) -> float:
    """For fixed q, k, b, g, outputs are jointly linear in (S0, w*v):
    F(S0a + 2 S0b, v_a + 2 v_b) = F(S0a, v_a) + 2 F(S0b, v_b)  (w = 1)."""
    rng = np.random.default_rng(1010)
    q, k, va, b, w, g, S0a = rand_problem(rng, B=2, T=6, H=2, dk=5, dv=4)
    vb = rng.standard_normal(va.shape)
    S0b = rng.standard_normal(S0a.shape)
    w[:] = 1.0
    oa, Sa = fwd(q, k, va, b, w, g, S0a)
    ob, Sb = fwd(q, k, vb, b, w, g, S0b)
    oc, Sc = fwd(q, k, va + 2 * vb, b, w, g, S0a + 2 * S0b)
    return max(rel_err(oc, oa + 2 * ob), rel_err(Sc, Sa + 2 * Sb))


def pin_split(fwd) -> float:
    """Running [0, T1) then [T1, T) from the carried state equals one pass."""
    rng = np.random.default_rng(1111)
    p = rand_problem(rng, B=2, T=11, H=2, dk=5, dv=4)
    q, k, v, b, w, g, S0 = p
    o, ST = fwd(*p)
    T1 = 4
    sl = lambda x, a, z: x[:, a:z]
    o1, S1 = fwd(*(sl(x, 0, T1) for x in (q, k, v, b, w, g)), S0)
    o2, S2 = fwd(*(sl(x, T1, 11) for x in (q, k, v, b, w, g)), S1)
    return max(rel_err(np.concatenate([o1, o2], axis=1), o), rel_err(S2, ST))


PINS = {
    "golden": pin_golden,
    "bruteforce": pin_bruteforce,
    "kda": pin_kda,
    "gdn": pin_gdn,
    "exact_recall": pin_exact_recall,
    "general_recall": pin_general_recall,
    "noop": pin_noop,
    "pure_decay": pin_pure_decay,
    "linear_attention": pin_linear_attention,
    "gla": pin_gla,
    "linearity": pin_linearity,
    "split": pin_split,
}
