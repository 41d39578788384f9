"""Pins for the sparse-write oracle: facts that the pages and plain mathematics
fix, each written independently of the oracle's gather / scatter loop.

Every pin takes ``sfwd(idx, q, k, v, b, w, g, S0) -> (o, S_T)`` (float64 NumPy
in and out; idx, q, k, b, g [B, T, H, K]; v, w [B, T, H, dv]; S0 [B, H, M, dv])
and returns the largest relative error it sees.  ``test_oracle_sparse`` checks
that the oracle stays below ``TOL`` on every pin and that plausible mistakes
planted in a CPU copy push at least one pin far above it.
"""
from __future__ import annotations

import json
import os

import numpy as np

import oracle
from pins import GOLDEN_DIR, rel_err, unit_rows

TOL = 1e-11


def rand_sparse(rng, B=2, T=6, H=2, M=9, K=3, dv=4, *, distinct=True):
    """Small random problem; K distinct slots per token (a random subset)."""
    if distinct:
        idx = np.stack([rng.permutation(M)[:K] for _ in range(B * T * H)]).reshape(B, T, H, K)
    else:
        idx = rng.integers(0, M, size=(B, T, H, K))
    q = unit_rows(rng.standard_normal((B, T, H, K))) if K else np.zeros((B, T, H, 0))
    k = unit_rows(rng.standard_normal((B, T, H, K))) if K else np.zeros((B, T, H, 0))
    v = rng.standard_normal((B, T, H, dv))
    b = 2.0 * rng.random((B, T, H, K))
    w = rng.random((B, T, H, dv))
    g = -rng.random((B, T, H, K))
    S0 = rng.standard_normal((B, H, M, dv))
    return idx, q, k, v, b, w, g, S0


def scatter(idx, vals, M):
    """Dense [B, T, H, M] array holding vals at the selected slots, 0 elsewhere."""
    B, T, H, K = idx.shape
    out = np.zeros((B, T, H, M))
    for bb in range(B):
        for t in range(T):
            for h in range(H):
                for j in range(K):
                    s = idx[bb, t, h, j]
                    if 0 <= s < M:
                        out[bb, t, h, s] = vals[bb, t, h, j]
    return out


# --------------------------------------------------------------------------
# the hand-computed worked example (tests/golden/sparse_example_*.json)
# --------------------------------------------------------------------------
def pin_golden(sfwd) -> float:
    worst = 0.0
    path = os.path.join(GOLDEN_DIR, "sparse_example_T2_M3.json")
    with open(path) as f:
        c = json.load(f)
    B, T, H, M, K, dv = c["B"], c["T"], c["H"], c["M"], c["K"], c["dv"]
    sel = lambda key, d: np.array(c[key], dtype=np.float64).reshape(B, T, H, d)
    idx = np.array(c["idx"]).reshape(B, T, H, K)
    S0 = np.array(c["S0"], dtype=np.float64).reshape(B, H, M, dv)
    o, ST = sfwd(idx, sel("q", K), sel("k", K), sel("v", dv), sel("b", K), sel("w", dv),
                 sel("log_decay", K), S0)
    return max(rel_err(o, sel("o", dv)), rel_err(ST, np.array(c["S_T"]).reshape(B, H, M, dv)))


# --------------------------------------------------------------------------
# every slot selected: the dense Gated DeltaNet-2 recurrence (slot = key channel)
# --------------------------------------------------------------------------
def pin_all_slots_dense(sfwd) -> float:
    rng = np.random.default_rng(11)
    worst = 0.0
    for M in (1, 4, 7):
        idx, q, k, v, b, w, g, S0 = rand_sparse(rng, T=5, M=M, K=M)
        o, ST = sfwd(idx, q, k, v, b, w, g, S0)
        dense = [scatter(idx, x, M) for x in (q, k, b, g)]
        ro, rS = oracle.forward(dense[0], dense[1], v, dense[2], w, dense[3], S0)
        worst = max(worst, rel_err(o, ro), rel_err(ST, rS))
    return worst


# --------------------------------------------------------------------------
# any selection: the dense recurrence with k, b, q scattered (zero elsewhere)
# and log_decay scattered with zero elsewhere (unselected slots: no decay)
# --------------------------------------------------------------------------
def pin_scattered_dense(sfwd) -> float:
    rng = np.random.default_rng(12)
    worst = 0.0
    for M, K in ((6, 1), (9, 3), (12, 5)):
        idx, q, k, v, b, w, g, S0 = rand_sparse(rng, T=7, M=M, K=K)
        o, ST = sfwd(idx, q, k, v, b, w, g, S0)
        dense = [scatter(idx, x, M) for x in (q, k, b, g)]
        ro, rS = oracle.forward(dense[0], dense[1], v, dense[2], w, dense[3], S0)
        worst = max(worst, rel_err(o, ro), rel_err(ST, rS))
    return worst


# --------------------------------------------------------------------------
# brute force (T <= 8): the routing-slot recurrence with M x M matrices,
#   S_t = (1 - r_t) * S_{t-1} + r_t * (A_t S_{t-1} + k_t (w_t * v_t)^T),
#   A_t = (I - k_t (b_t * k_t)^T) diag(exp g_t),   o_t = S_t^T q_t,
# r_t the 0/1 selection vector (scattered key-side vectors)
# --------------------------------------------------------------------------
def pin_bruteforce(sfwd) -> float:
    rng = np.random.default_rng(13)
    idx, q, k, v, b, w, g, S0 = rand_sparse(rng, B=1, T=8, H=1, M=5, K=2, dv=3)
    o, ST = sfwd(idx, q, k, v, b, w, g, S0)
    M = 5
    S = S0[0, 0].copy()
    ref_o = np.zeros((8, 3))
    for t in range(8):
        r = np.zeros(M)
        kh, bh, qh, gh = (np.zeros(M) for _ in range(4))
        for j in range(2):
            s = idx[0, t, 0, j]
            r[s], kh[s], bh[s], qh[s], gh[s] = 1.0, k[0, t, 0, j], b[0, t, 0, j], q[0, t, 0, j], g[0, t, 0, j]
        A = (np.eye(M) - np.outer(kh, bh * kh)) @ np.diag(np.exp(gh))
        upd = A @ S + np.outer(kh, w[0, t, 0] * v[0, t, 0])
        S = (1.0 - r)[:, None] * S + r[:, None] * upd
        ref_o[t] = S.T @ qh
    return max(rel_err(o[0, :, 0], ref_o), rel_err(ST[0, 0], S))


# --------------------------------------------------------------------------
# nothing selected: the memory is unchanged and every read is zero
# --------------------------------------------------------------------------
def pin_nothing_selected(sfwd) -> float:
    rng = np.random.default_rng(14)
    idx, q, k, v, b, w, g, S0 = rand_sparse(rng, M=6, K=0)
    o, ST = sfwd(idx, q, k, v, b, w, g, S0)
    return max(rel_err(ST, S0), float(np.max(np.abs(o))) if o.size else 0.0)


# --------------------------------------------------------------------------
# b = 0 and w = 0: pure decay of the selected slots only, in closed form
#   S_t[s] = S0[s] * exp(sum of the log decays s received up to t)
# --------------------------------------------------------------------------
def pin_pure_decay(sfwd) -> float:
    rng = np.random.default_rng(15)
    idx, q, k, v, b, w, g, S0 = rand_sparse(rng, T=9, M=7, K=3)
    b = np.zeros_like(b)
    w = np.zeros_like(w)
    o, ST = sfwd(idx, q, k, v, b, w, g, S0)
    B, T, H, K = idx.shape
    M = S0.shape[2]
    ref_o = np.zeros_like(o)
    ref_S = np.zeros_like(S0)
    for bb in range(B):
        for h in range(H):
            cum = np.zeros(M)   # accumulated log decay per slot
            for t in range(T):
                for j in range(K):
                    cum[idx[bb, t, h, j]] += g[bb, t, h, j]
                for j in range(K):
                    ref_o[bb, t, h] += q[bb, t, h, j] * S0[bb, h, idx[bb, t, h, j]] * np.exp(cum[idx[bb, t, h, j]])
            ref_S[bb, h] = S0[bb, h] * np.exp(cum)[:, None]
    return max(rel_err(o, ref_o), rel_err(ST, ref_S))


# --------------------------------------------------------------------------
# slots that are never selected keep their initial contents bit for bit
# --------------------------------------------------------------------------
def pin_frozen_rows(sfwd) -> float:
    rng = np.random.default_rng(16)
    idx, q, k, v, b, w, g, S0 = rand_sparse(rng, T=6, M=20, K=2)
    o, ST = sfwd(idx, q, k, v, b, w, g, S0)
    worst = 0.0
    for bb in range(idx.shape[0]):
        for h in range(idx.shape[2]):
            untouched = np.setdiff1d(np.arange(20), idx[bb, :, h].ravel())
            if untouched.size:
                d = np.max(np.abs(ST[bb, h, untouched] - S0[bb, h, untouched]))
                worst = max(worst, float(d) if d == 0 else float("inf"))
    return worst


# --------------------------------------------------------------------------
# an index outside [0, M) selects nothing: the same as leaving that entry out
# --------------------------------------------------------------------------
def pin_invalid_index(sfwd) -> float:
    rng = np.random.default_rng(17)
    idx, q, k, v, b, w, g, S0 = rand_sparse(rng, T=5, M=8, K=3)
    bad = idx.copy()
    bad[..., 1] = np.where(rng.random(bad[..., 1].shape) < 0.5, -1, 8)
    o, ST = sfwd(bad, q, k, v, b, w, g, S0)
    keep = [0, 2]
    ro, rS = sfwd(idx[..., keep], q[..., keep], k[..., keep], v, b[..., keep], w, g[..., keep], S0)
    return max(rel_err(o, ro), rel_err(ST, rS))


PINS = {
    "golden": pin_golden,
    "all_slots_dense": pin_all_slots_dense,
    "scattered_dense": pin_scattered_dense,
    "bruteforce": pin_bruteforce,
    "nothing_selected": pin_nothing_selected,
    "pure_decay": pin_pure_decay,
    "frozen_rows": pin_frozen_rows,
    "invalid_index": pin_invalid_index,
}
