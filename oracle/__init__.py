"""CPU oracle for the Gated Delta Rule-2 recurrence -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline legs of
``bench.py`` may import this package.  The product library
(``gated_delta_rule_166_b300``) never imports it, and nothing here imports the
product: the two share no code.

Two independent fp64 implementations of the same definition are provided:

* :func:`forward` -- the plain sequential C loop in ``gdr2_oracle.c`` (threaded
  over independent (batch, head) pairs), loaded through ctypes.
* :func:`forward_np` -- a NumPy restatement that forms the d_k x d_k transition
  matrix ``A_t = (I - k_t (b_t * k_t)^T) D_t`` explicitly every step.

Both follow the update equation of the "Gated DeltaNet-2: Decoupling Erase and
Write in Linear Attention" page (section "Gated Delta Rule-2 update equation")
with the readout ``o_t = S_t^T q_t`` after the update.  Layouts: token tensors
``[B, T, H, d]``, states ``[B, H, d_k, d_v]``.

A third function, :func:`sparse_write`, is the gated delta write restricted
to selected slots of a larger slot memory (the "Sparse Delta Memory" review
page, section "3. Method & Key Results", with the routing-slot recurrence of
the Raven summary page, section "2.1 RSM framework"): a NumPy fp64 token loop
that gathers, updates and scatters the selected rows.

Every function is pinned by the ``-m "not gpu"`` tests (closed forms, brute
force, hand-computed worked examples, reductions to KDA / Gated DeltaNet /
(gated) linear attention, invariants); none is "parity unpinned".
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gdr2_oracle.c")
_LIB_PATH = os.path.join(_HERE, "libgdr2_oracle.so")
_lib = None


def build(force: bool = False) -> str:
    """Compile the C oracle (plain -O2, no fast-math) into oracle/libgdr2_oracle.so."""
    if force or not os.path.exists(_LIB_PATH) or (
        os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC)
    ):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.check_call(
            ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread",
             "-fno-fast-math", "-ffp-contract=off", _SRC, "-o", tmp, "-lm"]
        )
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    if _lib is None:
        build()
        lib = ctypes.CDLL(_LIB_PATH)
        dp = ctypes.POINTER(ctypes.c_double)
        lib.gdr2_oracle_forward.argtypes = [dp] * 9 + [ctypes.c_long] * 5 + [ctypes.c_int]
        lib.gdr2_oracle_forward.restype = ctypes.c_int
        _lib = lib
    return _lib


def _f64(x):
    """Exact upcast of a NumPy array or torch tensor (bf16/fp16/fp32/fp64) to a
    C-contiguous float64 NumPy array."""
    if x is None:
        return None
    if hasattr(x, "detach"):  # torch tensor, possibly bf16
        import torch

        x = x.detach().to("cpu", torch.float64).contiguous().numpy()
    return np.ascontiguousarray(np.asarray(x, dtype=np.float64))


def _ptr(a):
    if a is None:
        return ctypes.POINTER(ctypes.c_double)()
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def default_threads() -> int:
    try:
        return max(1, len(os.sched_getaffinity(0)))
    except AttributeError:  # pragma: no cover
        return max(1, os.cpu_count() or 1)


def forward(q, k, v, b, w, g, S0=None, nthreads: int | None = None):
    """Sequential fp64 recurrence (C).  Returns ``(o, S_T)`` as float64 arrays.

    q, k, b, g: [B, T, H, dk]; v, w: [B, T, H, dv]; S0: [B, H, dk, dv] or None.
    """
    lib = _load()
    q, k, v, b, w, g, S0 = (_f64(t) for t in (q, k, v, b, w, g, S0))
    B, T, H, dk = q.shape
    dv = v.shape[-1]
    for name, t, d in (("k", k, dk), ("b", b, dk), ("log_decay", g, dk),
                       ("v", v, dv), ("w", w, dv)):
        if t.shape != (B, T, H, d):
            raise ValueError(f"{name} has shape {t.shape}, expected {(B, T, H, d)}")
    if S0 is not None and S0.shape != (B, H, dk, dv):
        raise ValueError(f"S0 has shape {S0.shape}, expected {(B, H, dk, dv)}")
    o = np.empty((B, T, H, dv), dtype=np.float64)
    ST = np.empty((B, H, dk, dv), dtype=np.float64)
    rc = lib.gdr2_oracle_forward(
        _ptr(q), _ptr(k), _ptr(v), _ptr(b), _ptr(w), _ptr(g), _ptr(S0),
        _ptr(o), _ptr(ST), B, T, H, dk, dv,
        int(nthreads if nthreads is not None else default_threads()))
    if rc != 0:
        raise RuntimeError(f"gdr2_oracle_forward failed with code {rc}")
    return o, ST


def decode_step(q, k, v, b, w, g, S):
    """One recurrence step per (batch, head).  Token tensors are [B, H, d];
    S is [B, H, dk, dv].  Returns ``(o [B, H, dv], S_new)`` in float64.  This
    is :func:`forward` with T = 1 (the decode step applies the same update)."""
    q, k, v, b, w, g = (_f64(t)[:, None] for t in (q, k, v, b, w, g))
    o, S_new = forward(q, k, v, b, w, g, S0=_f64(S))
    return o[:, 0], S_new


def forward_np(q, k, v, b, w, g, S0=None):
    """Independent NumPy fp64 restatement: per step, form the d_k x d_k
    transition ``A_t = (I - k_t (b_t * k_t)^T) diag(exp g_t)`` and apply
    ``S_t = A_t S_{t-1} + k_t (w_t * v_t)^T``; read out ``o_t = S_t^T q_t``.
    Vectorised over (batch, head); intended for small cases."""
    q, k, v, b, w, g, S0 = (_f64(t) for t in (q, k, v, b, w, g, S0))
    B, T, H, dk = q.shape
    dv = v.shape[-1]
    S = np.zeros((B, H, dk, dv)) if S0 is None else S0.copy()
    eye = np.eye(dk)
    o = np.empty((B, T, H, dv))
    for t in range(T):
        kt, bt, gt, qt = k[:, t], b[:, t], g[:, t], q[:, t]
        erase = eye - kt[..., :, None] * (bt * kt)[..., None, :]      # I - k (b*k)^T
        A = erase * np.exp(gt)[..., None, :]                           # (...) D_t
        S = A @ S + kt[..., :, None] * (w[:, t] * v[:, t])[..., None, :]
        o[:, t] = np.einsum("bhij,bhi->bhj", S, qt)
    return o, S


def backward(q, k, v, b, w, g, S0, do, dST=None):
    """Gradients of the recurrence, fp64, by reverse-mode automatic
    differentiation of the plain sequential loop (PyTorch CPU autograd).

    The scalar being differentiated is ``L = sum_t <o_t, do_t> + <S_T, dST>``:
    ``do`` [B, T, H, dv] is the gradient arriving at o, ``dST`` [B, H, dk, dv]
    (or None = zero) the one arriving at the final state.  The loop is the
    update equation of the "Gated DeltaNet-2: Decoupling Erase and Write in
    Linear Attention" page (section "Gated Delta Rule-2 update equation"),
    written out per token,
        X = diag(exp g_t) S,  S = X - k_t ((b_t * k_t)^T X) + k_t (w_t * v_t)^T,
        o_t = S^T q_t,
    with S0 = None taken as a zero initial state (its gradient is still
    returned).  Returns float64 arrays (dq, dk, dv, db, dw, dg, dS0), where dg
    is the gradient with respect to log_decay."""
    import torch

    q, k, v, b, w, g, S0, do, dST = (_f64(t) for t in (q, k, v, b, w, g, S0, do, dST))
    B, T, H, dk = q.shape
    dv = v.shape[-1]
    if S0 is None:
        S0 = np.zeros((B, H, dk, dv))
    leaves = [torch.tensor(a, dtype=torch.float64, requires_grad=True) for a in (q, k, v, b, w, g, S0)]
    tq, tk, tv, tb, tw, tg, tS0 = leaves
    S = tS0
    outs = []
    for t in range(T):
        kt = tk[:, t]                                              # [B, H, dk]
        X = torch.exp(tg[:, t])[..., :, None] * S                  # D_t S_{t-1}
        erase_read = torch.einsum("bhi,bhij->bhj", tb[:, t] * kt, X)
        write = tw[:, t] * tv[:, t]
        S = X + kt[..., :, None] * (write - erase_read)[..., None, :]
        outs.append(torch.einsum("bhij,bhi->bhj", S, tq[:, t]))
    loss = torch.zeros((), dtype=torch.float64)
    if T > 0:
        o = torch.stack(outs, dim=1)
        loss = loss + (o * torch.from_numpy(do)).sum()
    if dST is not None:
        loss = loss + (S * torch.from_numpy(dST)).sum()
    grads = torch.autograd.grad(loss, leaves, allow_unused=True)
    return tuple(np.zeros(leaf.shape) if gr is None else gr.numpy() for gr, leaf in zip(grads, leaves))


def sparse_write(idx, q, k, v, b, w, g, S0):
    """Gated delta write on selected slots of a slot memory, fp64.

    The memory S [M, d_v] per (batch, head) holds M slots.  At token t a router
    has selected the K slots ``idx[b, t, h, :]`` (distinct; an index outside
    [0, M) selects nothing), and the key-side inputs q, k, b, log_decay carry
    one value per selected slot.  Reading of the pages (the "Sparse Delta
    Memory" review page performs the Gated DeltaNet-2 write only on the slots a
    product-key memory selects; the routing-slot recurrence of the Raven page,
    S_t = (1 - r_t) * S_{t-1} + r_t * (update), leaves unselected slots as they
    are, with no decay):

        R   = the selected rows,  Sd = diag(exp g_t) S_{t-1}[R]     (decay)
        x   = (b_t * k_t)^T Sd                                       (erase read)
        S_t[R] = Sd - k_t x + k_t (w_t * v_t)^T                      (erase, write)
        S_t[other rows] = S_{t-1}[other rows]
        o_t = S_t[R]^T q_t                                           (read the selected slots)

    which is the dense update of the Gated DeltaNet-2 page with k, b, q
    scattered to the selected slots (zero elsewhere) and log_decay scattered
    with zero elsewhere.  Shapes: idx, q, k, b, g [B, T, H, K]; v, w [B, T, H,
    dv]; S0 [B, H, M, dv].  Returns ``(o [B, T, H, dv], S_T [B, H, M, dv])``.
    Vectorised over (batch, head); one Python step per token."""
    if hasattr(idx, "detach"):
        idx = idx.detach().cpu().numpy()
    idx = np.asarray(idx, dtype=np.int64)
    q, k, v, b, w, g, S0 = (_f64(t) for t in (q, k, v, b, w, g, S0))
    B, T, H, K = idx.shape
    dv = v.shape[-1]
    M = S0.shape[2]
    for name, t, d in (("q", q, K), ("k", k, K), ("b", b, K), ("log_decay", g, K),
                       ("v", v, dv), ("w", w, dv)):
        if t.shape != (B, T, H, d):
            raise ValueError(f"{name} has shape {t.shape}, expected {(B, T, H, d)}")
    if S0.shape != (B, H, M, dv):
        raise ValueError(f"S0 has shape {S0.shape}, expected {(B, H, M, dv)}")
    n = B * H
    S = S0.reshape(n, M, dv).copy()
    o = np.zeros((B, T, H, dv))
    heads = np.arange(n)[:, None]
    for t in range(T):
        sel = idx[:, t].reshape(n, K)
        valid = (sel >= 0) & (sel < M)
        rows = np.where(valid, sel, 0)
        kt = np.where(valid, k[:, t].reshape(n, K), 0.0)
        bt = np.where(valid, b[:, t].reshape(n, K), 0.0)
        qt = np.where(valid, q[:, t].reshape(n, K), 0.0)
        gt = np.where(valid, g[:, t].reshape(n, K), 0.0)
        Sd = np.exp(gt)[..., None] * S[heads, rows]                  # decay of the selected rows
        x = np.einsum("nk,nkd->nd", bt * kt, Sd)                      # (b * k)^T Sd
        u = (w[:, t] * v[:, t]).reshape(n, dv)
        new = Sd + kt[..., None] * (u - x)[:, None, :]                # erase and write
        hv, kv = np.nonzero(valid)
        S[hv, sel[hv, kv]] = new[hv, kv]                              # scatter the selected rows
        o[:, t] = np.einsum("nk,nkd->nd", qt, new).reshape(B, H, dv)  # read the selected slots
    return o, S.reshape(B, H, M, dv)
