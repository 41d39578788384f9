"""Sensitivity of the gradient oracle's pins: each plausible mistake, planted in
a CPU copy of the autograd loop (never in the product and never on a GPU),
must fail at least one pin of tests/pins_backward.py by a wide margin, and the
unmutated copy must pass them all."""
import numpy as np
import pytest
import torch

import pins_backward


def _mutant(kind):
    def bwd(q, k, v, b, w, g, S0, do, dST=None):
        B, T, H, dk = q.shape
        dv = v.shape[-1]
        S0 = np.zeros((B, H, dk, dv)) if S0 is None else S0
        leaves = [torch.tensor(np.asarray(a, dtype=np.float64), requires_grad=True) for a in (q, k, v, b, w, g, S0)]
        tq, tk, tv, tb, tw, tg, tS0 = leaves
        S = tS0.detach() if kind == "S0_detached" else tS0
        outs = []
        for t in range(T):
            kt = tk[:, t]
            decay = torch.exp(tg[:, t])[..., :, None]
            X = S if kind == "decay_after" else decay * S
            c = kt if kind == "erase_drops_b" else tb[:, t] * kt
            erase_read = torch.einsum("bhi,bhij->bhj", c, X)
            write = tv[:, t] if kind == "write_drops_w" else tw[:, t] * tv[:, t]
            sign = 1.0 if kind == "erase_sign" else -1.0
            Snew = X + kt[..., :, None] * (write + sign * erase_read)[..., None, :]
            if kind == "decay_after":
                Snew = decay * Snew
            outs.append(torch.einsum("bhij,bhi->bhj", S if kind == "readout_before" else Snew, tq[:, t]))
            S = Snew
        dO = np.roll(do, 1, axis=1) if kind == "do_shifted" else do
        loss = (torch.stack(outs, dim=1) * torch.from_numpy(np.asarray(dO, dtype=np.float64))).sum()
        if dST is not None and kind != "drop_dST_term":
            loss = loss + (S * torch.from_numpy(np.asarray(dST, dtype=np.float64))).sum()
        grads = torch.autograd.grad(loss, leaves, allow_unused=True)
        out = [np.zeros(leaf.shape) if gr is None else gr.numpy() for gr, leaf in zip(grads, leaves)]
        if kind == "swap_db_dw" and dk == dv:
            out[3], out[4] = out[4], out[3]
        elif kind == "swap_db_dw":
            out[3] = out[4][..., :dk] if dv >= dk else np.pad(out[4], [(0, 0)] * 3 + [(0, dk - dv)])
        if kind == "dg_wrt_decay_factor":   # gradient with respect to e^g instead of g
            out[5] = out[5] / np.exp(np.asarray(g, dtype=np.float64))
        return tuple(out)

    return bwd


MUTANTS = [
    "erase_drops_b",        # erase read from k instead of b * k
    "write_drops_w",        # write gate ignored
    "erase_sign",           # I + k (b*k)^T
    "decay_after",          # D applied after erase and write
    "readout_before",       # o_t = S_{t-1}^T q_t
    "drop_dST_term",        # the gradient at S_T left out of the loss
    "do_shifted",           # the gradient at o paired with the previous token
    "S0_detached",          # no gradient for S0
    "swap_db_dw",           # outputs in the wrong order (db holds dw)
    "dg_wrt_decay_factor",  # d/d(e^g) returned as d/dg
]


def _scores(bwd):
    out = {}
    for name, pin in pins_backward.PINS.items():
        try:
            out[name] = pin(bwd)
        except Exception:
            out[name] = float("inf")
    return out


@pytest.mark.parametrize("kind", MUTANTS)
def test_backward_mutant_is_caught(kind):
    scores = _scores(_mutant(kind))
    assert max(scores.values()) > 1e-3, f"mutant {kind} slips through every pin: {scores}"


def test_unmutated_copy_passes_every_backward_pin():
    scores = _scores(_mutant("none"))
    for name, s in scores.items():
        assert s <= pins_backward.TOL[name], (name, s)
