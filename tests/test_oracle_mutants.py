"""Sensitivity of the oracle pins: each plausible mistake, planted in a CPU
copy of the recurrence (never in the product and never on a GPU), must fail
at least one pin by a wide margin."""
import numpy as np
import pytest

import pins


def _mutant(kind):
    def fwd(q, k, v, b, w, g, S0):
        B, T, H, dk = q.shape
        dv = v.shape[-1]
        S = np.zeros((B, H, dk, dv)) if S0 is None or kind == "ignore_S0" else S0.copy()
        o = np.zeros((B, T, H, dv))
        for t in range(T):
            kt, bt, qt, gt = k[:, t], b[:, t], q[:, t], g[:, t]
            bb = np.clip(bt, 0.0, 1.0) if kind == "clamp_b" else bt
            u = v[:, t] if kind == "drop_w" else w[:, t] * v[:, t]
            c = kt if kind == "drop_b" else bb * kt
            if kind == "value_side_decay":
                P = S * np.exp(gt)[..., None, :]
            elif kind in ("decay_after",):
                P = S
            else:
                P = np.exp(gt)[..., :, None] * S
            src = S if kind == "erase_reads_undecayed" else P
            if kind == "transposed_erase":
                x = np.einsum("bhi,bhij->bhj", kt, src)
                Snew = P - c[..., :, None] * x[..., None, :]
            else:
                x = np.einsum("bhi,bhij->bhj", c, src)
                sign = 1.0 if kind == "erase_sign" else -1.0
                Snew = P + sign * kt[..., :, None] * x[..., None, :]
            Snew = Snew + kt[..., :, None] * u[..., None, :]
            if kind == "decay_after":
                Snew = np.exp(gt)[..., :, None] * Snew
            if kind == "readout_before":
                o[:, t] = np.einsum("bhij,bhi->bhj", S, qt)
            elif kind == "readout_untransposed":
                o[:, t] = np.einsum("bhij,bhj->bhi", Snew, qt) if dk == dv else np.nan
            else:
                o[:, t] = np.einsum("bhij,bhi->bhj", Snew, qt)
            S = Snew
        return o, S

    return fwd


MUTANTS = [
    "transposed_erase",        # I - (b*k) k^T instead of I - k (b*k)^T
    "erase_sign",              # I + k (b*k)^T
    "drop_b",                  # erase gate ignored
    "drop_w",                  # write gate ignored
    "clamp_b",                 # erase gate clamped to [0, 1]
    "value_side_decay",        # S D instead of D S
    "decay_after",             # D applied after erase/write
    "erase_reads_undecayed",   # erase read from S_{t-1} instead of D_t S_{t-1}
    "readout_before",          # o_t = S_{t-1}^T q_t
    "readout_untransposed",    # o_t = S_t q_t
    "ignore_S0",               # initial state dropped
]


def _score(fwd):
    out = {}
    for name, pin in pins.PINS.items():
        try:
            out[name] = pin(fwd)
        except Exception:
            out[name] = float("inf")
    return out


@pytest.mark.parametrize("kind", MUTANTS)
def test_mutant_is_caught(kind):
    scores = _score(_mutant(kind))
    worst = max(scores.values())
    assert worst > 1e-3, f"mutant {kind} slips through every pin: {scores}"


def test_unmutated_copy_passes_all_pins():
    scores = _score(_mutant("none"))
    assert max(scores.values()) < pins.TOL, scores
