"""The sparse-write oracle against its pins (tests/pins_sparse.py), and the
pins' sensitivity: each plausible mistake, planted in a CPU copy of the token
loop (never in the product and never on a GPU), must fail at least one pin by
a wide margin."""
import numpy as np
import pytest

import oracle
import pins_sparse


@pytest.mark.parametrize("name", sorted(pins_sparse.PINS))
def test_sparse_oracle_meets_pin(name):
    err = pins_sparse.PINS[name](oracle.sparse_write)
    assert err <= pins_sparse.TOL, f"{name}: {err:.3e}"


def _mutant(kind):
    def sfwd(idx, q, k, v, b, w, g, S0):
        B, T, H, K = idx.shape
        M, dv = S0.shape[2], S0.shape[3]
        S = S0.copy()
        o = np.zeros((B, T, H, dv))
        for bb in range(B):
            for h in range(H):
                for t in range(T):
                    sel = []
                    for j in range(K):
                        s = int(idx[bb, t, h, j])
                        if kind == "invalid_wraps":
                            s %= M
                        if 0 <= s < M:
                            sel.append((j, s))
                    old = {s: S[bb, h, s].copy() for _, s in sel}
                    dec = {s: (old[s] if kind == "no_decay" else np.exp(g[bb, t, h, j]) * old[s]) for j, s in sel}
                    src = old if kind == "erase_undecayed" else dec
                    bj = (lambda j: 1.0) if kind == "drop_b" else (lambda j: b[bb, t, h, j])
                    x = sum((bj(j) * k[bb, t, h, j] * src[s] for j, s in sel), np.zeros(dv))
                    u = w[bb, t, h] * v[bb, t, h]
                    sign = 1.0 if kind == "erase_sign" else -1.0
                    new = {s: dec[s] + k[bb, t, h, j] * (u + sign * x) for j, s in sel}
                    if kind == "decay_after":
                        new = {s: np.exp(g[bb, t, h, j]) * (old[s] + k[bb, t, h, j] * (u - x)) for j, s in sel}
                    for n, (j, s) in enumerate(sel):
                        if kind == "scatter_first_only" and n > 0:
                            continue
                        S[bb, h, s] = new[s]
                    for j, s in sel:
                        o[bb, t, h] += q[bb, t, h, j] * (old[s] if kind == "readout_before" else S[bb, h, s])
        return o, S

    return sfwd


MUTANTS = [
    "no_decay",            # selected slots not decayed
    "decay_after",         # decay applied after the erase and write
    "erase_undecayed",     # erase read from the undecayed rows
    "erase_sign",          # + k x instead of - k x
    "drop_b",              # erase gate ignored
    "scatter_first_only",  # only one selected row written back
    "readout_before",      # o_t read from S_{t-1}
    "invalid_wraps",       # out-of-range indices wrap around instead of selecting nothing
]


def test_faithful_copy_passes_every_pin():
    f = _mutant("none")
    for name, pin in pins_sparse.PINS.items():
        assert pin(f) <= 1e-10, name


@pytest.mark.parametrize("kind", MUTANTS)
def test_each_mutant_fails_a_pin(kind):
    f = _mutant(kind)
    worst = max(pin(f) for pin in pins_sparse.PINS.values())
    assert worst > 1e-3, f"{kind} passes every pin (worst {worst:.2e})"
