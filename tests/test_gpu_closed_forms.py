"""The special cases of the update equation that have a closed form, run
through the GPU path at GPU head sizes and compared with that closed form (not
with the oracle), at the same bars as the oracle comparisons: max|err| /
RMS(ref) <= 1e-4 for fp32 inputs (the token-recurrent kernel), 2e-2 for bf16
inputs (the chunked tensor-core kernels).  The oracle's own pins
(tests/pins.py) check the same facts on tiny sizes:

* no-op: b = w = 0 and D = I leave S unchanged, o_t = S0^T q_t;
* pure decay: b = w = 0 gives S_t = diag(exp(G_t)) S0, G_t = sum_{s<=t} g_s;
* linear attention: b = 0, w = 1, D = I gives O = tril(Q K^T) V + Q S0 and
  S_T = S0 + K^T V;
* gated linear attention: b = 0, w = 1, any D gives
  o_t = sum_{i<=t} (sum_j q_t[j] k_i[j] e^{G_t[j] - G_i[j]}) v_i + S0^T (q_t e^{G_t})
  and S_T = diag(e^{G_T}) S0 + sum_i (k_i e^{G_T - G_i}) v_i^T.

The closed forms are written here in fp64 NumPy from the inputs' exact values.
Lengths leave a partial last chunk, and S0 is non-zero so that it stays
visible in o and S_T."""
import numpy as np
import pytest
import torch

import gated_delta_rule_166_b300 as gdr2
from gated_delta_rule_166_b300.inputs import PrefillInputs, make_prefill_inputs
from gpu_util import TOL_BF16, TOL_F32, err_over_rms

pytestmark = pytest.mark.gpu

CASES = [(torch.float32, 64, 64, TOL_F32), (torch.bfloat16, 128, 128, TOL_BF16), (torch.bfloat16, 64, 32, TOL_BF16)]


def _problem(dtype, dk, dv, seed, *, b, w, decay):
    """q, k, v of the usual distributions; b, w constant; log decays zero or drawn
    (slow regime, so that S0 survives to the end)."""
    x = make_prefill_inputs(2, 200, 2, dk, dv, dtype=dtype, seed=seed, s0_std=0.5, decay_regime="slow")
    bt = torch.full_like(x.b, b)
    wt = torch.full_like(x.w, w)
    g = x.log_decay if decay else torch.zeros_like(x.log_decay)
    return PrefillInputs(x.q, x.k, x.v, bt, wt, g, x.S0)


def _f64(t):
    return t.double().numpy()


def _run(x):
    d = x.to("cuda")
    o, ST = gdr2.forward(*d.tensors(), d.S0)
    torch.cuda.synchronize()
    assert gdr2.gdr2_device_status() == 0
    return o.float().cpu().numpy(), ST.cpu().numpy()


def _check(got, ref, tol, label):
    for name, gv, rv in zip(("o", "S_T"), got, ref):
        e = err_over_rms(gv, rv)
        assert e <= tol, f"{label}: {name} {e:.3e} (bar {tol})"


@pytest.mark.parametrize("dtype,dk,dv,tol", CASES)
def test_noop_leaves_the_state_unchanged(dtype, dk, dv, tol):
    x = _problem(dtype, dk, dv, 1400, b=0.0, w=0.0, decay=False)
    q, S0 = _f64(x.q), _f64(x.S0)
    ro = np.einsum("bhij,bthi->bthj", S0, q)
    _check(_run(x), (ro, S0), tol, "no-op")


@pytest.mark.parametrize("dtype,dk,dv,tol", CASES)
def test_pure_decay_closed_form(dtype, dk, dv, tol):
    x = _problem(dtype, dk, dv, 1410, b=0.0, w=0.0, decay=True)
    q, g, S0 = _f64(x.q), _f64(x.log_decay), _f64(x.S0)
    G = np.cumsum(g, axis=1)                                    # [B, T, H, dk]
    ro = np.einsum("bthi,bhij,bthi->bthj", np.exp(G), S0, q)    # (e^{G_t} S0)^T q_t
    rS = np.exp(G[:, -1])[..., None] * S0
    _check(_run(x), (ro, rS), tol, "pure decay")


@pytest.mark.parametrize("dtype,dk,dv,tol", CASES)
def test_linear_attention_closed_form(dtype, dk, dv, tol):
    x = _problem(dtype, dk, dv, 1420, b=0.0, w=1.0, decay=False)
    q, k, v = (_f64(t).transpose(0, 2, 1, 3) for t in (x.q, x.k, x.v))   # [B, H, T, d]
    S0 = _f64(x.S0)
    ro = (np.tril(q @ k.transpose(0, 1, 3, 2)) @ v + q @ S0).transpose(0, 2, 1, 3)
    rS = S0 + k.transpose(0, 1, 3, 2) @ v
    _check(_run(x), (ro, rS), tol, "linear attention")


@pytest.mark.parametrize("dtype,dk,dv,tol", CASES)
def test_gated_linear_attention_closed_form(dtype, dk, dv, tol):
    x = _problem(dtype, dk, dv, 1430, b=0.0, w=1.0, decay=True)
    q, k, v, g = (_f64(t).transpose(0, 2, 1, 3) for t in (x.q, x.k, x.v, x.log_decay))   # [B, H, T, d]
    S0 = _f64(x.S0)
    G = np.cumsum(g, axis=2)
    T = q.shape[2]
    # A[t, i] = sum_j q_t[j] k_i[j] e^{G_t[j] - G_i[j]} for i <= t (exponents <= 0 there)
    diff = np.minimum(G[:, :, :, None, :] - G[:, :, None, :, :], 0.0)             # [B, H, T, T, dk]
    A = np.einsum("bhtj,bhij,bhtij->bhti", q, k, np.exp(diff)) * np.tril(np.ones((T, T)))
    ro = A @ v + np.einsum("bhtj,bhtj,bhjc->bhtc", q, np.exp(G), S0)
    kd = k * np.exp(G[:, :, -1:, :] - G)                                          # k_i e^{G_T - G_i}
    rS = np.exp(G[:, :, -1])[..., None] * S0 + kd.transpose(0, 1, 3, 2) @ v
    _check(_run(x), (ro.transpose(0, 2, 1, 3), rS), tol, "gated linear attention")
