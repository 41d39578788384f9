"""gdr2_backward (and the differentiable gdr2_apply) against the fp64 gradient
oracle, element by element on the same seeded inputs.  The kernels compute in
fp32 on the exact input values (fp32 or bf16), so every gradient -- dq, dk, dv,
db, dw, dlog_decay, dS0 -- must meet the fp32 bar, max|err| / RMS(ref) <= 1e-4."""
import numpy as np
import pytest
import torch

import gated_delta_rule_166_b300 as gdr2
import oracle
from gated_delta_rule_166_b300.inputs import make_prefill_inputs
from gpu_util import err_over_rms

pytestmark = pytest.mark.gpu

TOL = 1e-4
NAMES = ("dq", "dk", "dv", "db", "dw", "dlog_decay", "dS0")


def upstream(x, seed, with_dst=True):
    gen = torch.Generator().manual_seed(seed)
    B, T, H, dk = x.q.shape
    dv = x.v.shape[-1]
    d_o = torch.randn(B, T, H, dv, generator=gen)
    d_ST = torch.randn(B, H, dk, dv, generator=gen) if with_dst else None
    return d_o, d_ST


def check(x, d_o, d_ST, label, tol=TOL):
    d = x.to("cuda")
    got = gdr2.backward(*d.tensors(), d.S0, d_o.cuda(), None if d_ST is None else d_ST.cuda())
    torch.cuda.synchronize()
    assert gdr2.gdr2_device_status() == 0
    ref = oracle.backward(*x.tensors(), x.S0, d_o, d_ST)
    errs = {}
    for name, gt, rf in zip(NAMES, got, ref):
        errs[name] = err_over_rms(gt.cpu().numpy(), rf)
    bad = {k: v for k, v in errs.items() if not v <= tol}
    assert not bad, f"{label}: " + ", ".join(f"{k}={v:.3e}" for k, v in errs.items())
    return errs


@pytest.mark.parametrize("dk,dv", [(32, 32), (64, 64), (128, 128), (128, 64), (32, 128)])
def test_backward_fp32_head_dims(dk, dv):
    x = make_prefill_inputs(2, 45, 2, dk, dv, dtype=torch.float32, seed=500 + dk + dv,
                            decay_regime="mixed", s0_std=0.3, b_scale=2.0)
    check(x, *upstream(x, 1), f"fp32 dk={dk} dv={dv}")


@pytest.mark.parametrize("T", [1, 7, 8, 9, 64, 203])
def test_backward_bf16_lengths(T):
    x = make_prefill_inputs(1, T, 3, 128, 128, dtype=torch.bfloat16, seed=600 + T,
                            decay_regime="slow", s0_std=0.5)
    check(x, *upstream(x, 2), f"bf16 T={T}")


@pytest.mark.parametrize("regime", ["fast", "zero", "mixed"])
def test_backward_decay_regimes_without_final_gradient(regime):
    x = make_prefill_inputs(2, 300, 2, 128, 128, dtype=torch.bfloat16, seed=700,
                            decay_regime=regime, s0_std=0.2)
    check(x, *upstream(x, 3, with_dst=False), f"bf16 {regime}, no dS_T")


def test_backward_without_initial_state_and_tied_gates():
    x = make_prefill_inputs(2, 130, 2, 64, 64, dtype=torch.bfloat16, seed=701,
                            gates="tied", decay="scalar", decay_regime="slow")
    assert x.S0 is None
    check(x, *upstream(x, 4), "bf16 no S0, tied/scalar gates")


def test_backward_long_sequence():
    x = make_prefill_inputs(1, 2048, 4, 128, 128, dtype=torch.bfloat16, seed=702,
                            decay_regime="slow", s0_std=0.02)
    check(x, *upstream(x, 5), "bf16 T=2048")


def test_autograd_function_matches_oracle():
    """gdr2_apply: forward by gdr2_forward, backward by gdr2_backward, through
    torch.autograd, for a loss that uses both o and S_T."""
    x = make_prefill_inputs(2, 150, 2, 64, 64, dtype=torch.float32, seed=703,
                            decay_regime="mixed", s0_std=0.3)
    d_o, d_ST = upstream(x, 6)
    leaves = [t.cuda().requires_grad_(True) for t in (*x.tensors(), x.S0)]
    o, S_T = gdr2.gdr2_apply(*leaves)
    loss = (o * d_o.cuda()).sum() + (S_T * d_ST.cuda()).sum()
    loss.backward()
    ref = oracle.backward(*x.tensors(), x.S0, d_o, d_ST)
    for name, leaf, rf in zip(NAMES, leaves, ref):
        e = err_over_rms(leaf.grad.cpu().numpy(), rf)
        assert e <= TOL, f"{name}: {e:.3e}"
    ro, rS = oracle.forward(*x.tensors(), x.S0)
    assert err_over_rms(o.detach().cpu().numpy(), ro) <= TOL
    assert err_over_rms(S_T.detach().cpu().numpy(), rS) <= TOL


def test_backward_empty_sequence():
    x = make_prefill_inputs(2, 0, 2, 64, 64, dtype=torch.float32, seed=704, s0_std=0.1)
    d = x.to("cuda")
    d_ST = torch.randn(2, 2, 64, 64, device="cuda")
    g = gdr2.backward(*d.tensors(), d.S0, torch.empty(2, 0, 2, 64, device="cuda"), d_ST)
    torch.cuda.synchronize()
    assert torch.equal(g[6], d_ST)
    assert all(t.numel() == 0 for t in g[:6])
    assert np.isfinite(g[6].cpu().numpy()).all()


def test_autograd_function_bf16_inputs():
    """gdr2_apply on bf16 inputs: the chunked tensor-core forward (fp32 o) and the
    fp32 backward, gradients returned in bf16 -- bar 2e-2 plus one bf16 rounding."""
    x = make_prefill_inputs(1, 300, 2, 128, 128, dtype=torch.bfloat16, seed=705,
                            decay_regime="slow", s0_std=0.2)
    d_o, d_ST = upstream(x, 7)
    leaves = [t.cuda().requires_grad_(True) for t in (*x.tensors(), x.S0)]
    o, S_T = gdr2.gdr2_apply(*leaves)
    ((o * d_o.cuda()).sum() + (S_T * d_ST.cuda()).sum()).backward()
    ref = oracle.backward(*x.tensors(), x.S0, d_o, d_ST)
    for name, leaf, rf in zip(NAMES, leaves, ref):
        assert leaf.grad.dtype == leaf.dtype
        e = err_over_rms(leaf.grad.float().cpu().numpy(), rf)
        bar = 2e-2 + float(np.abs(rf).max()) * 2.0 ** -8 / float(np.sqrt(np.mean(rf * rf)))
        assert e <= bar, f"{name}: {e:.3e} (bar {bar:.3g})"
