"""GPU decode step vs the fp64 CPU oracle, and decode == prefill."""
import numpy as np
import pytest
import torch

import oracle
import gated_delta_rule_166_b300 as gdr2
from gated_delta_rule_166_b300.inputs import (DECODE_WORKLOAD, make_decode_state,
                                              make_decode_token, make_prefill_inputs)
from gpu_util import TOL_BF16, TOL_F32, err_over_rms

pytestmark = pytest.mark.gpu


def _decode_run(B, H, dk, dv, steps, dtype, seed, pool=None, out_dtype=torch.float32):
    """Run `steps` decode steps on the GPU; returns per-step o (CPU), final S,
    the initial S and the token list (CPU) the oracle replays."""
    S_init = make_decode_state(B, H, dk, dv, seed=seed)
    pool = pool or steps
    toks = [make_decode_token(B, H, dk, dv, seed=seed, step=s, dtype=dtype) for s in range(pool)]
    dtoks = [t.to("cuda") for t in toks]
    S = S_init.cuda()
    outs = []
    for s in range(steps):
        o = gdr2.decode_step(*dtoks[s % pool].tensors(), S, out_dtype=out_dtype)
        outs.append(o)
    torch.cuda.synchronize()
    assert gdr2.gdr2_device_status() == 0
    return [o.float().cpu().numpy() for o in outs], S.cpu().numpy(), S_init, toks


def test_decode_full_batch_first_steps():
    W = DECODE_WORKLOAD
    B, H, dk, dv = W["B"], W["H"], W["dk"], W["dv"]
    outs, S_gpu, S_init, toks = _decode_run(B, H, dk, dv, 4, torch.bfloat16, W["seed"])
    S_ref = S_init
    for s in range(4):
        o_ref, S_ref = oracle.decode_step(*toks[s].tensors(), S_ref)
        assert err_over_rms(outs[s], o_ref) <= TOL_BF16
    assert err_over_rms(S_gpu, S_ref) <= TOL_BF16


def test_decode_1024_steps_sampled_heads():
    """The bench's configuration (B=256, H=16, d=128, 1024 in-place steps, inputs
    cycled from a pool of 16 drawn steps); the oracle replays sampled heads."""
    W = DECODE_WORKLOAD
    B, H, dk, dv, steps = W["B"], W["H"], W["dk"], W["dv"], W["steps"]
    pool = 16
    outs, S_gpu, S_init, toks = _decode_run(B, H, dk, dv, steps, torch.bfloat16, W["seed"], pool)
    heads = [(0, 0), (17, 5), (128, 15), (255, 9)]
    for (bi, h) in heads:
        S_ref = S_init[bi:bi + 1, h:h + 1].double().numpy()
        worst_o = 0.0
        for s in range(steps):
            t = toks[s % pool]
            sel = [x[bi:bi + 1, h:h + 1] for x in t.tensors()]
            o_ref, S_ref = oracle.decode_step(*sel, S_ref)
            worst_o = max(worst_o, err_over_rms(outs[s][bi:bi + 1, h:h + 1], o_ref))
        assert worst_o <= TOL_BF16, (bi, h, worst_o)
        assert err_over_rms(S_gpu[bi:bi + 1, h:h + 1], S_ref) <= TOL_BF16, (bi, h)


@pytest.mark.parametrize("dk,dv", [(32, 32), (64, 64), (128, 128), (32, 128), (128, 64)])
def test_decode_fp32_head_dims(dk, dv):
    outs, S_gpu, S_init, toks = _decode_run(3, 5, dk, dv, 6, torch.float32, seed=dk * dv)
    S_ref = S_init
    for s in range(6):
        o_ref, S_ref = oracle.decode_step(*toks[s].tensors(), S_ref)
        assert err_over_rms(outs[s], o_ref) <= TOL_F32
    assert err_over_rms(S_gpu, S_ref) <= TOL_F32


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_decode_steps_equal_prefill(dtype):
    """T decode steps from S0 give the prefill's o_t and S_T (both GPU paths,
    and each against the oracle)."""
    B, T, H, d = 2, 70, 3, 128
    x = make_prefill_inputs(B, T, H, d, d, dtype=dtype, seed=31, decay_regime="mixed", s0_std=0.3)
    xd = x.to("cuda")
    o_pf, S_pf = gdr2.forward(*xd.tensors(), xd.S0)
    S = xd.S0.clone()
    o_dec = []
    for t in range(T):
        o_dec.append(gdr2.decode_step(*(z[:, t].contiguous() for z in xd.tensors()), S))
    torch.cuda.synchronize()
    o_dec = torch.stack(o_dec, dim=1)
    ro, rS = oracle.forward(*x.tensors(), x.S0)
    tol = TOL_F32 if dtype == torch.float32 else TOL_BF16
    assert err_over_rms(o_dec.float().cpu().numpy(), ro) <= tol
    assert err_over_rms(S.cpu().numpy(), rS) <= tol
    assert err_over_rms(o_pf.float().cpu().numpy(), o_dec.float().cpu().numpy()) <= tol
    assert err_over_rms(S_pf.cpu().numpy(), S.cpu().numpy()) <= tol


def test_decode_bf16_output():
    outs, S_gpu, S_init, toks = _decode_run(16, 4, 128, 128, 3, torch.bfloat16, seed=3,
                                            out_dtype=torch.bfloat16)
    from gpu_util import bf16_output_bar
    S_ref = S_init
    for s in range(3):
        o_ref, S_ref = oracle.decode_step(*toks[s].tensors(), S_ref)
        assert err_over_rms(outs[s], o_ref) <= bf16_output_bar(o_ref, TOL_BF16)
    assert err_over_rms(S_gpu, S_ref) <= TOL_BF16
