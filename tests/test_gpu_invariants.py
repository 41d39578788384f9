"""Properties of the GPU prefill that hold at any size: split composability,
generalised recall, empty sequences, in-place state, optional outputs."""
import numpy as np
import pytest
import torch

import oracle
import gated_delta_rule_166_b300 as gdr2
from gated_delta_rule_166_b300.inputs import make_prefill_inputs
from gpu_util import TOL_BF16, TOL_F32, err_over_rms

pytestmark = pytest.mark.gpu


def _np(t):
    return t.float().cpu().numpy()


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("T1", [100, 64, 1])
def test_split_composability(dtype, T1):
    T = 300
    x = make_prefill_inputs(2, T, 2, 128, 128, dtype=dtype, seed=41, decay_regime="slow",
                            s0_std=0.3).to("cuda")
    o, ST = gdr2.forward(*x.tensors(), x.S0)
    a = [t[:, :T1].contiguous() for t in x.tensors()]
    z = [t[:, T1:].contiguous() for t in x.tensors()]
    o1, S1 = gdr2.forward(*a, x.S0)
    o2, S2 = gdr2.forward(*z, S1)
    tol = TOL_F32 if dtype == torch.float32 else TOL_BF16
    assert err_over_rms(_np(torch.cat([o1, o2], 1)), _np(o)) <= tol
    assert err_over_rms(_np(S2), _np(ST)) <= tol


def test_general_recall_on_gpu():
    """||k|| = 1, b = 1, any decay: S_t^T k_t = w_t * v_t.  Reading the last
    token with q_T = k_T must return w_T * v_T."""
    x = make_prefill_inputs(2, 200, 4, 128, 128, dtype=torch.bfloat16, seed=43,
                            decay_regime="mixed", s0_std=0.3)
    x.b.fill_(1.0)
    x.q[:, -1] = x.k[:, -1]
    o, _ = gdr2.forward(*x.to("cuda").tensors(), x.S0.cuda())
    want = (x.w[:, -1].float() * x.v[:, -1].float()).numpy()
    assert err_over_rms(_np(o[:, -1]), want) <= TOL_BF16


def test_empty_sequence():
    x = make_prefill_inputs(2, 0, 3, 128, 128, dtype=torch.bfloat16, seed=1, s0_std=1.0).to("cuda")
    o, ST = gdr2.forward(*x.tensors(), x.S0)
    torch.cuda.synchronize()
    assert o.shape == (2, 0, 3, 128)
    assert torch.equal(ST, x.S0)
    o, ST = gdr2.forward(*x.tensors(), None)
    assert torch.count_nonzero(ST).item() == 0


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_in_place_state_and_optional_outputs(dtype):
    x = make_prefill_inputs(1, 130, 2, 128, 128, dtype=dtype, seed=45, s0_std=0.5).to("cuda")
    o_ref, S_ref = gdr2.forward(*x.tensors(), x.S0)
    S = x.S0.clone()
    o_ip, S_ip = gdr2.forward(*x.tensors(), S, S_T=S)
    assert S_ip.data_ptr() == S.data_ptr()
    o_ns, S_ns = gdr2.forward(*x.tensors(), x.S0, return_state=False)
    torch.cuda.synchronize()
    assert S_ns is None
    assert torch.equal(o_ip, o_ref) and torch.equal(S, S_ref) and torch.equal(o_ns, o_ref)


def test_nan_input_propagates_without_error():
    x = make_prefill_inputs(1, 200, 2, 128, 128, dtype=torch.bfloat16, seed=47)
    x.v[0, 150, 1, 3] = float("nan")
    o, ST = gdr2.forward(*x.to("cuda").tensors(), None)
    torch.cuda.synchronize()
    assert gdr2.gdr2_device_status() == 0
    o = o.float().cpu()
    # tokens before the 64-token chunk holding the NaN are untouched (inside a
    # chunk, tensor-core products multiply the NaN by the causal mask's zeros)
    assert torch.isfinite(o[0, :128]).all()
    assert torch.isfinite(o[0, :, 0]).all()           # the other head never sees it
    assert torch.isnan(o[0, 150:, 1]).any()


def test_oracle_agrees_on_general_recall():
    # the same property on the oracle, on the very inputs used above
    x = make_prefill_inputs(1, 50, 2, 128, 128, dtype=torch.bfloat16, seed=43,
                            decay_regime="mixed", s0_std=0.3)
    x.b.fill_(1.0)
    x.q[:, -1] = x.k[:, -1]
    o, _ = oracle.forward(*x.tensors(), x.S0)
    want = (x.w[:, -1].float() * x.v[:, -1].float()).double().numpy()
    # k is rounded to bf16, so ||k|| = 1 only to bf16 precision
    assert err_over_rms(o[:, -1], want) <= 1e-2
