"""gdr2_forward_cached: the state kept at the end of every segment of
cache_chunks 64-token chunks, against the fp64 oracle run segment by segment
(each segment started from the previous one's end state), and o / S_T against
the plain call.  Bars: bf16 inputs 2e-2, fp32 inputs 1e-4 (max|err| / RMS)."""
import numpy as np
import pytest
import torch

import gated_delta_rule_166_b300 as gdr2
import oracle
from gated_delta_rule_166_b300.inputs import make_prefill_inputs
from gpu_util import err_over_rms, tol_for

pytestmark = pytest.mark.gpu


def oracle_segment_states(x, seg_tokens, n):
    """S after tokens seg_tokens - 1, 2 seg_tokens - 1, ...: the oracle over one
    segment at a time, each from the previous segment's end state."""
    S = None if x.S0 is None else x.S0.double().numpy()
    out = []
    for m in range(n):
        sl = slice(m * seg_tokens, (m + 1) * seg_tokens)
        _, S = oracle.forward(*(t[:, sl] for t in x.tensors()), S)
        out.append(S)
    return np.stack(out, axis=2) if out else np.zeros((x.q.shape[0], x.q.shape[2], 0, x.q.shape[3], x.v.shape[3]))


@pytest.mark.parametrize("cache_chunks", [1, 4, 7])
def test_cached_states_bf16(cache_chunks):
    x = make_prefill_inputs(2, 1000, 3, 128, 128, dtype=torch.bfloat16, seed=800 + cache_chunks,
                            decay_regime="slow", s0_std=0.4)
    d = x.to("cuda")
    o, S_T, S_cache = gdr2.forward_cached(*d.tensors(), d.S0, cache_chunks=cache_chunks)
    torch.cuda.synchronize()
    assert gdr2.gdr2_device_status() == 0
    n = 1000 // (cache_chunks * 64)
    assert S_cache.shape == (2, 3, n, 128, 128)
    ref = oracle_segment_states(x, cache_chunks * 64, n)
    e = err_over_rms(S_cache.cpu().numpy(), ref)
    assert e <= tol_for(x.q.dtype), f"cache_chunks={cache_chunks}: {e:.3e}"
    # o and S_T are those of the plain sequential pass, bit for bit
    o1, S1 = gdr2.forward(*d.tensors(), d.S0, segments=1)
    torch.cuda.synchronize()
    assert torch.equal(o, o1) and torch.equal(S_T, S1)


def test_cached_states_fp32_token_kernel_and_short_sequence():
    x = make_prefill_inputs(1, 300, 2, 64, 64, dtype=torch.float32, seed=810, decay_regime="mixed", s0_std=0.3)
    d = x.to("cuda")
    o, S_T, S_cache = gdr2.forward_cached(*d.tensors(), d.S0, cache_chunks=1)
    torch.cuda.synchronize()
    ref = oracle_segment_states(x, 64, 4)
    assert err_over_rms(S_cache.cpu().numpy(), ref) <= tol_for(x.q.dtype)
    ro, rS = oracle.forward(*x.tensors(), x.S0)
    assert err_over_rms(o.cpu().numpy(), ro) <= 1e-4 and err_over_rms(S_T.cpu().numpy(), rS) <= 1e-4
    # shorter than one segment: nothing to keep
    y = make_prefill_inputs(1, 100, 2, 128, 128, dtype=torch.bfloat16, seed=811, s0_std=0.1).to("cuda")
    _, _, C = gdr2.forward_cached(*y.tensors(), y.S0, cache_chunks=2)
    torch.cuda.synchronize()
    assert C.shape[2] == 0 and gdr2.gdr2_device_status() == 0


@pytest.mark.parametrize("dk,dv", [(64, 32), (32, 128)])
def test_cached_states_small_head_dims(dk, dv):
    """Small bf16 head sizes (zero-padded channels in the chunked kernels)."""
    x = make_prefill_inputs(1, 700, 2, dk, dv, dtype=torch.bfloat16, seed=880 + dk + dv, s0_std=0.4)
    d = x.to("cuda")
    o, S_T, S_cache = gdr2.forward_cached(*d.tensors(), d.S0, cache_chunks=2)
    torch.cuda.synchronize()
    assert gdr2.gdr2_device_status() == 0
    n = 700 // 128
    ref = oracle_segment_states(x, 128, n)
    assert err_over_rms(S_cache.cpu().numpy(), ref) <= tol_for(torch.bfloat16)
    o1, S1 = gdr2.forward(*d.tensors(), d.S0, segments=1)
    assert torch.equal(o, o1) and torch.equal(S_T, S1)
