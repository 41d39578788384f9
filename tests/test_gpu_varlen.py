"""Packed variable-length prefill (gdr2_forward_varlen) on the GPU: every
sequence of a ragged batch matches the fp64 oracle run on that sequence alone,
and an equal-length batch reproduces gdr2_forward exactly."""
import numpy as np
import pytest
import torch

import oracle
import gated_delta_rule_166_b300 as gdr2
from gated_delta_rule_166_b300.inputs import make_prefill_inputs
from gpu_util import TOL_BF16, TOL_F32, err_over_rms

pytestmark = pytest.mark.gpu


def _packed(lengths, H, dk, dv, dtype, seed, **kw):
    """One independent draw per sequence, packed along the token axis."""
    seqs = [make_prefill_inputs(1, max(L, 0), H, dk, dv, dtype=dtype, seed=seed + 17 * i, s0_std=0.4, **kw)
            for i, L in enumerate(lengths)]
    cat = lambda i: torch.cat([s.tensors()[i][0] for s in seqs], dim=0).contiguous()
    toks = [cat(i) for i in range(6)]
    S0 = torch.stack([s.S0[0] for s in seqs]).contiguous()
    cu = torch.tensor(np.concatenate([[0], np.cumsum(lengths)]), dtype=torch.int32)
    return seqs, toks, S0, cu


@pytest.mark.parametrize("dtype,dk,dv,regime", [(torch.bfloat16, 128, 128, "mixed"),
                                                 (torch.bfloat16, 128, 64, "fast"),
                                                 (torch.bfloat16, 32, 32, "mixed"),
                                                 (torch.float32, 64, 32, "slow")])
def test_ragged_batch_matches_oracle_per_sequence(dtype, dk, dv, regime):
    lengths = [1, 63, 64, 65, 0, 200, 1000, 130]
    H = 3
    seqs, toks, S0, cu = _packed(lengths, H, dk, dv, dtype, seed=5, decay_regime=regime)
    d = [t.cuda() for t in toks]
    o, ST = gdr2.forward_varlen(*d, cu.cuda(), S0.cuda())
    torch.cuda.synchronize()
    assert gdr2.gdr2_device_status() == 0
    o, ST = o.float().cpu().numpy(), ST.cpu().numpy()
    tol = TOL_F32 if dtype == torch.float32 else TOL_BF16
    for i, (s, L) in enumerate(zip(seqs, lengths)):
        ro, rS = oracle.forward(*s.tensors(), s.S0)
        a, e = int(cu[i]), int(cu[i + 1])
        if L > 0:
            assert err_over_rms(o[a:e], ro[0]) <= tol, (i, L)
        assert err_over_rms(ST[i:i + 1], rS) <= tol, (i, L)


def test_equal_lengths_reproduce_fixed_length_call():
    B, T, H = 3, 150, 2
    x = make_prefill_inputs(B, T, H, 128, 128, dtype=torch.bfloat16, seed=21, s0_std=0.3).to("cuda")
    o_f, S_f = gdr2.forward(*x.tensors(), x.S0)
    cu = torch.arange(0, (B + 1) * T, T, dtype=torch.int32, device="cuda")
    packed = [t.reshape(B * T, H, -1) for t in x.tensors()]
    o_v, S_v = gdr2.forward_varlen(*packed, cu, x.S0)
    torch.cuda.synchronize()
    assert torch.equal(o_v.reshape(B, T, H, -1), o_f)
    assert torch.equal(S_v, S_f)


def test_malformed_offsets_are_clamped():
    """A decreasing pair gives an empty sequence (S_T = S0) instead of an
    out-of-range access; the first sequence's state is unaffected.  (The third
    sequence then starts at row 30 and overlaps the first, so only rows 0..29 of
    o have a single writer.)"""
    H, total = 2, 100
    x = make_prefill_inputs(1, total, H, 128, 128, dtype=torch.bfloat16, seed=23, s0_std=0.3)
    S0 = torch.randn(3, H, 128, 128) * 0.3
    cu = torch.tensor([0, 50, 30, 100], dtype=torch.int32)
    toks = [t[0].cuda() for t in x.tensors()]
    o, ST = gdr2.forward_varlen(*toks, cu.cuda(), S0.cuda())
    torch.cuda.synchronize()
    assert gdr2.gdr2_device_status() == 0
    assert torch.equal(ST[1].cpu(), S0[1])
    ro, rS = oracle.forward(*(t[:, :50] for t in x.tensors()), S0[0:1])
    assert err_over_rms(o[:30].float().cpu().numpy(), ro[0, :30]) <= TOL_BF16
    assert err_over_rms(ST[0:1].cpu().numpy(), rS) <= TOL_BF16


def test_overlapping_offsets_stay_within_the_workspace():
    """Offsets [0, 640, 0, 640, 0, 640] over 640 rows: sequences 0, 2 and 4 each
    claim all 10 chunks, 30 in all, where the workspace holds ceil(640 / 64) + 5 =
    15.  The chunk offsets are capped there: sequence 0 keeps its 10 chunks (its o
    rows past the overlap and its S_T match the oracle), sequence 2 gets 5 (its S_T
    is the state after its first 320 tokens), sequence 4 none (S_T = S0), and the
    call stays inside its workspace."""
    H, total = 2, 640
    x = make_prefill_inputs(1, total, H, 128, 128, dtype=torch.bfloat16, seed=24, s0_std=0.3,
                            decay_regime="slow")
    S0 = torch.randn(5, H, 128, 128) * 0.3
    cu = torch.tensor([0, 640, 0, 640, 0, 640], dtype=torch.int32)
    toks = [t[0].cuda() for t in x.tensors()]
    o, ST = gdr2.forward_varlen(*toks, cu.cuda(), S0.cuda())
    torch.cuda.synchronize()
    assert gdr2.gdr2_device_status() == 0
    ST = ST.cpu()
    for i in (1, 3, 4):
        assert torch.equal(ST[i], S0[i]), i
    ro, rS = oracle.forward(*x.tensors(), S0[0:1])
    assert err_over_rms(o[320:].float().cpu().numpy(), ro[0, 320:]) <= TOL_BF16
    assert err_over_rms(ST[0:1].numpy(), rS) <= TOL_BF16
    _, rS2 = oracle.forward(*(t[:, :320] for t in x.tensors()), S0[2:3])
    assert err_over_rms(ST[2:3].numpy(), rS2) <= TOL_BF16
