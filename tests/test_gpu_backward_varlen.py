"""gdr2_backward_varlen, gdr2_backward_chunked_varlen and the differentiable
gdr2_apply_varlen on the GPU: the gradients of every sequence of a packed
ragged batch match the fp64 gradient oracle run on that sequence alone -- at
the fp32 bar of the exact backward (max|err| / RMS(ref) <= 1e-4, fp32 or bf16
inputs), and at the bf16 bar (2e-2) for the tensor-core path; an equal-length
batch reproduces gdr2_backward (gdr2_backward_chunked) bit for bit; rows that
belong to no sequence are not written; malformed offsets stay in bounds."""
import ctypes

import numpy as np
import pytest
import torch

import gated_delta_rule_166_b300 as gdr2
import oracle
from gated_delta_rule_166_b300 import _lib
from gated_delta_rule_166_b300.inputs import PrefillInputs, make_prefill_inputs
from gpu_util import err_over_rms

pytestmark = pytest.mark.gpu

TOL = 1e-4
NAMES = ("dq", "dk", "dv", "db", "dw", "dlog_decay")


def _packed(lengths, H, dk, dv, dtype, seed, **kw):
    """One independent draw per sequence, packed along the token axis, with a
    seeded upstream gradient at o (packed) and at every final state."""
    seqs = [make_prefill_inputs(1, L, H, dk, dv, dtype=dtype, seed=seed + 17 * i, s0_std=0.4, **kw)
            for i, L in enumerate(lengths)]
    cat = lambda i: torch.cat([s.tensors()[i][0] for s in seqs], dim=0).contiguous()  # noqa: E731
    toks = [cat(i) for i in range(6)]
    S0 = torch.stack([s.S0[0] for s in seqs]).contiguous()
    cu = torch.tensor(np.concatenate([[0], np.cumsum(lengths)]), dtype=torch.int32)
    gen = torch.Generator().manual_seed(seed + 1)
    d_o = torch.randn(int(cu[-1]), H, dv, generator=gen)
    d_ST = torch.randn(len(lengths), H, dk, dv, generator=gen)
    return seqs, toks, S0, cu, d_o, d_ST


def _check_sequence(got, s, i, a, e, S0, d_o, d_ST, label):
    """Sequence i (rows a .. e - 1) of the packed gradients against the oracle
    run on that sequence alone."""
    L = e - a
    gS0 = got[6].cpu().numpy()
    if L == 0:
        assert np.array_equal(gS0[i], d_ST[i].numpy()), f"{label}: empty sequence {i}"
        return
    ref = oracle.backward(*s.tensors(), S0[i:i + 1], d_o[a:e].unsqueeze(0), d_ST[i:i + 1])
    errs = {n: err_over_rms(g[a:e].cpu().numpy(), r[0]) for n, g, r in zip(NAMES, got[:6], ref[:6])}
    errs["dS0"] = err_over_rms(gS0[i:i + 1], ref[6])
    bad = {k: v for k, v in errs.items() if not v <= TOL}
    assert not bad, f"{label}, sequence {i} (T={L}): " + ", ".join(f"{k}={v:.3e}" for k, v in errs.items())


@pytest.mark.parametrize("dtype,dk,dv,regime", [(torch.float32, 64, 32, "mixed"),
                                                 (torch.bfloat16, 128, 128, "slow"),
                                                 (torch.bfloat16, 32, 64, "fast")])
def test_ragged_batch_gradients_match_oracle_per_sequence(dtype, dk, dv, regime):
    lengths = [1, 5, 0, 64, 131, 9, 203]   # ragged against the 4-token checkpoint blocks
    H = 2
    seqs, toks, S0, cu, d_o, d_ST = _packed(lengths, H, dk, dv, dtype, seed=810 + dk + dv, decay_regime=regime,
                                            b_scale=2.0)
    got = gdr2.backward_varlen(*[t.cuda() for t in toks], cu.cuda(), S0.cuda(), d_o.cuda(), d_ST.cuda())
    torch.cuda.synchronize()
    assert gdr2.gdr2_device_status() == 0
    for i, s in enumerate(seqs):
        _check_sequence(got, s, i, int(cu[i]), int(cu[i + 1]), S0, d_o, d_ST, f"{dtype} dk={dk} dv={dv}")


def test_equal_lengths_reproduce_fixed_length_backward():
    """The same arithmetic per sequence: equal lengths give gdr2_backward's
    gradients bit for bit."""
    B, T, H = 3, 150, 2
    x = make_prefill_inputs(B, T, H, 128, 64, dtype=torch.bfloat16, seed=830, s0_std=0.3).to("cuda")
    gen = torch.Generator().manual_seed(831)
    d_o = torch.randn(B, T, H, 64, generator=gen).cuda()
    d_ST = torch.randn(B, H, 128, 64, generator=gen).cuda()
    ref = gdr2.backward(*x.tensors(), x.S0, d_o, d_ST)
    cu = torch.arange(0, (B + 1) * T, T, dtype=torch.int32, device="cuda")
    packed = [t.reshape(B * T, H, -1) for t in x.tensors()]
    got = gdr2.backward_varlen(*packed, cu, x.S0, d_o.reshape(B * T, H, -1), d_ST)
    torch.cuda.synchronize()
    for n, g, r in zip(NAMES + ("dS0",), got, ref):
        assert torch.equal(g.reshape(r.shape), r), n


def test_rows_outside_every_sequence_are_not_written():
    """Offsets that leave rows 0-2 and 40-47 to no sequence: those rows of every
    gradient keep the caller's contents (checked through the C ABI with sentinel
    values); the covered rows match the oracle."""
    H, dk, dv, total = 2, 64, 64, 48
    x = make_prefill_inputs(1, total, H, dk, dv, dtype=torch.float32, seed=840, s0_std=0.2)
    toks = [t[0].contiguous().cuda() for t in x.tensors()]
    cu = torch.tensor([3, 20, 20, 40], dtype=torch.int32)
    N = 3
    gen = torch.Generator().manual_seed(841)
    S0 = torch.randn(N, H, dk, dv, generator=gen) * 0.2
    d_o = torch.randn(total, H, dv, generator=gen)
    d_ST = torch.randn(N, H, dk, dv, generator=gen)
    sentinel = 7.25
    outs = [torch.full((total, H, d), sentinel, device="cuda") for d in (dk, dk, dv, dk, dv, dk)]
    gq, gk, gv, gb, gw, gg = outs
    gS0 = torch.empty(N, H, dk, dv, device="cuda")
    S0d, d_od, d_STd, cud = S0.cuda(), d_o.cuda(), d_ST.cuda(), cu.cuda()
    p = _lib._ptr
    st = _lib.lib().gdr2_backward_varlen(*(p(t) for t in toks), p(S0d), p(d_od), p(d_STd), p(gq), p(gk), p(gv),
                                         p(gb), p(gw), p(gg), p(gS0), p(cud), N, total, H, dk, dv, 0,
                                         ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == 0
    torch.cuda.synchronize()
    assert gdr2.gdr2_device_status() == 0
    for t in outs:
        assert torch.all(t[:3] == sentinel) and torch.all(t[40:] == sentinel)
    got = (gq, gk, gv, gb, gw, gg, gS0)
    for i, (a, e) in enumerate([(3, 20), (20, 20), (20, 40)]):
        s = PrefillInputs(*(t[:, a:e] for t in x.tensors()), None)
        _check_sequence(got, s, i, a, e, S0, d_o, d_ST, "partial cover")


def test_malformed_offsets_stay_in_bounds():
    """A decreasing pair gives an empty sequence (dS0 = dS_T) and a sequence that
    overlaps an earlier one; a later sequence that overlaps nothing is still exact
    and the call reports no error."""
    H, dk, dv, total = 2, 128, 128, 100
    x = make_prefill_inputs(1, total, H, dk, dv, dtype=torch.bfloat16, seed=850, s0_std=0.3)
    toks = [t[0].contiguous().cuda() for t in x.tensors()]
    cu = torch.tensor([0, 40, 20, 60, 100], dtype=torch.int32)
    gen = torch.Generator().manual_seed(851)
    S0 = torch.randn(4, H, dk, dv, generator=gen) * 0.3
    d_o = torch.randn(total, H, dv, generator=gen)
    d_ST = torch.randn(4, H, dk, dv, generator=gen)
    got = gdr2.backward_varlen(*toks, cu.cuda(), S0.cuda(), d_o.cuda(), d_ST.cuda())
    torch.cuda.synchronize()
    assert gdr2.gdr2_device_status() == 0
    assert torch.equal(got[6][1].cpu(), d_ST[1])
    s = PrefillInputs(*(t[:, 60:100] for t in x.tensors()), None)
    _check_sequence(got, s, 3, 60, 100, S0, d_o, d_ST, "malformed offsets")


def test_autograd_varlen_matches_oracle():
    """gdr2_apply_varlen: forward by gdr2_forward_varlen, backward by
    gdr2_backward_varlen, through torch.autograd, for a loss on o and S_T."""
    lengths = [70, 0, 33, 128]
    H, dk, dv = 2, 64, 64
    seqs, toks, S0, cu, d_o, d_ST = _packed(lengths, H, dk, dv, torch.float32, seed=860, decay_regime="mixed")
    leaves = [t.cuda().requires_grad_(True) for t in toks] + [S0.cuda().requires_grad_(True)]
    o, S_T = gdr2.gdr2_apply_varlen(*leaves[:6], cu.cuda(), leaves[6])
    ((o * d_o.cuda()).sum() + (S_T * d_ST.cuda()).sum()).backward()
    got = tuple(leaf.grad for leaf in leaves)
    for i, s in enumerate(seqs):
        a, e = int(cu[i]), int(cu[i + 1])
        _check_sequence(got, s, i, a, e, S0, d_o, d_ST, "autograd")
        if e > a:
            ro, rS = oracle.forward(*s.tensors(), S0[i:i + 1])
            assert err_over_rms(o[a:e].detach().cpu().numpy(), ro[0]) <= TOL
            assert err_over_rms(S_T[i:i + 1].detach().cpu().numpy(), rS) <= TOL


# ---- gdr2_backward_chunked_varlen: the chunkwise WY form on tensor cores -----------------
# fp16 operands (tf32 for the decay-weighted products) with fp32 accumulation, as in
# gdr2_backward_chunked, so the bar is the bf16 one on every gradient; the regimes
# here are those where gdr2_backward_chunked meets 2e-2 on all of them.
TOL_CHUNKED = 2e-2


def _check_sequence_chunked(got, s, i, a, e, S0, d_o, d_ST, label):
    L = e - a
    gS0 = got[6].cpu().numpy()
    if L == 0:
        assert np.array_equal(gS0[i], d_ST[i].numpy()), f"{label}: empty sequence {i}"
        return
    ref = oracle.backward(*s.tensors(), S0[i:i + 1], d_o[a:e].unsqueeze(0), d_ST[i:i + 1])
    errs = {n: err_over_rms(g[a:e].cpu().numpy(), r[0]) for n, g, r in zip(NAMES, got[:6], ref[:6])}
    errs["dS0"] = err_over_rms(gS0[i:i + 1], ref[6])
    bad = {k: v for k, v in errs.items() if not v <= TOL_CHUNKED}
    assert not bad, f"{label}, sequence {i} (T={L}): " + ", ".join(f"{k}={v:.3e}" for k, v in errs.items())


@pytest.mark.parametrize("regime,seed", [("slow", 870), ("mixed", 871)])
def test_chunked_ragged_batch_matches_oracle_per_sequence(regime, seed):
    """Ragged against the 64-token chunks: a single token, an empty sequence, exact
    multiples and partial last chunks, so global chunks of different sequences sit
    side by side in every workspace region."""
    lengths = [1, 64, 0, 65, 130, 7, 257]
    H = 2
    seqs, toks, S0, cu, d_o, d_ST = _packed(lengths, H, 128, 128, torch.bfloat16, seed=seed, decay_regime=regime)
    got = gdr2.backward_chunked_varlen(*[t.cuda() for t in toks], cu.cuda(), S0.cuda(), d_o.cuda(), d_ST.cuda())
    torch.cuda.synchronize()
    assert gdr2.gdr2_device_status() == 0
    for i, s in enumerate(seqs):
        _check_sequence_chunked(got, s, i, int(cu[i]), int(cu[i + 1]), S0, d_o, d_ST, f"chunked {regime}")


def test_chunked_equal_lengths_reproduce_fixed_length_backward():
    """The same kernels and arithmetic per chunk: equal lengths give
    gdr2_backward_chunked's gradients bit for bit (T = 150 leaves a partial chunk)."""
    B, T, H = 3, 150, 2
    x = make_prefill_inputs(B, T, H, 128, 128, dtype=torch.bfloat16, seed=880, s0_std=0.3,
                            decay_regime="slow").to("cuda")
    gen = torch.Generator().manual_seed(881)
    d_o = torch.randn(B, T, H, 128, generator=gen).cuda()
    d_ST = torch.randn(B, H, 128, 128, generator=gen).cuda()
    ref = gdr2.backward_chunked(*x.tensors(), x.S0, d_o, d_ST)
    cu = torch.arange(0, (B + 1) * T, T, dtype=torch.int32, device="cuda")
    packed = [t.reshape(B * T, H, -1) for t in x.tensors()]
    got = gdr2.backward_chunked_varlen(*packed, cu, x.S0, d_o.reshape(B * T, H, -1), d_ST)
    torch.cuda.synchronize()
    for n, g, r in zip(NAMES + ("dS0",), got, ref):
        assert torch.equal(g.reshape(r.shape), r), n


def test_chunked_varlen_without_initial_state_or_final_gradient_and_unsupported_shapes():
    lengths = [100, 28]
    H = 2
    seqs, toks, _, cu, d_o, _ = _packed(lengths, H, 128, 128, torch.bfloat16, seed=890, decay_regime="slow")
    d = [t.cuda() for t in toks]
    got = gdr2.backward_chunked_varlen(*d, cu.cuda(), None, d_o.cuda(), None)
    torch.cuda.synchronize()
    assert gdr2.gdr2_device_status() == 0
    zeros = torch.zeros(len(lengths), H, 128, 128)
    for i, s in enumerate(seqs):
        _check_sequence_chunked(got, s, i, int(cu[i]), int(cu[i + 1]), zeros, d_o, zeros, "S0 = 0, dS_T = 0")
    with pytest.raises(gdr2.GDR2Error):   # fp32 inputs: the exact path only
        gdr2.backward_chunked_varlen(*[t.float() for t in d], cu.cuda(), None, d_o.cuda(), None)


def test_chunked_varlen_small_head_sizes():
    """Packed sequences with d_k = 64, d_v = 32 on the zero-padded tensor-core path:
    per-sequence oracle parity at the bf16 bar."""
    lengths = [70, 129, 1]
    H = 2
    seqs, toks, S0, cu, d_o, d_ST = _packed(lengths, H, 64, 32, torch.bfloat16, seed=893, decay_regime="slow")
    got = gdr2.backward_chunked_varlen(*[t.cuda() for t in toks], cu.cuda(), S0.cuda(), d_o.cuda(), d_ST.cuda())
    torch.cuda.synchronize()
    assert gdr2.gdr2_device_status() == 0
    for i, s in enumerate(seqs):
        _check_sequence_chunked(got, s, i, int(cu[i]), int(cu[i + 1]), S0, d_o, d_ST, "chunked dk=64 dv=32")


def test_autograd_varlen_chunked_backward():
    """gdr2_apply_varlen(chunked_backward=True) on bf16 inputs: gradients through
    the tensor-core path, returned in bf16 (bar 2e-2 plus one bf16 rounding)."""
    lengths = [90, 0, 200]
    H = 2
    seqs, toks, S0, cu, d_o, d_ST = _packed(lengths, H, 128, 128, torch.bfloat16, seed=895, decay_regime="slow")
    leaves = [t.cuda().requires_grad_(True) for t in toks] + [S0.cuda().requires_grad_(True)]
    o, S_T = gdr2.gdr2_apply_varlen(*leaves[:6], cu.cuda(), leaves[6], chunked_backward=True)
    ((o * d_o.cuda()).sum() + (S_T * d_ST.cuda()).sum()).backward()
    for i, s in enumerate(seqs):
        a, e = int(cu[i]), int(cu[i + 1])
        if e == a:
            assert torch.equal(leaves[6].grad[i].cpu(), d_ST[i])
            continue
        ref = oracle.backward(*s.tensors(), S0[i:i + 1], d_o[a:e].unsqueeze(0), d_ST[i:i + 1])
        for name, leaf, rf in zip(NAMES + ("dS0",), leaves, ref):
            g = leaf.grad[i:i + 1] if name == "dS0" else leaf.grad[a:e].unsqueeze(0)
            assert g.dtype == leaf.dtype
            bar = TOL_CHUNKED + float(np.abs(rf).max()) * 2.0 ** -8 / float(np.sqrt(np.mean(rf * rf)))
            err = err_over_rms(g.float().cpu().numpy(), rf)
            assert err <= bar, f"sequence {i} {name}: {err:.3e} (bar {bar:.3g})"


def test_chunked_overlapping_offsets_stay_within_the_workspace():
    """Offsets [0, 640, 0, 640, 0, 640] claim 30 chunks where the workspace holds 15
    (see the forward's test of the same offsets): sequence 0 keeps its 10 chunks,
    sequence 2 gets its first 5 and sequence 4 none.  dS0 of each follows from the
    chunks it was given: the full sequence, the first 320 tokens with dS_T at their
    end, and dS_T itself."""
    H, total = 2, 640
    x = make_prefill_inputs(1, total, H, 128, 128, dtype=torch.bfloat16, seed=896, s0_std=0.3,
                            decay_regime="slow")
    gen = torch.Generator().manual_seed(897)
    S0 = torch.randn(5, H, 128, 128, generator=gen) * 0.3
    d_o = torch.randn(total, H, 128, generator=gen)
    d_ST = torch.randn(5, H, 128, 128, generator=gen)
    cu = torch.tensor([0, 640, 0, 640, 0, 640], dtype=torch.int32)
    toks = [t[0].contiguous().cuda() for t in x.tensors()]
    got = gdr2.backward_chunked_varlen(*toks, cu.cuda(), S0.cuda(), d_o.cuda(), d_ST.cuda())
    torch.cuda.synchronize()
    assert gdr2.gdr2_device_status() == 0
    dS0 = got[6].cpu()
    for i in (1, 3, 4):
        assert torch.equal(dS0[i], d_ST[i]), i
    for i, L in ((0, 640), (2, 320)):
        ref = oracle.backward(*(t[:, :L] for t in x.tensors()), S0[i:i + 1], d_o[:L].unsqueeze(0), d_ST[i:i + 1])
        err = err_over_rms(dS0[i:i + 1].numpy(), ref[6])
        assert err <= TOL_CHUNKED, f"sequence {i}: dS0 {err:.3e}"
