"""gdr2_forward_train and gdr2_backward_from_context: the chunked backward split
where its forward recomputation ends, the per-chunk context kept by the caller.
The same kernels run on the same values, so the results are those of
gdr2_forward (o, S_T) and gdr2_backward_chunked (every gradient) bit for bit;
the chunked backward's own parity against the fp64 oracle is tested in
test_gpu_backward_chunked.py, and the autograd path against the oracle here."""
import numpy as np
import pytest
import torch

import gated_delta_rule_166_b300 as gdr2
import oracle
from gated_delta_rule_166_b300.inputs import make_prefill_inputs
from gpu_util import err_over_rms

pytestmark = pytest.mark.gpu

NAMES = ("dq", "dk", "dv", "db", "dw", "dlog_decay", "dS0")


def _upstream(x, seed):
    gen = torch.Generator().manual_seed(seed)
    B, T, H, dk = x.q.shape
    dv = x.v.shape[-1]
    return torch.randn(B, T, H, dv, generator=gen).cuda(), torch.randn(B, H, dk, dv, generator=gen).cuda()


@pytest.mark.parametrize("dk,dv,T", [(128, 128, 300), (64, 32, 130), (128, 64, 64)])
def test_train_context_reproduces_forward_and_chunked_backward(dk, dv, T):
    x = make_prefill_inputs(2, T, 2, dk, dv, dtype=torch.bfloat16, seed=1200 + dk + dv + T, s0_std=0.3,
                            decay_regime="slow").to("cuda")
    o_f, S_f = gdr2.forward(*x.tensors(), x.S0)
    o_t, S_t, kept = gdr2.forward_train(*x.tensors(), x.S0)
    torch.cuda.synchronize()
    assert kept.numel() == gdr2.gdr2_train_context_bytes(2, T, 2, dk, dv)
    assert torch.equal(o_t, o_f) and torch.equal(S_t, S_f)
    for seed in (1, 2):   # the context is only read: two backward calls from it
        d_o, d_ST = _upstream(x, 1210 + seed)
        ref = gdr2.backward_chunked(*x.tensors(), x.S0, d_o, d_ST)
        got = gdr2.backward_from_context(kept, *x.tensors(), x.S0, d_o, d_ST)
        torch.cuda.synchronize()
        assert gdr2.gdr2_device_status() == 0
        for n, g, r in zip(NAMES, got, ref):
            assert torch.equal(g, r), (n, seed)


def test_train_context_bf16_output_no_state_and_no_initial_state():
    x = make_prefill_inputs(1, 200, 2, 128, 128, dtype=torch.bfloat16, seed=1220, decay_regime="mixed").to("cuda")
    assert x.S0 is None
    o_f, S_f = gdr2.forward(*x.tensors(), None, out_dtype=torch.bfloat16)
    o_t, S_t, kept = gdr2.forward_train(*x.tensors(), None, out_dtype=torch.bfloat16)
    torch.cuda.synchronize()
    assert o_t.dtype == torch.bfloat16 and torch.equal(o_t, o_f) and torch.equal(S_t, S_f)
    d_o, _ = _upstream(x, 1221)
    ref = gdr2.backward_chunked(*x.tensors(), None, d_o, None, want_dS0=False)
    got = gdr2.backward_from_context(kept, *x.tensors(), None, d_o, None, want_dS0=False)
    torch.cuda.synchronize()
    for n, g, r in zip(NAMES[:6], got[:6], ref[:6]):
        assert torch.equal(g, r), n
    assert got[6] is None


def test_train_context_empty_sequence_and_errors():
    x = make_prefill_inputs(1, 0, 2, 128, 128, dtype=torch.bfloat16, seed=1230, s0_std=0.2).to("cuda")
    o, S_T, kept = gdr2.forward_train(*x.tensors(), x.S0)
    torch.cuda.synchronize()
    assert gdr2.gdr2_train_context_bytes(1, 0, 2, 128, 128) == 0 and torch.equal(S_T, x.S0)
    y = make_prefill_inputs(1, 70, 2, 128, 128, dtype=torch.bfloat16, seed=1231).to("cuda")
    with pytest.raises(gdr2.GDR2Error):   # fp32 inputs: the exact path only
        gdr2.forward_train(*(t.float() for t in y.tensors()), None)
    with pytest.raises(ValueError):       # a context too small for these sizes
        gdr2.forward_train(*y.tensors(), None, ctx=torch.empty(1000, dtype=torch.uint8, device="cuda"))
    _, _, kept = gdr2.forward_train(*y.tensors(), None)
    d_o = torch.zeros(1, 70, 2, 128, device="cuda")
    with pytest.raises(gdr2.GDR2Error):   # a context for fewer tokens than these
        z = make_prefill_inputs(1, 700, 2, 128, 128, dtype=torch.bfloat16, seed=1232).to("cuda")
        gdr2.backward_from_context(kept, *z.tensors(), None, torch.zeros(1, 700, 2, 128, device="cuda"), None)


def test_autograd_keep_context_and_recompute_agree_and_match_oracle():
    """gdr2_apply(chunked_backward=True) keeps the context by default; with
    keep_context=False it recomputes it: the same gradients bit for bit, and both
    within the bf16 bar of the oracle (plus one bf16 rounding of the returned
    gradients)."""
    x = make_prefill_inputs(1, 260, 2, 128, 128, dtype=torch.bfloat16, seed=1240, decay_regime="slow", s0_std=0.2)
    gen = torch.Generator().manual_seed(1241)
    d_o = torch.randn(1, 260, 2, 128, generator=gen)
    d_ST = torch.randn(1, 2, 128, 128, generator=gen)
    grads = []
    for keep in (True, False):
        leaves = [t.cuda().requires_grad_(True) for t in (*x.tensors(), x.S0)]
        o, S_T = gdr2.gdr2_apply(*leaves, chunked_backward=True, keep_context=keep)
        ((o * d_o.cuda()).sum() + (S_T * d_ST.cuda()).sum()).backward()
        grads.append([leaf.grad for leaf in leaves])
    for n, a, b in zip(NAMES, *grads):
        assert torch.equal(a, b), n
    ref = oracle.backward(*x.tensors(), x.S0, d_o, d_ST)
    for n, g, rf in zip(NAMES, grads[0], ref):
        bar = 2e-2 + float(np.abs(rf).max()) * 2.0 ** -8 / float(np.sqrt(np.mean(rf * rf)))
        e = err_over_rms(g.float().cpu().numpy(), rf)
        assert e <= bar, f"{n}: {e:.3e} (bar {bar:.3g})"


def test_packed_train_context_reproduces_varlen_forward_and_chunked_backward():
    """Packed sequences (an empty one and ragged chunks among them): the training
    forward's o and S_T are gdr2_forward_varlen's and the gradients from its context
    gdr2_backward_chunked_varlen's, bit for bit; gdr2_apply_varlen with the default
    kept context gives the recomputing path's gradients."""
    lengths = [130, 0, 64, 257, 1]
    H = 2
    seqs = [make_prefill_inputs(1, L, H, 128, 64, dtype=torch.bfloat16, seed=1250 + 7 * i, s0_std=0.3,
                                decay_regime="slow") for i, L in enumerate(lengths)]
    toks = [torch.cat([s.tensors()[i][0] for s in seqs]).contiguous().cuda() for i in range(6)]
    S0 = torch.stack([s.S0[0] for s in seqs]).contiguous().cuda()
    cu = torch.tensor(np.concatenate([[0], np.cumsum(lengths)]), dtype=torch.int32, device="cuda")
    total = int(cu[-1])
    o_f, S_f = gdr2.forward_varlen(*toks, cu, S0)
    o_t, S_t, kept = gdr2.forward_train_varlen(*toks, cu, S0)
    torch.cuda.synchronize()
    assert torch.equal(o_t, o_f) and torch.equal(S_t, S_f)
    gen = torch.Generator().manual_seed(1260)
    d_o = torch.randn(total, H, 64, generator=gen).cuda()
    d_ST = torch.randn(len(lengths), H, 128, 64, generator=gen).cuda()
    ref = gdr2.backward_chunked_varlen(*toks, cu, S0, d_o, d_ST)
    got = gdr2.backward_from_context_varlen(kept, *toks, cu, S0, d_o, d_ST)
    torch.cuda.synchronize()
    assert gdr2.gdr2_device_status() == 0
    for n, g, r in zip(NAMES, got, ref):
        assert torch.equal(g, r), n
    grads = []
    for keep in (True, False):
        leaves = [t.clone().requires_grad_(True) for t in toks] + [S0.clone().requires_grad_(True)]
        o, S_T = gdr2.gdr2_apply_varlen(*leaves[:6], cu, leaves[6], chunked_backward=True, keep_context=keep)
        ((o * d_o).sum() + (S_T * d_ST).sum()).backward()
        grads.append([leaf.grad for leaf in leaves])
    for n, a, b in zip(NAMES, *grads):
        assert torch.equal(a, b), n
