"""The chunk-parallel scan over sequence segments for packed sequences
(gdr2_forward_varlen_segmented, and the library's own choice in
gdr2_forward_varlen) against the fp64 oracle run on each sequence alone, at
the bf16 bar (max|err| / RMS(ref) <= 2e-2 for o and S_T).  Slow and mixed
decays with a non-zero S0 keep every segment's start state visible; ragged
lengths give segments of different lengths per sequence, partial last chunks
and empty segments (sequences shorter than G chunks); one long sequence is
bit for bit the fixed-length segmented call."""
import numpy as np
import pytest
import torch

import gated_delta_rule_166_b300 as gdr2
import oracle
from gated_delta_rule_166_b300.inputs import make_prefill_inputs
from gpu_util import TOL_BF16, err_over_rms

pytestmark = pytest.mark.gpu


def _packed(lengths, H, dv, seed, **kw):
    seqs = [make_prefill_inputs(1, L, H, 128, dv, dtype=torch.bfloat16, seed=seed + 17 * i, s0_std=0.5, **kw)
            for i, L in enumerate(lengths)]
    cat = lambda i: torch.cat([s.tensors()[i][0] for s in seqs], dim=0).contiguous()  # noqa: E731
    toks = [cat(i) for i in range(6)]
    S0 = torch.stack([s.S0[0] for s in seqs]).contiguous()
    cu = torch.tensor(np.concatenate([[0], np.cumsum(lengths)]), dtype=torch.int32)
    return seqs, toks, S0, cu


def _check(seqs, cu, o, ST, label, tol=TOL_BF16):
    o, ST = o.float().cpu().numpy(), ST.cpu().numpy()
    for i, s in enumerate(seqs):
        a, e = int(cu[i]), int(cu[i + 1])
        ro, rS = oracle.forward(*s.tensors(), s.S0)
        if e > a:
            err = err_over_rms(o[a:e], ro[0])
            assert err <= tol, f"{label}: sequence {i} (T={e - a}) o {err:.3e}"
        err = err_over_rms(ST[i:i + 1], rS)
        assert err <= tol, f"{label}: sequence {i} (T={e - a}) S_T {err:.3e}"


@pytest.mark.parametrize("segments", [2, 3, 5])
@pytest.mark.parametrize("regime", ["slow", "mixed"])
def test_ragged_segments_vs_oracle(segments, regime):
    # 1 and 100 tokens leave most of their segments empty; 2085 and 1200 split
    # into runs of different lengths with partial last chunks
    lengths = [2085, 1, 1200, 100, 640]
    seqs, toks, S0, cu = _packed(lengths, 2, 128, seed=500 + segments, decay_regime=regime)
    o, ST = gdr2.forward_varlen(*[t.cuda() for t in toks], cu.cuda(), S0.cuda(), segments=segments)
    torch.cuda.synchronize()
    assert gdr2.gdr2_device_status() == 0
    _check(seqs, cu, o, ST, f"segments={segments} {regime}")


def test_value_width_64_bf16_output_and_empty_sequence():
    lengths = [1500, 0, 777]
    seqs, toks, S0, cu = _packed(lengths, 3, 64, seed=520, decay_regime="slow")
    d = [t.cuda() for t in toks]
    o, ST = gdr2.forward_varlen(*d, cu.cuda(), S0.cuda(), segments=3, out_dtype=torch.bfloat16)
    torch.cuda.synchronize()
    assert gdr2.gdr2_device_status() == 0
    assert torch.equal(ST[1].cpu(), S0[1])
    # bf16 o: the bar plus one bf16 rounding of the output (the fp32-o call meets 2e-2)
    o32, _ = gdr2.forward_varlen(*d, cu.cuda(), S0.cuda(), segments=3)
    _check(seqs, cu, o32, ST, "dv=64 segments=3")
    diff = (o.float() - o32).abs().max().item()
    assert diff <= o32.abs().max().item() * 2.0 ** -8


def test_one_sequence_matches_fixed_length_segments_bit_for_bit():
    """One packed sequence with G = 2 runs the same chunk runs, scan and products as
    gdr2_forward(segments=2) on the same tokens (L even there, ceil(chunks / 2) here:
    32 chunks give 16 either way)."""
    T, H = 2048, 2
    x = make_prefill_inputs(1, T, H, 128, 128, dtype=torch.bfloat16, seed=530, decay_regime="mixed",
                            s0_std=0.4).to("cuda")
    o_f, S_f = gdr2.forward(*x.tensors(), x.S0, segments=2)
    cu = torch.tensor([0, T], dtype=torch.int32, device="cuda")
    o_v, S_v = gdr2.forward_varlen(*[t[0] for t in x.tensors()], cu, x.S0, segments=2)
    torch.cuda.synchronize()
    assert torch.equal(o_v, o_f[0])
    assert torch.equal(S_v, S_f)


def test_library_choice_takes_segments_for_one_long_sequence():
    """gdr2_forward_varlen on one long sequence of a few heads: the library's own
    choice runs the segmented scan (launch list) and matches the oracle."""
    T, H = 4096 + 21, 4
    seqs, toks, S0, cu = _packed([T], H, 128, seed=540, decay_regime="slow")
    d = [t.cuda() for t in toks]
    from torch.profiler import ProfilerActivity, profile

    with profile(activities=[ProfilerActivity.CUDA]) as prof:
        o, ST = gdr2.forward_varlen(*d, cu.cuda(), S0.cuda())
        torch.cuda.synchronize()
    names = {e.name for e in prof.events()}
    assert any("correct_kernel" in n for n in names) and any("seg_plan_kernel" in n for n in names), sorted(names)
    assert gdr2.gdr2_device_status() == 0
    _check(seqs, cu, o, ST, "library choice")


def test_overlapping_offsets_stay_within_the_workspace_with_segments():
    """The capped chunk offsets of overlapping malformed offsets (see the one-pass
    test) with segments: sequence 0 is exact, sequence 2 keeps its first 5 chunks,
    the empty ones keep S0, and nothing leaves the workspace."""
    H, total = 2, 640
    x = make_prefill_inputs(1, total, H, 128, 128, dtype=torch.bfloat16, seed=550, s0_std=0.3,
                            decay_regime="slow")
    S0 = torch.randn(5, H, 128, 128) * 0.3
    cu = torch.tensor([0, 640, 0, 640, 0, 640], dtype=torch.int32)
    toks = [t[0].cuda() for t in x.tensors()]
    o, ST = gdr2.forward_varlen(*toks, cu.cuda(), S0.cuda(), segments=3)
    torch.cuda.synchronize()
    assert gdr2.gdr2_device_status() == 0
    ST = ST.cpu()
    for i in (1, 3, 4):
        assert torch.equal(ST[i], S0[i]), i
    _, rS = oracle.forward(*x.tensors(), S0[0:1])
    assert err_over_rms(ST[0:1].numpy(), rS) <= TOL_BF16
    _, rS2 = oracle.forward(*(t[:, :320] for t in x.tensors()), S0[2:3])
    assert err_over_rms(ST[2:3].numpy(), rS2) <= TOL_BF16


def test_segments_rejected_for_fp32_and_small_heads():
    x = make_prefill_inputs(1, 300, 2, 64, 64, dtype=torch.bfloat16, seed=560, s0_std=0.3)
    cu = torch.tensor([0, 300], dtype=torch.int32, device="cuda")
    toks = [t[0].cuda() for t in x.tensors()]
    with pytest.raises(gdr2.GDR2Error):
        gdr2.forward_varlen(*toks, cu, None, segments=2)
    with pytest.raises(gdr2.GDR2Error):
        gdr2.forward_varlen(*[t.float() for t in toks], cu, None, segments=2)
