"""The chunk-parallel scan over sequence segments (gdr2_forward_segmented and
the library's own choice in gdr2_forward) against the fp64 CPU oracle, at the
bf16 bar (max|err| / RMS(ref) <= 2e-2 for o and S_T).  Slow and mixed decays
with a non-zero S0 keep the start state of every segment visible in o and S_T;
ragged lengths leave a partial last chunk in the last segment."""
import numpy as np
import pytest
import torch

import gated_delta_rule_166_b300 as gdr2
from gated_delta_rule_166_b300 import GDR2Error
from gated_delta_rule_166_b300.inputs import make_prefill_inputs, make_workload
from gpu_util import compare, err_over_rms, run_gpu, run_oracle

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("segments", [1, 2, 3, 5])
@pytest.mark.parametrize("T", [2048 + 37, 1024])
@pytest.mark.parametrize("regime", ["slow", "mixed"])
def test_segments_vs_oracle(segments, T, regime):
    x = make_prefill_inputs(2, T, 2, 128, 128, dtype=torch.bfloat16, seed=300 + T + segments,
                            decay_regime=regime, s0_std=0.5)
    compare(x, f"segments={segments} T={T} {regime}", segments=segments)


def test_segments_more_than_one_wave_and_capped():
    # 8 segments of 16 heads: 480 CTAs, several waves; 1000 segments are capped at the chunk count
    x = make_prefill_inputs(1, 4096 + 5, 16, 128, 128, dtype=torch.bfloat16, seed=41,
                            decay_regime="mixed", s0_std=0.3)
    ref = run_oracle(x)
    compare(x, "segments=8", segments=8, ref=ref)
    y = make_prefill_inputs(1, 700, 2, 128, 128, dtype=torch.bfloat16, seed=42,
                            decay_regime="zero", s0_std=0.3)
    compare(y, "segments=1000 (capped at 11 chunks)", segments=1000)


def test_segments_value_width_64_and_bf16_output():
    x = make_prefill_inputs(2, 1500, 3, 128, 64, dtype=torch.bfloat16, seed=43,
                            decay_regime="slow", s0_std=0.4)
    ref = run_oracle(x)
    compare(x, "dv=64 segments=3", segments=3, ref=ref)
    compare(x, "dv=64 segments=4 bf16 o", segments=4, ref=ref, out_dtype=torch.bfloat16)
    y = make_prefill_inputs(1, 1300, 2, 128, 128, dtype=torch.bfloat16, seed=44,
                            decay_regime="slow", s0_std=0.4)
    compare(y, "dv=128 segments=3 bf16 o", segments=3, out_dtype=torch.bfloat16)


def test_segments_state_in_place_and_no_state():
    x = make_prefill_inputs(1, 1200, 2, 128, 128, dtype=torch.bfloat16, seed=45,
                            decay_regime="slow", s0_std=0.5)
    ro, rS = run_oracle(x)
    d = x.to("cuda")
    S = d.S0.clone()
    o, ST = gdr2.forward(*d.tensors(), S, S_T=S, segments=3)   # S_T is S0: updated in place
    torch.cuda.synchronize()
    assert ST is S and gdr2.gdr2_device_status() == 0
    assert err_over_rms(o.cpu().numpy(), ro) <= 2e-2
    assert err_over_rms(S.cpu().numpy(), rS) <= 2e-2
    o2, ST2 = gdr2.forward(*d.tensors(), d.S0, return_state=False, segments=3)
    torch.cuda.synchronize()
    assert ST2 is None
    assert err_over_rms(o2.cpu().numpy(), ro) <= 2e-2


def test_segments_rejected_where_unsupported():
    x = make_prefill_inputs(1, 200, 2, 64, 64, dtype=torch.float32, seed=46).to("cuda")
    with pytest.raises(GDR2Error) as e:
        gdr2.forward(*x.tensors(), x.S0, segments=2)
    assert e.value.status == -4   # GDR2_ERR_UNSUPPORTED: fp32 inputs take the token-recurrent kernel
    o, _ = gdr2.forward(*x.tensors(), x.S0, segments=1)   # one segment is the plain path
    torch.cuda.synchronize()
    ro, _ = run_oracle(x.to("cpu"))
    assert err_over_rms(o.cpu().numpy(), ro) <= 1e-4


def test_long_context_sequential_and_segmented_agree_with_oracle():
    """The long-context workload (1 x 16 heads x 65536 tokens) with slow decay:
    the library's choice (2 segments on a 148-SM part) and the sequential pass
    (segments=1) against one oracle run, and against each other."""
    x = make_workload("long_T65536", decay_regime="slow")
    ref = run_oracle(x)
    go1, gS1 = run_gpu(x, segments=1)
    goa, gSa = run_gpu(x)
    for label, (go, gS) in (("sequential", (go1, gS1)), ("auto", (goa, gSa))):
        eo, eS = err_over_rms(go, ref[0]), err_over_rms(gS, ref[1])
        assert eo <= 2e-2 and eS <= 2e-2, f"{label}: o={eo:.3e} S_T={eS:.3e}"
    assert err_over_rms(goa, go1) <= 2e-2 and err_over_rms(gSa, gS1) <= 2e-2
    assert np.isfinite(goa).all()
