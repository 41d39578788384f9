"""GPU prefill vs the fp64 CPU oracle, element by element on the same seeded
inputs.  Bars: max|err| / RMS(ref) <= 1e-4 (fp32 inputs), <= 2e-2 (bf16
inputs, fp32 state), for o and for S_T."""
import pytest
import torch

import gated_delta_rule_166_b300 as gdr2

from gated_delta_rule_166_b300.inputs import WORKLOADS, make_prefill_inputs, make_workload
from gpu_util import compare

pytestmark = pytest.mark.gpu


def test_tiny_fp32_workload():
    compare(make_workload("tiny_f32"), "tiny_f32")


# The full-size workloads, in the launch configuration the bench uses.
@pytest.mark.parametrize("name", ["gdn2_layer_T4096", "kda_T2048", "gdn_T2048", "long_T65536"])
def test_full_size_workload(name):
    compare(make_workload(name), name)


# Carry-exercising variants: slow / zero / mixed decay make S0 and the
# chunk-to-chunk state visible in o and S_T; ragged T leaves a partial chunk.
@pytest.mark.parametrize("regime", ["slow", "zero", "mixed", "fast"])
@pytest.mark.parametrize("T", [1000, 193])
def test_carry_regimes_bf16(regime, T):
    x = make_prefill_inputs(2, T, 4, 128, 128, dtype=torch.bfloat16, seed=11 + T,
                            decay_regime=regime, s0_std=0.5)
    compare(x, f"bf16 {regime} T={T}")


@pytest.mark.parametrize("dk,dv", [(32, 32), (64, 64), (128, 128), (32, 128), (128, 64)])
@pytest.mark.parametrize("regime", ["fast", "slow"])
def test_fp32_head_dims(dk, dv, regime):
    x = make_prefill_inputs(2, 150, 3, dk, dv, dtype=torch.float32, seed=dk + dv,
                            decay_regime=regime, s0_std=0.3)
    compare(x, f"fp32 dk={dk} dv={dv} {regime}")


@pytest.mark.parametrize("dk,dv", [(64, 64), (32, 128), (128, 32), (32, 32), (64, 32), (32, 64)])
def test_bf16_small_head_dims(dk, dv):
    x = make_prefill_inputs(2, 130, 2, dk, dv, dtype=torch.bfloat16, seed=5 * dk + dv, s0_std=0.2)
    compare(x, f"bf16 dk={dk} dv={dv}")
    compare(x, f"bf16 dk={dk} dv={dv} (bf16 o)", out_dtype=torch.bfloat16)


def _kernel_names(fn):
    """Names of the CUDA kernels that ``fn`` launches (torch profiler)."""
    from torch.profiler import ProfilerActivity, profile

    with profile(activities=[ProfilerActivity.CUDA]) as prof:
        fn()
        torch.cuda.synchronize()
    return {e.name for e in prof.events() if e.device_type == torch.autograd.DeviceType.CUDA}


@pytest.mark.parametrize("dk,dv", [(32, 32), (64, 128), (128, 32)])
def test_bf16_small_head_dims_run_the_chunked_kernels(dk, dv):
    """Small bf16 head sizes take the chunked tensor-core kernels (with zero-padded
    channels), not the token-recurrent one."""
    x = make_prefill_inputs(2, 200, 2, dk, dv, dtype=torch.bfloat16, seed=3, s0_std=0.2).to("cuda")
    names = _kernel_names(lambda: gdr2.forward(*x.tensors(), x.S0))
    assert any("prep2_kernel" in n for n in names), names
    assert any("chain_kernel" in n for n in names), names
    assert not any("recurrent" in n for n in names), names


@pytest.mark.parametrize("T", [1, 2, 63, 64, 65, 127, 128, 129])
def test_chunk_boundaries_bf16(T):
    x = make_prefill_inputs(1, T, 3, 128, 128, dtype=torch.bfloat16, seed=100 + T,
                            decay_regime="mixed", s0_std=0.5)
    compare(x, f"bf16 T={T}")


def test_erase_gate_up_to_two():
    # the page's ablation widens the erase range to [0, 2]: no clamp anywhere
    x = make_prefill_inputs(2, 300, 4, 128, 128, dtype=torch.bfloat16, seed=77, b_scale=2.0,
                            decay_regime="mixed", s0_std=0.2)
    compare(x, "b in [0,2]")
    x = make_prefill_inputs(1, 100, 2, 32, 32, dtype=torch.float32, seed=78, b_scale=2.0)
    compare(x, "fp32 b in [0,2]")


def test_tied_and_scalar_gates_small():
    for gates, decay in (("tied", "channel"), ("tied", "scalar"), ("channel", "scalar")):
        x = make_prefill_inputs(2, 257, 2, 128, 128, dtype=torch.bfloat16, seed=9,
                                gates=gates, decay=decay, decay_regime="slow", s0_std=0.1)
        compare(x, f"{gates}/{decay}")


@pytest.mark.parametrize("name", ["gdn2_layer_T4096"])
def test_bf16_output_mode(name):
    """o stored in bf16: the bar grows by one bf16 rounding of max|o|."""
    compare(make_workload(name), name + " (bf16 o)", out_dtype=torch.bfloat16)
    x = make_prefill_inputs(2, 300, 4, 128, 128, dtype=torch.bfloat16, seed=5,
                            decay_regime="mixed", s0_std=0.3)
    compare(x, "mixed (bf16 o)", out_dtype=torch.bfloat16)


def test_extreme_decays_and_resets():
    """Per-token log decays far below the chunked path's floor of -10 (-30, and
    -1e4 as a hard reset) stay within the bar: the floor changes the state
    carried across such a token by at most e^-10 of itself."""
    x = make_prefill_inputs(2, 400, 3, 128, 128, dtype=torch.bfloat16, seed=91, decay_regime="slow",
                            s0_std=0.5)
    gen = torch.Generator().manual_seed(92)
    g = x.log_decay.float()
    hard = torch.rand(g.shape, generator=gen) < 0.05
    g[hard] = -30.0
    reset = torch.rand(g.shape[:3], generator=gen) < 0.02          # whole-token resets
    g[reset] = -1e4
    x.log_decay = g.to(torch.bfloat16)
    compare(x, "extreme decays")


# The carry-exercising variants at the full shapes of the GDN-2 layer and
# long-context workloads: slow, zero and mixed decays with a non-zero S0 keep
# the chunk-to-chunk state and S0 visible in o and S_T over every chunk.
@pytest.mark.parametrize("regime", ["slow", "zero", "mixed"])
def test_full_size_carry_variants_layer(regime):
    x = make_workload("gdn2_layer_T4096", decay_regime=regime, s0_std=0.02)
    compare(x, f"gdn2_layer_T4096 {regime}")


def test_full_size_carry_variant_long():
    x = make_workload("long_T65536", decay_regime="slow")
    compare(x, "long_T65536 slow")
