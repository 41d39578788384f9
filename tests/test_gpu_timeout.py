"""The bounded-wait failure path on the device.

Every handshake wait of the prefill's chain kernel is bounded.  With the
testing hook gdr2_set_wait_limit(1) a wait gives up at its first miss, so a
call on one head of four chunks must stop early.  The kernel then still lets
its copies land and its tensor-core products complete, frees its tensor memory
and records the failure, and the next normal call must find a working
context: gdr2_device_status reports GDR2_ERR_TIMEOUT exactly once, and a call
with the default limit matches the fp64 oracle."""
import pytest
import torch

import gated_delta_rule_166_b300 as gdr2
from gated_delta_rule_166_b300.inputs import make_prefill_inputs

from gpu_util import TOL_BF16, bf16_output_bar, err_over_rms, run_oracle

pytestmark = pytest.mark.gpu

GDR2_ERR_TIMEOUT = -6


def _np(t):
    return t.float().cpu().numpy()


@pytest.mark.parametrize("out_dtype", [torch.bfloat16, torch.float32])
def test_chain_wait_gives_up_reports_and_recovers(out_dtype):
    xh = make_prefill_inputs(1, 256, 1, 128, 128, seed=31, s0_std=0.3)
    x = xh.to("cuda")
    assert gdr2.gdr2_device_status() == 0
    prev = gdr2.gdr2_set_wait_limit(1)
    try:
        gdr2.forward(*x.tensors(), x.S0, out_dtype=out_dtype)
        status = gdr2.gdr2_device_status()
    finally:
        gdr2.gdr2_set_wait_limit(prev)
    assert status == GDR2_ERR_TIMEOUT
    assert gdr2.gdr2_device_status() == 0   # reading cleared the record

    o, S = gdr2.forward(*x.tensors(), x.S0, out_dtype=out_dtype)
    torch.cuda.synchronize()
    assert gdr2.gdr2_device_status() == 0
    ro, rS = run_oracle(xh)
    assert err_over_rms(_np(S), rS) <= TOL_BF16
    tol_o = TOL_BF16 if out_dtype == torch.float32 else bf16_output_bar(ro, TOL_BF16)
    assert err_over_rms(_np(o), ro) <= tol_o
