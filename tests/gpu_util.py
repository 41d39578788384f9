"""Helpers shared by the GPU parity tests: run the CUDA library and the CPU
oracle on the same seeded inputs and compare element by element."""
from __future__ import annotations

import numpy as np
import torch

import oracle
import gated_delta_rule_166_b300 as gdr2

# Parity bars: max |gpu - ref| / RMS(ref) over the whole tensor, for o and S_T.
TOL_F32 = 1e-4     # fp32 inputs
TOL_BF16 = 2e-2    # bf16 inputs, fp32 state


def err_over_rms(got, ref) -> float:
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape, (got.shape, ref.shape)
    if ref.size == 0:
        return 0.0
    rms = float(np.sqrt(np.mean(ref * ref)))
    diff = np.abs(got - ref)
    if not np.all(np.isfinite(got)):
        return float("inf")
    return float(diff.max()) / max(rms, 1e-30)


def tol_for(dtype) -> float:
    return TOL_F32 if dtype == torch.float32 else TOL_BF16


def bf16_output_bar(ref, base_tol) -> float:
    """Bar for bf16 o: the fp32-output bar plus one bf16 rounding of the
    largest output (relative 2^-9 of max|ref|), expressed against RMS(ref)."""
    ref = np.asarray(ref, dtype=np.float64)
    rms = float(np.sqrt(np.mean(ref * ref)))
    return base_tol + float(np.abs(ref).max()) * 2.0 ** -9 / max(rms, 1e-30)


def run_gpu(x, S0=None, device="cuda", out_dtype=torch.float32, segments=None):
    d = x.to(device)
    S0d = None if S0 is None else S0.to(device)
    o, ST = gdr2.forward(*d.tensors(), S0d if S0 is not None else d.S0, out_dtype=out_dtype,
                         segments=segments)
    torch.cuda.synchronize()
    assert gdr2.gdr2_device_status() == 0
    return o.float().cpu().numpy(), ST.cpu().numpy()


def run_oracle(x, S0=None):
    return oracle.forward(*x.tensors(), S0 if S0 is not None else x.S0)


def compare(x, label="", tol=None, out_dtype=torch.float32, segments=None, ref=None):
    """Run both sides on the prefill inputs x; return (err_o, err_S).  With a
    bf16 o the bar on o grows by exactly the output rounding term.  `segments`
    is passed to gdr2.forward; `ref` = (o, S_T) of the oracle if already known."""
    tol = tol if tol is not None else tol_for(x.q.dtype)
    go, gS = run_gpu(x, out_dtype=out_dtype, segments=segments)
    ro, rS = ref if ref is not None else run_oracle(x)
    eo, eS = err_over_rms(go, ro), err_over_rms(gS, rS)
    tol_o = tol if out_dtype == torch.float32 else bf16_output_bar(ro, tol)
    assert eo <= tol_o and eS <= tol, (
        f"{label}: err/RMS o={eo:.3e} (bar {tol_o:.3g}) S_T={eS:.3e} (bar {tol:g})")
    return eo, eS
