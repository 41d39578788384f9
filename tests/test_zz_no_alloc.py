"""gdr2_forward_noalloc: the prefill entry point that allocates no device memory.

Some callers cannot allocate device memory when they call the library: a
serving runtime that reserves all memory at start-up and forbids allocation on
its request path, or a host whose device memory belongs to someone else and
that may not draw from the stream-ordered workspace pool that gdr2_forward
uses.  This entry point keeps the workspace in a fixed array inside the
library and runs the prefill over ranges of chunks that fit it.

Checked here, on two calls in a row (the array keeps the previous call's
contents): the results match the fp64 oracle within the bf16 bar and are bit
for bit those of the same kernels run over the whole sequence at once, and a
call leaves both the library's workspace pool and the device's default pool
untouched (a control call of gdr2_forward does draw on the library's pool).

This file is collected last so that a run stopping at the first failure has
already run every other test."""
import ctypes

import numpy as np
import pytest
import torch

import gated_delta_rule_166_b300 as gdr2
from gated_delta_rule_166_b300 import _lib
from gated_delta_rule_166_b300.inputs import make_prefill_inputs, make_workload

from gpu_util import TOL_BF16, err_over_rms, run_oracle

pytestmark = pytest.mark.gpu

GDR2_ERR_SCRATCH = -8
_USED_MEM_HIGH = 8   # cudaMemPoolAttrUsedMemHigh


def _np(t):
    return t.float().cpu().numpy()


def _cudart():
    """The CUDA runtime that torch loaded (its default-pool queries see the same
    driver pool as the library's)."""
    for name in ("libcudart.so.13", "libcudart.so"):
        try:
            return ctypes.CDLL(name)
        except OSError:
            continue
    pytest.skip("no CUDA runtime library to query the default memory pool")


def _default_pool_used_high(reset=False):
    rt = _cudart()
    pool = ctypes.c_void_p()
    dev = torch.cuda.current_device()
    assert rt.cudaDeviceGetDefaultMemPool(ctypes.byref(pool), ctypes.c_int(dev)) == 0
    val = ctypes.c_uint64(0)
    assert rt.cudaMemPoolGetAttribute(pool, ctypes.c_int(_USED_MEM_HIGH), ctypes.byref(val)) == 0
    if reset:
        zero = ctypes.c_uint64(0)
        assert rt.cudaMemPoolSetAttribute(pool, ctypes.c_int(_USED_MEM_HIGH), ctypes.byref(zero)) == 0
    return val.value


def _noalloc_twice(x, return_state=True):
    """Two calls in a row with preallocated outputs; each checked for device
    errors and for allocations; returns both results."""
    outs = []
    for _ in range(2):
        o = torch.empty(x.v.shape, dtype=torch.float32, device="cuda")
        S = torch.empty((*x.q.shape[:1], x.q.shape[2], x.q.shape[3], x.v.shape[3]),
                        dtype=torch.float32, device="cuda") if return_state else None
        torch.cuda.synchronize()
        gdr2.gdr2_workspace_stats(reset=True)
        _default_pool_used_high(reset=True)
        o, S = gdr2.forward_noalloc(*x.tensors(), x.S0, o=o, S_T=S, return_state=return_state)
        torch.cuda.synchronize()
        assert gdr2.gdr2_device_status() == 0
        assert gdr2.gdr2_workspace_stats()[1] == 0, "the no-allocation call drew on the workspace pool"
        assert _default_pool_used_high() == 0, "the no-allocation call drew on the default pool"
        outs.append((o, S))
    return outs


@pytest.mark.parametrize("case", ["layer_with_S0", "ragged_many_heads", "small_head_dims"])
def test_noalloc_matches_oracle_and_forward_on_two_calls(case):
    if case == "layer_with_S0":
        # B*H = 64: ranges of 14 chunks, the state carried in S_T across 5 ranges
        xh = make_workload("gdn2_layer_T4096", s0_std=0.02)
    elif case == "ragged_many_heads":
        # B*H = 128: ranges of 7 chunks over 16 chunks, the last one partial
        xh = make_prefill_inputs(8, 1000, 16, 128, 128, seed=11, decay_regime="slow", s0_std=0.3)
    else:
        # d_k = 64, d_v = 32 (zero-padded channels); B*H = 480: ranges of 1 chunk
        xh = make_prefill_inputs(30, 300, 16, 64, 32, seed=12, s0_std=0.3)
    x = xh.to("cuda")
    # the same kernels over the whole sequence at once (one sequential state pass)
    ref_o, ref_S = gdr2.forward(*x.tensors(), x.S0, segments=1)
    torch.cuda.synchronize()
    assert gdr2.gdr2_device_status() == 0
    ro, rS = run_oracle(xh)
    for o, S in _noalloc_twice(x):
        assert err_over_rms(_np(o), ro) <= TOL_BF16
        assert err_over_rms(_np(S), rS) <= TOL_BF16
        assert torch.equal(o, ref_o) and torch.equal(S, ref_S)


def test_noalloc_without_final_state():
    """S_T = NULL: the state between chunk ranges lives in the scratch."""
    xh = make_prefill_inputs(4, 777, 16, 128, 128, seed=5, s0_std=0.5)
    x = xh.to("cuda")
    ro, _ = run_oracle(xh)
    ref_o, _ = gdr2.forward(*x.tensors(), x.S0, segments=1)
    torch.cuda.synchronize()
    for o, S in _noalloc_twice(x, return_state=False):
        assert S is None
        assert err_over_rms(_np(o), ro) <= TOL_BF16
        assert torch.equal(o, ref_o)


def test_forward_control_draws_on_workspace_pool():
    """The control for the checks above: gdr2_forward's workspace comes from the
    library's pool, and the high-water mark sees it."""
    x = make_prefill_inputs(2, 256, 4, 128, 128, seed=3).to("cuda")
    torch.cuda.synchronize()
    gdr2.gdr2_workspace_stats(reset=True)
    gdr2.forward(*x.tensors(), x.S0)
    torch.cuda.synchronize()
    assert gdr2.gdr2_workspace_stats()[1] > 0


def test_noalloc_rejects_too_many_heads():
    """B*H beyond the fixed scratch is refused before anything is enqueued (the
    addresses below are never dereferenced)."""
    base, gap = 1 << 40, 1 << 34
    p = [ctypes.c_void_p(base + i * gap) for i in range(9)]
    st = _lib.lib().gdr2_forward_noalloc(*p, 1, 64, 1024, 128, 128, 1, 0, None)
    assert st == GDR2_ERR_SCRATCH
    assert "scratch" in _lib.status_string(st)
