"""gdr2_sparse_write on the GPU against the fp64 sparse-write oracle: slot
counts that do and do not fill the kernel's unrolled slot loop, ragged token
chunks, slots shared by consecutive tokens, out-of-range indices, K = 0, and
the full slot-memory workload (B4 H16 T4096, 2048 slots, 32 selected).  Slots
that no token selects must come back bit for bit."""
import numpy as np
import pytest
import torch

import oracle
import gated_delta_rule_166_b300 as gdr2
from gated_delta_rule_166_b300.inputs import make_sparse_inputs, make_sparse_workload

from gpu_util import TOL_BF16, TOL_F32, bf16_output_bar, err_over_rms

pytestmark = pytest.mark.gpu


def _run(x, out_dtype=torch.float32):
    d = x.to("cuda")
    S = d.S0.clone()
    o = gdr2.sparse_write(*d.tensors(), S, out_dtype=out_dtype)
    torch.cuda.synchronize()
    assert gdr2.gdr2_device_status() == 0
    return o.float().cpu().numpy(), S.cpu().numpy()


def _check(x, tol, out_dtype=torch.float32):
    o, S = _run(x, out_dtype)
    ro, rS = oracle.sparse_write(*x.tensors(), x.S0)
    assert err_over_rms(S, rS) <= tol
    tol_o = tol if out_dtype == torch.float32 else bf16_output_bar(ro, tol)
    assert err_over_rms(o, ro) <= tol_o
    return o, S, ro, rS


CASES = [
    # B, T, H, M, K, dv
    (1, 1, 1, 16, 1, 32),
    (2, 37, 3, 64, 8, 32),
    (1, 100, 2, 200, 17, 64),
    (2, 300, 2, 2048, 32, 128),
    (1, 50, 2, 100, 64, 128),
    (1, 40, 1, 8, 8, 64),       # every slot selected at every token
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "B{}T{}H{}M{}K{}dv{}".format(*c))
@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_sparse_matches_oracle(case, dtype):
    B, T, H, M, K, dv = case
    x = make_sparse_inputs(B, T, H, M, K, dv, dtype=dtype, seed=40 + T, s0_std=0.3)
    _check(x, TOL_F32 if dtype == torch.float32 else TOL_BF16)


def test_sparse_bf16_output():
    x = make_sparse_inputs(2, 130, 2, 512, 16, 128, seed=7, s0_std=0.3)
    _check(x, TOL_BF16, out_dtype=torch.bfloat16)


def test_sparse_untouched_slots_bit_exact():
    x = make_sparse_inputs(1, 20, 2, 1000, 4, 64, dtype=torch.float32, seed=9, s0_std=0.5)
    _, S = _run(x)
    sel = x.idx.numpy()
    for h in range(2):
        untouched = np.setdiff1d(np.arange(1000), sel[0, :, h].ravel())
        assert untouched.size > 0
        assert np.array_equal(S[0, h, untouched], x.S0.numpy()[0, h, untouched])


def test_sparse_out_of_range_indices_select_nothing():
    x = make_sparse_inputs(2, 70, 2, 96, 6, 32, dtype=torch.float32, seed=12, s0_std=0.3)
    rng = np.random.default_rng(3)
    idx = x.idx.numpy().copy()
    hit = rng.random(idx.shape) < 0.3
    idx[hit] = np.where(rng.random(int(hit.sum())) < 0.5, -7, 96 + 5)
    x.idx = torch.from_numpy(idx).to(torch.int32)
    _check(x, TOL_F32)


def test_sparse_nothing_selected():
    x = make_sparse_inputs(1, 33, 2, 50, 0, 64, dtype=torch.float32, seed=13, s0_std=0.3)
    o, S = _run(x)
    assert np.array_equal(S, x.S0.numpy())
    assert not np.any(o)


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_sparse_memory_beyond_shared_memory(dtype):
    """60,000 slots: too many for a one-column tile in shared memory, so the
    kernel that gathers from and scatters to global memory runs."""
    x = make_sparse_inputs(1, 45, 2, 60000, 24, 32, dtype=dtype, seed=21, s0_std=0.3)
    _check(x, TOL_F32 if dtype == torch.float32 else TOL_BF16)


def test_sparse_full_workload():
    """2048 slots x 128 value columns per head, 32 slots per token, B4 H16
    T4096, bf16 inputs: the whole output and memory against the oracle."""
    x = make_sparse_workload()
    _check(x, TOL_BF16)
