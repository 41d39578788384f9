"""Property tests of the C ABI's host-side validation (CPU only): every entry
point, given extreme or malformed sizes, misaligned or overlapping pointers and
unknown dtypes, returns one of the documented status codes and never crashes.
No device is touched: the module is skipped where a CUDA device is visible, and
without one even valid arguments stop at the device check, so the fake
addresses are never dereferenced."""
import ctypes

import pytest
import torch
from hypothesis import given, settings, strategies as st

from gated_delta_rule_166_b300 import _lib

# Generated argument sets can be valid; with a reachable GPU they would launch
# kernels on the fake addresses below, so these tests run only where no CUDA
# device is visible (there, valid arguments stop at the library's device check).
pytestmark = pytest.mark.skipif(torch.cuda.is_available(), reason="uses fake device addresses")

STATUSES = {0, -1, -2, -3, -4, -5, -6, -7, -8}
BASE = 1 << 40
GAP = 1 << 34

sizes = st.one_of(st.integers(-3, 5), st.integers(0, 1 << 20), st.sampled_from([1 << 31, 1 << 40, (1 << 62) - 1]))
dims = st.sampled_from([-1, 0, 16, 32, 48, 64, 96, 128, 256])
dtypes = st.sampled_from([-1, 0, 1, 2])
# fake device addresses: far apart, or overlapping, or misaligned, or null
ptr_kind = st.sampled_from(["ok", "null", "odd", "same"])


def fake(i, kind):
    if kind == "null":
        return None
    if kind == "odd":
        return ctypes.c_void_p(BASE + i * GAP + 4)
    if kind == "same":
        return ctypes.c_void_p(BASE)
    return ctypes.c_void_p(BASE + i * GAP)


@settings(max_examples=300, deadline=None)
@given(B=sizes, T=sizes, H=sizes, dk=dims, dv=dims, din=dtypes, dout=dtypes,
       kinds=st.lists(ptr_kind, min_size=9, max_size=9), seg=st.integers(-2, 9), cache=st.integers(-2, 9))
def test_forward_family_validation(B, T, H, dk, dv, din, dout, kinds, seg, cache):
    L = _lib.lib()
    p = [fake(i, k) for i, k in enumerate(kinds)]
    assert L.gdr2_forward(*p, B, T, H, dk, dv, din, dout, None) in STATUSES
    assert L.gdr2_forward_noalloc(*p, B, T, H, dk, dv, din, dout, None) in STATUSES
    assert L.gdr2_forward_segmented(*p, B, T, H, dk, dv, din, dout, seg, None) in STATUSES
    assert L.gdr2_forward_cached(*p, fake(9, kinds[0]), cache, B, T, H, dk, dv, din, dout, None) in STATUSES
    if B < 0 or T < 0 or H < 0:
        assert L.gdr2_forward(*p, B, T, H, dk, dv, din, dout, None) != 0


@settings(max_examples=200, deadline=None)
@given(N=sizes, total=sizes, H=sizes, dk=dims, dv=dims, din=dtypes, dout=dtypes,
       kinds=st.lists(ptr_kind, min_size=10, max_size=10))
def test_varlen_validation(N, total, H, dk, dv, din, dout, kinds):
    L = _lib.lib()
    p = [fake(i, k) for i, k in enumerate(kinds)]
    assert L.gdr2_forward_varlen(*p, N, total, H, dk, dv, din, dout, None) in STATUSES


@settings(max_examples=200, deadline=None)
@given(B=sizes, T=sizes, H=sizes, dk=dims, dv=dims, din=dtypes,
       kinds=st.lists(ptr_kind, min_size=16, max_size=16))
def test_backward_validation(B, T, H, dk, dv, din, kinds):
    L = _lib.lib()
    p = [fake(i, k) for i, k in enumerate(kinds)]
    rc = L.gdr2_backward(*p, B, T, H, dk, dv, din, None)
    assert rc in STATUSES
    if din not in (0, 1) and B >= 0 and T >= 0 and H >= 0:
        assert rc == -4


@settings(max_examples=200, deadline=None)
@given(B=sizes, H=sizes, dk=dims, dv=dims, din=dtypes, dout=dtypes,
       kinds=st.lists(ptr_kind, min_size=8, max_size=8))
def test_decode_validation(B, H, dk, dv, din, dout, kinds):
    L = _lib.lib()
    p = [fake(i, k) for i, k in enumerate(kinds)]
    assert L.gdr2_decode_step(*p, B, H, dk, dv, din, dout, None) in STATUSES
