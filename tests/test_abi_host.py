"""The C ABI on the host: the library loads, exports every entry point that
include/gdr2.h declares, and rejects bad arguments before touching a device.
No CUDA device is needed: the pointers below are never dereferenced because
validation fails first."""
import ctypes
import os
import re

import pytest

from gated_delta_rule_166_b300 import _lib

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "gdr2.h")

OK, ARG, SHAPE, ALIGN, UNSUP, CUDA, TIMEOUT, ALIAS, SCRATCH = 0, -1, -2, -3, -4, -5, -6, -7, -8


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(gdr2_[a-z_0-9]+)\s*\(", text)))


def test_library_exports_every_declared_symbol():
    L = _lib.lib()
    names = declared_functions()
    assert {"gdr2_forward", "gdr2_decode_step", "gdr2_device_status"} <= set(names)
    for n in names:
        assert hasattr(L, n), f"libgdr2.so does not export {n}"


def test_status_strings_and_version():
    for s in (OK, ARG, SHAPE, ALIGN, UNSUP, CUDA, TIMEOUT, ALIAS, SCRATCH):
        assert _lib.status_string(s).startswith("GDR2")
    assert _lib.gdr2_version() >= 100


def test_wait_limit_hook_swaps_and_restores():
    """The testing hook is host state only: it returns the previous limit and
    non-positive values mean the default (reported as 0)."""
    prev = _lib.gdr2_set_wait_limit(1234)
    try:
        assert _lib.gdr2_set_wait_limit(-5) == 1234
        assert _lib.gdr2_set_wait_limit(0) == 0
    finally:
        _lib.gdr2_set_wait_limit(prev)


# fake, never-dereferenced device addresses (16-byte aligned, far apart)
BASE = 1 << 40
GAP = 1 << 32


def fwd_args(B=1, T=4, H=2, dk=64, dv=64, dtype=1, out_dtype=0, **over):
    p = {n: ctypes.c_void_p(BASE + i * GAP) for i, n in
         enumerate(["q", "k", "v", "b", "w", "g", "S0", "o", "ST"])}
    p.update(over)
    return ([p[n] for n in ["q", "k", "v", "b", "w", "g", "S0", "o", "ST"]]
            + [B, T, H, dk, dv, dtype, out_dtype, None])


def call_fwd(**kw):
    return _lib.lib().gdr2_forward(*fwd_args(**kw))


@pytest.mark.parametrize("dk,dv", [(16, 64), (64, 96), (256, 128), (0, 32)])
def test_forward_rejects_head_dims(dk, dv):
    assert call_fwd(dk=dk, dv=dv) == SHAPE


def test_forward_rejects_negative_sizes_and_dtype():
    assert call_fwd(B=-1) == ARG
    assert call_fwd(T=-3) == ARG
    assert call_fwd(dtype=7) == UNSUP
    assert call_fwd(out_dtype=3) == UNSUP


def test_forward_rejects_null_token_pointer():
    for n in ("q", "k", "v", "b", "w", "g", "o"):
        assert call_fwd(**{n: None}) == ARG, n


def test_forward_rejects_misaligned_pointer():
    for n in ("q", "v", "S0", "o", "ST"):
        assert call_fwd(**{n: ctypes.c_void_p(BASE + 7 * GAP + 8)}) == ALIGN, n


def test_forward_rejects_aliasing():
    # o overlapping q, o overlapping S0, S_T overlapping a token input, S_T straddling S0
    assert call_fwd(o=ctypes.c_void_p(BASE)) == ALIAS
    assert call_fwd(o=ctypes.c_void_p(BASE + 6 * GAP)) == ALIAS
    assert call_fwd(ST=ctypes.c_void_p(BASE + 1 * GAP + 64)) == ALIAS
    assert call_fwd(ST=ctypes.c_void_p(BASE + 6 * GAP + 16)) == ALIAS


def test_forward_size_overflow():
    assert call_fwd(B=1 << 40, T=1 << 30) == SHAPE


def test_decode_rejects_bad_args():
    L = _lib.lib()
    p = [ctypes.c_void_p(BASE + i * GAP) for i in range(8)]
    assert L.gdr2_decode_step(*p, 4, 2, 48, 64, 1, 0, None) == SHAPE
    assert L.gdr2_decode_step(*p, -1, 2, 64, 64, 1, 0, None) == ARG
    assert L.gdr2_decode_step(*p, 4, 2, 64, 64, 1, 5, None) == UNSUP
    bad = list(p)
    bad[6] = None  # S
    assert L.gdr2_decode_step(*bad, 4, 2, 64, 64, 1, 0, None) == ARG
    bad = list(p)
    bad[7] = p[0]  # o aliases q
    assert L.gdr2_decode_step(*bad, 4, 2, 64, 64, 1, 0, None) == ALIAS
    bad = list(p)
    bad[2] = ctypes.c_void_p(BASE + 2 * GAP + 4)
    assert L.gdr2_decode_step(*bad, 4, 2, 64, 64, 1, 0, None) == ALIGN


def test_binding_rejects_cpu_tensors():
    torch = pytest.importorskip("torch")
    x = torch.zeros(1, 2, 1, 32)
    with pytest.raises(ValueError):
        _lib.gdr2_forward(x, x, x, x, x, x)


def varlen_args(N=3, total=10, H=2, dk=64, dv=64, dtype=1, out_dtype=0, **over):
    names = ["q", "k", "v", "b", "w", "g", "S0", "o", "ST", "cu"]
    p = {n: ctypes.c_void_p(BASE + i * GAP) for i, n in enumerate(names)}
    p.update(over)
    return [p[n] for n in names] + [N, total, H, dk, dv, dtype, out_dtype, None]


def test_varlen_rejects_bad_args():
    L = _lib.lib()
    assert L.gdr2_forward_varlen(*varlen_args(cu=None)) == ARG
    assert L.gdr2_forward_varlen(*varlen_args(cu=ctypes.c_void_p(BASE + 9 * GAP + 2))) == ALIGN
    assert L.gdr2_forward_varlen(*varlen_args(o=ctypes.c_void_p(BASE + 9 * GAP))) == ALIAS   # o over cu
    assert L.gdr2_forward_varlen(*varlen_args(ST=ctypes.c_void_p(BASE + 9 * GAP))) == ALIAS  # S_T over cu
    assert L.gdr2_forward_varlen(*varlen_args(dk=48)) == SHAPE
    assert L.gdr2_forward_varlen(*varlen_args(N=-1)) == ARG
    assert L.gdr2_forward_varlen(*varlen_args(total=1 << 31)) == SHAPE


def test_varlen_segmented_rejects_bad_args():
    L = _lib.lib()
    seg = lambda n, **kw: L.gdr2_forward_varlen_segmented(*(varlen_args(**kw)[:-1] + [n, None]))  # noqa: E731
    assert seg(-1) == ARG
    assert seg(2, cu=None) == ARG
    assert seg(2, dk=48) == SHAPE
    assert seg(2, total=1 << 31) == SHAPE
    assert seg(2, o=ctypes.c_void_p(BASE + 9 * GAP)) == ALIAS   # o over cu


def test_segmented_rejects_bad_args():
    L = _lib.lib()

    def seg(n, **kw):   # gdr2_forward's arguments with `segments` before the stream
        return L.gdr2_forward_segmented(*(fwd_args(**kw)[:-1] + [n, None]))

    assert seg(-1) == ARG
    assert seg(2, dk=16) == SHAPE
    assert seg(3, B=-1) == ARG
    assert seg(0, o=None) == ARG
    assert seg(2, o=ctypes.c_void_p(BASE)) == ALIAS


def bwd_args(B=1, T=4, H=2, dk=64, dv=64, dtype=1, **over):
    names = ["q", "k", "v", "b", "w", "g", "S0", "do", "dST",
             "gq", "gk", "gv", "gb", "gw", "gg", "gS0"]
    p = {n: ctypes.c_void_p(BASE + i * GAP) for i, n in enumerate(names)}
    p.update(over)
    return [p[n] for n in names] + [B, T, H, dk, dv, dtype, None]


def test_backward_rejects_bad_args():
    L = _lib.lib()
    call = lambda **kw: L.gdr2_backward(*bwd_args(**kw))  # noqa: E731
    assert call(B=-1) == ARG
    assert call(dk=48) == SHAPE
    assert call(dv=16) == SHAPE
    assert call(dtype=5) == UNSUP
    for n in ("q", "do", "gq", "gv", "gg"):
        assert call(**{n: None}) == ARG, n
    assert call(gk=ctypes.c_void_p(BASE + 11 * GAP + 4)) == ALIGN
    assert call(gq=ctypes.c_void_p(BASE)) == ALIAS                 # d_q over q
    assert call(gb=ctypes.c_void_p(BASE + 9 * GAP)) == ALIAS       # d_b over d_q
    assert call(gS0=ctypes.c_void_p(BASE + 6 * GAP)) == ALIAS      # d_S0 over S0


def bwd_varlen_args(N=3, total=10, H=2, dk=64, dv=64, dtype=1, **over):
    names = ["q", "k", "v", "b", "w", "g", "S0", "do", "dST",
             "gq", "gk", "gv", "gb", "gw", "gg", "gS0", "cu"]
    p = {n: ctypes.c_void_p(BASE + i * GAP) for i, n in enumerate(names)}
    p.update(over)
    return [p[n] for n in names] + [N, total, H, dk, dv, dtype, None]


def test_backward_varlen_rejects_bad_args():
    L = _lib.lib()
    call = lambda **kw: L.gdr2_backward_varlen(*bwd_varlen_args(**kw))  # noqa: E731
    assert call(cu=None) == ARG
    assert call(N=-1) == ARG
    assert call(total=-5) == ARG
    assert call(total=1 << 31) == SHAPE
    assert call(dk=48) == SHAPE
    assert call(dtype=5) == UNSUP
    assert call(gq=None) == ARG
    assert call(cu=ctypes.c_void_p(BASE + 16 * GAP + 2)) == ALIGN
    assert call(gg=ctypes.c_void_p(BASE + 16 * GAP)) == ALIAS      # d_log_decay over cu_seqlens
    assert call(gS0=ctypes.c_void_p(BASE + 16 * GAP)) == ALIAS     # d_S0 over cu_seqlens
    assert call(gv=ctypes.c_void_p(BASE + 2 * GAP)) == ALIAS       # d_v over v


def test_backward_chunked_varlen_rejects_bad_args():
    L = _lib.lib()
    call = lambda **kw: L.gdr2_backward_chunked_varlen(*bwd_varlen_args(**kw))  # noqa: E731
    assert call(cu=None) == ARG
    assert call(N=-1) == ARG
    assert call(total=1 << 31) == SHAPE
    assert call(dk=48) == SHAPE
    assert call(dtype=0, dk=128, dv=128) == UNSUP            # fp32 inputs
    assert call(cu=ctypes.c_void_p(BASE + 16 * GAP + 2), dk=128, dv=128) == ALIGN
    assert call(gq=ctypes.c_void_p(BASE + 16 * GAP), dk=128, dv=128) == ALIAS   # d_q over cu_seqlens


def test_train_context_bytes_by_hand_and_bad_sizes():
    L = _lib.lib()
    L.gdr2_train_context_bytes.restype = ctypes.c_int64
    # one 64-token chunk of one head: the forward slot (74,240 B), the backward record
    # (49,152 B) and one fp32 start state (65,536 B), each region rounded to 256 B
    assert L.gdr2_train_context_bytes(1, 64, 1, 128, 128) == 74240 + 49152 + 65536
    # a ragged second chunk adds a slot and a record but no cached state (the state after
    # the last, partial chunk is never a start state)
    assert L.gdr2_train_context_bytes(1, 65, 1, 128, 128) == 2 * 74240 + 2 * 49152 + 65536
    assert L.gdr2_train_context_bytes(1, 0, 3, 128, 128) == 0
    assert L.gdr2_train_context_bytes(-1, 64, 1, 128, 128) == ARG
    assert L.gdr2_train_context_bytes(1, 64, 1, 48, 128) == SHAPE


def test_forward_train_and_backward_from_context_reject_bad_args():
    L = _lib.lib()
    names = ["q", "k", "v", "b", "w", "g", "S0", "o", "ST", "ctx"]
    p = {n: ctypes.c_void_p(BASE + i * GAP) for i, n in enumerate(names)}

    def fwd(ctx_bytes=1 << 30, dtype=1, **over):
        q = dict(p)
        q.update(over)
        return L.gdr2_forward_train(*[q[n] for n in names], ctx_bytes, 1, 64, 2, 128, 128, dtype, 0, None)

    assert fwd(ctx=None) == ARG
    assert fwd(ctx_bytes=100) == ARG                              # smaller than the context
    assert fwd(ctx=ctypes.c_void_p(BASE + 9 * GAP + 8)) == ALIGN
    assert fwd(ctx=ctypes.c_void_p(BASE + 1 * GAP)) == ALIAS       # over k
    assert fwd(ctx=ctypes.c_void_p(BASE + 7 * GAP)) == ALIAS       # over o
    assert fwd(dtype=0) == UNSUP                                   # fp32 inputs
    bnames = ["q", "k", "v", "b", "w", "g", "S0", "do", "dST", "ctx",
              "gq", "gk", "gv", "gb", "gw", "gg", "gS0"]
    bp = {n: ctypes.c_void_p(BASE + i * GAP) for i, n in enumerate(bnames)}

    def bwd(ctx_bytes=1 << 30, **over):
        q = dict(bp)
        q.update(over)
        a = [q[n] for n in bnames]
        return L.gdr2_backward_from_context(*a[:10], ctx_bytes, *a[10:], 1, 64, 2, 128, 128, 1, None)

    assert bwd(ctx=None, ctx_bytes=0) == ARG
    assert bwd(ctx_bytes=100) == ARG
    assert bwd(gq=ctypes.c_void_p(BASE + 9 * GAP)) == ALIAS       # d_q over the context


def test_packed_train_context_bytes_and_bad_args():
    L = _lib.lib()
    L.gdr2_train_context_bytes_varlen.restype = ctypes.c_int64
    # 2 sequences over 65 rows: ceil(65 / 64) + 2 = 4 chunk slots, records and states per
    # head, plus the sequences' first chunks (3 ints, one 256-byte region)
    assert L.gdr2_train_context_bytes_varlen(2, 65, 1, 128, 128) == 4 * (74240 + 49152 + 65536) + 256
    assert L.gdr2_train_context_bytes_varlen(0, 65, 1, 128, 128) == 0
    assert L.gdr2_train_context_bytes_varlen(-1, 65, 1, 128, 128) == ARG
    names = ["q", "k", "v", "b", "w", "g", "S0", "o", "ST", "cu", "ctx"]
    p = {n: ctypes.c_void_p(BASE + i * GAP) for i, n in enumerate(names)}

    def fwd(**over):
        q = dict(p)
        q.update(over)
        return L.gdr2_forward_train_varlen(*[q[n] for n in names], 1 << 30, 2, 100, 2, 128, 128, 1, 0, None)

    assert fwd(cu=None) == ARG
    assert fwd(ctx=None) == ARG
    assert fwd(cu=ctypes.c_void_p(BASE + 9 * GAP + 2)) == ALIGN
    assert fwd(ctx=ctypes.c_void_p(BASE + 9 * GAP)) == ALIAS      # context over cu_seqlens


def test_cached_rejects_bad_args():
    L = _lib.lib()

    def cached(n, S_cache=ctypes.c_void_p(BASE + 12 * GAP), **kw):   # T = 128: two cache points at n = 1
        a = fwd_args(T=128, **kw)
        return L.gdr2_forward_cached(*(a[:9] + [S_cache, n] + a[9:]))

    assert cached(0) == ARG
    assert cached(-2) == ARG
    assert cached(1, S_cache=None) == ARG                         # two states to keep, no buffer
    assert cached(1, S_cache=ctypes.c_void_p(BASE + 12 * GAP + 4)) == ALIGN
    assert cached(1, S_cache=ctypes.c_void_p(BASE + 7 * GAP)) == ALIAS   # over o
    assert cached(1, dk=48) == SHAPE
