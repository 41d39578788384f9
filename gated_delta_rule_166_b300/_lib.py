"""ctypes binding over libgdr2.so (the C ABI declared in include/gdr2.h).

Argument marshalling only: tensors are checked for device, dtype, shape and
contiguity, their device pointers and the current CUDA stream are passed to
the C entry points, and a non-zero status becomes an exception.  Every step of
the computation runs in the library's CUDA kernels; there is no CPU path.  If
the library is missing the call fails loudly (GDR2LibraryError).
"""
from __future__ import annotations

import ctypes
import os

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libgdr2.so")

GDR2_F32, GDR2_BF16 = 0, 1
_DTYPES = {torch.float32: GDR2_F32, torch.bfloat16: GDR2_BF16}
_lib = None


class GDR2LibraryError(RuntimeError):
    """libgdr2.so is missing or cannot be loaded."""


class GDR2Error(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {status_string(status)} ({status})")


def lib():
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise GDR2LibraryError(
                f"{LIB_PATH} not found: build it with `python -m gated_delta_rule_166_b300.build`")
        try:
            L = ctypes.CDLL(LIB_PATH)
        except OSError as e:  # pragma: no cover
            raise GDR2LibraryError(f"cannot load {LIB_PATH}: {e}") from e
        vp, i64, ci = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int
        L.gdr2_forward.argtypes = [vp] * 9 + [i64] * 5 + [ci, ci, vp]
        L.gdr2_forward.restype = ci
        L.gdr2_forward_noalloc.argtypes = [vp] * 9 + [i64] * 5 + [ci, ci, vp]
        L.gdr2_forward_noalloc.restype = ci
        L.gdr2_forward_segmented.argtypes = [vp] * 9 + [i64] * 5 + [ci, ci, i64, vp]
        L.gdr2_forward_segmented.restype = ci
        L.gdr2_forward_varlen.argtypes = [vp] * 10 + [i64] * 5 + [ci, ci, vp]
        L.gdr2_forward_varlen.restype = ci
        L.gdr2_forward_varlen_segmented.argtypes = [vp] * 10 + [i64] * 5 + [ci, ci, i64, vp]
        L.gdr2_forward_varlen_segmented.restype = ci
        L.gdr2_forward_cached.argtypes = [vp] * 10 + [i64] * 6 + [ci, ci, vp]
        L.gdr2_forward_cached.restype = ci
        L.gdr2_backward.argtypes = [vp] * 16 + [i64] * 5 + [ci, vp]
        L.gdr2_backward.restype = ci
        L.gdr2_backward_varlen.argtypes = [vp] * 17 + [i64] * 5 + [ci, vp]
        L.gdr2_backward_varlen.restype = ci
        L.gdr2_backward_chunked_varlen.argtypes = [vp] * 17 + [i64] * 5 + [ci, vp]
        L.gdr2_backward_chunked_varlen.restype = ci
        L.gdr2_train_context_bytes.argtypes = [i64] * 5
        L.gdr2_train_context_bytes.restype = i64
        L.gdr2_forward_train.argtypes = [vp] * 10 + [i64] * 6 + [ci, ci, vp]
        L.gdr2_forward_train.restype = ci
        L.gdr2_backward_from_context.argtypes = [vp] * 10 + [i64] + [vp] * 7 + [i64] * 5 + [ci, vp]
        L.gdr2_backward_from_context.restype = ci
        L.gdr2_train_context_bytes_varlen.argtypes = [i64] * 5
        L.gdr2_train_context_bytes_varlen.restype = i64
        L.gdr2_forward_train_varlen.argtypes = [vp] * 11 + [i64] * 6 + [ci, ci, vp]
        L.gdr2_forward_train_varlen.restype = ci
        L.gdr2_backward_from_context_varlen.argtypes = [vp] * 11 + [i64] + [vp] * 7 + [i64] * 5 + [ci, vp]
        L.gdr2_backward_from_context_varlen.restype = ci
        L.gdr2_backward_chunked.argtypes = [vp] * 16 + [i64] * 5 + [ci, vp]
        L.gdr2_backward_chunked.restype = ci
        L.gdr2_decode_step.argtypes = [vp] * 8 + [i64] * 4 + [ci, ci, vp]
        L.gdr2_decode_step.restype = ci
        L.gdr2_device_status.argtypes = [vp]
        L.gdr2_device_status.restype = ci
        L.gdr2_status_string.argtypes = [ci]
        L.gdr2_status_string.restype = ctypes.c_char_p
        L.gdr2_version.argtypes = []
        L.gdr2_version.restype = ci
        L.gdr2_workspace_stats.argtypes = [ctypes.POINTER(i64), ctypes.POINTER(i64), ci]
        L.gdr2_workspace_stats.restype = ci
        L.gdr2_release_workspace.argtypes = []
        L.gdr2_release_workspace.restype = ci
        L.gdr2_sparse_write.argtypes = [vp] * 9 + [i64] * 6 + [ci, ci, vp]
        L.gdr2_sparse_write.restype = ci
        L.gdr2_set_wait_limit.argtypes = [i64]
        L.gdr2_set_wait_limit.restype = i64
        _lib = L
    return _lib


def status_string(status: int) -> str:
    return lib().gdr2_status_string(int(status)).decode()


def _stream_handle(stream) -> int:
    if stream is None:
        stream = torch.cuda.current_stream()
    return int(stream.cuda_stream)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _check_tokens(name, t, shape, dtype, device):
    if t.device != device:
        raise ValueError(f"{name} is on {t.device}, expected {device}")
    if t.dtype != dtype:
        raise ValueError(f"{name} has dtype {t.dtype}, expected {dtype}")
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {tuple(shape)}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def gdr2_forward(q, k, v, b, w, log_decay, S0=None, *, o=None, S_T=None,
                 out_dtype=torch.float32, return_state: bool = True, stream=None, segments=None):
    """Chunked prefill.  q, k, b, log_decay: [B, T, H, dk]; v, w: [B, T, H, dv]
    (all fp32 or all bf16, on one CUDA device); S0: [B, H, dk, dv] fp32 or None.
    Returns ``(o, S_T)`` with o in ``out_dtype`` (fp32 by default, or bf16);
    S_T is None when ``return_state`` is False.  ``o`` and ``S_T`` may be passed
    in to reuse buffers (``S_T is S0`` updates in place).  ``segments`` (an int)
    fixes the number of sequence segments of the chunk-parallel scan
    (gdr2_forward_segmented; 1 = the sequential state pass); None leaves the
    choice to the library."""
    if segments is not None:
        if int(segments) < 0:
            raise ValueError("segments must be >= 0")
        return _forward("gdr2_forward_segmented", q, k, v, b, w, log_decay, S0, o, S_T, out_dtype, return_state,
                        stream, extra=(int(segments),))
    return _forward("gdr2_forward", q, k, v, b, w, log_decay, S0, o, S_T, out_dtype, return_state, stream)


def gdr2_forward_noalloc(q, k, v, b, w, log_decay, S0=None, *, o=None, S_T=None,
                         out_dtype=torch.float32, return_state: bool = True, stream=None):
    """gdr2_forward through the entry point that allocates no device memory (its
    workspace is a fixed array inside the library; see include/gdr2.h), for
    callers that may not allocate at call time.  The outputs ``o`` (and ``S_T``
    when requested) are still allocated here unless passed in."""
    return _forward("gdr2_forward_noalloc", q, k, v, b, w, log_decay, S0, o, S_T, out_dtype, return_state,
                    stream)


def _forward(entry, q, k, v, b, w, log_decay, S0, o, S_T, out_dtype, return_state, stream, extra=(),
             cache=None):
    if q.dim() != 4 or v.dim() != 4:
        raise ValueError("q and v must be [B, T, H, d]")
    B, T, H, dk = q.shape
    dv = v.shape[-1]
    dtype, dev = q.dtype, q.device
    if dev.type != "cuda":
        raise ValueError(f"{entry} runs on CUDA tensors only")
    if dtype not in _DTYPES:
        raise ValueError(f"unsupported dtype {dtype}")
    for name, t, d in (("k", k, dk), ("b", b, dk), ("log_decay", log_decay, dk),
                       ("v", v, dv), ("w", w, dv)):
        _check_tokens(name, t, (B, T, H, d), dtype, dev)
    if S0 is not None:
        _check_tokens("S0", S0, (B, H, dk, dv), torch.float32, dev)
    if o is None:
        if out_dtype not in _DTYPES:
            raise ValueError(f"unsupported out_dtype {out_dtype}")
        o = torch.empty((B, T, H, dv), dtype=out_dtype, device=dev)
    else:
        if o.dtype not in _DTYPES:
            raise ValueError(f"unsupported o dtype {o.dtype}")
        _check_tokens("o", o, (B, T, H, dv), o.dtype, dev)
    if S_T is None and return_state:
        S_T = torch.empty((B, H, dk, dv), dtype=torch.float32, device=dev)
    elif S_T is not None:
        _check_tokens("S_T", S_T, (B, H, dk, dv), torch.float32, dev)
    with torch.cuda.device(dev):
        cache_args = () if cache is None else (_ptr(cache[0]) if cache[0].numel() else None, cache[1])
        st = getattr(lib(), entry)(_ptr(q), _ptr(k), _ptr(v), _ptr(b), _ptr(w), _ptr(log_decay),
                                   _ptr(S0), _ptr(o), _ptr(S_T), *cache_args, B, T, H, dk, dv,
                                   _DTYPES[dtype], _DTYPES[o.dtype], *extra,
                                   ctypes.c_void_p(_stream_handle(stream)))
    if st != 0:
        raise GDR2Error(st, entry)
    return o, S_T


def gdr2_forward_cached(q, k, v, b, w, log_decay, S0=None, *, cache_chunks: int, o=None, S_T=None,
                        out_dtype=torch.float32, return_state: bool = True, stream=None):
    """gdr2_forward that also returns the state at the end of every segment of
    ``cache_chunks`` 64-token chunks: ``(o, S_T, S_cache)`` with S_cache
    [B, H, T // (cache_chunks * 64), dk, dv] fp32 (the states after tokens
    cache_chunks * 64 - 1, 2 * cache_chunks * 64 - 1, ...)."""
    if int(cache_chunks) < 1:
        raise ValueError("cache_chunks must be >= 1")
    B, T, H, dk = q.shape
    dv = v.shape[-1]
    n_cache = T // (int(cache_chunks) * 64)
    S_cache = torch.empty((B, H, n_cache, dk, dv), dtype=torch.float32, device=q.device)
    o, S_T = _forward("gdr2_forward_cached", q, k, v, b, w, log_decay, S0, o, S_T, out_dtype, return_state,
                      stream, cache=(S_cache, int(cache_chunks)))
    return o, S_T, S_cache


def gdr2_forward_varlen(q, k, v, b, w, log_decay, cu_seqlens, S0=None, *, o=None, S_T=None,
                        out_dtype=torch.float32, return_state: bool = True, segments=None, stream=None):
    """Prefill over N packed sequences of different lengths.  q, k, b,
    log_decay: [total_T, H, dk]; v, w: [total_T, H, dv]; cu_seqlens: int32
    [N + 1] on the same device (sequence n owns rows cu_seqlens[n] ..
    cu_seqlens[n+1] - 1); S0: [N, H, dk, dv] fp32 or None.  ``segments`` (None:
    the library's choice) fixes the segments per sequence of the chunk-parallel
    scan (gdr2_forward_varlen_segmented).  Returns
    ``(o [total_T, H, dv], S_T [N, H, dk, dv])``.  Offsets from 0 to total_T
    cover every row; rows that other offsets leave to no sequence are not
    written in ``o`` (a new ``o`` holds whatever its memory held there)."""
    if q.dim() != 3 or v.dim() != 3:
        raise ValueError("q and v must be [total_T, H, d]")
    total, H, dk = q.shape
    dv = v.shape[-1]
    dtype, dev = q.dtype, q.device
    if dev.type != "cuda":
        raise ValueError("gdr2_forward_varlen runs on CUDA tensors only")
    if dtype not in _DTYPES:
        raise ValueError(f"unsupported dtype {dtype}")
    for name, t, d in (("k", k, dk), ("b", b, dk), ("log_decay", log_decay, dk),
                       ("v", v, dv), ("w", w, dv)):
        _check_tokens(name, t, (total, H, d), dtype, dev)
    if cu_seqlens.dim() != 1 or cu_seqlens.numel() < 1:
        raise ValueError("cu_seqlens must be a 1-D tensor of N + 1 offsets")
    _check_tokens("cu_seqlens", cu_seqlens, cu_seqlens.shape, torch.int32, dev)
    N = cu_seqlens.numel() - 1
    if S0 is not None:
        _check_tokens("S0", S0, (N, H, dk, dv), torch.float32, dev)
    if o is None:
        if out_dtype not in _DTYPES:
            raise ValueError(f"unsupported out_dtype {out_dtype}")
        o = torch.empty((total, H, dv), dtype=out_dtype, device=dev)
    else:
        if o.dtype not in _DTYPES:
            raise ValueError(f"unsupported o dtype {o.dtype}")
        _check_tokens("o", o, (total, H, dv), o.dtype, dev)
    if S_T is None and return_state:
        S_T = torch.empty((N, H, dk, dv), dtype=torch.float32, device=dev)
    elif S_T is not None:
        _check_tokens("S_T", S_T, (N, H, dk, dv), torch.float32, dev)
    entry = "gdr2_forward_varlen" if segments is None else "gdr2_forward_varlen_segmented"
    extra = () if segments is None else (int(segments),)
    with torch.cuda.device(dev):
        st = getattr(lib(), entry)(_ptr(q), _ptr(k), _ptr(v), _ptr(b), _ptr(w), _ptr(log_decay),
                                   _ptr(S0), _ptr(o), _ptr(S_T), _ptr(cu_seqlens), N, total, H,
                                   dk, dv, _DTYPES[dtype], _DTYPES[o.dtype], *extra,
                                   ctypes.c_void_p(_stream_handle(stream)))
    if st != 0:
        raise GDR2Error(st, entry)
    return o, S_T


def gdr2_backward(q, k, v, b, w, log_decay, S0, d_o, d_S_T=None, *, want_dS0: bool = True, stream=None):
    """Gradients of gdr2_forward.  Forward inputs as for gdr2_forward (q, k, b,
    log_decay: [B, T, H, dk]; v, w: [B, T, H, dv]; all fp32 or all bf16; S0 fp32
    [B, H, dk, dv] or None); d_o: [B, T, H, dv] gradient at o; d_S_T: [B, H, dk,
    dv] gradient at S_T or None.  Returns fp32 tensors (dq, dk, dv, db, dw,
    dlog_decay, dS0), dS0 None when ``want_dS0`` is False."""
    return _backward("gdr2_backward", q, k, v, b, w, log_decay, S0, d_o, d_S_T, want_dS0, stream)


def gdr2_backward_chunked(q, k, v, b, w, log_decay, S0, d_o, d_S_T=None, *, want_dS0: bool = True,
                          stream=None):
    """gdr2_backward through the chunkwise WY form on tensor cores: bf16 inputs
    (dk, dv in {32, 64, 128}), the same arguments and outputs."""
    return _backward("gdr2_backward_chunked", q, k, v, b, w, log_decay, S0, d_o, d_S_T, want_dS0, stream)


def gdr2_train_context_bytes(B: int, T: int, H: int, dk: int, dv: int) -> int:
    """Bytes of the context gdr2_forward_train keeps for these sizes."""
    n = lib().gdr2_train_context_bytes(B, T, H, dk, dv)
    if n < 0:
        raise GDR2Error(int(n), "gdr2_train_context_bytes")
    return int(n)


def gdr2_forward_train(q, k, v, b, w, log_decay, S0=None, *, o=None, S_T=None, out_dtype=torch.float32,
                       ctx=None, stream=None):
    """gdr2_forward that also keeps, in a device buffer, what the chunked backward
    would recompute: every chunk's maps, backward records and start state (bf16
    inputs).  Returns ``(o, S_T, ctx)``; ``ctx`` (uint8, or the given buffer) goes
    to gdr2_backward_from_context with the same, unchanged inputs."""
    if q.dim() != 4 or v.dim() != 4:
        raise ValueError("q and v must be [B, T, H, d]")
    B, T, H, dk = q.shape
    dv = v.shape[-1]
    dtype, dev = q.dtype, q.device
    if dev.type != "cuda":
        raise ValueError("gdr2_forward_train runs on CUDA tensors only")
    if dtype not in _DTYPES:
        raise ValueError(f"unsupported dtype {dtype}")
    for name, t, d in (("k", k, dk), ("b", b, dk), ("log_decay", log_decay, dk),
                       ("v", v, dv), ("w", w, dv)):
        _check_tokens(name, t, (B, T, H, d), dtype, dev)
    if S0 is not None:
        _check_tokens("S0", S0, (B, H, dk, dv), torch.float32, dev)
    if o is None:
        if out_dtype not in _DTYPES:
            raise ValueError(f"unsupported out_dtype {out_dtype}")
        o = torch.empty((B, T, H, dv), dtype=out_dtype, device=dev)
    else:
        _check_tokens("o", o, (B, T, H, dv), o.dtype, dev)
    if S_T is None:
        S_T = torch.empty((B, H, dk, dv), dtype=torch.float32, device=dev)
    else:
        _check_tokens("S_T", S_T, (B, H, dk, dv), torch.float32, dev)
    need = gdr2_train_context_bytes(B, T, H, dk, dv)
    if ctx is None:
        ctx = torch.empty(max(need, 1), dtype=torch.uint8, device=dev)
    elif ctx.device != dev or ctx.dtype != torch.uint8 or not ctx.is_contiguous() or ctx.numel() < need:
        raise ValueError(f"ctx must be a contiguous uint8 tensor of at least {need} bytes on {dev}")
    with torch.cuda.device(dev):
        st = lib().gdr2_forward_train(_ptr(q), _ptr(k), _ptr(v), _ptr(b), _ptr(w), _ptr(log_decay), _ptr(S0),
                                      _ptr(o), _ptr(S_T), _ptr(ctx), ctx.numel(), B, T, H, dk, dv,
                                      _DTYPES[dtype], _DTYPES[o.dtype], ctypes.c_void_p(_stream_handle(stream)))
    if st != 0:
        raise GDR2Error(st, "gdr2_forward_train")
    return o, S_T, ctx


def gdr2_backward_from_context(ctx, q, k, v, b, w, log_decay, S0, d_o, d_S_T=None, *, want_dS0: bool = True,
                               stream=None):
    """gdr2_backward_chunked from the context gdr2_forward_train kept for these
    inputs: the same arguments and fp32 outputs (dq, dk, dv, db, dw, dlog_decay,
    dS0), without recomputing the forward."""
    if ctx.dtype != torch.uint8 or not ctx.is_contiguous() or ctx.device != q.device:
        raise ValueError("ctx must be the contiguous uint8 context of gdr2_forward_train")
    return _backward("gdr2_backward_from_context", q, k, v, b, w, log_decay, S0, d_o, d_S_T, want_dS0, stream,
                     ctx=ctx)


def _backward(fn, q, k, v, b, w, log_decay, S0, d_o, d_S_T, want_dS0, stream, ctx=None):
    if q.dim() != 4 or v.dim() != 4:
        raise ValueError("q and v must be [B, T, H, d]")
    B, T, H, dk = q.shape
    dv = v.shape[-1]
    dtype, dev = q.dtype, q.device
    if dev.type != "cuda":
        raise ValueError(f"{fn} runs on CUDA tensors only")
    if dtype not in _DTYPES:
        raise ValueError(f"unsupported dtype {dtype}")
    for name, t, d in (("k", k, dk), ("b", b, dk), ("log_decay", log_decay, dk),
                       ("v", v, dv), ("w", w, dv)):
        _check_tokens(name, t, (B, T, H, d), dtype, dev)
    _check_tokens("d_o", d_o, (B, T, H, dv), torch.float32, dev)
    for name, t in (("S0", S0), ("d_S_T", d_S_T)):
        if t is not None:
            _check_tokens(name, t, (B, H, dk, dv), torch.float32, dev)
    f32 = dict(dtype=torch.float32, device=dev)
    gq, gk, gb, gg = (torch.empty((B, T, H, dk), **f32) for _ in range(4))
    gv, gw = (torch.empty((B, T, H, dv), **f32) for _ in range(2))
    gS0 = torch.empty((B, H, dk, dv), **f32) if want_dS0 else None
    ctx_args = () if ctx is None else (_ptr(ctx), ctx.numel())
    with torch.cuda.device(dev):
        st = getattr(lib(), fn)(_ptr(q), _ptr(k), _ptr(v), _ptr(b), _ptr(w), _ptr(log_decay), _ptr(S0),
                                _ptr(d_o), _ptr(d_S_T), *ctx_args, _ptr(gq), _ptr(gk), _ptr(gv), _ptr(gb),
                                _ptr(gw), _ptr(gg), _ptr(gS0), B, T, H, dk, dv, _DTYPES[dtype],
                                ctypes.c_void_p(_stream_handle(stream)))
    if st != 0:
        raise GDR2Error(st, fn)
    return gq, gk, gv, gb, gw, gg, gS0


def gdr2_backward_varlen(q, k, v, b, w, log_decay, cu_seqlens, S0, d_o, d_S_T=None, *, want_dS0: bool = True,
                         stream=None):
    """Gradients of gdr2_forward_varlen.  Forward inputs as for
    gdr2_forward_varlen (q, k, b, log_decay: [total_T, H, dk]; v, w: [total_T, H,
    dv]; cu_seqlens int32 [N + 1] on the device; S0 fp32 [N, H, dk, dv] or None);
    d_o: [total_T, H, dv] fp32; d_S_T: [N, H, dk, dv] fp32 or None.  Returns fp32
    (dq, dk, dv, db, dw, dlog_decay, dS0), dS0 None when ``want_dS0`` is False.
    Rows that belong to no sequence are returned as zeros."""
    return _backward_varlen("gdr2_backward_varlen", q, k, v, b, w, log_decay, cu_seqlens, S0, d_o, d_S_T,
                            want_dS0, stream)


def gdr2_backward_chunked_varlen(q, k, v, b, w, log_decay, cu_seqlens, S0, d_o, d_S_T=None, *,
                                 want_dS0: bool = True, stream=None):
    """gdr2_backward_varlen through the chunkwise WY form on tensor cores: bf16
    inputs (dk, dv in {32, 64, 128}), the same arguments and outputs."""
    return _backward_varlen("gdr2_backward_chunked_varlen", q, k, v, b, w, log_decay, cu_seqlens, S0, d_o,
                            d_S_T, want_dS0, stream)


def gdr2_forward_train_varlen(q, k, v, b, w, log_decay, cu_seqlens, S0=None, *, out_dtype=torch.float32,
                              ctx=None, stream=None):
    """gdr2_forward_varlen that keeps the per-chunk context for
    gdr2_backward_from_context_varlen (bf16 inputs; the packed form of
    gdr2_forward_train).  Returns ``(o, S_T, ctx)``."""
    if q.dim() != 3 or v.dim() != 3:
        raise ValueError("q and v must be [total_T, H, d]")
    total, H, dk = q.shape
    dv = v.shape[-1]
    dtype, dev = q.dtype, q.device
    if dev.type != "cuda":
        raise ValueError("gdr2_forward_train_varlen runs on CUDA tensors only")
    if dtype not in _DTYPES:
        raise ValueError(f"unsupported dtype {dtype}")
    for name, t, d in (("k", k, dk), ("b", b, dk), ("log_decay", log_decay, dk),
                       ("v", v, dv), ("w", w, dv)):
        _check_tokens(name, t, (total, H, d), dtype, dev)
    if cu_seqlens.dim() != 1 or cu_seqlens.numel() < 1:
        raise ValueError("cu_seqlens must be a 1-D tensor of N + 1 offsets")
    _check_tokens("cu_seqlens", cu_seqlens, cu_seqlens.shape, torch.int32, dev)
    N = cu_seqlens.numel() - 1
    if S0 is not None:
        _check_tokens("S0", S0, (N, H, dk, dv), torch.float32, dev)
    if out_dtype not in _DTYPES:
        raise ValueError(f"unsupported out_dtype {out_dtype}")
    o = torch.empty((total, H, dv), dtype=out_dtype, device=dev)
    S_T = torch.empty((N, H, dk, dv), dtype=torch.float32, device=dev)
    need = int(lib().gdr2_train_context_bytes_varlen(N, total, H, dk, dv))
    if need < 0:
        raise GDR2Error(need, "gdr2_train_context_bytes_varlen")
    if ctx is None:
        ctx = torch.empty(max(need, 1), dtype=torch.uint8, device=dev)
    elif ctx.device != dev or ctx.dtype != torch.uint8 or not ctx.is_contiguous() or ctx.numel() < need:
        raise ValueError(f"ctx must be a contiguous uint8 tensor of at least {need} bytes on {dev}")
    with torch.cuda.device(dev):
        st = lib().gdr2_forward_train_varlen(_ptr(q), _ptr(k), _ptr(v), _ptr(b), _ptr(w), _ptr(log_decay), _ptr(S0),
                                             _ptr(o), _ptr(S_T), _ptr(cu_seqlens), _ptr(ctx), ctx.numel(), N, total,
                                             H, dk, dv, _DTYPES[dtype], _DTYPES[out_dtype],
                                             ctypes.c_void_p(_stream_handle(stream)))
    if st != 0:
        raise GDR2Error(st, "gdr2_forward_train_varlen")
    return o, S_T, ctx


def gdr2_backward_from_context_varlen(ctx, q, k, v, b, w, log_decay, cu_seqlens, S0, d_o, d_S_T=None, *,
                                      want_dS0: bool = True, stream=None):
    """gdr2_backward_chunked_varlen from the context gdr2_forward_train_varlen kept."""
    if ctx.dtype != torch.uint8 or not ctx.is_contiguous() or ctx.device != q.device:
        raise ValueError("ctx must be the contiguous uint8 context of gdr2_forward_train_varlen")
    return _backward_varlen("gdr2_backward_from_context_varlen", q, k, v, b, w, log_decay, cu_seqlens, S0, d_o,
                            d_S_T, want_dS0, stream, ctx=ctx)


def _backward_varlen(fn, q, k, v, b, w, log_decay, cu_seqlens, S0, d_o, d_S_T, want_dS0, stream, ctx=None):
    if q.dim() != 3 or v.dim() != 3:
        raise ValueError("q and v must be [total_T, H, d]")
    total, H, dk = q.shape
    dv = v.shape[-1]
    dtype, dev = q.dtype, q.device
    if dev.type != "cuda":
        raise ValueError(f"{fn} runs on CUDA tensors only")
    if dtype not in _DTYPES:
        raise ValueError(f"unsupported dtype {dtype}")
    for name, t, d in (("k", k, dk), ("b", b, dk), ("log_decay", log_decay, dk),
                       ("v", v, dv), ("w", w, dv)):
        _check_tokens(name, t, (total, H, d), dtype, dev)
    if cu_seqlens.dim() != 1 or cu_seqlens.numel() < 1:
        raise ValueError("cu_seqlens must be a 1-D tensor of N + 1 offsets")
    _check_tokens("cu_seqlens", cu_seqlens, cu_seqlens.shape, torch.int32, dev)
    N = cu_seqlens.numel() - 1
    _check_tokens("d_o", d_o, (total, H, dv), torch.float32, dev)
    for name, t in (("S0", S0), ("d_S_T", d_S_T)):
        if t is not None:
            _check_tokens(name, t, (N, H, dk, dv), torch.float32, dev)
    f32 = dict(dtype=torch.float32, device=dev)
    # rows outside every sequence are left to the caller: zero, as their gradients
    # are.  One fill over one buffer of the six (disjoint, 16-byte-aligned views)
    # runs at full bandwidth; six small fills do not.
    nk, nv = total * H * dk, total * H * dv
    flat = torch.zeros(4 * nk + 2 * nv, **f32)
    gq, gk, gb, gg = (flat[i * nk:(i + 1) * nk].view(total, H, dk) for i in range(4))
    gv, gw = (flat[4 * nk + i * nv:4 * nk + (i + 1) * nv].view(total, H, dv) for i in range(2))
    gS0 = torch.empty((N, H, dk, dv), **f32) if want_dS0 else None
    if ctx is None:
        ptrs = (_ptr(gq), _ptr(gk), _ptr(gv), _ptr(gb), _ptr(gw), _ptr(gg), _ptr(gS0), _ptr(cu_seqlens))
    else:   # the context entry takes cu_seqlens and the context before the outputs
        ptrs = (_ptr(cu_seqlens), _ptr(ctx), ctx.numel(), _ptr(gq), _ptr(gk), _ptr(gv), _ptr(gb), _ptr(gw),
                _ptr(gg), _ptr(gS0))
    with torch.cuda.device(dev):
        st = getattr(lib(), fn)(_ptr(q), _ptr(k), _ptr(v), _ptr(b), _ptr(w), _ptr(log_decay), _ptr(S0),
                                _ptr(d_o), _ptr(d_S_T), *ptrs, N, total, H, dk, dv,
                                _DTYPES[dtype], ctypes.c_void_p(_stream_handle(stream)))
    if st != 0:
        raise GDR2Error(st, fn)
    return gq, gk, gv, gb, gw, gg, gS0


class GatedDeltaRule2(torch.autograd.Function):
    """(o, S_T) = gdr2_forward(q, k, v, b, w, log_decay, S0) as a differentiable
    operation: the forward pass is gdr2_forward (fp32 o), the backward pass
    gdr2_backward, or the chunked tensor-core backward when ``chunked`` is set and
    the inputs are bf16.  The chunked backward either recomputes the forward's
    per-chunk context (gdr2_backward_chunked) or, with ``keep_context``, the
    forward pass is gdr2_forward_train and keeps it for
    gdr2_backward_from_context (faster, 773 MB more memory per B4 H16 T4096 d128
    call).  Gradients are fp32 and cast to each input's dtype."""

    @staticmethod
    def forward(ctx, q, k, v, b, w, log_decay, S0=None, chunked=False, keep_context=True):
        ctx.has_s0 = S0 is not None
        ctx.chunked = bool(chunked) and q.dtype == torch.bfloat16
        kept = None
        if ctx.chunked and keep_context and q.shape[0] * q.shape[1] * q.shape[2] > 0:
            o, S_T, kept = gdr2_forward_train(q, k, v, b, w, log_decay, S0)
        else:
            o, S_T = gdr2_forward(q, k, v, b, w, log_decay, S0)
        ctx.save_for_backward(q, k, v, b, w, log_decay, S0, kept)
        return o, S_T

    @staticmethod
    def backward(ctx, d_o, d_S_T):
        q, k, v, b, w, log_decay, S0, kept = ctx.saved_tensors
        d_o = torch.zeros((*v.shape[:3], v.shape[-1]), dtype=torch.float32, device=q.device) if d_o is None \
            else d_o.float().contiguous()
        d_S_T = None if d_S_T is None else d_S_T.float().contiguous()
        if kept is not None:
            g = gdr2_backward_from_context(kept, q, k, v, b, w, log_decay, S0, d_o, d_S_T, want_dS0=ctx.has_s0)
        else:
            fn = gdr2_backward_chunked if ctx.chunked else gdr2_backward
            g = fn(q, k, v, b, w, log_decay, S0, d_o, d_S_T, want_dS0=ctx.has_s0)
        cast = [g[i].to(t.dtype) for i, t in enumerate((q, k, v, b, w, log_decay))]
        return (*cast, g[6] if ctx.has_s0 else None, None, None)


def gdr2_apply(q, k, v, b, w, log_decay, S0=None, *, chunked_backward: bool = False, keep_context: bool = True):
    """Differentiable prefill: ``(o, S_T)`` with gradients through gdr2_backward
    (exact fp32), or through the chunked tensor-core backward (bf16 inputs, else
    the exact path) when ``chunked_backward`` is set: from a context the forward
    keeps (gdr2_forward_train, the default) or, with ``keep_context=False``,
    recomputed by gdr2_backward_chunked."""
    return GatedDeltaRule2.apply(q, k, v, b, w, log_decay, S0, chunked_backward, keep_context)


class GatedDeltaRule2Varlen(torch.autograd.Function):
    """(o, S_T) = gdr2_forward_varlen(q, k, v, b, w, log_decay, cu_seqlens, S0) as
    a differentiable operation over packed sequences: the forward pass is
    gdr2_forward_varlen (fp32 o), the backward pass gdr2_backward_varlen, or the
    chunked tensor-core backward when ``chunked`` is set and the inputs are bf16
    (from the context gdr2_forward_train_varlen keeps with ``keep_context``, else
    recomputed by gdr2_backward_chunked_varlen).  Gradients are fp32 and cast to
    each input's dtype; cu_seqlens gets none."""

    @staticmethod
    def forward(ctx, q, k, v, b, w, log_decay, cu_seqlens, S0=None, chunked=False, keep_context=True):
        ctx.has_s0 = S0 is not None
        ctx.chunked = bool(chunked) and q.dtype == torch.bfloat16
        kept = None
        if ctx.chunked and keep_context and q.shape[0] * q.shape[1] > 0 and cu_seqlens.numel() > 1:
            o, S_T, kept = gdr2_forward_train_varlen(q, k, v, b, w, log_decay, cu_seqlens, S0)
        else:
            o, S_T = gdr2_forward_varlen(q, k, v, b, w, log_decay, cu_seqlens, S0)
        ctx.save_for_backward(q, k, v, b, w, log_decay, cu_seqlens, S0, kept)
        return o, S_T

    @staticmethod
    def backward(ctx, d_o, d_S_T):
        q, k, v, b, w, log_decay, cu_seqlens, S0, kept = ctx.saved_tensors
        d_o = torch.zeros(v.shape, dtype=torch.float32, device=q.device) if d_o is None \
            else d_o.float().contiguous()
        d_S_T = None if d_S_T is None else d_S_T.float().contiguous()
        if kept is not None:
            g = gdr2_backward_from_context_varlen(kept, q, k, v, b, w, log_decay, cu_seqlens, S0, d_o, d_S_T,
                                                  want_dS0=ctx.has_s0)
        else:
            fn = gdr2_backward_chunked_varlen if ctx.chunked else gdr2_backward_varlen
            g = fn(q, k, v, b, w, log_decay, cu_seqlens, S0, d_o, d_S_T, want_dS0=ctx.has_s0)
        cast = [g[i].to(t.dtype) for i, t in enumerate((q, k, v, b, w, log_decay))]
        return (*cast, None, g[6] if ctx.has_s0 else None, None, None)


def gdr2_apply_varlen(q, k, v, b, w, log_decay, cu_seqlens, S0=None, *, chunked_backward: bool = False,
                      keep_context: bool = True):
    """Differentiable prefill over packed sequences: ``(o, S_T)`` of
    gdr2_forward_varlen with gradients through gdr2_backward_varlen (exact fp32),
    or through the chunked tensor-core backward (bf16 inputs, else the exact path)
    when ``chunked_backward`` is set: from a context the forward keeps
    (gdr2_forward_train_varlen, the default) or recomputed
    (gdr2_backward_chunked_varlen, ``keep_context=False``)."""
    return GatedDeltaRule2Varlen.apply(q, k, v, b, w, log_decay, cu_seqlens, S0, chunked_backward, keep_context)


def gdr2_decode_step(q, k, v, b, w, log_decay, S, *, o=None, out_dtype=torch.float32,
                     stream=None):
    """One decode step, S updated in place.  q, k, b, log_decay: [B, H, dk];
    v, w: [B, H, dv]; S: [B, H, dk, dv] fp32.  Returns o [B, H, dv] in
    ``out_dtype`` (fp32 by default, or bf16)."""
    if q.dim() != 3 or v.dim() != 3:
        raise ValueError("q and v must be [B, H, d]")
    B, H, dk = q.shape
    dv = v.shape[-1]
    dtype, dev = q.dtype, q.device
    if dev.type != "cuda":
        raise ValueError("gdr2_decode_step runs on CUDA tensors only")
    if dtype not in _DTYPES:
        raise ValueError(f"unsupported dtype {dtype}")
    for name, t, d in (("k", k, dk), ("b", b, dk), ("log_decay", log_decay, dk),
                       ("v", v, dv), ("w", w, dv)):
        _check_tokens(name, t, (B, H, d), dtype, dev)
    _check_tokens("S", S, (B, H, dk, dv), torch.float32, dev)
    if o is None:
        if out_dtype not in _DTYPES:
            raise ValueError(f"unsupported out_dtype {out_dtype}")
        o = torch.empty((B, H, dv), dtype=out_dtype, device=dev)
    else:
        if o.dtype not in _DTYPES:
            raise ValueError(f"unsupported o dtype {o.dtype}")
        _check_tokens("o", o, (B, H, dv), o.dtype, dev)
    with torch.cuda.device(dev):
        st = lib().gdr2_decode_step(_ptr(q), _ptr(k), _ptr(v), _ptr(b), _ptr(w), _ptr(log_decay),
                                    _ptr(S), _ptr(o), B, H, dk, dv, _DTYPES[dtype],
                                    _DTYPES[o.dtype], ctypes.c_void_p(_stream_handle(stream)))
    if st != 0:
        raise GDR2Error(st, "gdr2_decode_step")
    return o


def gdr2_sparse_write(idx, q, k, v, b, w, log_decay, S, *, o=None, out_dtype=torch.float32,
                      stream=None):
    """Gated delta write on the selected slots of a slot memory, S updated in
    place.  idx: int32 [B, T, H, K] (distinct slots per token; outside [0, M):
    nothing); q, k, b, log_decay: [B, T, H, K]; v, w: [B, T, H, dv]; S: [B, H,
    M, dv] fp32.  Returns o [B, T, H, dv] in ``out_dtype`` (fp32 by default, or
    bf16)."""
    if idx.dim() != 4 or v.dim() != 4 or S.dim() != 4:
        raise ValueError("idx and v must be [B, T, H, *], S [B, H, M, dv]")
    B, T, H, K = idx.shape
    dv = v.shape[-1]
    M = S.shape[2]
    dtype, dev = q.dtype, q.device
    if dev.type != "cuda":
        raise ValueError("gdr2_sparse_write runs on CUDA tensors only")
    if dtype not in _DTYPES:
        raise ValueError(f"unsupported dtype {dtype}")
    _check_tokens("idx", idx, (B, T, H, K), torch.int32, dev)
    for name, t, d in (("q", q, K), ("k", k, K), ("b", b, K), ("log_decay", log_decay, K),
                       ("v", v, dv), ("w", w, dv)):
        _check_tokens(name, t, (B, T, H, d), dtype, dev)
    _check_tokens("S", S, (B, H, M, dv), torch.float32, dev)
    if o is None:
        if out_dtype not in _DTYPES:
            raise ValueError(f"unsupported out_dtype {out_dtype}")
        o = torch.empty((B, T, H, dv), dtype=out_dtype, device=dev)
    else:
        if o.dtype not in _DTYPES:
            raise ValueError(f"unsupported o dtype {o.dtype}")
        _check_tokens("o", o, (B, T, H, dv), o.dtype, dev)
    with torch.cuda.device(dev):
        st = lib().gdr2_sparse_write(_ptr(idx), _ptr(q), _ptr(k), _ptr(v), _ptr(b), _ptr(w), _ptr(log_decay),
                                     _ptr(S), _ptr(o), B, T, H, M, K, dv, _DTYPES[dtype], _DTYPES[o.dtype],
                                     ctypes.c_void_p(_stream_handle(stream)))
    if st != 0:
        raise GDR2Error(st, "gdr2_sparse_write")
    return o


def gdr2_device_status(stream=None) -> int:
    """Synchronise the stream and return (and clear) the device-side status."""
    return lib().gdr2_device_status(ctypes.c_void_p(_stream_handle(stream)))


def gdr2_version() -> int:
    return lib().gdr2_version()


def gdr2_workspace_stats(reset: bool = False):
    """(reserved, used_high) bytes of the library's workspace pool on the current
    device; ``reset`` sets the high-water mark back to zero after reading it."""
    r, u = ctypes.c_int64(0), ctypes.c_int64(0)
    st = lib().gdr2_workspace_stats(ctypes.byref(r), ctypes.byref(u), 1 if reset else 0)
    if st != 0:
        raise GDR2Error(st, "gdr2_workspace_stats")
    return r.value, u.value


def gdr2_release_workspace() -> None:
    """Return the workspace pool's unused memory on the current device to the system."""
    st = lib().gdr2_release_workspace()
    if st != 0:
        raise GDR2Error(st, "gdr2_release_workspace")


def gdr2_set_wait_limit(cycles: int) -> int:
    """Testing hook: the chain kernel's handshake waits give up after ``cycles`` SM
    cycles (<= 0: the default of about 2 s).  Returns the previous limit (0 = default)."""
    return lib().gdr2_set_wait_limit(int(cycles))
