"""B300-native (sm_103a) Gated Delta Rule-2: chunked prefill and decode.

    S_t = (I - k_t (b_t * k_t)^T) D_t S_{t-1} + k_t (w_t * v_t)^T,   o_t = S_t^T q_t

The computation lives in libgdr2.so (hand-written CUDA, C ABI in
include/gdr2.h); this package is its thin Python binding plus the seeded
synthetic input generators used by the tests and the bench.
"""
from ._lib import (  # noqa: F401
    GDR2Error,
    GDR2LibraryError,
    GatedDeltaRule2,
    GatedDeltaRule2Varlen,
    gdr2_apply,
    gdr2_apply_varlen,
    gdr2_backward,
    gdr2_backward_chunked,
    gdr2_backward_chunked_varlen,
    gdr2_backward_from_context,
    gdr2_backward_from_context_varlen,
    gdr2_backward_varlen,
    gdr2_decode_step,
    gdr2_device_status,
    gdr2_forward,
    gdr2_forward_cached,
    gdr2_forward_noalloc,
    gdr2_forward_train,
    gdr2_forward_train_varlen,
    gdr2_forward_varlen,
    gdr2_release_workspace,
    gdr2_set_wait_limit,
    gdr2_sparse_write,
    gdr2_train_context_bytes,
    gdr2_version,
    gdr2_workspace_stats,
)

forward = gdr2_forward
forward_varlen = gdr2_forward_varlen
forward_noalloc = gdr2_forward_noalloc
forward_cached = gdr2_forward_cached
decode_step = gdr2_decode_step
backward = gdr2_backward
backward_chunked = gdr2_backward_chunked
backward_varlen = gdr2_backward_varlen
backward_chunked_varlen = gdr2_backward_chunked_varlen
forward_train = gdr2_forward_train
backward_from_context = gdr2_backward_from_context
forward_train_varlen = gdr2_forward_train_varlen
backward_from_context_varlen = gdr2_backward_from_context_varlen
apply_varlen = gdr2_apply_varlen
sparse_write = gdr2_sparse_write
