/*
 * gdr2.h -- C ABI of the B300 (sm_103a) Gated Delta Rule-2 library (libgdr2.so).
 *
 * The operation ("Gated DeltaNet-2: Decoupling Erase and Write in Linear
 * Attention" page, section "Gated Delta Rule-2 update equation", and the
 * symbol table under it):
 *
 *     S_t = (I - k_t (b_t (.) k_t)^T) D_t S_{t-1} + k_t (w_t (.) v_t)^T
 *     o_t = S_t^T q_t                       (readout after the update)
 *
 *   S_t       per-head d_k x d_v fast-weight memory, fp32 in this library
 *   k_t, q_t  key / query, d_k channels (keys are expected L2-normalised by the
 *             caller, as the page's symbol table states; nothing is normalised
 *             or scaled inside)
 *   b_t       erase gate over the d_k key channels   (used as given: no
 *             sigmoid, no clamp -- the page's ablation widens it to [0, 2])
 *   w_t       write gate over the d_v value channels (used as given)
 *   D_t       diag(exp(log_decay_t)), log_decay_t over the d_k key channels
 *
 * Special cases named on the same page: b = w = one scalar gives KDA; a scalar
 * decay in addition gives Gated DeltaNet.  Both run through the same calls.
 *
 * Conventions shared by every call
 * --------------------------------
 * - All tensor pointers are DEVICE pointers on the current CUDA device,
 *   row-major and contiguous, 16-byte aligned.  The caller owns every buffer
 *   and the library keeps no pointer after return.  Workspaces come from a
 *   stream-ordered memory pool that the library creates on each device it is
 *   called on (allocated and released on `stream`); the pool keeps freed memory
 *   reserved for later calls until gdr2_release_workspace() is called, so a call
 *   after a synchronisation does not map its workspace again.  The chunked
 *   bf16 prefill in one pass takes 74,240 bytes per
 *   (64-token chunk, head) -- the maps of each chunk's state update that its
 *   two kernels exchange (plus 4 bytes per packed sequence) -- or, when it splits
 *   sequences into segments, the segment scratch described at
 *   gdr2_forward_segmented; gdr2_backward takes its checkpoints and partial
 *   sums.  gdr2_forward_noalloc and gdr2_decode_step allocate nothing.
 * - in_dtype selects the element type of the six token inputs and out_dtype
 *   that of o: GDR2_F32 (float) or GDR2_BF16 (__nv_bfloat16).  States are
 *   always fp32.  All arithmetic is fp32 (bf16 only as tensor-core operands
 *   on the chunked bf16 path).  out_dtype = GDR2_F32 keeps o at accumulation
 *   precision; GDR2_BF16 halves its bytes at the cost of one bf16 rounding
 *   (relative 2^-9) per element.
 * - Supported head dims: d_k, d_v in {32, 64, 128}.
 * - Calls are asynchronous on `stream` (0 = legacy default stream): they
 *   validate on the host, enqueue kernels and return.  Argument errors are
 *   reported before anything is enqueued and leave every buffer untouched.
 * - Device-side failures (a bounded wait that timed out) are recorded in a
 *   per-library device word and reported by gdr2_device_status().
 * - Nothing throws across the ABI; every call returns a gdr2_status.
 */
#ifndef GDR2_H_
#define GDR2_H_

#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    GDR2_F32 = 0,
    GDR2_BF16 = 1
} gdr2_dtype;

typedef enum {
    GDR2_OK = 0,
    GDR2_ERR_ARG = -1,          /* null pointer where one is required, negative size */
    GDR2_ERR_SHAPE = -2,        /* head dims outside {32, 64, 128}, size overflow     */
    GDR2_ERR_ALIGN = -3,        /* a pointer is not 16-byte aligned                   */
    GDR2_ERR_UNSUPPORTED = -4,  /* unknown in/out dtype; device is not sm_103         */
    GDR2_ERR_CUDA = -5,         /* a CUDA runtime call failed (launch, attribute)     */
    GDR2_ERR_TIMEOUT = -6,      /* a bounded device-side wait gave up                 */
    GDR2_ERR_ALIAS = -7,        /* o overlaps an input, or S_T overlaps a token input */
    GDR2_ERR_SCRATCH = -8       /* gdr2_forward_noalloc: B*H exceeds its fixed scratch */
} gdr2_status;

/*
 * gdr2_forward -- chunked prefill over a whole sequence.
 *
 * Applies the update above for t = 0 .. T-1 to every (batch, head) pair,
 * starting from S0, writes every o_t and (optionally) the final state.
 * The page's "efficient implementation" section (WY form with decay
 * absorption, chunkwise algorithm) describes the method used for bf16 inputs:
 * fixed 64-token chunks, a per-chunk UT/WY transform with the cumulative
 * channel decay folded into the rank-1 erase factors (computed for all chunks
 * in parallel), and an fp32 state carried across the chunks of a sequence on
 * chip.  Head sizes below 128 key channels or 64 value columns run the same
 * kernels on zero-padded channels.  fp32 inputs run a token-sequential fp32
 * kernel.
 *
 *   q, k, b, log_decay : [B, T, H, dk]  (in_dtype)
 *   v, w               : [B, T, H, dv]  (in_dtype)
 *   S0                 : [B, H, dk, dv] fp32, or NULL for a zero initial state
 *   o                  : [B, T, H, dv]  (out_dtype), written
 *   S_T                : [B, H, dk, dv] fp32, written, or NULL (not stored)
 *
 * T = 0 is allowed: S_T receives S0 (or zeros) and o is untouched.
 * S0 == S_T (in-place state update) is allowed; any other overlap between S_T
 * or o and another argument is rejected with GDR2_ERR_ALIAS.
 * Preconditions (not checked): log_decay <= 0 and finite.  The chunked bf16
 * path forms per-channel decay factors about the middle token of each
 * 16-token sub-chunk and takes log_decay values below -10 as -10 (a per-token
 * decay factor of 4.5e-5 instead of a smaller one, e.g. a hard reset at
 * -inf): the state carried across such a token then differs from the exact
 * one by at most 4.5e-5 of itself.  The fp32 path and the decode step use
 * log_decay as given.
 */
int gdr2_forward(const void* q, const void* k, const void* v,
                 const void* b, const void* w, const void* log_decay,
                 const float* S0, void* o, float* S_T,
                 int64_t B, int64_t T, int64_t H, int64_t dk, int64_t dv,
                 int in_dtype, int out_dtype, cudaStream_t stream);

/*
 * gdr2_forward_varlen -- gdr2_forward over N packed sequences of different
 * lengths (the serving layout): sequence n owns token rows
 * [cu_seqlens[n], cu_seqlens[n+1]) of the packed tensors and its own initial
 * and final state.  Each sequence is an independent recurrence, so the result
 * for sequence n equals gdr2_forward on that sequence alone.
 *
 *   q, k, b, log_decay : [total_T, H, dk]  (in_dtype)
 *   v, w               : [total_T, H, dv]  (in_dtype)
 *   cu_seqlens         : [N + 1] int32 DEVICE offsets, non-decreasing, with
 *                        cu_seqlens[0] = 0 and cu_seqlens[N] = total_T.  The
 *                        kernels clamp each offset to [0, total_T] and each end
 *                        to at least its start, so malformed offsets cannot
 *                        cause out-of-range accesses (they give empty or
 *                        truncated sequences instead).
 *   S0                 : [N, H, dk, dv] fp32, or NULL (zeros)
 *   o                  : [total_T, H, dv] (out_dtype), written for every row
 *                        that belongs to a sequence
 *   S_T                : [N, H, dk, dv] fp32, or NULL
 *
 * An empty sequence gives S_T = S0 (or zeros).  Errors and aliasing rules are
 * those of gdr2_forward; o and S_T must not overlap cu_seqlens, and a null
 * cu_seqlens with N > 0 is GDR2_ERR_ARG.
 */
int gdr2_forward_varlen(const void* q, const void* k, const void* v,
                        const void* b, const void* w, const void* log_decay,
                        const float* S0, void* o, float* S_T, const int32_t* cu_seqlens,
                        int64_t N, int64_t total_T, int64_t H, int64_t dk, int64_t dv,
                        int in_dtype, int out_dtype, cudaStream_t stream);

/*
 * gdr2_forward_noalloc -- gdr2_forward that allocates no device memory.
 *
 * The page has no counterpart to this call; it exists for callers that must
 * not allocate at call time: a serving runtime that reserves all device memory
 * when it starts and forbids allocations on its request path, or an embedding
 * host whose memory is managed by someone else and that may not draw from the
 * library's stream-ordered workspace pool (which gdr2_forward uses).
 *
 * Same arguments, layouts, results and error codes as gdr2_forward.  For bf16
 * inputs the two prefill kernels run over ranges of chunks whose per-chunk
 * maps fit a fixed 64 MiB device array inside the library (file-scope memory
 * that every GPU which loads the library holds until the process exits): a
 * range covers min(all, floor(scratch / (B*H*74,240 B))) chunks of every
 * sequence, and the state is carried between ranges in S_T (in the scratch
 * when S_T is NULL).  The results are bit for bit those of gdr2_forward_segmented
 * with one segment.  B*H above about 900 (fewer when S_T is NULL) returns
 * GDR2_ERR_SCRATCH before anything is enqueued.  fp32 inputs run the
 * token-sequential kernel, which needs no scratch.
 *
 * Every call shares the one array per device: two calls that overlap on the
 * GPU (on different streams, or from different host threads without ordering)
 * race on it and give wrong results; calls on one stream are ordered and safe.
 * Nothing in the array needs to start at zero: each call writes every byte it
 * reads.  The first call on a device looks up the array's device address (with
 * that device current); make that first call before any stream capture.
 */
int gdr2_forward_noalloc(const void* q, const void* k, const void* v,
                         const void* b, const void* w, const void* log_decay,
                         const float* S0, void* o, float* S_T,
                         int64_t B, int64_t T, int64_t H, int64_t dk, int64_t dv,
                         int in_dtype, int out_dtype, cudaStream_t stream);

/*
 * gdr2_forward_segmented -- gdr2_forward with an explicit number of sequence
 * segments for the chunk-parallel scan.
 *
 * The state update is affine in the state, so a run of chunks (a segment) maps
 * its start state S to M S + N and adds S^T r_t to each of its outputs o_t
 * (the page's "efficient implementation" section: chunkwise algorithm; the
 * segment form follows from the same recurrence).  With G segments per
 * sequence, the state pass runs every segment at once -- segment 0 from S0, the
 * others from a zero state and, for M and r, from the identity -- then chains
 * the segments' maps (G - 1 products of 128 x 128 by 128 x dv per head) and
 * adds each later segment's start-state term to its o rows.  It shortens the
 * chunk-to-chunk chain G-fold at the cost of (1 + 2/(dv/64)) times the state
 * work and an fp32 scratch of (T - L*64) x H x (dk + dv) x 4 bytes per sequence
 * (L = chunks per segment).  gdr2_forward chooses G itself: the most segments,
 * each of at least 16 chunks, whose work still fits one wave of the GPU's SMs
 * (with 148 SMs and dk = dv = 128: 2 for B*H = 16 heads at T = 65536, and 1
 * whenever B*H >= 25).
 *
 *   segments : 0 = the library's choice (as gdr2_forward); n >= 1 = n segments
 *              (capped at the number of 64-token chunks and rounded so that
 *              none is empty; 1 = the plain sequential pass).
 *
 * Arguments, layouts, results and error codes as gdr2_forward, plus
 * GDR2_ERR_ARG for segments < 0 and GDR2_ERR_UNSUPPORTED for segments > 1 on
 * inputs that the chunked path does not take (fp32 inputs, d_k != 128).
 */
int gdr2_forward_segmented(const void* q, const void* k, const void* v,
                           const void* b, const void* w, const void* log_decay,
                           const float* S0, void* o, float* S_T,
                           int64_t B, int64_t T, int64_t H, int64_t dk, int64_t dv,
                           int in_dtype, int out_dtype, int64_t segments, cudaStream_t stream);

/*
 * gdr2_forward_varlen_segmented -- gdr2_forward_varlen with an explicit number of
 * segments per sequence for the chunk-parallel scan (see gdr2_forward_segmented).
 * Sequence n's chunks are split into G runs of ceil(chunks_n / G) (runs past its
 * last chunk are empty), the plan made on the device from cu_seqlens; the state
 * pass runs every (sequence, segment) at once, then a scan over each sequence's
 * segments and a tensor-core correction of the later segments' rows.  The
 * results are those of the one-pass call within the bf16 bar.
 *   segments : 0 = the library's choice (as gdr2_forward_varlen, which takes
 *              segments only when few long sequences would leave SMs idle);
 *              n >= 1 = n segments per sequence (1 = the sequential state pass)
 * Workspace (the library's pool): the one-pass slots plus, per (sequence,
 * segment, head), a state and a map (fp32), and fp32 partial outputs and r rows
 * for every token row: total_T*H*(dk + dv)*4 bytes.  GDR2_ERR_ARG for segments
 * < 0; GDR2_ERR_UNSUPPORTED for segments > 1 with fp32 inputs or head sizes
 * other than dk = 128, dv in {64, 128}.
 */
int gdr2_forward_varlen_segmented(const void* q, const void* k, const void* v,
                                  const void* b, const void* w, const void* log_decay,
                                  const float* S0, void* o, float* S_T, const int32_t* cu_seqlens,
                                  int64_t N, int64_t total_T, int64_t H, int64_t dk, int64_t dv,
                                  int in_dtype, int out_dtype, int64_t segments, cudaStream_t stream);

/*
 * gdr2_forward_cached -- gdr2_forward that also keeps the state at segment ends.
 *
 * The "Memory Caching (MC)" page ("caching the memory" section) splits a
 * sequence into segments and keeps each segment's final memory state as a
 * cached memory, so that later tokens can read the past through the cached
 * states as well as the online one.  This call provides those states for this
 * recurrence: S_cache[b][h][m] = the state after token (m + 1) * cache_chunks * 64
 * - 1 of sequence b, for m = 0 .. n_cache - 1 with n_cache = floor(T /
 * (cache_chunks * 64)) (segments of cache_chunks 64-token chunks; a final
 * partial segment is not cached -- its end state is S_T).  How the cached
 * states are combined with the readout is the caller's; the library computes o
 * and S_T as gdr2_forward_segmented with one segment does, bit for bit (the
 * chain kernel writes the cached states as it passes them).
 *
 *   S_cache      : [B, H, n_cache, dk, dv] fp32, written (may be NULL when n_cache = 0)
 *   cache_chunks : >= 1, segment length in 64-token chunks
 *
 * Other arguments, layouts and errors as gdr2_forward (fixed-length sequences;
 * the state pass is the sequential one, without sequence segments).
 * GDR2_ERR_ARG for cache_chunks < 1 or a NULL S_cache with n_cache > 0;
 * S_cache may overlap no other argument (GDR2_ERR_ALIAS).
 */
int gdr2_forward_cached(const void* q, const void* k, const void* v,
                        const void* b, const void* w, const void* log_decay,
                        const float* S0, void* o, float* S_T, float* S_cache, int64_t cache_chunks,
                        int64_t B, int64_t T, int64_t H, int64_t dk, int64_t dv,
                        int in_dtype, int out_dtype, cudaStream_t stream);

/*
 * gdr2_backward -- gradients of gdr2_forward (the training half).
 *
 * Differentiates L = sum_t <o_t, d_o_t> + <S_T, d_S_T> with respect to every
 * input of the update equation above (the page's "Gated Delta Rule-2 update
 * equation" section): q, k, v, b, w, log_decay and S0.  With X_t = D_t S_{t-1},
 * c_t = b_t (.) k_t, delta_t = w_t (.) v_t - X_t^T c_t and G the gradient at S_t
 * (later tokens, d_S_T, and q_t d_o_t^T from the readout):
 *     dq_t = S_t d_o_t,  ddelta = G^T k_t,  dv_t = ddelta (.) w_t,  dw_t = ddelta (.) v_t,
 *     dc = -X_t ddelta,  db_t = dc (.) k_t,  dk_t = G delta_t + dc (.) b_t,
 *     dX = G - c_t ddelta^T,  dlog_decay_t = rowsum(dX (.) X_t),  dS_{t-1} = D_t dX.
 * The kernels run the recurrence token by token in fp32: a forward sweep keeps
 * the state every 4 tokens, the backward sweep recomputes each 4-token block
 * from its checkpoint and walks it in reverse.
 *
 *   q, k, b, log_decay : [B, T, H, dk]  (in_dtype), the forward's inputs
 *   v, w               : [B, T, H, dv]  (in_dtype)
 *   S0                 : [B, H, dk, dv] fp32, or NULL (zero initial state)
 *   d_o                : [B, T, H, dv] fp32, gradient arriving at o
 *   d_S_T              : [B, H, dk, dv] fp32, gradient arriving at S_T, or NULL (zero)
 *   d_q, d_k, d_b, d_log_decay : [B, T, H, dk] fp32, written
 *   d_v, d_w           : [B, T, H, dv] fp32, written
 *   d_S0               : [B, H, dk, dv] fp32, written, or NULL (not stored)
 *
 * dk, dv in {32, 64, 128}.  Workspace (the library's pool, released on the
 * stream): B*H*ceil(T/4)*dk*dv*4 bytes of checkpoints plus
 * B*T*H*(dv/32)*4*dk*4 bytes of per-tile partial sums.  Outputs may overlap
 * no input and no other output (GDR2_ERR_ALIAS).  T = 0 gives d_S0 = d_S_T (or
 * zeros).  The page has no equations for the backward pass; these follow from
 * the update equation by the chain rule.
 */
int gdr2_backward(const void* q, const void* k, const void* v,
                  const void* b, const void* w, const void* log_decay,
                  const float* S0, const float* d_o, const float* d_S_T,
                  float* d_q, float* d_k, float* d_v, float* d_b, float* d_w,
                  float* d_log_decay, float* d_S0,
                  int64_t B, int64_t T, int64_t H, int64_t dk, int64_t dv,
                  int in_dtype, cudaStream_t stream);

/*
 * gdr2_backward_varlen -- gdr2_backward over N packed sequences of different
 * lengths: the gradients of gdr2_forward_varlen.  Sequence n owns token rows
 * [cu_seqlens[n], cu_seqlens[n+1]) and its own S0[n], d_S_T[n] and d_S0[n];
 * each sequence is an independent recurrence, so its gradients are those of
 * gdr2_backward on that sequence alone, with the same fp32 arithmetic.
 *
 *   q, k, b, log_decay : [total_T, H, dk]  (in_dtype), the forward's inputs
 *   v, w               : [total_T, H, dv]  (in_dtype)
 *   S0                 : [N, H, dk, dv] fp32, or NULL (zero initial states)
 *   d_o                : [total_T, H, dv] fp32, gradient arriving at o
 *   d_S_T              : [N, H, dk, dv] fp32, or NULL (zero)
 *   d_q, d_k, d_b, d_log_decay : [total_T, H, dk] fp32, written for every row
 *                        that belongs to a sequence (other rows are left as they are)
 *   d_v, d_w           : [total_T, H, dv] fp32, likewise
 *   d_S0               : [N, H, dk, dv] fp32, written, or NULL (not stored)
 *   cu_seqlens         : [N + 1] int32 DEVICE offsets, as for gdr2_forward_varlen
 *                        (non-decreasing, from 0 to total_T; clamped on the device,
 *                        so malformed offsets give empty, truncated or unspecified
 *                        sequences, never out-of-range accesses)
 *
 * dk, dv in {32, 64, 128}.  Workspace (the library's pool, released on the
 * stream): H*(dv/32)*(total_T/4 + N + 2)*dk*32*4 bytes of checkpoints plus
 * total_T*H*(dv/32)*4*dk*4 bytes of per-tile partial sums.  An empty sequence
 * gives d_S0[n] = d_S_T[n] (or zeros).  Errors and aliasing rules are those of
 * gdr2_backward; no output may overlap cu_seqlens, and a null cu_seqlens with
 * N > 0 is GDR2_ERR_ARG.
 */
int gdr2_backward_varlen(const void* q, const void* k, const void* v,
                         const void* b, const void* w, const void* log_decay,
                         const float* S0, const float* d_o, const float* d_S_T,
                         float* d_q, float* d_k, float* d_v, float* d_b, float* d_w,
                         float* d_log_decay, float* d_S0, const int32_t* cu_seqlens,
                         int64_t N, int64_t total_T, int64_t H, int64_t dk, int64_t dv,
                         int in_dtype, cudaStream_t stream);

/*
 * gdr2_backward_chunked -- the gradients of gdr2_backward (same arguments, same
 * outputs) through the chunkwise WY form on tensor cores, for bf16 inputs
 * (GDR2_ERR_UNSUPPORTED for fp32); dk, dv in {32, 64, 128}, head sizes below 128
 * computed on channels zero-padded to 128 as in the forward.  Per 64-token chunk, with
 * start state S, the gradient dS' at its end state and dO at its outputs
 * (Cb = c e^G, Qb = q e^G, Kb = k e^{G_C - G}, Kh = k e^{-G}, u = w (.) v,
 * A_kk = strict_tril(Cb Kh^T), A_qk = tril(Qb Kh^T), T = (I + A_kk)^-1,
 * W = T Cb, E = T u - W S):
 *     dE = A_qk^T dO + Kb dS',   dA_qk = tril(dO E^T),   dKb = E dS'^T,
 *     dW = -dE S^T,   du = T^T dE,   dT = dE u^T + dW Cb^T,
 *     dA_kk = strict_tril(-T^T dT T^T),   dCb = T^T dW + dA_kk Kh,
 *     dQb = dO S^T + dA_qk Kh,   dKh = dA_kk^T Cb + dA_qk^T Qb,
 * then through the exponential factors and the prefix sums of log_decay; dS'
 * runs from chunk to chunk as dS = diag(e^{G_C}) dS' + Qb^T dO - W^T dE.  The
 * products take fp16 operands (tf32 for the decay-weighted ones) with fp32
 * accumulation, like the chunked forward, where gdr2_backward keeps fp32
 * throughout (max|err| / RMS within 1e-4).  Against exact gradients the chunked
 * ones stay within 2e-2 (max|err| / RMS) except db and dlog_decay under fast
 * decays (about e^-2 per token in every channel): there both are heavy-tailed
 * (max / RMS of 40-55) and formed from chunk terms several times their size, so
 * an element accuracy near 1e-3 relative reaches 2-5e-2 of RMS (measured at
 * B4 H16 T4096).  Per-token log decays below -10 count as -10, as in the chunked
 * forward.  Workspace (the library's pool, released on the stream): per
 * (chunk, head) 123,392 bytes (the forward's maps and backward record) plus
 * 128 KB of start state and end-state gradient, plus B*T*H*dv*2 bytes of o
 * that the recomputed forward writes.  The page gives no backward equations;
 * these follow from its chunkwise form by the chain rule.
 */
int gdr2_backward_chunked(const void* q, const void* k, const void* v,
                          const void* b, const void* w, const void* log_decay,
                          const float* S0, const float* d_o, const float* d_S_T,
                          float* d_q, float* d_k, float* d_v, float* d_b, float* d_w,
                          float* d_log_decay, float* d_S0,
                          int64_t B, int64_t T, int64_t H, int64_t dk, int64_t dv,
                          int in_dtype, cudaStream_t stream);

/*
 * Training with a kept context.  gdr2_backward_chunked recomputes the forward's
 * per-chunk maps and states before its backward products.  A training step that
 * runs the forward anyway can keep them instead: gdr2_forward_train is
 * gdr2_forward that also writes, into a caller-owned device buffer `ctx`, every
 * chunk's maps and backward record and its start state, and
 * gdr2_backward_from_context takes the gradients from that context (the same
 * kernels on the same values as gdr2_backward_chunked, so the same results bit
 * for bit).  The trade is memory for time: the context holds, per (64-token
 * chunk, head), 123,392 bytes of maps and records and a 64 KB fp32 state, 773 MB
 * at B4 H16 T4096 d128.
 *
 * gdr2_train_context_bytes -- the bytes `ctx` must hold for a fixed-length call
 * of these sizes (0 without tokens), or a negative status (GDR2_ERR_ARG,
 * GDR2_ERR_SHAPE).
 *
 * gdr2_forward_train -- gdr2_forward's arguments and results (o in out_dtype,
 * S_T or NULL) plus ctx (device, 16-byte aligned, ctx_bytes >= the size above,
 * overlapping no input or output).  bf16 inputs, dk, dv in {32, 64, 128}
 * (GDR2_ERR_UNSUPPORTED for fp32).  It always runs the one-pass chunked kernels
 * (no sequence segments).  The context stays valid while the caller keeps the
 * inputs unchanged.
 *
 * gdr2_backward_from_context -- gdr2_backward_chunked's arguments and results,
 * plus the ctx (and its size) that gdr2_forward_train wrote for the same inputs
 * and sizes.  Outputs may not overlap the context (GDR2_ERR_ALIAS); a NULL ctx
 * with tokens is GDR2_ERR_ARG.  Workspace (the library's pool): the end-state
 * gradients, 64 KB per (chunk, head).  What they compute is what
 * gdr2_forward and gdr2_backward_chunked compute (the page's update equation,
 * its chunkwise WY form and the chain rule through it); the two calls only split
 * gdr2_backward_chunked where its forward recomputation ends.
 */
int64_t gdr2_train_context_bytes(int64_t B, int64_t T, int64_t H, int64_t dk, int64_t dv);
int gdr2_forward_train(const void* q, const void* k, const void* v,
                       const void* b, const void* w, const void* log_decay,
                       const float* S0, void* o, float* S_T, void* ctx, int64_t ctx_bytes,
                       int64_t B, int64_t T, int64_t H, int64_t dk, int64_t dv,
                       int in_dtype, int out_dtype, cudaStream_t stream);
int gdr2_backward_from_context(const void* q, const void* k, const void* v,
                               const void* b, const void* w, const void* log_decay,
                               const float* S0, const float* d_o, const float* d_S_T,
                               const void* ctx, int64_t ctx_bytes,
                               float* d_q, float* d_k, float* d_v, float* d_b, float* d_w,
                               float* d_log_decay, float* d_S0,
                               int64_t B, int64_t T, int64_t H, int64_t dk, int64_t dv,
                               int in_dtype, cudaStream_t stream);

/*
 * The same over N packed sequences (layouts, offsets and row ownership as in
 * gdr2_forward_varlen and gdr2_backward_varlen; the context also keeps each
 * sequence's first chunk).  The context holds ceil(total_T / 64) + N chunks (an
 * upper bound: each sequence adds at most one partial chunk), 0 bytes without
 * tokens or sequences.  The backward's gradients are gdr2_backward_chunked_varlen's
 * bit for bit.
 */
int64_t gdr2_train_context_bytes_varlen(int64_t N, int64_t total_T, int64_t H, int64_t dk, int64_t dv);
int gdr2_forward_train_varlen(const void* q, const void* k, const void* v,
                              const void* b, const void* w, const void* log_decay,
                              const float* S0, void* o, float* S_T, const int32_t* cu_seqlens,
                              void* ctx, int64_t ctx_bytes,
                              int64_t N, int64_t total_T, int64_t H, int64_t dk, int64_t dv,
                              int in_dtype, int out_dtype, cudaStream_t stream);
int gdr2_backward_from_context_varlen(const void* q, const void* k, const void* v,
                                      const void* b, const void* w, const void* log_decay,
                                      const float* S0, const float* d_o, const float* d_S_T,
                                      const int32_t* cu_seqlens, const void* ctx, int64_t ctx_bytes,
                                      float* d_q, float* d_k, float* d_v, float* d_b, float* d_w,
                                      float* d_log_decay, float* d_S0,
                                      int64_t N, int64_t total_T, int64_t H, int64_t dk, int64_t dv,
                                      int in_dtype, cudaStream_t stream);

/*
 * gdr2_backward_chunked_varlen -- gdr2_backward_chunked over N packed sequences:
 * the gradients of gdr2_forward_varlen through the chunkwise WY form on tensor
 * cores, for bf16 inputs (dk, dv in {32, 64, 128}; GDR2_ERR_UNSUPPORTED for fp32).
 * Arguments, layouts and row ownership are those of gdr2_backward_varlen; the
 * precision is that of gdr2_backward_chunked, sequence by sequence.  Workspace
 * (the library's pool, released on the stream): per (chunk, head) 123,392
 * bytes plus 128 KB of start state and end-state gradient, counting
 * ceil(total_T / 64) + N chunks (each sequence adds at most one partial chunk),
 * plus total_T*H*dv*2 bytes of o that the recomputed forward writes.
 */
int gdr2_backward_chunked_varlen(const void* q, const void* k, const void* v,
                                 const void* b, const void* w, const void* log_decay,
                                 const float* S0, const float* d_o, const float* d_S_T,
                                 float* d_q, float* d_k, float* d_v, float* d_b, float* d_w,
                                 float* d_log_decay, float* d_S0, const int32_t* cu_seqlens,
                                 int64_t N, int64_t total_T, int64_t H, int64_t dk, int64_t dv,
                                 int in_dtype, cudaStream_t stream);

/*
 * gdr2_sparse_write -- the gated delta write on selected slots of a slot
 * memory ("Sparse Delta Memory" review page, section "3. Method & Key
 * Results": the write is applied only to the slots a product-key memory
 * selects; routing-slot recurrence of the Raven summary page, section "2.1
 * RSM framework": unselected slots keep their contents).  Per (sequence, head)
 * the memory S is M x dv; token t has selected the K slots R = idx[t] and
 *
 *     Sd = diag(exp log_decay_t) S[R],   x = (b_t (.) k_t)^T Sd,
 *     S[R] <- Sd + k_t (w_t (.) v_t - x)^T,   o_t = S[R]^T q_t,
 *
 * the dense update with k, b, q scattered to the selected slots and the decay
 * applied to those slots only.  Tokens run in order; the state is updated in
 * place.
 *
 *   idx                : [B, T, H, K] int32 slot indices; the K slots of one
 *                        token must be distinct (otherwise the result is
 *                        unspecified, accesses stay in bounds); an index outside
 *                        [0, M) selects nothing
 *   q, k, b, log_decay : [B, T, H, K]  (in_dtype), values at the selected slots
 *   v, w               : [B, T, H, dv] (in_dtype)
 *   S                  : [B, H, M, dv] fp32, read (S0) and overwritten (S_T)
 *   o                  : [B, T, H, dv] (out_dtype), written
 *
 * dv in {32, 64, 128}; 0 <= K <= min(M, 64) (GDR2_ERR_SHAPE otherwise).  o
 * and S may overlap no input and not each other (GDR2_ERR_ALIAS).  K = 0 writes
 * o = 0 and leaves S as it is; T = 0 does nothing.  Allocates nothing.
 * Asynchronous on `stream`.
 */
int gdr2_sparse_write(const int32_t* idx, const void* q, const void* k, const void* v,
                      const void* b, const void* w, const void* log_decay, float* S, void* o,
                      int64_t B, int64_t T, int64_t H, int64_t M, int64_t K, int64_t dv,
                      int in_dtype, int out_dtype, cudaStream_t stream);

/*
 * gdr2_decode_step -- one autoregressive step for every (batch, head), the
 * state updated in place (same equation, one token):
 *
 *     S' = D S,  r = S'^T (b (.) k),  p = S'^T q,  delta = w (.) v - r,
 *     S  <- S' + k delta^T,           o = p + (k . q) delta  ( = S^T q )
 *
 *   q, k, b, log_decay : [B, H, dk]  (in_dtype)
 *   v, w               : [B, H, dv]  (in_dtype)
 *   S                  : [B, H, dk, dv] fp32, read and overwritten
 *   o                  : [B, H, dv]  (out_dtype), written
 *
 * The fp32 state is streamed once from HBM and written once (128-bit
 * accesses); o must not overlap any other argument.
 */
int gdr2_decode_step(const void* q, const void* k, const void* v,
                     const void* b, const void* w, const void* log_decay,
                     float* S, void* o,
                     int64_t B, int64_t H, int64_t dk, int64_t dv,
                     int in_dtype, int out_dtype, cudaStream_t stream);

/*
 * gdr2_device_status -- synchronises `stream`, then returns GDR2_OK, the
 * recorded device-side failure (GDR2_ERR_TIMEOUT) or GDR2_ERR_CUDA if the
 * stream reports a CUDA error.  Reading clears the recorded failure.
 */
int gdr2_device_status(cudaStream_t stream);

/*
 * gdr2_workspace_stats -- the library's workspace pool on the current device:
 * *reserved = device memory it holds now, *used_high = the most of it in use at
 * once since the pool was created or last reset (bytes).  reset != 0 sets the
 * high-water mark back to zero after reading it.  GDR2_ERR_ARG for a NULL output.
 */
int gdr2_workspace_stats(int64_t* reserved, int64_t* used_high, int reset);

/*
 * gdr2_release_workspace -- synchronises the current device and returns the
 * memory that the library's workspace pool holds but does not use to the system.
 */
int gdr2_release_workspace(void);

/*
 * gdr2_set_wait_limit -- testing hook.  Every handshake wait inside the prefill's
 * chain kernel (between its elementwise warps and its copy / tensor-core
 * thread) gives up after `cycles` SM clock cycles instead of about 4e9
 * (about 2 s); cycles <= 0 restores that default.  A wait that gives up makes
 * the kernel stop: it lets its own copies in flight land and its products
 * complete (with the default limit), frees its tensor memory, records
 * GDR2_ERR_TIMEOUT for gdr2_device_status and returns; o and S_T of that call
 * are then incomplete.  Process-wide, read at each launch; not for concurrent
 * use with other calls.  Returns the previous limit (0 = the default).
 */
int64_t gdr2_set_wait_limit(int64_t cycles);

/* Human-readable name of a gdr2_status value (static storage). */
const char* gdr2_status_string(int status);

/* Library ABI version: major * 10000 + minor * 100 + patch.  0.2.0 added the
 * backward over packed sequences (both paths), segments for packed sequences,
 * the training forward and backward around a kept context, and the chunked
 * backward for head sizes below 128; every 0.1.0 entry point is unchanged. */
int gdr2_version(void);

#ifdef __cplusplus
}
#endif

#endif /* GDR2_H_ */
