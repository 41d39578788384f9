// Internal declarations shared by the libgdr2 translation units.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace gdr2 {

// Element conversions for the two supported token dtypes.
__device__ __forceinline__ float to_f32(float x) { return x; }
__device__ __forceinline__ float to_f32(__nv_bfloat16 x) { return __bfloat162float(x); }
template <typename T> __device__ __forceinline__ T from_f32(float x);
template <> __device__ __forceinline__ float from_f32<float>(float x) { return x; }
template <> __device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float x) {
    return __float2bfloat16_rn(x);
}

// Packed sequence `seq` of a call with token offsets cu and chunk offsets cb (the
// first global chunk of each sequence, capped at the workspace's chunk bound): its
// rows a .. a + Ts - 1 are the ones its `given` = cb[seq + 1] - cb[seq] chunks cover
// (offsets clamped into [0, total], the end to at least the start).  With G segments
// each holds Lc = ceil(given / G) chunks and segment g starts at chunk cs (segments
// past the last chunk are empty).
struct PackedSegment {
    int a, Ts, given, Lc, cs;
};
__device__ __forceinline__ PackedSegment packed_segment(const int* cu, const int* cb, int total, int seq, int G,
                                                        int g) {
    PackedSegment p;
    p.a = min(max(cu[seq], 0), total);
    const int e = min(max(cu[seq + 1], p.a), total);
    p.given = cb[seq + 1] - cb[seq];
    p.Ts = static_cast<int>(min(static_cast<long long>(e - p.a), static_cast<long long>(p.given) * 64));
    p.Lc = G > 1 ? (p.given + G - 1) / G : p.given;
    p.cs = G > 1 ? min(g * p.Lc, p.given) : 0;
    return p;
}

// Device-side failure codes written to the library's error word.
enum : int { kDevOk = 0, kDevTimeout = 1 };

struct ForwardArgs {
    const void *q, *k, *v, *b, *w, *g;
    const float* S0;
    void* o;
    float* ST;
    int64_t B, T, H, dk, dv;   // B sequences; T their common length when cu is null
    const int* cu;             // packed sequences: start offsets [B + 1] on the device, or null
    int64_t total;             // token rows of the packed tensors (cu != null)
    int in_dtype;        // GDR2_F32 / GDR2_BF16: q, k, v, b, w, log_decay
    int out_dtype;       // GDR2_F32 / GDR2_BF16: o
    // fixed-length calls only: the state after every cache_chunks 64-token chunks,
    // [B][H][n_cache][dk][dv] with n_cache = T / (cache_chunks * 64); null: none
    float* S_cache = nullptr;
    int64_t cache_chunks = 0;
};

struct BackwardArgs {
    const void *q, *k, *v, *b, *w, *g;   // forward inputs (in_dtype)
    const float* S0;                     // [B, H, dk, dv] or null (zero)
    const float* dO;                     // [B, T, H, dv] gradient at o
    const float* dST;                    // [B, H, dk, dv] gradient at S_T, or null (zero)
    float *d_q, *d_k, *d_v, *d_b, *d_w, *d_g;   // fp32 gradients, layouts of the inputs
    float* d_S0;                         // [B, H, dk, dv] or null (not stored)
    int64_t B, T, H, dk, dv;   // B sequences; T their common length when cu is null
    int in_dtype;
    const int* cu = nullptr;   // packed sequences: start offsets [B + 1] on the device, or null
    int64_t total = 0;         // token rows of the packed tensors (cu != null)
};

struct DecodeArgs {
    const void *q, *k, *v, *b, *w, *g;
    float* S;
    void* o;
    int64_t B, H, dk, dv;
    int in_dtype;
    int out_dtype;
};

// Sparse gated delta write over a slot memory (gdr2_sparse.cu).
constexpr int64_t kSparseMaxK = 64;   // selected slots per token
struct SparseArgs {
    const int* idx;
    const void *q, *k, *v, *b, *w, *g;
    float* S;
    void* o;
    int64_t B, T, H, M, K, dv;
    int in_dtype;
    int out_dtype;
};
int launch_sparse(const SparseArgs& a, cudaStream_t stream);

// Launchers; each returns a gdr2_status value.  `err` is the device address
// of the library's error word (bounded waits record failures there).
int launch_recurrent(const ForwardArgs& a, cudaStream_t stream);
int launch_decode(const DecodeArgs& a, cudaStream_t stream);
// Gradients (token-sequential fp32 kernels); the workspace holds state
// checkpoints and the per-tile row-vector partials.
size_t backward_workspace_bytes(int64_t B, int64_t T, int64_t H, int64_t dk, int64_t dv, bool packed = false,
                                int64_t total = 0);
int launch_backward(const BackwardArgs& a, void* ws, cudaStream_t stream);
// Chunked gradients (bf16 inputs, d_k = d_v = 128, T > 0): the forward's prep2 (with
// backward records) and chain kernels keep every chunk's maps and start state, the
// reverse chain carries dS across the chunks, one CTA per (chunk, head) forms the
// token gradients (gdr2_bwd_chunk.cu).
size_t backward_chunked_workspace_bytes(int64_t B, int64_t T, int64_t H, bool packed = false, int64_t total = 0);
int launch_backward_chunked(const BackwardArgs& a, void* ws, cudaStream_t stream, int* err);
// The chunked backward in two halves around a context kept by the caller: the forward
// part (writing o and S_T as gdr2_forward does) and the backward part from it.
size_t chunked_context_bytes(int64_t B, int64_t T, int64_t H, bool packed = false, int64_t total = 0);
int launch_forward_train(const BackwardArgs& a, void* o, int out_dtype, float* S_T, void* ctx, cudaStream_t stream,
                         int* err);
size_t backward_from_context_workspace_bytes(int64_t B, int64_t T, int64_t H, bool packed = false, int64_t total = 0);
int launch_backward_from_context(const BackwardArgs& a, const void* ctx, void* ws, cudaStream_t stream, int* err);

// ---- chunked prefill in affine form (bf16 inputs) -----------------------------------
// prep2 writes, for every 64-token chunk of every (sequence, head), the maps of the
// chunk's state update
//     S' = diag(gamma) S + M' S + Y U,      O = P S + X U      (U = w * v)
// into one workspace slot, as fp16 images that the chain kernel copies to shared
// memory unchanged: K-major (rows = M index), 128-byte swizzle, 64-element K blocks.
// The chain kernel then carries the state across the chunks of each sequence.
// Slot index = (global chunk) * H + head, where a sequence's chunks are numbered
// consecutively from chunk_base[sequence] (packed sequences) or from sequence *
// chunks per sequence.
constexpr int kPrepC = 64;     // chunk length
constexpr int kPrepDK = 128;   // key channels (smaller d_k: zero-padded channels)
constexpr uint32_t kSlotM = 0;         // M' [d_k out (M)][d_k in (K)]: 2 K blocks x 128 rows x 128 B
constexpr uint32_t kSlotY = 32768;     // Y  [d_k (M)][token (K)]:       1 K block x 128 rows x 128 B
constexpr uint32_t kSlotP = 49152;     // P  [token (M)][d_k (K)]:       2 K blocks x 64 rows x 128 B
constexpr uint32_t kSlotX = 65536;     // X  [token (M)][token (K)]:     1 K block x 64 rows x 128 B
constexpr uint32_t kSlotGam = 73728;   // gamma = e^{G_C} [d_k] fp32
constexpr size_t kSlot2Bytes = 74240;
// Backward record of a (chunk, head) item, written by prep2 in its backward mode:
// the fp16 images of W^T [d_k (rows)][token], A_qk [token][token], T [token][token]
// (K-major, one 64-element K block) and Kb [token][d_k] (two K blocks), with
// Kb = k e^{G_C - G}, T = (I + A_kk)^-1 and W = T (b k) e^{G}.
constexpr uint32_t kWyWt = 0, kWyAq = 16384, kWyT = 24576, kWyKb = 32768;
constexpr uint32_t kWyBytes = 49152;
// Global chunks of a call: exact for fixed-length sequences, an upper bound
// (ceil(total / 64) + N) for packed ones.
int64_t prep_chunk_bound(const ForwardArgs& a);
// bf16 inputs, d_k = 128, d_v in {64, 128} (the unpadded shapes; others run padded)
bool two_kernel_supports(const ForwardArgs& a);
// Chunk-parallel scan over segments of the sequences (fixed-length calls): G
// segments of L chunks per sequence, L even (the last may be shorter, none is
// empty).  The chain kernel runs every segment at once: value tiles from S0
// (segment 0) or zero, transfer tiles from the identity with U = 0; launch_scan
// chains the segments' affine maps S -> M S + N and launch_correct adds each later
// segment's start-state term S_start^T r_t to its o rows.  G = 1: no segments.
struct SegArgs {
    int G = 1, L = 0;            // packed sequences: L unused (ceil(chunks / G) per sequence)
    int64_t Tr = 0;              // T - L * 64: rows per sequence of o32 and r (packed: o32 and r
                                 // hold every global row, Tr unused)
    const int* chunk_base = nullptr;   // packed: first global chunk of each sequence
    int* tile_base = nullptr;    // packed: [N (G - 1) + 1] first correction tile of each
                                 // (sequence, segment g >= 1), then the total
    float* seg_state = nullptr;  // [B][H][G][d_k][dv] value tiles' end states
    float* seg_m = nullptr;      // [B][H][G][d_k][d_k] transfer tiles' end states (g >= 1)
    float* o32 = nullptr;        // [B * Tr][H][dv] o of segments g >= 1 from a zero start
    float* r = nullptr;          // [B * Tr][H][d_k] r_t = M_t^T q_t of segments g >= 1
    float* sT = nullptr;         // [B][H][G][dv][d_k] S_start(g)^T (g >= 1)
};
// S_start of every segment and the final state (into a.ST when non-null); then o of
// segments g >= 1 = o32 + S_start^T r in the output dtype.
int launch_scan(const ForwardArgs& a, const SegArgs& seg, cudaStream_t stream);
int launch_correct(const ForwardArgs& a, const SegArgs& seg, cudaStream_t stream, int* err);
// packed sequences: the correction tiles of each (sequence, segment) into seg.tile_base
int launch_seg_plan(const ForwardArgs& a, const SegArgs& seg, cudaStream_t stream);
// Fixed-length calls may prepare chunks [c0, c0 + cpiece) of every sequence only
// (cpiece > 0; `chunks` = N * cpiece, slots numbered from 0 per sequence).
// wy (non-null): also the backward record of every item, [chunks * H][kWyBytes].
int launch_prep2(const ForwardArgs& a, uint8_t* slots, const int* chunk_base, int64_t chunks, cudaStream_t stream,
                 int* err, int c0 = 0, int cpiece = 0, uint8_t* wy = nullptr);
// One CTA per (sequence * head, 64-column d_v tile): the chunk-to-chunk chain over the
// slots of prep2, o and S_T.  Packed sequences pass the chunk_base that prep2 used.
// With seg.G > 1 (fixed-length, d_k = 128) the chain runs over segments as the
// segmented state pass does (value and transfer tiles, then launch_scan and
// launch_correct).
// Fixed-length calls may run chunks [c0, c0 + cpiece) of every sequence (cpiece > 0;
// the slots then hold only those chunks, numbered from 0 per sequence): S0 is the
// state before chunk c0, and S_T receives the state after the range.  a.S_cache
// (fixed-length, one pass) keeps the state after every a.cache_chunks chunks.
int launch_chain(const ForwardArgs& a, const uint8_t* slots, const int* chunk_base, cudaStream_t stream, int* err,
                 const SegArgs& seg = SegArgs{}, int c0 = 0, int cpiece = 0);
// Limit of the chain kernel's handshake waits for later launches (0: the default);
// returns the previous value.
int64_t set_chain_wait_limit(int64_t cycles);
// chunk_base[s] (s = 0 .. N) of packed sequences, offsets clamped to [0, total].
int launch_chunk_base(const int* cu, int64_t N, int64_t total, int* chunk_base, cudaStream_t stream);

}  // namespace gdr2
