// C ABI of libgdr2: host-side validation, dispatch, and the device error word.
#include <algorithm>
#include <mutex>

#include "gdr2.h"
#include "gdr2_internal.cuh"

namespace gdr2 {
namespace {

// Device word where bounded waits record a failure (kDevTimeout).  It lives in
// the module's static device memory: nothing is allocated for it.
__device__ int g_error_word;

constexpr int kMaxDevices = 64;
std::mutex g_mu;
int* g_err_addr[kMaxDevices] = {};
int g_cc_ok[kMaxDevices] = {};   // 0 unknown, 1 sm_103, -1 other

// Address of the error word on the current device (looked up once per device,
// with that device current) and a check that the device is an sm_103 part.
int device_setup(int** err_out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return GDR2_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_mu);
    if (g_cc_ok[dev] == 0) {
        int major = 0, minor = 0;
        if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
            return GDR2_ERR_CUDA;
        g_cc_ok[dev] = (major == 10 && minor == 3) ? 1 : -1;
    }
    if (g_cc_ok[dev] != 1) return GDR2_ERR_UNSUPPORTED;
    if (!g_err_addr[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_error_word) != cudaSuccess) return GDR2_ERR_CUDA;
        g_err_addr[dev] = static_cast<int*>(p);
    }
    if (err_out) *err_out = g_err_addr[dev];
    return GDR2_OK;
}

// Scratch of gdr2_forward_noalloc: file-scope device memory that every device
// loading the library holds until exit, shared by all calls of that entry point.
constexpr size_t kNoAllocScratchBytes = size_t(64) << 20;   // 64 MiB
static __device__ __align__(256) uint8_t g_noalloc_scratch[kNoAllocScratchBytes];
void* g_scratch_addr[kMaxDevices] = {};

// Device address of the scratch on the current device, looked up once per device
// with that device current (the host-side name of the array is not a device address).
int scratch_setup(void** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return GDR2_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_mu);
    if (!g_scratch_addr[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return GDR2_ERR_CUDA;
        g_scratch_addr[dev] = p;
    }
    *out = g_scratch_addr[dev];
    return GDR2_OK;
}

// Stream-ordered pool of the library's workspaces on each device.  Its release
// threshold is unlimited: memory freed at the end of a call stays mapped for the
// next one, so a call that follows a synchronisation does not pay to map its
// workspace again (a pool that trims at every synchronisation made the first
// call after one slower than the rest).  gdr2_release_workspace() trims it.
cudaMemPool_t g_pool[kMaxDevices] = {};

int workspace_pool(cudaMemPool_t* out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return GDR2_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_mu);
    if (!g_pool[dev]) {
        cudaMemPoolProps props = {};
        props.allocType = cudaMemAllocationTypePinned;
        props.handleTypes = cudaMemHandleTypeNone;
        props.location.type = cudaMemLocationTypeDevice;
        props.location.id = dev;
        cudaMemPool_t p = nullptr;
        if (cudaMemPoolCreate(&p, &props) != cudaSuccess) return GDR2_ERR_CUDA;
        uint64_t keep = UINT64_MAX;
        if (cudaMemPoolSetAttribute(p, cudaMemPoolAttrReleaseThreshold, &keep) != cudaSuccess) {
            cudaMemPoolDestroy(p);
            return GDR2_ERR_CUDA;
        }
        g_pool[dev] = p;
    }
    *out = g_pool[dev];
    return GDR2_OK;
}

// Workspace of `bytes` from the library's pool, stream-ordered on `stream`.
int ws_alloc(void** p, size_t bytes, cudaStream_t stream) {
    cudaMemPool_t pool = nullptr;
    const int st = workspace_pool(&pool);
    if (st != GDR2_OK) return st;
    return cudaMallocFromPoolAsync(p, bytes, pool, stream) == cudaSuccess ? GDR2_OK : GDR2_ERR_CUDA;
}

int g_sm_count[kMaxDevices] = {};

// Streaming multiprocessors of the current device (looked up once per device).
int sm_count() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return 0;
    std::lock_guard<std::mutex> lock(g_mu);
    if (!g_sm_count[dev] && cudaDeviceGetAttribute(&g_sm_count[dev], cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        g_sm_count[dev] = 0;
    return g_sm_count[dev];
}

// Segments per sequence for the chunk-parallel scan when the caller leaves the
// choice to the library: the most segments (each of at least kMinSegChunks chunks)
// whose value and transfer tiles still fit one CTA per SM in a single wave.  The
// state pass is a chain of dependent steps per chunk, so splitting the sequences
// pays only while the unsplit pass leaves SMs idle.
constexpr int64_t kMinSegChunks = 16;
int auto_segments(int64_t BH, int64_t dv, int64_t nch) {
    const int64_t sms = sm_count();
    const int64_t tv = dv / 64, tk = kPrepDK / 64;
    int G = 1;
    for (int64_t g = 2; g <= 64; ++g) {
        if (g * BH * tv + (g - 1) * BH * tk > sms || nch < g * kMinSegChunks) break;
        G = static_cast<int>(g);
    }
    return G;
}

size_t round256(size_t x) { return (x + 255) / 256 * 256; }

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool overlaps(const void* a, size_t na, const void* b, size_t nb) {
    if (!a || !b || na == 0 || nb == 0) return false;
    const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
    return x < y + nb && y < x + na;
}

bool head_dim_ok(int64_t d) { return d == 32 || d == 64 || d == 128; }
bool dtype_ok(int t) { return t == GDR2_F32 || t == GDR2_BF16; }

bool mul_ok(int64_t a, int64_t b, int64_t* out) {
    if (a < 0 || b < 0) return false;
    if (a != 0 && b > INT64_MAX / a) return false;
    *out = a * b;
    return true;
}

}  // namespace
}  // namespace gdr2

using namespace gdr2;

namespace {

// Shared by the fixed-length and the packed-sequence prefill: N sequences of
// `total` token rows in all; cu (device, N + 1 offsets) or null for N x T rows.
int forward_impl(const void* q, const void* k, const void* v, const void* b, const void* w,
                 const void* log_decay, const float* S0, void* o, float* S_T, const int32_t* cu,
                 int64_t N, int64_t T, int64_t total, int64_t H, int64_t dk, int64_t dv, int in_dtype,
                 int out_dtype, cudaStream_t stream, bool noalloc = false, int64_t segments = 0,
                 float* S_cache = nullptr, int64_t cache_chunks = 0) {
    if (N < 0 || T < 0 || total < 0 || H < 0 || segments < 0 || cache_chunks < 0) return GDR2_ERR_ARG;
    if (!dtype_ok(in_dtype) || !dtype_ok(out_dtype)) return GDR2_ERR_UNSUPPORTED;
    if (!head_dim_ok(dk) || !head_dim_ok(dv)) return GDR2_ERR_SHAPE;
    const size_t esz = in_dtype == GDR2_F32 ? 4 : 2;
    const size_t osz = out_dtype == GDR2_F32 ? 4 : 2;
    int64_t rows = 0, bh = 0, nk = 0, nv = 0, ns = 0;
    if (!mul_ok(total, H, &rows) || !mul_ok(N, H, &bh) || !mul_ok(rows, dk, &nk) || !mul_ok(rows, dv, &nv) ||
        !mul_ok(bh, dk * dv, &ns) || nk > INT64_MAX / 4 || ns > INT64_MAX / 4)
        return GDR2_ERR_SHAPE;
    const bool has_tokens = rows > 0;
    if (has_tokens && (!q || !k || !v || !b || !w || !log_decay || !o)) return GDR2_ERR_ARG;
    for (const void* p : {q, k, v, b, w, log_decay, (const void*)S0, (const void*)o, (const void*)S_T})
        if (p && !aligned16(p)) return GDR2_ERR_ALIGN;
    if (cu && (reinterpret_cast<uintptr_t>(cu) & 3u)) return GDR2_ERR_ALIGN;

    const size_t bk = (size_t)nk * esz, bv = (size_t)nv * esz, bs = (size_t)ns * 4;
    const size_t bo = (size_t)nv * osz, bc = cu ? (size_t)(N + 1) * 4 : 0;
    const void* tok_in[6] = {q, k, b, log_decay, v, w};
    const size_t tok_bytes[6] = {bk, bk, bk, bk, bv, bv};
    if (has_tokens) {
        for (int i = 0; i < 6; ++i)
            if (overlaps(o, bo, tok_in[i], tok_bytes[i])) return GDR2_ERR_ALIAS;
        if (overlaps(o, bo, S0, bs) || overlaps(o, bo, S_T, bs) || overlaps(o, bo, cu, bc)) return GDR2_ERR_ALIAS;
    }
    for (int i = 0; i < 6; ++i)
        if (has_tokens && overlaps(S_T, bs, tok_in[i], tok_bytes[i])) return GDR2_ERR_ALIAS;
    if (S_T && S0 && S_T != S0 && overlaps(S_T, bs, S0, bs)) return GDR2_ERR_ALIAS;
    if (overlaps(S_T, bs, cu, bc)) return GDR2_ERR_ALIAS;
    // cached states: [N][H][T / (cache_chunks * 64)][dk][dv], fixed-length calls only
    const int64_t n_cache = cache_chunks > 0 ? T / (cache_chunks * 64) : 0;
    size_t bcache = 0;
    if (cache_chunks > 0) {
        if (cu || noalloc) return GDR2_ERR_ARG;
        int64_t nc = 0;
        if (!mul_ok(ns, n_cache, &nc) || nc > INT64_MAX / 4) return GDR2_ERR_SHAPE;
        bcache = static_cast<size_t>(nc) * 4;
        if (bcache > 0 && !S_cache) return GDR2_ERR_ARG;
        if (S_cache && !aligned16(S_cache)) return GDR2_ERR_ALIGN;
        for (int i = 0; i < 6; ++i)
            if (overlaps(S_cache, bcache, tok_in[i], tok_bytes[i])) return GDR2_ERR_ALIAS;
        if (overlaps(S_cache, bcache, o, bo) || overlaps(S_cache, bcache, S0, bs) ||
            overlaps(S_cache, bcache, S_T, bs))
            return GDR2_ERR_ALIAS;
    }

    int* err = nullptr;
    int st = device_setup(&err);
    if (st != GDR2_OK) return st;
    if (bh == 0) return GDR2_OK;

    if (!has_tokens) {   // no tokens at all: S_T = S0 (or zeros)
        if (!S_T) return GDR2_OK;
        cudaError_t e = S0 ? (S0 == S_T ? cudaSuccess
                                        : cudaMemcpyAsync(S_T, S0, bs, cudaMemcpyDeviceToDevice, stream))
                           : cudaMemsetAsync(S_T, 0, bs, stream);
        return e == cudaSuccess ? GDR2_OK : GDR2_ERR_CUDA;
    }

    ForwardArgs a{q, k, v, b, w, log_decay, S0, o, S_T, N, T, H, dk, dv,
                  reinterpret_cast<const int*>(cu), total, in_dtype, out_dtype};
    if (bcache > 0) {
        a.S_cache = S_cache;
        a.cache_chunks = cache_chunks;
    }
    // bf16 inputs run the affine-form kernels.  Head sizes below d_k = 128 or d_v =
    // 64 run them with zero-padded channels: TMA fills key channels past d_k with
    // zeros (k = b = q = 0, log decay 0), so those state rows stay zero and add
    // nothing; value columns past d_v are computed and never stored.
    ForwardArgs full = a;
    full.dk = kPrepDK;
    full.dv = 128;
    const bool exact = two_kernel_supports(a);
    const bool padded = !exact && two_kernel_supports(full);
    if (exact || padded) {
        const int64_t nch = (T + 63) / 64;
        if (noalloc) {
            // chunk ranges whose slots fit the fixed scratch; the state between ranges is
            // carried in S_T (or, when the caller wants no S_T, in the scratch)
            void* scratch = nullptr;
            if ((st = scratch_setup(&scratch)) != GDR2_OK) return st;
            const size_t carry = S_T ? 0 : (static_cast<size_t>(ns) * 4 + 255) / 256 * 256;
            const size_t per_chunk = static_cast<size_t>(N) * static_cast<size_t>(H) * kSlot2Bytes;
            const int64_t cpiece = carry < kNoAllocScratchBytes
                                       ? std::min<int64_t>(nch, static_cast<int64_t>((kNoAllocScratchBytes - carry) / per_chunk))
                                       : 0;
            if (cpiece == 0) return GDR2_ERR_SCRATCH;
            float* state = S_T ? S_T : reinterpret_cast<float*>(scratch);
            uint8_t* slots = static_cast<uint8_t*>(scratch) + carry;
            for (int64_t c0 = 0; c0 < nch; c0 += cpiece) {
                const int64_t cp = nch - c0 < cpiece ? nch - c0 : cpiece;
                ForwardArgs ap = a;
                ap.S0 = c0 == 0 ? S0 : state;
                ap.ST = state;
                int rc = launch_prep2(ap, slots, nullptr, N * cp, stream, err, static_cast<int>(c0), static_cast<int>(cp));
                if (rc == GDR2_OK)
                    rc = launch_chain(ap, slots, nullptr, stream, err, SegArgs{}, static_cast<int>(c0), static_cast<int>(cp));
                if (rc != GDR2_OK) return rc;
            }
            return GDR2_OK;
        }
        if (segments > 1 && padded) return GDR2_ERR_UNSUPPORTED;
        if (exact && cu && bcache == 0 && segments != 1) {
            // Packed sequences, few and long: the same segments per sequence (each
            // sequence's chunks in G runs of ceil(chunks / G)), planned on the device.
            // The library's choice takes the mean sequence length.
            const int64_t nch_bound = (total + 63) / 64;
            int64_t G = segments > 0 ? segments : auto_segments(bh, dv, (nch_bound + N - 1) / std::max<int64_t>(N, 1));
            G = std::min<int64_t>(G, std::max<int64_t>(nch_bound, 1));
            if (G > 1) {
                SegArgs seg;
                seg.G = static_cast<int>(G);
                const int64_t chunks = prep_chunk_bound(a);
                const size_t slot_bytes = round256(static_cast<size_t>(chunks) * static_cast<size_t>(H) * kSlot2Bytes);
                const size_t nb_state = round256(static_cast<size_t>(N * G * H) * dk * dv * 4);   // also sT
                const size_t nb_m = round256(static_cast<size_t>(N * G * H) * dk * dk * 4);
                const size_t nb_o32 = round256(static_cast<size_t>(total * H) * dv * 4);
                const size_t nb_r = round256(static_cast<size_t>(total * H) * dk * 4);
                const size_t nb_cb = round256(static_cast<size_t>(N + 1) * 4);
                const size_t nb_tb = round256(static_cast<size_t>(N * (G - 1) + 1) * 4);
                void* ws = nullptr;
                if ((st = ws_alloc(&ws, slot_bytes + 2 * nb_state + nb_m + nb_o32 + nb_r + nb_cb + nb_tb, stream)) !=
                    GDR2_OK)
                    return st;
                uint8_t* p = static_cast<uint8_t*>(ws) + slot_bytes;
                seg.seg_state = reinterpret_cast<float*>(p);
                seg.sT = reinterpret_cast<float*>(p + nb_state);
                seg.seg_m = reinterpret_cast<float*>(p + 2 * nb_state);
                seg.o32 = reinterpret_cast<float*>(p + 2 * nb_state + nb_m);
                seg.r = reinterpret_cast<float*>(p + 2 * nb_state + nb_m + nb_o32);
                int* cbp = reinterpret_cast<int*>(p + 2 * nb_state + nb_m + nb_o32 + nb_r);
                seg.chunk_base = cbp;
                seg.tile_base = reinterpret_cast<int*>(p + 2 * nb_state + nb_m + nb_o32 + nb_r + nb_cb);
                int rc = launch_chunk_base(a.cu, N, total, cbp, stream);
                if (rc == GDR2_OK) rc = launch_prep2(a, static_cast<uint8_t*>(ws), cbp, chunks, stream, err);
                if (rc == GDR2_OK) rc = launch_chain(a, static_cast<const uint8_t*>(ws), cbp, stream, err, seg);
                if (rc == GDR2_OK) rc = launch_seg_plan(a, seg, stream);
                if (rc == GDR2_OK) rc = launch_scan(a, seg, stream);
                if (rc == GDR2_OK) rc = launch_correct(a, seg, stream, err);
                if (cudaFreeAsync(ws, stream) != cudaSuccess && rc == GDR2_OK) rc = GDR2_ERR_CUDA;
                return rc;
            }
        }
        if (exact && !cu && bcache == 0 && segments != 1) {
            // Few long fixed-length sequences: segments of the chunk-parallel scan (prep2
            // over every chunk, the chain kernel over segments with value and transfer
            // tiles, then the scan and the correction).
            int64_t G = segments > 0 ? (segments < nch ? segments : nch) : auto_segments(bh, dv, nch);
            int64_t L = (nch + G - 1) / G;
            L += L & 1;              // even: 128-row tiles of the correction stay in one segment
            G = (nch + L - 1) / L;   // no empty segment
            if (G > 1) {
                SegArgs seg;
                seg.G = static_cast<int>(G);
                seg.L = static_cast<int>(L);
                seg.Tr = T - L * 64;
                const int64_t chunks = N * nch;
                const size_t slot_bytes = round256(static_cast<size_t>(chunks) * static_cast<size_t>(H) * kSlot2Bytes);
                const size_t nb_state = round256(static_cast<size_t>(N * G * H) * dk * dv * 4);   // also sT
                const size_t nb_m = round256(static_cast<size_t>(N * G * H) * dk * dk * 4);
                const size_t nb_o32 = round256(static_cast<size_t>(N * seg.Tr * H) * dv * 4);
                const size_t nb_r = round256(static_cast<size_t>(N * seg.Tr * H) * dk * 4);
                void* ws = nullptr;
                if ((st = ws_alloc(&ws, slot_bytes + 2 * nb_state + nb_m + nb_o32 + nb_r, stream)) != GDR2_OK) return st;
                uint8_t* p = static_cast<uint8_t*>(ws) + slot_bytes;
                seg.seg_state = reinterpret_cast<float*>(p);
                seg.sT = reinterpret_cast<float*>(p + nb_state);
                seg.seg_m = reinterpret_cast<float*>(p + 2 * nb_state);
                seg.o32 = reinterpret_cast<float*>(p + 2 * nb_state + nb_m);
                seg.r = reinterpret_cast<float*>(p + 2 * nb_state + nb_m + nb_o32);
                int rc = launch_prep2(a, static_cast<uint8_t*>(ws), nullptr, chunks, stream, err);
                if (rc == GDR2_OK) rc = launch_chain(a, static_cast<const uint8_t*>(ws), nullptr, stream, err, seg);
                if (rc == GDR2_OK) rc = launch_scan(a, seg, stream);
                if (rc == GDR2_OK) rc = launch_correct(a, seg, stream, err);
                if (cudaFreeAsync(ws, stream) != cudaSuccess && rc == GDR2_OK) rc = GDR2_ERR_CUDA;
                return rc;
            }
        }
        // One pass over the chunks: prep2 writes each chunk's maps, the chain kernel
        // carries the state (and keeps the cached states); workspace (slots, then
        // chunk_base of packed sequences) from the library's pool.
        const int64_t chunks = prep_chunk_bound(a);
        const size_t slot_bytes = round256(static_cast<size_t>(chunks) * static_cast<size_t>(H) * kSlot2Bytes);
        void* ws = nullptr;
        if ((st = ws_alloc(&ws, slot_bytes + (cu ? static_cast<size_t>(N + 1) * 4 : 0), stream)) != GDR2_OK)
            return st;
        uint8_t* slots = static_cast<uint8_t*>(ws);
        int* cb = cu ? reinterpret_cast<int*>(slots + slot_bytes) : nullptr;
        int rc = cu ? launch_chunk_base(a.cu, N, total, cb, stream) : GDR2_OK;
        if (rc == GDR2_OK) rc = launch_prep2(a, slots, cb, chunks, stream, err);
        if (rc == GDR2_OK) rc = launch_chain(a, slots, cb, stream, err);
        if (cudaFreeAsync(ws, stream) != cudaSuccess && rc == GDR2_OK) rc = GDR2_ERR_CUDA;
        return rc;
    }
    if (segments > 1) return GDR2_ERR_UNSUPPORTED;
    return launch_recurrent(a, stream);
}

}  // namespace

extern "C" int gdr2_forward(const void* q, const void* k, const void* v,
                            const void* b, const void* w, const void* log_decay,
                            const float* S0, void* o, float* S_T,
                            int64_t B, int64_t T, int64_t H, int64_t dk, int64_t dv,
                            int in_dtype, int out_dtype, cudaStream_t stream) {
    int64_t total = 0;
    if (B >= 0 && T >= 0 && !mul_ok(B, T, &total)) return GDR2_ERR_SHAPE;
    return forward_impl(q, k, v, b, w, log_decay, S0, o, S_T, nullptr, B, T, total, H, dk, dv, in_dtype,
                        out_dtype, stream);
}

extern "C" int gdr2_forward_varlen(const void* q, const void* k, const void* v,
                                   const void* b, const void* w, const void* log_decay,
                                   const float* S0, void* o, float* S_T, const int32_t* cu_seqlens,
                                   int64_t N, int64_t total_T, int64_t H, int64_t dk, int64_t dv,
                                   int in_dtype, int out_dtype, cudaStream_t stream) {
    if (N > 0 && !cu_seqlens) return GDR2_ERR_ARG;
    if (N >= 0x7fffffffLL || total_T >= 0x7fffffffLL) return GDR2_ERR_SHAPE;
    return forward_impl(q, k, v, b, w, log_decay, S0, o, S_T, cu_seqlens, N, 0, total_T, H, dk, dv,
                        in_dtype, out_dtype, stream);
}

extern "C" int gdr2_forward_varlen_segmented(const void* q, const void* k, const void* v,
                                             const void* b, const void* w, const void* log_decay,
                                             const float* S0, void* o, float* S_T, const int32_t* cu_seqlens,
                                             int64_t N, int64_t total_T, int64_t H, int64_t dk, int64_t dv,
                                             int in_dtype, int out_dtype, int64_t segments, cudaStream_t stream) {
    if (N > 0 && !cu_seqlens) return GDR2_ERR_ARG;
    if (N >= 0x7fffffffLL || total_T >= 0x7fffffffLL) return GDR2_ERR_SHAPE;
    return forward_impl(q, k, v, b, w, log_decay, S0, o, S_T, cu_seqlens, N, 0, total_T, H, dk, dv,
                        in_dtype, out_dtype, stream, /*noalloc=*/false, segments);
}

extern "C" int gdr2_forward_noalloc(const void* q, const void* k, const void* v,
                                    const void* b, const void* w, const void* log_decay,
                                    const float* S0, void* o, float* S_T,
                                    int64_t B, int64_t T, int64_t H, int64_t dk, int64_t dv,
                                    int in_dtype, int out_dtype, cudaStream_t stream) {
    int64_t total = 0;
    if (B >= 0 && T >= 0 && !mul_ok(B, T, &total)) return GDR2_ERR_SHAPE;
    return forward_impl(q, k, v, b, w, log_decay, S0, o, S_T, nullptr, B, T, total, H, dk, dv, in_dtype,
                        out_dtype, stream, /*noalloc=*/true);
}

extern "C" int gdr2_forward_segmented(const void* q, const void* k, const void* v,
                                      const void* b, const void* w, const void* log_decay,
                                      const float* S0, void* o, float* S_T,
                                      int64_t B, int64_t T, int64_t H, int64_t dk, int64_t dv,
                                      int in_dtype, int out_dtype, int64_t segments, cudaStream_t stream) {
    int64_t total = 0;
    if (B >= 0 && T >= 0 && !mul_ok(B, T, &total)) return GDR2_ERR_SHAPE;
    if (segments < 0) return GDR2_ERR_ARG;
    return forward_impl(q, k, v, b, w, log_decay, S0, o, S_T, nullptr, B, T, total, H, dk, dv, in_dtype,
                        out_dtype, stream, /*noalloc=*/false, segments);
}

namespace {

// Shared by the token-sequential and the chunked backward, fixed-length or packed
// (cu: device offsets [B + 1] of B sequences over `total` token rows; T unused):
// the same arguments, checks and empty-sequence behaviour.
int backward_impl(const void* q, const void* k, const void* v, const void* b, const void* w,
                  const void* log_decay, const float* S0, const float* d_o, const float* d_S_T, float* d_q,
                  float* d_k, float* d_v, float* d_b, float* d_w, float* d_log_decay, float* d_S0, int64_t B,
                  int64_t T, int64_t H, int64_t dk, int64_t dv, int in_dtype, cudaStream_t stream, bool chunked,
                  const int32_t* cu = nullptr, int64_t total = 0, const void* ctx = nullptr,
                  int64_t ctx_bytes = 0) {
    if (B < 0 || T < 0 || H < 0 || total < 0) return GDR2_ERR_ARG;
    if (!dtype_ok(in_dtype)) return GDR2_ERR_UNSUPPORTED;
    if (!head_dim_ok(dk) || !head_dim_ok(dv)) return GDR2_ERR_SHAPE;
    const size_t esz = in_dtype == GDR2_F32 ? 4 : 2;
    int64_t rows = cu ? total : 0, bh = 0, nk = 0, nv = 0, ns = 0;
    if ((!cu && !mul_ok(B, T, &rows)) || !mul_ok(rows, H, &rows) || !mul_ok(B, H, &bh) || !mul_ok(rows, dk, &nk) ||
        !mul_ok(rows, dv, &nv) || !mul_ok(bh, dk * dv, &ns) || nk > INT64_MAX / 8 || ns > INT64_MAX / 8 ||
        bh >= 0x7fffffffLL)
        return GDR2_ERR_SHAPE;
    const bool has_tokens = rows > 0;
    if (has_tokens && (!q || !k || !v || !b || !w || !log_decay || !d_o || !d_q || !d_k || !d_v || !d_b ||
                       !d_w || !d_log_decay))
        return GDR2_ERR_ARG;
    const void* all[] = {q, k, v, b, w, log_decay, S0, d_o, d_S_T, d_q, d_k, d_v, d_b, d_w, d_log_decay, d_S0};
    for (const void* ptr : all)
        if (ptr && !aligned16(ptr)) return GDR2_ERR_ALIGN;
    if (cu && (reinterpret_cast<uintptr_t>(cu) & 3u)) return GDR2_ERR_ALIGN;
    // outputs must not overlap any input or each other
    const size_t bk = (size_t)nk * esz, bv = (size_t)nv * esz, bs = (size_t)ns * 4;
    const size_t fk = (size_t)nk * 4, fv = (size_t)nv * 4;
    const void* ins[] = {q, k, b, log_decay, v, w, S0, d_o, d_S_T};
    const size_t in_bytes[] = {bk, bk, bk, bk, bv, bv, bs, fv, bs};
    const void* outs[] = {d_q, d_k, d_b, d_log_decay, d_v, d_w, d_S0};
    const size_t out_bytes[] = {fk, fk, fk, fk, fv, fv, bs};
    const size_t bc = cu ? static_cast<size_t>(B + 1) * 4 : 0;
    for (int i = 0; i < 7; ++i) {
        for (int j = 0; j < 9; ++j)
            if (overlaps(outs[i], out_bytes[i], ins[j], in_bytes[j])) return GDR2_ERR_ALIAS;
        for (int j = i + 1; j < 7; ++j)
            if (overlaps(outs[i], out_bytes[i], outs[j], out_bytes[j])) return GDR2_ERR_ALIAS;
        if (overlaps(outs[i], out_bytes[i], cu, bc)) return GDR2_ERR_ALIAS;
    }
    if (chunked && in_dtype != GDR2_BF16) return GDR2_ERR_UNSUPPORTED;
    // from a training forward's context: big enough, and no output inside it
    size_t need_ctx = 0;
    if (ctx || ctx_bytes) {
        if (has_tokens && bh > 0) need_ctx = chunked_context_bytes(B, cu ? 0 : T, H, cu != nullptr, cu ? total : 0);
        if ((need_ctx > 0 && !ctx) || ctx_bytes < 0 || static_cast<uint64_t>(ctx_bytes) < need_ctx) return GDR2_ERR_ARG;
        if (ctx && !aligned16(ctx)) return GDR2_ERR_ALIGN;
        for (int i = 0; i < 7; ++i)
            if (overlaps(outs[i], out_bytes[i], ctx, need_ctx)) return GDR2_ERR_ALIAS;
    }
    int* err = nullptr;
    int st = device_setup(&err);
    if (st != GDR2_OK) return st;
    if (bh == 0) return GDR2_OK;
    if (!has_tokens) {   // no tokens: dS0 = dS_T (or zero)
        if (!d_S0) return GDR2_OK;
        const cudaError_t e = d_S_T ? cudaMemcpyAsync(d_S0, d_S_T, bs, cudaMemcpyDeviceToDevice, stream)
                                    : cudaMemsetAsync(d_S0, 0, bs, stream);
        return e == cudaSuccess ? GDR2_OK : GDR2_ERR_CUDA;
    }
    BackwardArgs a{q, k, v, b, w, log_decay, S0, d_o, d_S_T, d_q, d_k, d_v, d_b, d_w, d_log_decay, d_S0,
                   B, cu ? 0 : T, H, dk, dv, in_dtype, reinterpret_cast<const int*>(cu), cu ? total : 0};
    void* ws = nullptr;
    const size_t wsb = ctx ? backward_from_context_workspace_bytes(B, a.T, H, cu != nullptr, a.total)
                     : chunked ? backward_chunked_workspace_bytes(B, a.T, H, cu != nullptr, a.total)
                               : backward_workspace_bytes(B, a.T, H, dk, dv, cu != nullptr, a.total);
    if ((st = ws_alloc(&ws, wsb, stream)) != GDR2_OK) return st;
    int rc = ctx       ? launch_backward_from_context(a, ctx, ws, stream, err)
             : chunked ? launch_backward_chunked(a, ws, stream, err)
                       : launch_backward(a, ws, stream);
    if (cudaFreeAsync(ws, stream) != cudaSuccess && rc == GDR2_OK) rc = GDR2_ERR_CUDA;
    return rc;
}

}  // namespace

extern "C" int gdr2_backward(const void* q, const void* k, const void* v,
                             const void* b, const void* w, const void* log_decay,
                             const float* S0, const float* d_o, const float* d_S_T,
                             float* d_q, float* d_k, float* d_v, float* d_b, float* d_w,
                             float* d_log_decay, float* d_S0,
                             int64_t B, int64_t T, int64_t H, int64_t dk, int64_t dv,
                             int in_dtype, cudaStream_t stream) {
    return backward_impl(q, k, v, b, w, log_decay, S0, d_o, d_S_T, d_q, d_k, d_v, d_b, d_w, d_log_decay, d_S0,
                         B, T, H, dk, dv, in_dtype, stream, false);
}

extern "C" int gdr2_backward_varlen(const void* q, const void* k, const void* v,
                                    const void* b, const void* w, const void* log_decay,
                                    const float* S0, const float* d_o, const float* d_S_T,
                                    float* d_q, float* d_k, float* d_v, float* d_b, float* d_w,
                                    float* d_log_decay, float* d_S0, const int32_t* cu_seqlens,
                                    int64_t N, int64_t total_T, int64_t H, int64_t dk, int64_t dv,
                                    int in_dtype, cudaStream_t stream) {
    if (N > 0 && !cu_seqlens) return GDR2_ERR_ARG;
    if (N >= 0x7fffffffLL || total_T >= 0x7fffffffLL) return GDR2_ERR_SHAPE;
    if (N < 0 || total_T < 0) return GDR2_ERR_ARG;
    return backward_impl(q, k, v, b, w, log_decay, S0, d_o, d_S_T, d_q, d_k, d_v, d_b, d_w, d_log_decay, d_S0,
                         N, 0, H, dk, dv, in_dtype, stream, false, N > 0 ? cu_seqlens : nullptr, total_T);
}

extern "C" int gdr2_backward_chunked_varlen(const void* q, const void* k, const void* v,
                                            const void* b, const void* w, const void* log_decay,
                                            const float* S0, const float* d_o, const float* d_S_T,
                                            float* d_q, float* d_k, float* d_v, float* d_b, float* d_w,
                                            float* d_log_decay, float* d_S0, const int32_t* cu_seqlens,
                                            int64_t N, int64_t total_T, int64_t H, int64_t dk, int64_t dv,
                                            int in_dtype, cudaStream_t stream) {
    if (N > 0 && !cu_seqlens) return GDR2_ERR_ARG;
    if (N >= 0x7fffffffLL || total_T >= 0x7fffffffLL) return GDR2_ERR_SHAPE;
    if (N < 0 || total_T < 0) return GDR2_ERR_ARG;
    return backward_impl(q, k, v, b, w, log_decay, S0, d_o, d_S_T, d_q, d_k, d_v, d_b, d_w, d_log_decay, d_S0,
                         N, 0, H, dk, dv, in_dtype, stream, true, N > 0 ? cu_seqlens : nullptr, total_T);
}

extern "C" int64_t gdr2_train_context_bytes(int64_t B, int64_t T, int64_t H, int64_t dk, int64_t dv) {
    if (B < 0 || T < 0 || H < 0) return GDR2_ERR_ARG;
    if (!head_dim_ok(dk) || !head_dim_ok(dv)) return GDR2_ERR_SHAPE;
    int64_t rows = 0, bh = 0;
    if (!mul_ok(B, T, &rows) || !mul_ok(rows, H, &rows) || !mul_ok(B, H, &bh) || rows >= (1ll << 40))
        return GDR2_ERR_SHAPE;
    return rows == 0 ? 0 : static_cast<int64_t>(chunked_context_bytes(B, T, H));
}

extern "C" int64_t gdr2_train_context_bytes_varlen(int64_t N, int64_t total_T, int64_t H, int64_t dk, int64_t dv) {
    if (N < 0 || total_T < 0 || H < 0) return GDR2_ERR_ARG;
    if (!head_dim_ok(dk) || !head_dim_ok(dv)) return GDR2_ERR_SHAPE;
    int64_t rows = 0, bh = 0;
    if (N >= 0x7fffffffLL || total_T >= 0x7fffffffLL || !mul_ok(total_T, H, &rows) || !mul_ok(N, H, &bh))
        return GDR2_ERR_SHAPE;
    return rows == 0 || N == 0 ? 0 : static_cast<int64_t>(chunked_context_bytes(N, 0, H, true, total_T));
}

namespace {

// gdr2_forward_train and its packed form (cu: device offsets [N + 1] over `total` rows).
int forward_train_impl(const void* q, const void* k, const void* v, const void* b, const void* w,
                       const void* log_decay, const float* S0, void* o, float* S_T, void* ctx, int64_t ctx_bytes,
                       const int32_t* cu, int64_t N, int64_t T, int64_t total, int64_t H, int64_t dk, int64_t dv,
                       int in_dtype, int out_dtype, cudaStream_t stream) {
    if (N < 0 || T < 0 || total < 0 || H < 0 || ctx_bytes < 0) return GDR2_ERR_ARG;
    if (!dtype_ok(in_dtype) || !dtype_ok(out_dtype)) return GDR2_ERR_UNSUPPORTED;
    if (!head_dim_ok(dk) || !head_dim_ok(dv)) return GDR2_ERR_SHAPE;
    if (in_dtype != GDR2_BF16) return GDR2_ERR_UNSUPPORTED;
    int64_t rows = cu ? total : 0, bh = 0, nk = 0, nv = 0, ns = 0;
    if ((!cu && !mul_ok(N, T, &rows)) || !mul_ok(rows, H, &rows) || !mul_ok(N, H, &bh) || !mul_ok(rows, dk, &nk) ||
        !mul_ok(rows, dv, &nv) || !mul_ok(bh, dk * dv, &ns) || nk > INT64_MAX / 8 || ns > INT64_MAX / 8 ||
        bh >= 0x7fffffffLL)
        return GDR2_ERR_SHAPE;
    const bool has_tokens = rows > 0;
    if (has_tokens && (!q || !k || !v || !b || !w || !log_decay || !o)) return GDR2_ERR_ARG;
    for (const void* p : {q, k, v, b, w, log_decay, (const void*)S0, (const void*)o, (const void*)S_T,
                          (const void*)ctx})
        if (p && !aligned16(p)) return GDR2_ERR_ALIGN;
    if (cu && (reinterpret_cast<uintptr_t>(cu) & 3u)) return GDR2_ERR_ALIGN;
    const size_t need = has_tokens && bh > 0 ? chunked_context_bytes(N, cu ? 0 : T, H, cu != nullptr, total) : 0;
    if ((need > 0 && !ctx) || static_cast<uint64_t>(ctx_bytes) < need) return GDR2_ERR_ARG;
    const size_t bk = (size_t)nk * 2, bv = (size_t)nv * 2, bs = (size_t)ns * 4;
    const size_t bo = (size_t)nv * (out_dtype == GDR2_F32 ? 4 : 2), bc = cu ? static_cast<size_t>(N + 1) * 4 : 0;
    const void* ins[8] = {q, k, b, log_decay, v, w, S0, cu};
    const size_t in_bytes[8] = {bk, bk, bk, bk, bv, bv, bs, bc};
    for (int i = 0; i < 8; ++i) {
        if (has_tokens && overlaps(o, bo, ins[i], in_bytes[i])) return GDR2_ERR_ALIAS;
        if (i != 6 && overlaps(S_T, bs, ins[i], in_bytes[i])) return GDR2_ERR_ALIAS;
        if (overlaps(ctx, need, ins[i], in_bytes[i])) return GDR2_ERR_ALIAS;
    }
    if (S_T && S0 && S_T != S0 && overlaps(S_T, bs, S0, bs)) return GDR2_ERR_ALIAS;
    if ((has_tokens && overlaps(o, bo, S_T, bs)) || overlaps(ctx, need, o, has_tokens ? bo : 0) ||
        overlaps(ctx, need, S_T, bs))
        return GDR2_ERR_ALIAS;
    int* err = nullptr;
    int st = device_setup(&err);
    if (st != GDR2_OK) return st;
    if (bh == 0) return GDR2_OK;
    if (!has_tokens) {   // no tokens: S_T = S0 (or zeros), nothing to keep
        if (!S_T) return GDR2_OK;
        const cudaError_t e = S0 ? (S0 == S_T ? cudaSuccess
                                              : cudaMemcpyAsync(S_T, S0, bs, cudaMemcpyDeviceToDevice, stream))
                                 : cudaMemsetAsync(S_T, 0, bs, stream);
        return e == cudaSuccess ? GDR2_OK : GDR2_ERR_CUDA;
    }
    BackwardArgs a{q, k, v, b, w, log_decay, S0, nullptr, nullptr, nullptr, nullptr, nullptr, nullptr, nullptr,
                   nullptr, nullptr, N, cu ? 0 : T, H, dk, dv, in_dtype, reinterpret_cast<const int*>(cu),
                   cu ? total : 0};
    return launch_forward_train(a, o, out_dtype, S_T, ctx, stream, err);
}

}  // namespace

extern "C" int gdr2_forward_train(const void* q, const void* k, const void* v,
                                  const void* b, const void* w, const void* log_decay,
                                  const float* S0, void* o, float* S_T, void* ctx, int64_t ctx_bytes,
                                  int64_t B, int64_t T, int64_t H, int64_t dk, int64_t dv,
                                  int in_dtype, int out_dtype, cudaStream_t stream) {
    return forward_train_impl(q, k, v, b, w, log_decay, S0, o, S_T, ctx, ctx_bytes, nullptr, B, T, 0, H, dk, dv,
                              in_dtype, out_dtype, stream);
}

extern "C" int gdr2_forward_train_varlen(const void* q, const void* k, const void* v,
                                         const void* b, const void* w, const void* log_decay,
                                         const float* S0, void* o, float* S_T, const int32_t* cu_seqlens,
                                         void* ctx, int64_t ctx_bytes,
                                         int64_t N, int64_t total_T, int64_t H, int64_t dk, int64_t dv,
                                         int in_dtype, int out_dtype, cudaStream_t stream) {
    if (N > 0 && !cu_seqlens) return GDR2_ERR_ARG;
    if (N >= 0x7fffffffLL || total_T >= 0x7fffffffLL) return GDR2_ERR_SHAPE;
    return forward_train_impl(q, k, v, b, w, log_decay, S0, o, S_T, ctx, ctx_bytes, N > 0 ? cu_seqlens : nullptr, N,
                              0, total_T, H, dk, dv, in_dtype, out_dtype, stream);
}

extern "C" int gdr2_backward_from_context_varlen(const void* q, const void* k, const void* v,
                                                 const void* b, const void* w, const void* log_decay,
                                                 const float* S0, const float* d_o, const float* d_S_T,
                                                 const int32_t* cu_seqlens, const void* ctx, int64_t ctx_bytes,
                                                 float* d_q, float* d_k, float* d_v, float* d_b, float* d_w,
                                                 float* d_log_decay, float* d_S0,
                                                 int64_t N, int64_t total_T, int64_t H, int64_t dk, int64_t dv,
                                                 int in_dtype, cudaStream_t stream) {
    if (N > 0 && !cu_seqlens) return GDR2_ERR_ARG;
    if (N >= 0x7fffffffLL || total_T >= 0x7fffffffLL) return GDR2_ERR_SHAPE;
    if (N < 0 || total_T < 0) return GDR2_ERR_ARG;
    if (!ctx && ctx_bytes == 0 && N > 0 && total_T > 0 && H > 0) return GDR2_ERR_ARG;
    return backward_impl(q, k, v, b, w, log_decay, S0, d_o, d_S_T, d_q, d_k, d_v, d_b, d_w, d_log_decay, d_S0,
                         N, 0, H, dk, dv, in_dtype, stream, true, N > 0 ? cu_seqlens : nullptr, total_T, ctx,
                         ctx_bytes);
}

extern "C" int gdr2_backward_from_context(const void* q, const void* k, const void* v,
                                          const void* b, const void* w, const void* log_decay,
                                          const float* S0, const float* d_o, const float* d_S_T,
                                          const void* ctx, int64_t ctx_bytes,
                                          float* d_q, float* d_k, float* d_v, float* d_b, float* d_w,
                                          float* d_log_decay, float* d_S0,
                                          int64_t B, int64_t T, int64_t H, int64_t dk, int64_t dv,
                                          int in_dtype, cudaStream_t stream) {
    if (!ctx && ctx_bytes == 0 && B > 0 && T > 0 && H > 0) return GDR2_ERR_ARG;
    return backward_impl(q, k, v, b, w, log_decay, S0, d_o, d_S_T, d_q, d_k, d_v, d_b, d_w, d_log_decay, d_S0,
                         B, T, H, dk, dv, in_dtype, stream, true, nullptr, 0, ctx, ctx_bytes);
}

extern "C" int gdr2_backward_chunked(const void* q, const void* k, const void* v,
                                     const void* b, const void* w, const void* log_decay,
                                     const float* S0, const float* d_o, const float* d_S_T,
                                     float* d_q, float* d_k, float* d_v, float* d_b, float* d_w,
                                     float* d_log_decay, float* d_S0,
                                     int64_t B, int64_t T, int64_t H, int64_t dk, int64_t dv,
                                     int in_dtype, cudaStream_t stream) {
    return backward_impl(q, k, v, b, w, log_decay, S0, d_o, d_S_T, d_q, d_k, d_v, d_b, d_w, d_log_decay, d_S0,
                         B, T, H, dk, dv, in_dtype, stream, true);
}


extern "C" int gdr2_forward_cached(const void* q, const void* k, const void* v,
                                   const void* b, const void* w, const void* log_decay,
                                   const float* S0, void* o, float* S_T, float* S_cache, int64_t cache_chunks,
                                   int64_t B, int64_t T, int64_t H, int64_t dk, int64_t dv,
                                   int in_dtype, int out_dtype, cudaStream_t stream) {
    int64_t total = 0;
    if (B >= 0 && T >= 0 && !mul_ok(B, T, &total)) return GDR2_ERR_SHAPE;
    if (cache_chunks < 1) return GDR2_ERR_ARG;
    return forward_impl(q, k, v, b, w, log_decay, S0, o, S_T, nullptr, B, T, total, H, dk, dv, in_dtype,
                        out_dtype, stream, /*noalloc=*/false, /*segments=*/1, S_cache, cache_chunks);
}

extern "C" int gdr2_decode_step(const void* q, const void* k, const void* v,
                                const void* b, const void* w, const void* log_decay,
                                float* S, void* o,
                                int64_t B, int64_t H, int64_t dk, int64_t dv,
                                int in_dtype, int out_dtype, cudaStream_t stream) {
    if (B < 0 || H < 0) return GDR2_ERR_ARG;
    if (!dtype_ok(in_dtype) || !dtype_ok(out_dtype)) return GDR2_ERR_UNSUPPORTED;
    if (!head_dim_ok(dk) || !head_dim_ok(dv)) return GDR2_ERR_SHAPE;
    int64_t bh = 0, tmp = 0;
    if (!mul_ok(B, H, &bh) || !mul_ok(bh, dk * dv, &tmp) || tmp > INT64_MAX / 4 ||
        bh > 0x7fffffffLL)
        return GDR2_ERR_SHAPE;
    if (bh > 0 && (!q || !k || !v || !b || !w || !log_decay || !S || !o)) return GDR2_ERR_ARG;
    for (const void* p : {q, k, v, b, w, log_decay, (const void*)S, (const void*)o})
        if (p && !aligned16(p)) return GDR2_ERR_ALIGN;
    const size_t esz = in_dtype == GDR2_F32 ? 4 : 2;
    const size_t osz = out_dtype == GDR2_F32 ? 4 : 2;
    const size_t bk = (size_t)(bh * dk) * esz, bv = (size_t)(bh * dv) * esz, bs = (size_t)tmp * 4;
    const size_t bo = (size_t)(bh * dv) * osz;
    const void* ins[6] = {q, k, b, log_decay, v, w};
    const size_t nb[6] = {bk, bk, bk, bk, bv, bv};
    for (int i = 0; i < 6; ++i)
        if (overlaps(o, bo, ins[i], nb[i]) || overlaps(S, bs, ins[i], nb[i])) return GDR2_ERR_ALIAS;
    if (overlaps(o, bo, S, bs)) return GDR2_ERR_ALIAS;

    int st = device_setup(nullptr);
    if (st != GDR2_OK) return st;
    if (bh == 0) return GDR2_OK;
    DecodeArgs a{q, k, v, b, w, log_decay, S, o, B, H, dk, dv, in_dtype, out_dtype};
    return launch_decode(a, stream);
}

extern "C" int gdr2_sparse_write(const int32_t* idx, const void* q, const void* k, const void* v,
                                 const void* b, const void* w, const void* log_decay, float* S, void* o,
                                 int64_t B, int64_t T, int64_t H, int64_t M, int64_t K, int64_t dv,
                                 int in_dtype, int out_dtype, cudaStream_t stream) {
    if (B < 0 || T < 0 || H < 0 || M < 0 || K < 0) return GDR2_ERR_ARG;
    if (!dtype_ok(in_dtype) || !dtype_ok(out_dtype)) return GDR2_ERR_UNSUPPORTED;
    if (dv != 32 && dv != 64 && dv != 128) return GDR2_ERR_SHAPE;
    if (K > kSparseMaxK || K > M) return GDR2_ERR_SHAPE;
    int64_t bh = 0, rows = 0, nsel = 0, nval = 0, nmem = 0;
    if (!mul_ok(B, H, &bh) || !mul_ok(bh, T, &rows) || !mul_ok(rows, K, &nsel) || !mul_ok(rows, dv, &nval) ||
        !mul_ok(bh, M, &nmem) || !mul_ok(nmem, dv, &nmem) || nmem > INT64_MAX / 4 || nval > INT64_MAX / 4 ||
        nsel > INT64_MAX / 4 || bh > 0x7fffffffLL || T > 0x7fffffffLL || M > 0x7fffffffLL)
        return GDR2_ERR_SHAPE;
    const bool has_tokens = rows > 0;
    if (has_tokens && (!v || !w || !o || (nsel > 0 && (!idx || !q || !k || !b || !log_decay || !S))))
        return GDR2_ERR_ARG;
    for (const void* p : {(const void*)idx, q, k, v, b, w, log_decay, (const void*)S, (const void*)o})
        if (p && !aligned16(p)) return GDR2_ERR_ALIGN;
    const size_t esz = in_dtype == GDR2_F32 ? 4 : 2;
    const size_t osz = out_dtype == GDR2_F32 ? 4 : 2;
    const size_t bsel = (size_t)nsel * esz, bval = (size_t)nval * esz, bmem = (size_t)nmem * 4;
    const size_t bo = (size_t)nval * osz, bidx = (size_t)nsel * 4;
    if (has_tokens) {
        const void* ins[7] = {idx, q, k, b, log_decay, v, w};
        const size_t nb[7] = {bidx, bsel, bsel, bsel, bsel, bval, bval};
        for (int i = 0; i < 7; ++i)
            if (overlaps(o, bo, ins[i], nb[i]) || overlaps(S, bmem, ins[i], nb[i])) return GDR2_ERR_ALIAS;
        if (overlaps(o, bo, S, bmem)) return GDR2_ERR_ALIAS;
    }

    int st = device_setup(nullptr);
    if (st != GDR2_OK) return st;
    if (!has_tokens) return GDR2_OK;
    SparseArgs a{idx, q, k, v, b, w, log_decay, S, o, B, T, H, M, K, dv, in_dtype, out_dtype};
    return launch_sparse(a, stream);
}

extern "C" int gdr2_device_status(cudaStream_t stream) {
    int* err = nullptr;
    int st = device_setup(&err);
    if (st != GDR2_OK) return st;
    if (cudaStreamSynchronize(stream) != cudaSuccess) return GDR2_ERR_CUDA;
    int h = 0;
    if (cudaMemcpy(&h, err, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) return GDR2_ERR_CUDA;
    if (h != kDevOk) {
        const int zero = 0;
        if (cudaMemcpy(err, &zero, sizeof(int), cudaMemcpyHostToDevice) != cudaSuccess)
            return GDR2_ERR_CUDA;
        return GDR2_ERR_TIMEOUT;
    }
    return GDR2_OK;
}

extern "C" int gdr2_workspace_stats(int64_t* reserved, int64_t* used_high, int reset) {
    if (!reserved || !used_high) return GDR2_ERR_ARG;
    cudaMemPool_t pool = nullptr;
    const int st = workspace_pool(&pool);
    if (st != GDR2_OK) return st;
    uint64_t r = 0, u = 0;
    if (cudaMemPoolGetAttribute(pool, cudaMemPoolAttrReservedMemCurrent, &r) != cudaSuccess ||
        cudaMemPoolGetAttribute(pool, cudaMemPoolAttrUsedMemHigh, &u) != cudaSuccess)
        return GDR2_ERR_CUDA;
    *reserved = static_cast<int64_t>(r);
    *used_high = static_cast<int64_t>(u);
    if (reset) {
        uint64_t zero = 0;
        if (cudaMemPoolSetAttribute(pool, cudaMemPoolAttrUsedMemHigh, &zero) != cudaSuccess) return GDR2_ERR_CUDA;
    }
    return GDR2_OK;
}

extern "C" int64_t gdr2_set_wait_limit(int64_t cycles) {
    return gdr2::set_chain_wait_limit(cycles > 0 ? cycles : 0);
}

extern "C" int gdr2_release_workspace(void) {
    cudaMemPool_t pool = nullptr;
    const int st = workspace_pool(&pool);
    if (st != GDR2_OK) return st;
    if (cudaDeviceSynchronize() != cudaSuccess) return GDR2_ERR_CUDA;
    return cudaMemPoolTrimTo(pool, 0) == cudaSuccess ? GDR2_OK : GDR2_ERR_CUDA;
}

extern "C" const char* gdr2_status_string(int status) {
    switch (status) {
        case GDR2_OK: return "GDR2_OK";
        case GDR2_ERR_ARG: return "GDR2_ERR_ARG: null pointer or negative size";
        case GDR2_ERR_SHAPE: return "GDR2_ERR_SHAPE: unsupported head dim or size overflow";
        case GDR2_ERR_ALIGN: return "GDR2_ERR_ALIGN: pointer not 16-byte aligned";
        case GDR2_ERR_UNSUPPORTED: return "GDR2_ERR_UNSUPPORTED: unknown dtype or device is not sm_103";
        case GDR2_ERR_CUDA: return "GDR2_ERR_CUDA: a CUDA runtime call failed";
        case GDR2_ERR_SCRATCH:
            return "GDR2_ERR_SCRATCH: B*H too large for the no-allocation scratch (gdr2_forward_noalloc)";
        case GDR2_ERR_TIMEOUT: return "GDR2_ERR_TIMEOUT: a bounded device-side wait gave up";
        case GDR2_ERR_ALIAS: return "GDR2_ERR_ALIAS: output buffer overlaps another argument";
        default: return "GDR2: unknown status";
    }
}

extern "C" int gdr2_version(void) { return 200; }
