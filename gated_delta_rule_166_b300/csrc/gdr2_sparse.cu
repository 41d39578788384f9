// Sparse gated delta write: the Gated Delta Rule-2 update applied only to the
// slots of a slot memory that a router selected for each token.
//
// Method: the "Sparse Delta Memory" review page (section "3. Method & Key
// Results": the gated delta write is performed on the slots a product-key
// memory selects, not on the whole state) with the routing-slot recurrence of
// the Raven summary page (section "2.1 RSM framework": unselected slots keep
// their contents, no decay).  Per (sequence, head) the memory S is M x d_v fp32;
// at token t the K selected slots R = idx_t carry key-side values q, k, b and
// log_decay g (one per selected slot) and
//     Sd = diag(exp g) S[R],   x = (b * k)^T Sd,   S[R] = Sd + k (w * v - x)^T,
//     o_t = S[R]^T q       (the selected slots read after the update).
//
// The value columns of the memory evolve independently (x and o are per
// column), so the work splits over (sequence, head, column tile) with no
// exchange.  Two kernels:
//
// * sparse_tile_kernel (every memory that fits): one warp per (sequence, head,
//   W-column tile) keeps its M x W tile of the memory in shared memory for the
//   whole sequence, so a token's gathers and scatters are shared-memory
//   accesses.  Lane = (slot group g, column c) with 32 / W slot groups; lane
//   (g, c) handles the selected slots j = g, g + 32/W, ... of each token, and
//   the x and o sums over the slots are shuffle reductions across the groups.
//   W = 8 when the tile fits (M up to about 6,800 slots), else 4, 2, 1.  The key-side
//   values of the next chunk of tokens (slot, e^g, b k, k, q) are loaded into
//   registers while the current chunk runs and staged in shared memory
//   between chunks.
// * sparse_kernel (memories too large for shared memory): one CTA per
//   (sequence, head), lane = value column, the memory gathered from and
//   scattered to global memory; the next token's gathers follow the scatter in
//   program order, so a slot selected twice in a row is read after its write.
#include "gdr2_internal.cuh"
#include "gdr2.h"

namespace gdr2 {
namespace {

constexpr int kTC = 16;   // tokens per staged chunk

struct SparseParams {
    const int* idx;
    const void *q, *k, *v, *b, *w, *g;
    float* S;
    void* o;
    int T, H, M, K, dv;
};

template <typename Tin, typename Tout, int KMAX>
__global__ void __launch_bounds__(128)
sparse_kernel(const SparseParams p) {
    // staged key-side values: slot (-1 = none) and {e^g, b k, k, q} per (token, slot)
    __shared__ int s_idx[2][kTC][KMAX];
    __shared__ float4 s_val[2][kTC][KMAX];

    const int bh = static_cast<int>(blockIdx.x);
    const int seq = bh / p.H, h = bh - seq * p.H;
    const int tid = static_cast<int>(threadIdx.x), nthr = static_cast<int>(blockDim.x);
    const int col = tid;   // value column of this thread (blockDim.x = d_v)
    const Tin* qi = static_cast<const Tin*>(p.q);
    const Tin* ki = static_cast<const Tin*>(p.k);
    const Tin* bi = static_cast<const Tin*>(p.b);
    const Tin* gi = static_cast<const Tin*>(p.g);
    const Tin* vi = static_cast<const Tin*>(p.v);
    const Tin* wi = static_cast<const Tin*>(p.w);
    Tout* oo = static_cast<Tout*>(p.o);
    float* Sh = p.S + static_cast<int64_t>(bh) * p.M * p.dv + col;
    const int K = p.K;

    auto stage = [&](int c, int buf) {
        const int t0 = c * kTC, nt = min(kTC, p.T - t0);
        for (int e = tid; e < kTC * K; e += nthr) {
            const int tt = e / K, j = e - tt * K;
            int s = -1;
            float4 val = make_float4(1.f, 0.f, 0.f, 0.f);
            if (tt < nt) {
                const int64_t off = ((static_cast<int64_t>(seq) * p.T + t0 + tt) * p.H + h) * K + j;
                s = p.idx[off];
                if (s >= 0 && s < p.M) {
                    const float kv = to_f32(ki[off]);
                    val = make_float4(expf(to_f32(gi[off])), to_f32(bi[off]) * kv, kv, to_f32(qi[off]));
                } else {
                    s = -1;
                }
            }
            s_idx[buf][tt][j] = s;
            s_val[buf][tt][j] = val;
        }
    };

    const int nchunks = (p.T + kTC - 1) / kTC;
    if (nchunks > 0) stage(0, 0);
    __syncthreads();
    // w * v of the next token, loaded one token ahead
    auto uoff = [&](int t) { return ((static_cast<int64_t>(seq) * p.T + t) * p.H + h) * p.dv + col; };
    float vn = 0.f, wn = 0.f;
    if (p.T > 0) {
        vn = to_f32(vi[uoff(0)]);
        wn = to_f32(wi[uoff(0)]);
    }
#pragma unroll 1
    for (int c = 0; c < nchunks; ++c) {
        const int buf = c & 1;
        if (c + 1 < nchunks) stage(c + 1, buf ^ 1);   // read two barriers later
        const int t0 = c * kTC, nt = min(kTC, p.T - t0);
#pragma unroll 1
        for (int tt = 0; tt < nt; ++tt) {
            const int t = t0 + tt;
            const float u = vn * wn;
            if (t + 1 < p.T) {
                vn = to_f32(vi[uoff(t + 1)]);
                wn = to_f32(wi[uoff(t + 1)]);
            }
            const int* si = s_idx[buf][tt];
            const float4* sv = s_val[buf][tt];
            // gathers first (all in flight), then decay and the erase read
            float sd[KMAX];
#pragma unroll
            for (int j = 0; j < KMAX; ++j) {
                const int s = j < K ? si[j] : -1;
                sd[j] = s >= 0 ? Sh[static_cast<int64_t>(s) * p.dv] : 0.f;
            }
            float x = 0.f;
#pragma unroll
            for (int j = 0; j < KMAX; ++j) {
                if (j < K) {
                    const float4 a = sv[j];
                    sd[j] *= a.x;
                    x = fmaf(a.y, sd[j], x);
                }
            }
            const float d = u - x;
            float ov = 0.f;
#pragma unroll
            for (int j = 0; j < KMAX; ++j) {
                if (j < K) {
                    const int s = si[j];
                    const float4 a = sv[j];
                    const float nv = fmaf(a.z, d, sd[j]);
                    if (s >= 0) Sh[static_cast<int64_t>(s) * p.dv] = nv;
                    ov = fmaf(a.w, nv, ov);
                }
            }
            oo[uoff(t)] = from_f32<Tout>(ov);
        }
        __syncthreads();   // chunk c + 1 staged; buffer buf free for chunk c + 2
    }
}

// ---- shared-memory tile kernel ------------------------------------------------------
// Raw element bits (read-only path) and their conversion, kept apart so that a
// prefetch does not wait for its loads.
__device__ __forceinline__ uint32_t raw_bits(const float* p) { return __float_as_uint(__ldg(p)); }
__device__ __forceinline__ uint32_t raw_bits(const __nv_bfloat16* p) {
    return static_cast<uint32_t>(__ldg(reinterpret_cast<const unsigned short*>(p)));
}
template <typename T> __device__ __forceinline__ float bits_f32(uint32_t x);
template <> __device__ __forceinline__ float bits_f32<float>(uint32_t x) { return __uint_as_float(x); }
template <> __device__ __forceinline__ float bits_f32<__nv_bfloat16>(uint32_t x) { return __uint_as_float(x << 16); }
// Shared-space accesses by 32-bit shared address (the token loop's pointers are
// computed, so their state space is stated explicitly).
__device__ __forceinline__ float lds_f(uint32_t a) {
    float v;
    asm volatile("ld.shared.f32 %0, [%1];" : "=f"(v) : "r"(a) : "memory");
    return v;
}
__device__ __forceinline__ int lds_i(uint32_t a) {
    int v;
    asm volatile("ld.shared.s32 %0, [%1];" : "=r"(v) : "r"(a) : "memory");
    return v;
}
__device__ __forceinline__ float4 lds_f4(uint32_t a) {
    float4 v;
    asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];" : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w) : "r"(a) : "memory");
    return v;
}
__device__ __forceinline__ void sts_f(uint32_t a, float v) {
    asm volatile("st.shared.f32 [%0], %1;" ::"r"(a), "f"(v) : "memory");
}

constexpr int kTileStageEntries = 256;   // staged (token, slot) entries per chunk
constexpr int kTileSmemMax = 227 * 1024;

// Slots per token padded to a multiple of the slot groups (padding entries
// and out-of-range indices point at a scratch row of the tile, with e^g = 1
// and b k = k = q = 0, so the token loop has no branches); tokens per chunk.
template <int KMAX, int W>
struct TileShape {
    static constexpr int G = 32 / W;                          // slot groups
    static constexpr int KPL = (KMAX + G - 1) / G;            // slots per lane
    static constexpr int KPAD = G * KPL;                      // staged slots per token
    static constexpr int TC = kTileStageEntries / KPAD;       // tokens per chunk
    static constexpr int E = kTileStageEntries / 32;          // staged entries per lane
    static constexpr int EV = (TC * W + 31) / 32;             // staged u values per lane
    static constexpr size_t stage_bytes =
        static_cast<size_t>(2 * TC * KPAD) * (sizeof(float4) + sizeof(int)) + static_cast<size_t>(2 * TC * W) * sizeof(float);
};

template <typename Tin, typename Tout, int W, int KMAX>
__global__ void __launch_bounds__(32)
sparse_tile_kernel(const SparseParams p) {
    using TS = TileShape<KMAX, W>;
    constexpr int G = TS::G, KPL = TS::KPL, KPAD = TS::KPAD, TC = TS::TC, E = TS::E, EV = TS::EV;
    static_assert(TC * KPAD == kTileStageEntries, "staging shape");
    extern __shared__ float4 smem4[];
    float4* sval = smem4;                                                   // [2][TC][KPAD] {e^g, b k, k, q}
    int* soff = reinterpret_cast<int*>(smem4 + 2 * TC * KPAD);              // [2][TC][KPAD] slot * W
    float* su = reinterpret_cast<float*>(soff + 2 * TC * KPAD);             // [2][TC][W]    w * v
    float* tile = su + 2 * TC * W;                                          // [M + 1][W]  (row M: scratch)
    const uint32_t a_sval = static_cast<uint32_t>(__cvta_generic_to_shared(sval));
    const uint32_t a_soff = static_cast<uint32_t>(__cvta_generic_to_shared(soff));
    const uint32_t a_su = static_cast<uint32_t>(__cvta_generic_to_shared(su));
    const uint32_t a_tile = static_cast<uint32_t>(__cvta_generic_to_shared(tile));

    const int ntiles = p.dv / W;
    const int bh = static_cast<int>(blockIdx.x) / ntiles;
    const int col0 = (static_cast<int>(blockIdx.x) - bh * ntiles) * W;
    const int seq = bh / p.H, h = bh - seq * p.H;
    const int lane = static_cast<int>(threadIdx.x);
    const int g = lane / W, c = lane - g * W;
    const int K = p.K, M = p.M;
    const Tin* qi = static_cast<const Tin*>(p.q);
    const Tin* ki = static_cast<const Tin*>(p.k);
    const Tin* bi = static_cast<const Tin*>(p.b);
    const Tin* gi = static_cast<const Tin*>(p.g);
    const Tin* vi = static_cast<const Tin*>(p.v);
    const Tin* wi = static_cast<const Tin*>(p.w);
    Tout* oo = static_cast<Tout*>(p.o);
    float* Sg = p.S + static_cast<int64_t>(bh) * M * p.dv + col0;

    // the memory tile into shared memory
#pragma unroll 4
    for (int m = lane; m < M; m += 32) {
#pragma unroll
        for (int e = 0; e < W; ++e) tile[m * W + e] = Sg[static_cast<int64_t>(m) * p.dv + e];
    }

    // key-side values and u of a chunk: raw bits loaded into registers (every
    // address clamped into range, nothing computed from them) while the previous
    // chunk runs, then masked, converted and staged between chunks
    struct Raw {
        int s[E];
        uint32_t kq[E][4];   // k, b, g, q (raw element bits)
        uint32_t vw[EV][2];  // v, w
    };
    auto fetch = [&](int ch, Raw& r) {
        const int t0 = ch * TC;
#pragma unroll
        for (int e = 0; e < EV; ++e) {
            const int n = lane + 32 * e, tt = min(n / W, TC - 1), cc = n % W;
            const int t = min(t0 + tt, p.T - 1);
            const int64_t off = ((static_cast<int64_t>(seq) * p.T + t) * p.H + h) * p.dv + col0 + cc;
            r.vw[e][0] = raw_bits(vi + off);
            r.vw[e][1] = raw_bits(wi + off);
        }
#pragma unroll
        for (int e = 0; e < E; ++e) {
            const int n = lane + 32 * e, tt = n / KPAD, j = min(n - tt * KPAD, K - 1);
            const int t = min(t0 + tt, p.T - 1);
            const int64_t off = ((static_cast<int64_t>(seq) * p.T + t) * p.H + h) * K + max(j, 0);
            r.s[e] = __ldg(p.idx + off);
            r.kq[e][0] = raw_bits(ki + off);
            r.kq[e][1] = raw_bits(bi + off);
            r.kq[e][2] = raw_bits(gi + off);
            r.kq[e][3] = raw_bits(qi + off);
        }
    };
    auto put = [&](int ch, int buf, const Raw& r) {
        const int t0 = ch * TC;
#pragma unroll
        for (int e = 0; e < E; ++e) {
            const int n = lane + 32 * e, tt = n / KPAD, j = n - tt * KPAD;
            const int s = r.s[e];
            const bool ok = j < K && t0 + tt < p.T && s >= 0 && s < M;
            const float kv = bits_f32<Tin>(r.kq[e][0]);
            soff[buf * TC * KPAD + n] = (ok ? s : M) * W;
            sval[buf * TC * KPAD + n] = ok ? make_float4(expf(bits_f32<Tin>(r.kq[e][2])), bits_f32<Tin>(r.kq[e][1]) * kv, kv,
                                                         bits_f32<Tin>(r.kq[e][3]))
                                           : make_float4(1.f, 0.f, 0.f, 0.f);
        }
#pragma unroll
        for (int e = 0; e < EV; ++e) {
            const int n = lane + 32 * e;
            if (n < TC * W) su[buf * TC * W + n] = bits_f32<Tin>(r.vw[e][0]) * bits_f32<Tin>(r.vw[e][1]);
        }
    };
    const int nchunks = (p.T + TC - 1) / TC;
    Raw raw;
    fetch(0, raw);
    put(0, 0, raw);
    __syncwarp();
    auto uoff = [&](int t) { return ((static_cast<int64_t>(seq) * p.T + t) * p.H + h) * p.dv + col0 + c; };
#pragma unroll 1
    for (int ch = 0; ch < nchunks; ++ch) {
        const int buf = ch & 1;
        if (ch + 1 < nchunks) fetch(ch + 1, raw);   // in flight during this chunk
        const int t0 = ch * TC, nt = min(TC, p.T - t0);
        // A token's slot offsets, key-side values and u come from the staging buffer,
        // not the memory tile, so the next token's are loaded while this one reduces;
        // only the gathers wait for the previous token's scatter.
        struct Staged {
            uint32_t ad[KPL];   // shared-memory address of each selected slot's column c
            float4 a[KPL];      // {e^g, b k, k, q} of each selected slot
            float u;            // w v of column c
        };
        auto stage_of = [&](int tt) {
            Staged x;
            x.u = lds_f(a_su + 4u * static_cast<uint32_t>((buf * TC + tt) * W + c));
            const uint32_t so = a_soff + 4u * static_cast<uint32_t>((buf * TC + tt) * KPAD + g);
            const uint32_t sv = a_sval + 16u * static_cast<uint32_t>((buf * TC + tt) * KPAD + g);
#pragma unroll
            for (int i = 0; i < KPL; ++i) {
                x.ad[i] = a_tile + 4u * static_cast<uint32_t>(lds_i(so + 4u * G * i) + c);
                x.a[i] = lds_f4(sv + 16u * G * i);
            }
            return x;
        };
        Staged cur = stage_of(0);   // nt >= 1: chunks hold at least one token
#pragma unroll 1
        for (int tt = 0; tt < nt; ++tt) {
            const int t = t0 + tt;
            const uint32_t (&ad)[KPL] = cur.ad;
            const float4 (&a)[KPL] = cur.a;
            const float u = cur.u;
            float sd[KPL];
#pragma unroll
            for (int i = 0; i < KPL; ++i) sd[i] = lds_f(ad[i]);
            const Staged nxt = stage_of(tt + 1 < nt ? tt + 1 : tt);   // the last token re-reads its own
            float x0 = 0.f, x1 = 0.f;   // two accumulators: half the dependent chain
#pragma unroll
            for (int i = 0; i < KPL; ++i) {
                sd[i] *= a[i].x;
                if (i & 1) x1 = fmaf(a[i].y, sd[i], x1); else x0 = fmaf(a[i].y, sd[i], x0);
            }
            float x = x0 + x1;
#pragma unroll
            for (int off = W; off < 32; off <<= 1) x += __shfl_xor_sync(0xffffffffu, x, off);
            const float d = u - x;
            float o0 = 0.f, o1 = 0.f;
#pragma unroll
            for (int i = 0; i < KPL; ++i) {
                const float nv = fmaf(a[i].z, d, sd[i]);
                sts_f(ad[i], nv);
                if (i & 1) o1 = fmaf(a[i].w, nv, o1); else o0 = fmaf(a[i].w, nv, o0);
            }
            float ov = o0 + o1;
#pragma unroll
            for (int off = W; off < 32; off <<= 1) ov += __shfl_xor_sync(0xffffffffu, ov, off);
            if (g == 0) oo[uoff(t)] = from_f32<Tout>(ov);
            __syncwarp();   // this token's scatter is visible to the next token's gathers
            cur = nxt;
        }
        if (ch + 1 < nchunks) {
            put(ch + 1, buf ^ 1, raw);
            __syncwarp();
        }
    }
    // the tile back to global memory
#pragma unroll 4
    for (int m = lane; m < M; m += 32) {
#pragma unroll
        for (int e = 0; e < W; ++e) Sg[static_cast<int64_t>(m) * p.dv + e] = tile[m * W + e];
    }
}

template <typename Tin, typename Tout, int W, int KMAX>
int launch_tile(const SparseParams& p, int64_t BH, cudaStream_t stream) {
    const size_t smem = TileShape<KMAX, W>::stage_bytes + static_cast<size_t>(p.M + 1) * W * sizeof(float);
    auto kern = sparse_tile_kernel<Tin, Tout, W, KMAX>;
    if (smem > 48 * 1024 && cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                 static_cast<int>(smem)) != cudaSuccess)
        return GDR2_ERR_CUDA;
    const int64_t grid = BH * (p.dv / W);
    if (grid > 0x7fffffffLL) return GDR2_ERR_SHAPE;
    kern<<<static_cast<unsigned>(grid), 32, smem, stream>>>(p);
    return cudaPeekAtLastError() == cudaSuccess ? GDR2_OK : GDR2_ERR_CUDA;
}

template <int KMAX, int W>
bool tile_fits(int64_t M) {
    return TileShape<KMAX, W>::stage_bytes + static_cast<size_t>(M + 1) * W * 4 <= kTileSmemMax;
}

template <typename Tin, typename Tout, int KMAX>
int launch_tile_k(const SparseParams& p, int64_t BH, cudaStream_t stream) {
    if (tile_fits<KMAX, 8>(p.M)) return launch_tile<Tin, Tout, 8, KMAX>(p, BH, stream);
    if (tile_fits<KMAX, 4>(p.M)) return launch_tile<Tin, Tout, 4, KMAX>(p, BH, stream);
    if (tile_fits<KMAX, 2>(p.M)) return launch_tile<Tin, Tout, 2, KMAX>(p, BH, stream);
    return launch_tile<Tin, Tout, 1, KMAX>(p, BH, stream);
}

template <typename Tin, typename Tout>
int launch_t(const SparseArgs& a, cudaStream_t stream) {
    const SparseParams p{a.idx, a.q, a.k, a.v, a.b, a.w, a.g, a.S, a.o,
                         static_cast<int>(a.T), static_cast<int>(a.H), static_cast<int>(a.M),
                         static_cast<int>(a.K), static_cast<int>(a.dv)};
    const int64_t BH = a.B * a.H;
    // the shared-memory tile kernel whenever a one-column tile fits
    if (a.K <= 8) {
        if (tile_fits<8, 1>(a.M)) return launch_tile_k<Tin, Tout, 8>(p, BH, stream);
    } else if (a.K <= 16) {
        if (tile_fits<16, 1>(a.M)) return launch_tile_k<Tin, Tout, 16>(p, BH, stream);
    } else if (a.K <= 32) {
        if (tile_fits<32, 1>(a.M)) return launch_tile_k<Tin, Tout, 32>(p, BH, stream);
    } else if (tile_fits<64, 1>(a.M)) {
        return launch_tile_k<Tin, Tout, 64>(p, BH, stream);
    }
    const dim3 grid(static_cast<unsigned>(BH)), block(static_cast<unsigned>(a.dv));
    if (a.K <= 8) sparse_kernel<Tin, Tout, 8><<<grid, block, 0, stream>>>(p);
    else if (a.K <= 16) sparse_kernel<Tin, Tout, 16><<<grid, block, 0, stream>>>(p);
    else if (a.K <= 32) sparse_kernel<Tin, Tout, 32><<<grid, block, 0, stream>>>(p);
    else sparse_kernel<Tin, Tout, 64><<<grid, block, 0, stream>>>(p);
    return cudaPeekAtLastError() == cudaSuccess ? GDR2_OK : GDR2_ERR_CUDA;
}

}  // namespace

int launch_sparse(const SparseArgs& a, cudaStream_t stream) {
    if (a.B * a.H == 0 || a.T == 0) return GDR2_OK;
    if (a.K == 0) {   // nothing selected: o = 0 (all-zero bits in both output types), S unchanged
        const size_t bytes = static_cast<size_t>(a.B * a.T * a.H * a.dv) * (a.out_dtype == GDR2_F32 ? 4 : 2);
        return cudaMemsetAsync(a.o, 0, bytes, stream) == cudaSuccess ? GDR2_OK : GDR2_ERR_CUDA;
    }
    const bool in32 = a.in_dtype == GDR2_F32, out32 = a.out_dtype == GDR2_F32;
    if (in32) return out32 ? launch_t<float, float>(a, stream) : launch_t<float, __nv_bfloat16>(a, stream);
    return out32 ? launch_t<__nv_bfloat16, float>(a, stream) : launch_t<__nv_bfloat16, __nv_bfloat16>(a, stream);
}

}  // namespace gdr2
