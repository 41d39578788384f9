// Token-sequential Gated Delta Rule-2 prefill in fp32 arithmetic.
//
// Serves fp32 inputs (where the tolerance calls for fp32 arithmetic at every
// step) and head dims the chunked tensor-core kernel does not cover.  It
// applies the update of the "Gated DeltaNet-2: Decoupling Erase and Write in
// Linear Attention" page (section "Gated Delta Rule-2 update equation") one
// token at a time:
//     P = D_t S,   x = P^T (b_t * k_t),   p = P^T q_t,   delta = w_t * v_t - x,
//     S = P + k_t delta^T,                o_t = p + (k_t . q_t) delta  (= S_t^T q_t)
//
// Work split: one CTA per (batch*head, d_v tile of DVT columns); the CTA's
// slice of S lives in registers for the whole sequence.  Each warp owns
// DVT/NW columns; lane l owns key rows l, l+32, ...; column reductions are
// warp shuffles, so tokens need no block-wide barrier.  Token inputs are
// staged through shared memory TB tokens at a time.
#include "gdr2_internal.cuh"
#include "gdr2.h"

namespace gdr2 {
namespace {

constexpr int kNW = 8;      // warps per CTA
constexpr int kDVT = 32;    // d_v columns per CTA
constexpr int kTB = 16;     // tokens staged per round

template <typename Tin, typename Tout, int DK>
__global__ void __launch_bounds__(kNW * 32)
recurrent_kernel(const Tin* __restrict__ q, const Tin* __restrict__ k,
                 const Tin* __restrict__ v, const Tin* __restrict__ b,
                 const Tin* __restrict__ w, const Tin* __restrict__ g,
                 const float* __restrict__ S0, Tout* __restrict__ o,
                 float* __restrict__ ST, int64_t Tfix, int H, int dv,
                 const int* __restrict__ cu, int64_t total,
                 float* __restrict__ cache, int64_t cache_every, int n_cache) {
    constexpr int RPL = DK / 32;          // key rows per lane
    constexpr int CPW = kDVT / kNW;       // value columns per warp
    __shared__ float sq[kTB][DK], sk[kTB][DK], sc[kTB][DK], sa[kTB][DK];
    __shared__ float su[kTB][kDVT], so[kTB][kDVT], skq[kTB];

    const int64_t bh = blockIdx.x;
    const int64_t seq = bh / H, h = bh % H;
    // this sequence's token rows [tok0, tok0 + T) of the packed [total, H, d] tensors
    int64_t tok0, T;
    if (cu) {   // offsets clamped to [0, total] and made non-decreasing
        const int64_t a = min(max(static_cast<int64_t>(cu[seq]), int64_t(0)), total);
        const int64_t e = min(max(static_cast<int64_t>(cu[seq + 1]), a), total);
        tok0 = a;
        T = e - a;
    } else {
        tok0 = seq * Tfix;
        T = Tfix;
    }
    const int j0 = blockIdx.y * kDVT;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int jw = warp * CPW;            // first column of this warp within the tile

    float S[RPL][CPW];
#pragma unroll
    for (int r = 0; r < RPL; ++r)
#pragma unroll
        for (int c = 0; c < CPW; ++c) {
            const int64_t idx = (bh * DK + lane + 32 * r) * dv + j0 + jw + c;
            S[r][c] = S0 ? S0[idx] : 0.f;
        }

    for (int64_t t0 = 0; t0 < T; t0 += kTB) {
        const int n = (T - t0) < kTB ? (int)(T - t0) : kTB;
        for (int e = threadIdx.x; e < kTB * DK; e += blockDim.x) {
            const int tt = e / DK, i = e % DK;
            if (tt < n) {
                const int64_t off = ((tok0 + t0 + tt) * H + h) * DK + i;
                const float kv = to_f32(k[off]);
                sq[tt][i] = to_f32(q[off]);
                sk[tt][i] = kv;
                sc[tt][i] = to_f32(b[off]) * kv;
                sa[tt][i] = expf(to_f32(g[off]));
            }
        }
        for (int e = threadIdx.x; e < kTB * kDVT; e += blockDim.x) {
            const int tt = e / kDVT, j = e % kDVT;
            if (tt < n) {
                const int64_t off = ((tok0 + t0 + tt) * H + h) * dv + j0 + j;
                su[tt][j] = to_f32(w[off]) * to_f32(v[off]);
            }
        }
        __syncthreads();
        for (int tt = warp; tt < n; tt += kNW) {      // k_t . q_t, one warp per token
            float acc = 0.f;
            for (int i = lane; i < DK; i += 32) acc += sk[tt][i] * sq[tt][i];
#pragma unroll
            for (int s = 16; s > 0; s >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, s);
            if (lane == 0) skq[tt] = acc;
        }
        __syncthreads();

        for (int tt = 0; tt < n; ++tt) {
#pragma unroll
            for (int c = 0; c < CPW; ++c) {
                float x = 0.f, p = 0.f;
#pragma unroll
                for (int r = 0; r < RPL; ++r) {
                    const int i = lane + 32 * r;
                    const float P = sa[tt][i] * S[r][c];
                    S[r][c] = P;
                    x = fmaf(sc[tt][i], P, x);
                    p = fmaf(sq[tt][i], P, p);
                }
#pragma unroll
                for (int s = 16; s > 0; s >>= 1) {
                    x += __shfl_xor_sync(0xffffffffu, x, s);
                    p += __shfl_xor_sync(0xffffffffu, p, s);
                }
                const float delta = su[tt][jw + c] - x;
#pragma unroll
                for (int r = 0; r < RPL; ++r) S[r][c] = fmaf(sk[tt][lane + 32 * r], delta, S[r][c]);
                if (lane == 0) so[tt][jw + c] = fmaf(skq[tt], delta, p);
            }
        }
        __syncthreads();
        for (int e = threadIdx.x; e < n * kDVT; e += blockDim.x) {
            const int tt = e / kDVT, j = e % kDVT;
            const int64_t off = ((tok0 + t0 + tt) * H + h) * dv + j0 + j;
            o[off] = from_f32<Tout>(so[tt][j]);
        }
        // the state at a cache point (cache_every is a multiple of the 16-token round)
        if (cache && (t0 + n) % cache_every == 0 && (t0 + n) / cache_every <= n_cache) {
            const int64_t m = (t0 + n) / cache_every - 1;
#pragma unroll
            for (int r = 0; r < RPL; ++r)
#pragma unroll
                for (int c = 0; c < CPW; ++c)
                    cache[((bh * n_cache + m) * DK + lane + 32 * r) * dv + j0 + jw + c] = S[r][c];
        }
        __syncthreads();
    }

    if (ST) {
#pragma unroll
        for (int r = 0; r < RPL; ++r)
#pragma unroll
            for (int c = 0; c < CPW; ++c)
                ST[(bh * DK + lane + 32 * r) * dv + j0 + jw + c] = S[r][c];
    }
}

template <typename Tin, typename Tout>
int launch_typed(const ForwardArgs& a, cudaStream_t stream) {
    const dim3 grid((unsigned)(a.B * a.H), (unsigned)(a.dv / kDVT));
    const dim3 block(kNW * 32);
    auto args = [&](auto kern) {
        kern<<<grid, block, 0, stream>>>(
            (const Tin*)a.q, (const Tin*)a.k, (const Tin*)a.v, (const Tin*)a.b,
            (const Tin*)a.w, (const Tin*)a.g, a.S0, (Tout*)a.o, a.ST, a.T, (int)a.H, (int)a.dv, a.cu,
            a.total, a.S_cache, a.cache_chunks * 64,
            a.S_cache ? static_cast<int>(a.T / (a.cache_chunks * 64)) : 0);
    };
    switch (a.dk) {
        case 32: args(recurrent_kernel<Tin, Tout, 32>); break;
        case 64: args(recurrent_kernel<Tin, Tout, 64>); break;
        case 128: args(recurrent_kernel<Tin, Tout, 128>); break;
        default: return GDR2_ERR_SHAPE;
    }
    return cudaPeekAtLastError() == cudaSuccess ? GDR2_OK : GDR2_ERR_CUDA;
}

}  // namespace

int launch_recurrent(const ForwardArgs& a, cudaStream_t stream) {
    using bf16 = __nv_bfloat16;
    if (a.in_dtype == GDR2_F32)
        return a.out_dtype == GDR2_F32 ? launch_typed<float, float>(a, stream)
                                       : launch_typed<float, bf16>(a, stream);
    return a.out_dtype == GDR2_F32 ? launch_typed<bf16, float>(a, stream)
                                   : launch_typed<bf16, bf16>(a, stream);
}

}  // namespace gdr2
