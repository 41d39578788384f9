// Memory-bound Gated Delta Rule-2 decode step: one token per (batch, head),
// fp32 state updated in place.
//
// Per head (update equation of the "Gated DeltaNet-2: Decoupling Erase and
// Write in Linear Attention" page, one token, readout o = S^T q):
//     S' = D S,   r = S'^T (b * k),   p = S'^T q,   delta = w * v - r,
//     S  <- S' + k delta^T,           o = p + (k . q) delta
//
// The state dominates the traffic (d_k * d_v * 4 bytes read and written per
// head; the token inputs are ~1% of it), so the kernel is built to stream it:
// one CTA per head, 256 threads, every thread holds DK*DV/1024 float4 of S in
// registers.  Element (row i, column 4c..4c+3) sits at float4 index
// i*DV/4 + c, and thread t loads float4 indices t, t+256, t+512, ... -- each
// warp instruction reads or writes 512 contiguous bytes.  The column
// reductions for r and p are a per-thread sum over its rows followed by one
// shared-memory reduction across the row groups.  S is read once and written
// once with streaming (evict-first) cache hints; no second pass.
#include "gdr2_internal.cuh"
#include "gdr2.h"

namespace gdr2 {
namespace {

constexpr int kThreads = 256;

template <typename Tin, typename Tout, int DK, int DV>
__global__ void __launch_bounds__(kThreads, 2)
decode_kernel(const Tin* __restrict__ q, const Tin* __restrict__ k,
              const Tin* __restrict__ v, const Tin* __restrict__ b,
              const Tin* __restrict__ w, const Tin* __restrict__ g,
              float* __restrict__ S, Tout* __restrict__ o) {
    constexpr int LPR = DV / 4;               // threads per state row (one float4 each)
    constexpr int RPP = kThreads / LPR;       // rows covered per pass
    constexpr int NP = DK / RPP;              // float4 per thread
    static_assert(NP >= 1 && DK % RPP == 0, "tile shape");

    __shared__ float sq[DK], sk[DK], sc[DK], sa[DK], su[DV];
    __shared__ float4 red_r[RPP][LPR], red_p[RPP][LPR];
    __shared__ float skq;

    const int64_t head = blockIdx.x;
    const int t = threadIdx.x;
    const int c4 = t % LPR, row0 = t / LPR;
    float4* Sh = reinterpret_cast<float4*>(S + head * DK * DV);

    // Issue every state load first; the token inputs are staged meanwhile.
    float4 s[NP];
#pragma unroll
    for (int m = 0; m < NP; ++m) s[m] = __ldcs(Sh + t + m * kThreads);

    const int64_t tk = head * DK, tv = head * DV;
    for (int i = t; i < DK; i += kThreads) {
        const float kv = to_f32(k[tk + i]);
        sq[i] = to_f32(q[tk + i]);
        sk[i] = kv;
        sc[i] = to_f32(b[tk + i]) * kv;
        sa[i] = expf(to_f32(g[tk + i]));
    }
    for (int j = t; j < DV; j += kThreads) su[j] = to_f32(w[tv + j]) * to_f32(v[tv + j]);
    __syncthreads();
    if (t < 32) {
        float acc = 0.f;
        for (int i = t; i < DK; i += 32) acc += sk[i] * sq[i];
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
        if (t == 0) skq = acc;
    }

    // S' = D S and the per-thread partial column sums of r and p.
    float4 r = make_float4(0.f, 0.f, 0.f, 0.f), p = r;
#pragma unroll
    for (int m = 0; m < NP; ++m) {
        const int i = row0 + m * RPP;
        const float a = sa[i], c = sc[i], qq = sq[i];
        float4 P = s[m];
        P.x *= a; P.y *= a; P.z *= a; P.w *= a;
        s[m] = P;
        r.x = fmaf(c, P.x, r.x); r.y = fmaf(c, P.y, r.y); r.z = fmaf(c, P.z, r.z); r.w = fmaf(c, P.w, r.w);
        p.x = fmaf(qq, P.x, p.x); p.y = fmaf(qq, P.y, p.y); p.z = fmaf(qq, P.z, p.z); p.w = fmaf(qq, P.w, p.w);
    }
    red_r[row0][c4] = r;
    red_p[row0][c4] = p;
    __syncthreads();
    r = make_float4(0.f, 0.f, 0.f, 0.f);
    p = r;
#pragma unroll
    for (int rr = 0; rr < RPP; ++rr) {
        const float4 x = red_r[rr][c4], y = red_p[rr][c4];
        r.x += x.x; r.y += x.y; r.z += x.z; r.w += x.w;
        p.x += y.x; p.y += y.y; p.z += y.z; p.w += y.w;
    }
    float4 d;
    d.x = su[4 * c4 + 0] - r.x;
    d.y = su[4 * c4 + 1] - r.y;
    d.z = su[4 * c4 + 2] - r.z;
    d.w = su[4 * c4 + 3] - r.w;

    // S <- S' + k delta^T, written back in place.
#pragma unroll
    for (int m = 0; m < NP; ++m) {
        const float kk = sk[row0 + m * RPP];
        float4 P = s[m];
        P.x = fmaf(kk, d.x, P.x); P.y = fmaf(kk, d.y, P.y);
        P.z = fmaf(kk, d.z, P.z); P.w = fmaf(kk, d.w, P.w);
        __stcs(Sh + t + m * kThreads, P);
    }
    if (row0 == 0) {
        const float kq = skq;
        Tout* oh = o + tv + 4 * c4;
        oh[0] = from_f32<Tout>(fmaf(kq, d.x, p.x));
        oh[1] = from_f32<Tout>(fmaf(kq, d.y, p.y));
        oh[2] = from_f32<Tout>(fmaf(kq, d.z, p.z));
        oh[3] = from_f32<Tout>(fmaf(kq, d.w, p.w));
    }
}

template <typename Tin, typename Tout, int DK>
int launch_dv(const DecodeArgs& a, cudaStream_t stream) {
    const dim3 grid((unsigned)(a.B * a.H));
    auto go = [&](auto kern) {
        kern<<<grid, kThreads, 0, stream>>>((const Tin*)a.q, (const Tin*)a.k, (const Tin*)a.v,
                                            (const Tin*)a.b, (const Tin*)a.w, (const Tin*)a.g,
                                            a.S, (Tout*)a.o);
    };
    switch (a.dv) {
        case 32: go(decode_kernel<Tin, Tout, DK, 32>); break;
        case 64: go(decode_kernel<Tin, Tout, DK, 64>); break;
        case 128: go(decode_kernel<Tin, Tout, DK, 128>); break;
        default: return GDR2_ERR_SHAPE;
    }
    return cudaPeekAtLastError() == cudaSuccess ? GDR2_OK : GDR2_ERR_CUDA;
}

template <typename Tin, typename Tout>
int launch_typed(const DecodeArgs& a, cudaStream_t stream) {
    switch (a.dk) {
        case 32: return launch_dv<Tin, Tout, 32>(a, stream);
        case 64: return launch_dv<Tin, Tout, 64>(a, stream);
        case 128: return launch_dv<Tin, Tout, 128>(a, stream);
        default: return GDR2_ERR_SHAPE;
    }
}

}  // namespace

int launch_decode(const DecodeArgs& a, cudaStream_t stream) {
    using bf16 = __nv_bfloat16;
    if (a.in_dtype == GDR2_F32)
        return a.out_dtype == GDR2_F32 ? launch_typed<float, float>(a, stream)
                                       : launch_typed<float, bf16>(a, stream);
    return a.out_dtype == GDR2_F32 ? launch_typed<bf16, float>(a, stream)
                                   : launch_typed<bf16, bf16>(a, stream);
}

}  // namespace gdr2
