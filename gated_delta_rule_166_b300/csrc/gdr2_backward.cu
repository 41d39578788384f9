// Gradients of the Gated Delta Rule-2 recurrence (fp32, token-sequential).
//
// Method: reverse-mode differentiation of the update of the "Gated DeltaNet-2:
// Decoupling Erase and Write in Linear Attention" page (section "Gated Delta
// Rule-2 update equation"), written per token with X_t = D_t S_{t-1},
// c_t = b_t * k_t, delta_t = w_t * v_t - X_t^T c_t:
//     S_t = X_t + k_t delta_t^T,      o_t = S_t^T q_t.
// With G the gradient arriving at S_t (from later tokens and dS_T) plus
// q_t do_t^T from the readout, one step back is
//     dq_t = S_t do_t,               ddelta = G^T k_t,
//     dv_t = ddelta * w_t,           dw_t = ddelta * v_t,
//     dc = -X_t ddelta,              db_t = dc * k_t,
//     dk_t = G delta_t + dc * b_t,   dX = G - c_t ddelta^T,
//     dlog_decay_t = rowsum(dX * X_t),   dS_{t-1} = D_t dX.
// The d_v columns of S evolve independently, so one CTA owns a 32-column tile
// of one (sequence, head): the tile of S, later of G, stays in registers (lane
// l of warp w: key rows l, l+32, ...; columns 4w .. 4w+3).  Column sums are
// warp shuffles; the row vectors (dq, dk, dc, dlog_decay) are summed over the
// CTA's warps in shared memory and over the tiles by a second kernel.
//
// States in reverse order come from recomputation: a forward sweep stores the
// tile at the start of every 4-token block (checkpoints in the workspace); the
// backward sweep reloads a block's checkpoint, recomputes its 4 states with the
// same arithmetic (so the same fp32 values), keeps X_t and delta_t in shared
// memory and walks the block backwards.  Each block's token inputs are fetched
// into registers while the previous block is computed.  Short blocks keep the
// shared memory at two CTAs per SM: the sweeps are chains of dependent steps,
// so the second CTA's warps hide latency.
#include <mutex>

#include "gdr2.h"
#include "gdr2_internal.cuh"

namespace gdr2 {
namespace {

constexpr int kNW = 8;            // warps per CTA
constexpr int kCPW = 4;           // value columns per warp
constexpr int kDVT = kNW * kCPW;  // value columns per CTA
constexpr int kCK = 4;            // tokens per checkpoint block
constexpr int kVec = 4;           // row vectors reduced over tiles: dq, G delta, dc, dlog_decay

struct BwdParams {
    const void *q, *k, *v, *b, *w, *g;
    const float *S0, *dO, *dST;
    float *dv, *dw, *dS0;
    float* ckpt;   // [B*H][tiles][blocks][DK * 32]; packed: [H][tiles][blk_stride][DK * 32]
    float* part;   // [token rows][H][tiles][kVec][DK]
    int64_t T;
    int H, dv_dim, tiles;
    // packed sequences (cu != null): sequence n owns rows cu[n] .. cu[n+1] - 1 of the
    // `total` token rows; its checkpoint blocks start at floor(cu[n] / kCK) + n
    const int* cu;
    int64_t total, blk_stride;
};

// Shared memory: the X_t stash of one block, its token inputs and two buffers of
// row-vector partials -- 106.5 KB at d_k = 128, so two CTAs share an SM.
template <int DK> constexpr size_t bwd_smem() {
    return sizeof(float) * (static_cast<size_t>(kCK) * DK * kDVT     // X_t stash
                            + 4 * kCK * DK                           // q, k, c, alpha
                            + 5 * kCK * kDVT                         // u, v, w, do, delta
                            + 2 * kNW * kVec * DK);                  // row-vector partials (two buffers)
}

template <typename Tin, int DK>
__global__ void __launch_bounds__(kNW * 32, 2) bwd_kernel(const BwdParams p) {
    constexpr int RPL = DK / 32;
    extern __shared__ __align__(16) float sm[];
    float* xs = sm;                                   // [kCK][kNW][RPL][kCPW][32]
    float* sq = xs + kCK * DK * kDVT;                 // [kCK][DK]
    float* sk = sq + kCK * DK;
    float* sc = sk + kCK * DK;
    float* sa = sc + kCK * DK;
    float* su = sa + kCK * DK;                        // [kCK][kDVT]
    float* sv = su + kCK * kDVT;
    float* sw = sv + kCK * kDVT;
    float* sdo = sw + kCK * kDVT;
    float* sdl = sdo + kCK * kDVT;                    // delta_t
    float* red = sdl + kCK * kDVT;                    // [2][kNW][kVec][DK]

    const Tin* q = static_cast<const Tin*>(p.q);
    const Tin* k = static_cast<const Tin*>(p.k);
    const Tin* v = static_cast<const Tin*>(p.v);
    const Tin* b = static_cast<const Tin*>(p.b);
    const Tin* w = static_cast<const Tin*>(p.w);
    const Tin* g = static_cast<const Tin*>(p.g);
    const int64_t bh = blockIdx.x;
    const int64_t seq = bh / p.H, h = bh % p.H;
    const int tile = blockIdx.y, j0 = tile * kDVT;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int cw = warp * kCPW;                       // first column of this warp in the tile
    int64_t T, tok0, ck_blk0;   // this sequence's rows and its first checkpoint block
    if (p.cu) {
        // offsets clamped into [0, total], the end to at least the start.  With
        // a <= e: floor(a / kCK) + ceil((e - a) / kCK) <= floor(e / kCK) + 1, so the
        // blocks of sequence n end at or before the first block of sequence n + 1 and
        // below floor(total / kCK) + N + 1 <= blk_stride, whatever the offsets are
        const int64_t a = min(max(static_cast<int64_t>(p.cu[seq]), static_cast<int64_t>(0)), p.total);
        const int64_t e = min(max(static_cast<int64_t>(p.cu[seq + 1]), a), p.total);
        T = e - a;
        tok0 = a;
        ck_blk0 = (h * p.tiles + tile) * p.blk_stride + a / kCK + seq;
    } else {
        T = p.T;
        tok0 = seq * T;
        ck_blk0 = (bh * p.tiles + tile) * ((T + kCK - 1) / kCK);
    }
    const int64_t nblk = (T + kCK - 1) / kCK;
    float* ck = p.ckpt + ck_blk0 * (DK * kDVT);

    // A block's token inputs: fetched into registers one block ahead (so the global
    // loads overlap the current block's arithmetic), then stored to shared memory.
    constexpr int NE = (kCK * DK + kNW * 32 - 1) / (kNW * 32);   // key-side elements per thread
    static_assert(kCK * kDVT <= kNW * 32, "at most one value-side element per thread");
    float fq[NE], fk[NE], fb[NE], fg[NE], fv, fw, fd;
    auto fetch = [&](int64_t t0, int n) {
#pragma unroll
        for (int u = 0; u < NE; ++u) {
            const int e = tid + u * kNW * 32, tt = e / DK, i = e % DK;
            fq[u] = fk[u] = fb[u] = fg[u] = 0.f;
            if (e < kCK * DK && tt < n) {
                const int64_t off = ((tok0 + t0 + tt) * p.H + h) * DK + i;
                fq[u] = to_f32(q[off]);
                fk[u] = to_f32(k[off]);
                fb[u] = to_f32(b[off]);
                fg[u] = to_f32(g[off]);
            }
        }
        const int tt = tid / kDVT, j = tid % kDVT;
        fv = fw = fd = 0.f;
        if (tid < kCK * kDVT && tt < n) {
            const int64_t off = ((tok0 + t0 + tt) * p.H + h) * p.dv_dim + j0 + j;
            fv = to_f32(v[off]);
            fw = to_f32(w[off]);
            fd = p.dO[off];
        }
    };
    auto stash = [&]() {
#pragma unroll
        for (int u = 0; u < NE; ++u) {
            const int e = tid + u * kNW * 32;
            if (e < kCK * DK) {
                sq[e] = fq[u];
                sk[e] = fk[u];
                sc[e] = fb[u] * fk[u];
                sa[e] = expf(fg[u]);
            }
        }
        if (tid < kCK * kDVT) {
            sv[tid] = fv;
            sw[tid] = fw;
            su[tid] = fw * fv;
            sdo[tid] = fd;
        }
    };
    // one forward step of token tt of the staged block: X = alpha * S, delta = u - X^T c,
    // S = X + k delta^T; X (optional) and delta are kept for the backward walk
    // Arithmetic runs on column pairs (packed f32x2 FMA / MUL, each lane rounded as its
    // scalar counterpart): S2[r][p] holds columns 2p, 2p+1 of row r.  The columns'
    // shuffle reductions run round by round together, so their latencies overlap, and
    // the token's per-row values are read into registers first (the stash stores could
    // otherwise force them to be reread for every column).
    constexpr int NP = kCPW / 2;
    auto dup = [](float a) { return make_float2(a, a); };
    auto fwd_step = [&](float2 (&S2)[RPL][NP], int tt, bool keep) {
        float2 x2[NP];
        float ar[RPL], cr[RPL], kr[RPL];
#pragma unroll
        for (int r = 0; r < RPL; ++r) {
            const int i = tt * DK + lane + 32 * r;
            ar[r] = sa[i];
            cr[r] = sc[i];
            kr[r] = sk[i];
        }
#pragma unroll
        for (int pp = 0; pp < NP; ++pp) x2[pp] = make_float2(0.f, 0.f);
#pragma unroll
        for (int r = 0; r < RPL; ++r)
#pragma unroll
            for (int pp = 0; pp < NP; ++pp) {
                const float2 X = __fmul2_rn(dup(ar[r]), S2[r][pp]);
                S2[r][pp] = X;
                x2[pp] = __ffma2_rn(dup(cr[r]), X, x2[pp]);
                if (keep) reinterpret_cast<float2*>(xs)[(((tt * kNW + warp) * RPL + r) * NP + pp) * 32 + lane] = X;
            }
#pragma unroll
        for (int s = 16; s > 0; s >>= 1)
#pragma unroll
            for (int pp = 0; pp < NP; ++pp)
                x2[pp] = __fadd2_rn(x2[pp], make_float2(__shfl_xor_sync(0xffffffffu, x2[pp].x, s),
                                                        __shfl_xor_sync(0xffffffffu, x2[pp].y, s)));
#pragma unroll
        for (int pp = 0; pp < NP; ++pp) {
            const float2 u2 = *reinterpret_cast<const float2*>(su + tt * kDVT + cw + 2 * pp);
            const float2 d2 = make_float2(u2.x - x2[pp].x, u2.y - x2[pp].y);
            if (keep && (lane >> 1) == pp) sdl[tt * kDVT + cw + lane] = (lane & 1) ? d2.y : d2.x;
#pragma unroll
            for (int r = 0; r < RPL; ++r) S2[r][pp] = __ffma2_rn(dup(kr[r]), d2, S2[r][pp]);
        }
    };
    auto ck_ptr = [&](int64_t blk, int r, int c) {
        return ck + blk * (DK * kDVT) + ((warp * RPL + r) * kCPW + c) * 32 + lane;
    };

    // ---- forward sweep: the tile at the start of every block ------------------------------
    float2 S2[RPL][NP];
#pragma unroll
    for (int r = 0; r < RPL; ++r)
#pragma unroll
        for (int pp = 0; pp < NP; ++pp) {
            const int64_t o = (bh * DK + lane + 32 * r) * p.dv_dim + j0 + cw + 2 * pp;
            S2[r][pp] = p.S0 ? make_float2(p.S0[o], p.S0[o + 1]) : make_float2(0.f, 0.f);
        }
    if (nblk > 1) fetch(0, kCK);
    for (int64_t blk = 0; blk < nblk; ++blk) {
#pragma unroll
        for (int r = 0; r < RPL; ++r)
#pragma unroll
            for (int pp = 0; pp < NP; ++pp) {
                *ck_ptr(blk, r, 2 * pp) = S2[r][pp].x;
                *ck_ptr(blk, r, 2 * pp + 1) = S2[r][pp].y;
            }
        if (blk + 1 == nblk) break;   // the last block is recomputed from its checkpoint
        __syncthreads();
        stash();
        __syncthreads();
        if (blk + 2 < nblk) fetch((blk + 1) * kCK, kCK);   // blocks before the last are full
        for (int tt = 0; tt < kCK; ++tt) fwd_step(S2, tt, false);
    }

    // ---- backward sweep ---------------------------------------------------------------------
    float2 G2[RPL][NP];
#pragma unroll
    for (int r = 0; r < RPL; ++r)
#pragma unroll
        for (int pp = 0; pp < NP; ++pp) {
            const int64_t o = (bh * DK + lane + 32 * r) * p.dv_dim + j0 + cw + 2 * pp;
            G2[r][pp] = p.dST ? make_float2(p.dST[o], p.dST[o + 1]) : make_float2(0.f, 0.f);
        }
    int buf = 0;
    if (nblk > 0) fetch((nblk - 1) * kCK, static_cast<int>(T - (nblk - 1) * kCK));
    for (int64_t blk = nblk - 1; blk >= 0; --blk) {
        const int64_t t0 = blk * kCK;
        const int n = static_cast<int>(T - t0 < kCK ? T - t0 : kCK);
        __syncthreads();
        stash();
        __syncthreads();
        if (blk > 0) fetch((blk - 1) * kCK, kCK);
#pragma unroll
        for (int r = 0; r < RPL; ++r)
#pragma unroll
            for (int pp = 0; pp < NP; ++pp) S2[r][pp] = make_float2(*ck_ptr(blk, r, 2 * pp), *ck_ptr(blk, r, 2 * pp + 1));
        for (int tt = 0; tt < n; ++tt) fwd_step(S2, tt, true);
        __syncwarp();
        for (int tt = n - 1; tt >= 0; --tt) {
            const int64_t row = tok0 + t0 + tt;
            float2 X2[RPL][NP], dl2[NP], do2[NP];
#pragma unroll
            for (int pp = 0; pp < NP; ++pp) {
                dl2[pp] = *reinterpret_cast<const float2*>(sdl + tt * kDVT + cw + 2 * pp);
                do2[pp] = *reinterpret_cast<const float2*>(sdo + tt * kDVT + cw + 2 * pp);
            }
            // per row: dq = S_t do and G delta over this warp's columns (two partial sums each)
            float pq[RPL], pk[RPL], pc[RPL], pg[RPL], kr[RPL];
#pragma unroll
            for (int r = 0; r < RPL; ++r) {
                const int i = tt * DK + lane + 32 * r;
                const float qi = sq[i], ki = sk[i];
                kr[r] = ki;
                float2 aq = make_float2(0.f, 0.f), ak = make_float2(0.f, 0.f);
#pragma unroll
                for (int pp = 0; pp < NP; ++pp) {
                    X2[r][pp] = reinterpret_cast<const float2*>(xs)[(((tt * kNW + warp) * RPL + r) * NP + pp) * 32 + lane];
                    const float2 St = __ffma2_rn(dup(ki), dl2[pp], X2[r][pp]);       // S_t
                    G2[r][pp] = __ffma2_rn(dup(qi), do2[pp], G2[r][pp]);             // + q_t do_t^T
                    aq = __ffma2_rn(St, do2[pp], aq);
                    ak = __ffma2_rn(G2[r][pp], dl2[pp], ak);
                }
                pq[r] = aq.x + aq.y;
                pk[r] = ak.x + ak.y;
            }
            float2 dd2[NP];   // ddelta = G^T k
#pragma unroll
            for (int pp = 0; pp < NP; ++pp) {
                dd2[pp] = make_float2(0.f, 0.f);
#pragma unroll
                for (int r = 0; r < RPL; ++r) dd2[pp] = __ffma2_rn(G2[r][pp], dup(kr[r]), dd2[pp]);
            }
#pragma unroll
            for (int s = 16; s > 0; s >>= 1)
#pragma unroll
                for (int pp = 0; pp < NP; ++pp)
                    dd2[pp] = __fadd2_rn(dd2[pp], make_float2(__shfl_xor_sync(0xffffffffu, dd2[pp].x, s),
                                                              __shfl_xor_sync(0xffffffffu, dd2[pp].y, s)));
            if (lane < kCPW) {
                const int c = lane;
                float ddc = 0.f;   // column c of ddelta (compile-time indices only)
#pragma unroll
                for (int pp = 0; pp < NP; ++pp) {
                    if (c == 2 * pp) ddc = dd2[pp].x;
                    if (c == 2 * pp + 1) ddc = dd2[pp].y;
                }
                const int64_t off = (row * p.H + h) * p.dv_dim + j0 + cw + c;
                p.dv[off] = ddc * sw[tt * kDVT + cw + c];
                p.dw[off] = ddc * sv[tt * kDVT + cw + c];
            }
            // per row: dc = -X ddelta, dlog_decay = rowsum(dX * X); G <- D_t dX
#pragma unroll
            for (int r = 0; r < RPL; ++r) {
                const int i = tt * DK + lane + 32 * r;
                const float ci = sc[i], ai = sa[i];
                float2 ac = make_float2(0.f, 0.f), ag = make_float2(0.f, 0.f);
#pragma unroll
                for (int pp = 0; pp < NP; ++pp) {
                    const float2 nX = make_float2(-X2[r][pp].x, -X2[r][pp].y);
                    ac = __ffma2_rn(nX, dd2[pp], ac);
                    const float2 dX = __ffma2_rn(dup(-ci), dd2[pp], G2[r][pp]);
                    ag = __ffma2_rn(dX, X2[r][pp], ag);
                    G2[r][pp] = __fmul2_rn(dup(ai), dX);                              // dS_{t-1}
                }
                pc[r] = ac.x + ac.y;
                pg[r] = ag.x + ag.y;
            }
            // row vectors: this warp's column partials -> shared memory -> sum over warps
            float* rb = red + buf * (kNW * kVec * DK);
#pragma unroll
            for (int r = 0; r < RPL; ++r) {
                const int i = lane + 32 * r;
                rb[(warp * kVec + 0) * DK + i] = pq[r];
                rb[(warp * kVec + 1) * DK + i] = pk[r];
                rb[(warp * kVec + 2) * DK + i] = pc[r];
                rb[(warp * kVec + 3) * DK + i] = pg[r];
            }
            __syncthreads();
            float* dst = p.part + ((row * p.H + h) * p.tiles + tile) * (kVec * DK);
            for (int e = tid; e < kVec * DK; e += kNW * 32) {
                float s = 0.f;
#pragma unroll
                for (int ww = 0; ww < kNW; ++ww) s += rb[ww * kVec * DK + e];
                dst[e] = s;
            }
            buf ^= 1;   // the other buffer takes the next token; this one is reread only
                        // after the next token's barrier
        }
    }
    if (p.dS0) {
#pragma unroll
        for (int r = 0; r < RPL; ++r)
#pragma unroll
            for (int pp = 0; pp < NP; ++pp) {
                const int64_t o = (bh * DK + lane + 32 * r) * p.dv_dim + j0 + cw + 2 * pp;
                p.dS0[o] = G2[r][pp].x;
                p.dS0[o + 1] = G2[r][pp].y;
            }
    }
}

// Packed sequences: whether token row `row` belongs to a sequence (offsets clamped
// as in bwd_kernel).  Valid offsets are non-decreasing, so the owner is the last
// sequence whose start is at or before the row; rows before the first start, after
// the last end or in no sequence are not written.  Malformed offsets only change
// which rows are written.
__device__ __forceinline__ bool row_in_sequence(const int* cu, int N, int64_t total, int64_t row) {
    auto start = [&](int n) { return min(max(static_cast<int64_t>(cu[n]), static_cast<int64_t>(0)), total); };
    if (N <= 0 || row < start(0)) return false;
    int lo = 0, hi = N;
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (start(mid) <= row) lo = mid; else hi = mid;
    }
    const int64_t a = start(lo);
    const int64_t e = min(max(static_cast<int64_t>(cu[lo + 1]), a), total);
    return row >= a && row < e;
}

// dq, dk, db, dlog_decay of one (token row, head) per DK threads: the tiles' row
// vectors summed, then db = dc * k and dk = G delta + dc * b.
template <typename Tin, int DK>
__global__ void __launch_bounds__(256) bwd_reduce_kernel(const float* __restrict__ part, const Tin* __restrict__ k,
                                                         const Tin* __restrict__ b, float* __restrict__ dq,
                                                         float* __restrict__ dk, float* __restrict__ db,
                                                         float* __restrict__ dg, int64_t items, int tiles,
                                                         const int* __restrict__ cu, int N, int64_t total, int H) {
    constexpr int kPer = 256 / DK;
    const int64_t item = static_cast<int64_t>(blockIdx.x) * kPer + threadIdx.x / DK;   // row * H + head
    const int j = threadIdx.x % DK;
    if (item >= items) return;
    if (cu && !row_in_sequence(cu, N, total, item / H)) return;
    const float* src = part + item * tiles * (kVec * DK) + j;
    float s[kVec] = {0.f, 0.f, 0.f, 0.f};
    for (int t = 0; t < tiles; ++t)
#pragma unroll
        for (int e = 0; e < kVec; ++e) s[e] += src[(t * kVec + e) * DK];
    const int64_t off = item * DK + j;
    const float kv = to_f32(k[off]), bv = to_f32(b[off]);
    dq[off] = s[0];
    db[off] = s[2] * kv;
    dk[off] = fmaf(s[2], bv, s[1]);
    dg[off] = s[3];
}

template <typename Tin, int DK>
int run_backward(const BwdParams& p, int64_t B, int64_t rows, const float* part, const void* k, const void* b,
                 float* dq, float* dk, float* db, float* dg, cudaStream_t stream) {
    static std::once_flag once;
    static cudaError_t attr = cudaSuccess;
    std::call_once(once, [] {
        attr = cudaFuncSetAttribute(bwd_kernel<Tin, DK>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    static_cast<int>(bwd_smem<DK>()));
    });
    if (attr != cudaSuccess) return GDR2_ERR_CUDA;
    const dim3 grid(static_cast<unsigned>(B * p.H), static_cast<unsigned>(p.tiles));
    bwd_kernel<Tin, DK><<<grid, kNW * 32, bwd_smem<DK>(), stream>>>(p);
    if (cudaPeekAtLastError() != cudaSuccess) return GDR2_ERR_CUDA;
    const int64_t items = rows * p.H;
    constexpr int kPer = 256 / DK;
    bwd_reduce_kernel<Tin, DK><<<static_cast<unsigned>((items + kPer - 1) / kPer), 256, 0, stream>>>(
        part, static_cast<const Tin*>(k), static_cast<const Tin*>(b), dq, dk, db, dg, items, p.tiles, p.cu,
        static_cast<int>(B), p.total, p.H);
    return cudaPeekAtLastError() == cudaSuccess ? GDR2_OK : GDR2_ERR_CUDA;
}

}  // namespace

namespace {
// checkpoint blocks per (sequence * head, tile), or per (head, tile) over all packed
// sequences (see bwd_kernel for why blocks from floor(start / kCK) + n fit)
int64_t ckpt_blocks(int64_t N, int64_t T, int64_t H, int64_t tiles, bool packed, int64_t total) {
    return packed ? H * tiles * (total / kCK + N + 2) : N * H * tiles * ((T + kCK - 1) / kCK);
}
}  // namespace

size_t backward_workspace_bytes(int64_t B, int64_t T, int64_t H, int64_t dk, int64_t dv, bool packed,
                                int64_t total) {
    const int64_t tiles = dv / kDVT, rows = packed ? total : B * T;
    const size_t ck = static_cast<size_t>(ckpt_blocks(B, T, H, tiles, packed, total)) * dk * kDVT * 4;
    const size_t part = static_cast<size_t>(rows * H * tiles) * kVec * dk * 4;
    return (ck + 255) / 256 * 256 + part;
}

int launch_backward(const BackwardArgs& a, void* ws, cudaStream_t stream) {
    if (a.dv % kDVT != 0 || a.B * a.H >= (1ll << 31) || a.dv / kDVT > 65535) return GDR2_ERR_SHAPE;
    const bool packed = a.cu != nullptr;
    const int64_t tiles = a.dv / kDVT, rows = packed ? a.total : a.B * a.T;
    const size_t ckb =
        (static_cast<size_t>(ckpt_blocks(a.B, a.T, a.H, tiles, packed, a.total)) * a.dk * kDVT * 4 + 255) / 256 * 256;
    BwdParams p{a.q, a.k, a.v, a.b, a.w, a.g, a.S0, a.dO, a.dST, a.d_v, a.d_w, a.d_S0,
                static_cast<float*>(ws), reinterpret_cast<float*>(static_cast<uint8_t*>(ws) + ckb),
                packed ? 0 : a.T, static_cast<int>(a.H), static_cast<int>(a.dv), static_cast<int>(tiles),
                a.cu, packed ? a.total : 0, packed ? a.total / kCK + a.B + 2 : 0};
    const bool bf = a.in_dtype == GDR2_BF16;
    using bf16 = __nv_bfloat16;
#define GDR2_BWD(DKV)                                                                                           \
    return bf ? run_backward<bf16, DKV>(p, a.B, rows, p.part, a.k, a.b, a.d_q, a.d_k, a.d_b, a.d_g, stream)    \
              : run_backward<float, DKV>(p, a.B, rows, p.part, a.k, a.b, a.d_q, a.d_k, a.d_b, a.d_g, stream)
    switch (a.dk) {
        case 32: GDR2_BWD(32);
        case 64: GDR2_BWD(64);
        case 128: GDR2_BWD(128);
        default: return GDR2_ERR_SHAPE;
    }
#undef GDR2_BWD
}

}  // namespace gdr2
