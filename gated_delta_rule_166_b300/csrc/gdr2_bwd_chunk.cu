// Chunked gradients of the Gated Delta Rule-2 prefill: bf16 inputs, d_k and d_v up to
// 128 (smaller head sizes on channels zero-padded to 128, as in the forward), tensor
// cores for every contraction; fixed-length batches or packed sequences.
//
// Method: reverse-mode differentiation of the chunkwise WY form of the "Gated
// DeltaNet-2: Decoupling Erase and Write in Linear Attention" page (update equation;
// "efficient implementation" section: WY form with decay absorption, chunkwise
// algorithm, gate-aware backward).  One 64-token chunk with start state S maps
//     E = T u - W S,     O = Qb S + A_qk E,     S' = diag(e^{G_C}) S + Kb^T E
// (Cb = c e^{G}, Qb = q e^{G}, Kb = k e^{G_C - G}, Kh = k e^{-G}, c = b k, u = w v,
// A_kk = strict_tril(Cb Kh^T), A_qk = tril(Qb Kh^T), T = (I + A_kk)^-1, W = T Cb).
// With dO the gradient at the chunk's outputs and dS' the one at S':
//     dE = A_qk^T dO + Kb dS'          dA_qk = tril(dO E^T)        dKb = E dS'^T
//     dW = -dE S^T                      du = T^T dE                 dT = dE u^T + dW Cb^T
//     dA_kk = strict_tril(-T^T dT T^T) = -strict_tril(du E^T)
//     dCb = T^T dW + dA_kk Kh,  dQb = dO S^T + dA_qk Kh,  dKh = dA_kk^T Cb + dA_qk^T Qb
// and, through the exponential factors, c = b k, u = w v and G's prefix sums,
//     dq = dQb e^{G},  dc = dCb e^{G},  db = dc k,  dk = dKb e^{G_C - G} + dKh e^{-G} + dc b,
//     dv = du w,  dw = du v,  dG = dc c + dq q - (dKb e^{G_C - G} + dKh e^{-G}) k,
//     dG_C += sum_r dKb_r Kb_r + e^{G_C} rowsum(dS' S),  dlog_decay = suffix sums of dG.
// Only dS crosses chunks:  dS = diag(e^{G_C}) dS' + M'^T dS' + P^T dO, the transpose of
// the forward chain's map S' = diag(e^{G_C}) S + M' S + Y U,  O = P S + X U.
//
// Kernels (after the forward's prep2, in its backward mode, and chain kernels have
// written the chunks' maps, backward records and start states):
//   rchain_kernel: one CTA per (sequence * head, 64-column d_v tile) carries dS from
//     the last chunk to the first on tcgen05 (M'^T and P^T are the forward slot's fp16
//     images read through MN-major descriptors; dO is an fp16 pair hi + lo), keeps the
//     gradient at every chunk's end state and writes dS0.
//   cgrad_kernel: one CTA per (chunk, head) forms all token gradients of the chunk from
//     its backward record (W^T, A_qk, T and Kb), S, dS' and dO:
//     - eleven fp16 products with fp32 accumulators in TMEM: E; then dA_qk, dKb, dE and
//       dO S^T; then dW and du; then du E^T and dW^T T.  dA_kk takes its one-product
//       form: T^T dW = -du S^T and T Cb = W give -T^T dT T^T = -du (T u)^T + du S^T W^T
//       = -du E^T, one rounding where the three-product form also rounds dT and dT T^T,
//       and no Cb.  dS', dO, u, dE, du and E enter as fp16 pairs hi + lo (a product
//       runs once per half);
//     - the decay-weighted products dA_kk Kh, dA_qk Kh and dKh on tf32 with the
//       stripe-referenced factors of the forward (e^{G_r - G_i} = e^{G_r - G_m}
//       e^{G_m - G_i}, m the middle token of a 16-token stripe; factors across stripes
//       are <= 1), the per-channel factors held in TMEM as the A operand (lane = key
//       channel);
//     - dG adds each token pair's product through dq q (or dc c) and subtracts it
//       through Y1 k; it multiplies those terms by the group factors exactly as the
//       MMAs saw them (rounded to tf32), so that a pair within a stripe enters both
//       sides as the same product and cancels.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <atomic>
#include <mutex>

#include "gdr2.h"
#include "gdr2_internal.cuh"
#include "gdr2_tc.cuh"

namespace gdr2 {
namespace {

using namespace tc;

constexpr int kC = kPrepC;
constexpr float kMinLogDecay = -10.f;   // the forward's floor of a per-token log decay

// ================================ reverse chain =====================================
namespace rch {
constexpr int kDVT = 64;
constexpr int kSimt = 512;
constexpr int kThreads = kSimt + 32;   // one more warp: lane 0 issues the copies and MMAs
// shared memory: two buffers of a chunk's M' (32 KB) and P (16 KB) images
constexpr uint32_t kBuf = 49152;
constexpr uint32_t kBM = 0, kBP = 32768;
constexpr uint32_t kSB = 2 * kBuf;     // two dS' operands, fp16 MN-major [128 K rows][64] (16 KB each)
constexpr uint32_t kUB = kSB + 32768;  // two [dO_hi^T | dO_lo^T] operands, fp16 K-major [64][64] x 2
constexpr uint32_t kMisc = kUB + 32768;
enum : uint32_t { kBarSlot0 = 0, kBarSlot1, kSRdy, kURdy0, kURdy1, kDS0, kDS1, kDrain, kNumBars };
constexpr uint32_t kTmemSlot = kMisc + 8 * kNumBars;
constexpr uint32_t kAbort = kTmemSlot + 4;
constexpr uint32_t kSmemBytes = kMisc + 128;
constexpr uint32_t kSmemAlloc = kSmemBytes + 1024;
static_assert(kAbort + 4 <= kSmemBytes && kSmemAlloc <= 232448, "shared memory");
constexpr int kTmCols = 256;   // per buffer b: 128 b + [0, 64) and + [64, 128), summed at read-out

struct Params {
    const uint8_t* slots;
    const float* dST;   // [B H][d_k][d_v] or null (zero)
    const float* dO;    // [token rows][H][d_v]
    float* dsn;         // [global chunk][H][d_k][d_v]: gradient at each chunk's end state
    float* dS0;         // [B H][d_k][d_v] or null
    int* err;
    int T, H, nch;
    long long wait_cycles;
    // packed sequences: token offsets [B + 1] and first global chunk of each sequence
    // (T and nch unused), or null
    const int* cu;
    const int* chunk_base;
    int total;
    int dk, dv;   // head sizes (up to 128; the state is zero-padded to 128 x 128 inside)
};

__global__ void __launch_bounds__(kThreads, 1) rchain_kernel(const Params prm) {
    const int bh = static_cast<int>(blockIdx.x);
    const int h = bh % prm.H, seq = bh / prm.H;
    const int j0 = static_cast<int>(blockIdx.y) * kDVT;
    // this sequence's token rows and its first global chunk (packed offsets clamped as
    // in the forward kernels)
    int n, T;
    int64_t tok0, chunk0;
    if (prm.cu) {
        const int a = min(max(prm.cu[seq], 0), prm.total);
        const int e = min(max(prm.cu[seq + 1], a), prm.total);
        // only the chunks this sequence was given (see chunk_base_kernel)
        T = static_cast<int>(min(static_cast<int64_t>(e - a),
                                     static_cast<int64_t>(prm.chunk_base[seq + 1] - prm.chunk_base[seq]) * kC));
        n = (T + kC - 1) / kC;
        tok0 = a;
        chunk0 = prm.chunk_base[seq];
    } else {
        T = prm.T;
        n = prm.nch;
        tok0 = static_cast<int64_t>(seq) * T;
        chunk0 = static_cast<int64_t>(seq) * n;
    }

    extern __shared__ uint8_t smem_raw[];
    const uint32_t base = (smem_u32(smem_raw) + 1023u) & ~1023u;
    uint8_t* sgen = smem_raw + (base - smem_u32(smem_raw));
    auto bar = [&](uint32_t i) { return base + kMisc + 8u * i; };
    volatile uint32_t* tmem_slot = reinterpret_cast<volatile uint32_t*>(sgen + kTmemSlot);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(sgen + kAbort);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, quarter = warp & 3;
    auto slot_of = [&](int c) {
        return prm.slots + ((chunk0 + c) * prm.H + h) * static_cast<int64_t>(kSlot2Bytes);
    };

    if (tid == 0) {
        for (uint32_t i = 0; i < kNumBars; ++i)
            mbar_init(bar(i), (i == kSRdy || i == kURdy0 || i == kURdy1) ? 16u : 1u);
        *abort_flag = 0;
        fence_mbar_init();
        fence_async_smem();
    }
    if (warp == 0) tmem_alloc<kTmCols>(base + kTmemSlot);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == kSimt / 32) {
        if (lane == 0) {
            // Step k handles chunk n - 1 - k in buffer k & 1: P^T [dO_hi; dO_lo]^T first
            // (issued a step ahead), then M'^T dS' once dS' is written; the slot buffer
            // takes chunk n - 3 - k when step k's products are done.
            uint32_t c_slot0 = 0, c_slot1 = 0, iss_slot0 = 0, iss_slot1 = 0;
            bool ok = true, issued = false;
            auto wait = [&](uint32_t b, uint32_t parity) {
                return mbar_wait_ab(bar(b), parity, abort_flag, prm.wait_cycles);
            };
            auto wait_slot = [&](uint32_t b) {
                uint32_t& cnt = b ? c_slot1 : c_slot0;
                const bool r = wait(kBarSlot0 + b, cnt & 1u);
                if (r) ++cnt;
                return r;
            };
            auto load_slot = [&](int k) {
                const uint32_t b = static_cast<uint32_t>(k & 1);
                const uint8_t* src = slot_of(n - 1 - k);
                mbar_expect_tx(bar(kBarSlot0 + b), kBuf);
                bulk_g2s(base + kBuf * b + kBM, src + kSlotM, 32768u, bar(kBarSlot0 + b));
                bulk_g2s(base + kBuf * b + kBP, src + kSlotP, 16384u, bar(kBarSlot0 + b));
                if (b) ++iss_slot1; else ++iss_slot0;
            };
            // M'^T: the K-major M' image read MN-major (its two 64-row K blocks are the MN
            // blocks, 16 KB apart); P^T likewise (8 KB apart).  A K step is 16 image rows.
            const uint64_t dMt0 = umma_desc2(base + kBM, 16384u, 1024u), dPt0 = umma_desc2(base + kBP, 8192u, 1024u);
            const uint64_t dS0d = umma_desc2(base + kSB, 16384u, 1024u), dU0 = umma_desc2(base + kUB, 16u, 1024u);
            constexpr uint32_t idC = idesc_f16x(128, 64, 0, 1, 1), idU = idesc_f16x(128, 128, 0, 1, 0);
            auto issue_do = [&](int k) {
                const uint32_t b = static_cast<uint32_t>(k & 1);
                const uint64_t dPt = dPt0 + (kBuf >> 4) * b, dU = dU0 + (16384u >> 4) * b;
                tc_fence_after();
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)
                    mma_ss_f16(tmem + 128u * b, dPt + 128u * kk, dU + 2u * kk, idU, kk > 0 ? 1u : 0u);
            };
            if (n > 0) {
                load_slot(0);
                if (n > 1) load_slot(1);
                ok = wait(kURdy0, 0u) && wait_slot(0u);
                if (ok) {
                    issue_do(0);
                    issued = true;
                }
            }
#pragma unroll 1
            for (int k = 0; k < n && ok; ++k) {
                const uint32_t b = static_cast<uint32_t>(k & 1);
                const uint64_t dMt = dMt0 + (kBuf >> 4) * b, dSd = dS0d + (16384u >> 4) * b;
                if (!(ok = wait(kSRdy, static_cast<uint32_t>(k) & 1u))) break;
                tc_fence_after();
                const uint32_t tS = tmem + 128u * b;
#pragma unroll
                for (int kk = 0; kk < 4; ++kk) {
                    mma_ss_f16(tS, dMt + 128u * kk, dSd + 128u * kk, idC, 1u);
                    mma_ss_f16(tS + 64u, dMt + 512u + 128u * kk, dSd + 512u + 128u * kk, idC, 1u);
                }
                mma_commit(bar(kDS0 + b));
                if (k + 1 < n) {
                    const uint32_t bn = b ^ 1u;
                    if (!(ok = wait(kURdy0 + bn, static_cast<uint32_t>((k + 1) >> 1) & 1u) && wait_slot(bn))) break;
                    issue_do(k + 1);
                }
                if (k + 2 < n) {
                    if (!(ok = wait(kDS0 + b, static_cast<uint32_t>(k >> 1) & 1u))) break;
                    load_slot(k + 2);
                }
            }
            if (!ok) {
                *abort_flag = 1;
                atomicExch(prm.err, kDevTimeout);
            }
            if (iss_slot0 > c_slot0) mbar_wait(bar(kBarSlot0), (iss_slot0 - 1u) & 1u);
            if (iss_slot1 > c_slot1) mbar_wait(bar(kBarSlot1), (iss_slot1 - 1u) & 1u);
            if (issued) {
                mma_commit(bar(kDrain));
                mbar_wait(bar(kDrain), 0u);
            }
        }
        __syncwarp();
    } else {
        const uint32_t lane_base = static_cast<uint32_t>(quarter * 32) << 16;
        const int R = warp >> 2;             // d_v columns j0 + 16 R .. + 15
        const int j = 32 * quarter + lane;   // state row (key channel)
        bool failed = false;
        auto arrive = [&](uint32_t b) {
            fence_async_smem();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(b));
        };
        auto put_st = [&](uint32_t buf, const float (&S)[16]) {
            uint8_t* img = sgen + kSB + 16384u * buf + static_cast<uint32_t>(j) * 128u;
            uint32_t w[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) w[e] = pack_h2(S[2 * e], S[2 * e + 1]);
#pragma unroll
            for (int q = 0; q < 2; ++q)
                *reinterpret_cast<uint4*>(img + ((static_cast<uint32_t>((2 * R + q) ^ (j & 7))) << 4)) =
                    make_uint4(w[4 * q], w[4 * q + 1], w[4 * q + 2], w[4 * q + 3]);
        };
        float* const dsn_row = prm.dsn + ((chunk0 * prm.H + h) * kPrepDK + j) * 128 + j0 + 16 * R;
        auto keep = [&](int c, const float (&S)[16]) {
            float* p = dsn_row + static_cast<int64_t>(c) * prm.H * kPrepDK * 128;
#pragma unroll
            for (int jj = 0; jj < 16; jj += 4)
                *reinterpret_cast<float4*>(p + jj) = make_float4(S[jj], S[jj + 1], S[jj + 2], S[jj + 3]);
        };
        // dO of chunk c for d_v column un, tokens 8 ug .. 8 ug + 7 (past the sequence end: 0)
        const int un = tid & 63, ug = tid >> 6;
        // (value columns past d_v read as zero)
        const int64_t rs = static_cast<int64_t>(prm.H) * prm.dv;
        const bool col_ok = j0 + un < prm.dv;
        const float* const dcol = prm.dO + (tok0 * prm.H + h) * prm.dv + (col_ok ? j0 + un : 0);
        auto fetch_do = [&](int c, float (&x)[8]) {
            const int t0 = c * kC + 8 * ug;
#pragma unroll
            for (int e = 0; e < 8; ++e) x[e] = col_ok && t0 + e < T ? __ldg(dcol + static_cast<int64_t>(t0 + e) * rs) : 0.f;
        };
        auto put_do = [&](int k, const float (&x)[8]) {
            uint4 hk, lk;
            __half2* hh = reinterpret_cast<__half2*>(&hk);
            __half2* lh = reinterpret_cast<__half2*>(&lk);
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const __half2 h2 = __floats2half2_rn(x[2 * e], x[2 * e + 1]);
                const float2 hf = __half22float2(h2);
                hh[e] = h2;
                lh[e] = __floats2half2_rn(x[2 * e] - hf.x, x[2 * e + 1] - hf.y);
            }
            uint8_t* ub = sgen + kUB + 16384u * static_cast<uint32_t>(k & 1);
            const uint32_t off = static_cast<uint32_t>(un) * 128u + ((static_cast<uint32_t>(ug) ^ (static_cast<uint32_t>(un) & 7u)) << 4);
            *reinterpret_cast<uint4*>(ub + off) = hk;
            *reinterpret_cast<uint4*>(ub + 8192u + off) = lk;
        };
        auto gamma_of = [&](int c) { return __ldg(reinterpret_cast<const float*>(slot_of(c) + kSlotGam) + j); };

        float S[16];
        {
            // d_S_T is [d_k][d_v]; rows past d_k and columns past d_v are zero padding
            const bool live = j < prm.dk && j0 + 16 * R < prm.dv;
            const float* s0 = prm.dST && live ? prm.dST + (static_cast<int64_t>(bh) * prm.dk + j) * prm.dv + j0 + 16 * R
                                              : nullptr;
#pragma unroll
            for (int jj = 0; jj < 16; jj += 4) {
                const float4 x = s0 ? *reinterpret_cast<const float4*>(s0 + jj) : make_float4(0.f, 0.f, 0.f, 0.f);
                S[jj] = x.x; S[jj + 1] = x.y; S[jj + 2] = x.z; S[jj + 3] = x.w;
            }
        }
        float xpre[8];
        float gam_next = n > 0 ? gamma_of(n - 1) : 1.f;
        if (n > 0) {
            keep(n - 1, S);
            put_st(0, S);
            arrive(kSRdy);
            fetch_do(n - 1, xpre);
            put_do(0, xpre);
            arrive(kURdy0);
            if (n > 1) {
                fetch_do(n - 2, xpre);
                put_do(1, xpre);
                arrive(kURdy1);
            }
            if (n > 2) fetch_do(n - 3, xpre);
        }
#pragma unroll 1
        for (int k = 0; k < n; ++k) {
            const uint32_t b = static_cast<uint32_t>(k & 1);
            const int c = n - 1 - k;
            const float gam = gam_next;
            if (k + 1 < n) gam_next = gamma_of(c - 1);
            if (!mbar_wait_ab(bar(kDS0 + b), static_cast<uint32_t>(k >> 1) & 1u, abort_flag, prm.wait_cycles)) {
                failed = true;
                break;
            }
            tc_fence_after();
            {
                float v[16];
                tmem_ld16_pair(tmem + lane_base + 128u * b + static_cast<uint32_t>(16 * R), v);
#pragma unroll
                for (int jj = 0; jj < 16; ++jj) S[jj] = fmaf(gam, S[jj], v[jj]);
            }
            if (k + 1 < n) {
                put_st(b ^ 1u, S);
                arrive(kSRdy);
                keep(c - 1, S);   // after the next chunk's operand is released
            }
            if (k + 2 < n) {
                put_do(k + 2, xpre);
                arrive(kURdy0 + b);
                if (k + 3 < n) fetch_do(c - 3, xpre);
            }
        }
        if (failed) {
            *abort_flag = 1;
            if (lane == 0) atomicExch(prm.err, kDevTimeout);
        } else if (prm.dS0 && j < prm.dk && j0 + 16 * R < prm.dv) {
            float* p = prm.dS0 + (static_cast<int64_t>(bh) * prm.dk + j) * prm.dv + j0 + 16 * R;
#pragma unroll
            for (int jj = 0; jj < 16; jj += 4)
                *reinterpret_cast<float4*>(p + jj) = make_float4(S[jj], S[jj + 1], S[jj + 2], S[jj + 3]);
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc<kTmCols>(tmem);
    }
}
}  // namespace rch

// ============================== chunk gradients ======================================
namespace cgr {
constexpr int kThreads = 512;
// ---- shared memory (bytes from a 1024-aligned base); fp16 images are 128-byte
// swizzled rows of 64 elements ("[rows][cols]": rows written by one thread each) ----
constexpr uint32_t kWt = 0, kAq = 16384, kT = 24576, kKb = 32768;   // the backward record (48 KB)
static_assert(kWt == kWyWt && kAq == kWyAq && kT == kWyT && kKb == kWyKb, "record layout");
constexpr uint32_t kdWt = kWt;            // dW^T [d_k][token] (after W^T is consumed)
constexpr uint32_t kScr = kAq;            // cross-warp sums, 2 x [4][128] fp32 (after A_qk)
constexpr uint32_t kdEtL = kKb;           // low half of dE^T (after Kb), then
constexpr uint32_t kdUt = kKb;            // du^T [d_v][token]
constexpr uint32_t kEtL = kKb + 16384;    // low half of E^T (the record ends at kKb + 16 KB)
constexpr uint32_t kS = 65536;            // S [d_k][d_v], two 64-column blocks 16 KB apart
constexpr uint32_t kdS = 98304;           // dS' [d_k][d_v]
constexpr uint32_t kRaw = kS;             // bf16 [token][128] tiles q, k, b, log decay (after S, dS')
constexpr uint32_t kdO = 131072;          // dO [token][d_v], two blocks 8 KB apart
constexpr uint32_t kU = 147456;           // u = w v [token][d_v]
constexpr uint32_t kG = kdO;              // G [token][d_k] fp32 (after dO, u)
constexpr uint32_t kEt = 163840;          // E^T [d_v][token]
constexpr uint32_t kdEt = 180224;         // dE^T [d_v][token]
constexpr uint32_t kAkk = kEt, kAkkT = kdEt;   // dA_kk [r][i], [i][r] tf32 (after E^T, dE^T)
constexpr uint32_t kAqk = 196608, kAqkT = 212992;   // dA_qk [r][i], [i][r] tf32
// Per-warp 2 KB transpose buffers for the token-gradient stores: during the third
// phase's read-out (where dO and u were), and from the fourth phase on (where T and
// du^T were)
constexpr uint32_t kXpA = kdO, kXpB = kT;
// Low halves x - fp16(x) of the pairs dS', dO and u (read by the first products only),
// in regions whose own contents are written after those products complete; du's low
// half where dE^T was (read by the fourth phase, before dA_kk^T is written there)
constexpr uint32_t kdSL = kAqk, kdOL = kdEt, kUL = kEt, kdUtL = kdEt;
constexpr uint32_t kMisc = 229376;
enum : uint32_t { kBarLd = 0, kBarMma, kBarDrain, kNumBars };
constexpr uint32_t kTmemSlot = kMisc + 8 * kNumBars;
constexpr uint32_t kGsum = kMisc + 64;    // rowsum(dS' * S) [d_k] fp32
constexpr uint32_t kSmemBytes = kGsum + 512;
constexpr uint32_t kSmemAlloc = kSmemBytes + 1024;
static_assert(kTmemSlot + 4 <= kGsum && kSmemAlloc <= 232448, "shared memory");
static_assert(kXpA + 16 * 2048 <= kEt && kXpB + 16 * 2048 <= kS && kXpB >= kScr + 8192, "transpose buffers");
static_assert(kEtL + 16384 <= kS && kEtL >= kKb + 16384, "low half of E^T");
// ---- TMEM columns (M = 128 accumulators: lane = row; M = 64: row r at lane 32 (r / 16) + r % 16) ----
constexpr uint32_t kTmEa = 0, kTmEb = 64;                              // u^T T^T, S^T W^T
constexpr uint32_t kTmAqk = 128, kTmKb = 192, kTmdE = 256, kTmQb = 320;   // dO E^T, dS' E^T, dE^T, S dO^T
constexpr uint32_t kTmdW = 0, kTmdu = 64;                              // S dE^T = -dW^T, du^T
constexpr uint32_t kTmAkk = 128, kTmCb0 = 256;                         // du E^T (= -dA_kk below the diagonal), dW^T T
constexpr uint32_t kTmX1 = 128, kTmX2 = 32;                            // dA_kk / dA_qk x K-groups (N = 16 per stripe)
__device__ __forceinline__ uint32_t col_kg(int R) { return R == 0 ? 496u : R == 1 ? 0u : R == 2 ? 448u : 384u; }
constexpr uint32_t kTmY = 320;                                         // C-, Q-groups x dA^T
__device__ __forceinline__ uint32_t col_cg(int s) { return s == 0 ? 0u : s == 1 ? 64u : s == 2 ? 112u : 144u; }
constexpr uint32_t kQgOff = 160;
constexpr int kTmCols = 512;

struct Params {
    const uint8_t* wy;          // backward records [items][kWyBytes]
    const float* Sc;            // state after chunk c (c < n_cache): [B H][n_cache][d_k][d_v];
                                // packed: after every global chunk, [global chunk][H][d_k][d_v]
    const float* S0;            // [B H][d_k][d_v] or null
    const float* dsn;           // [global chunk][H][d_k][d_v]
    const float* dO;            // [token rows][H][d_v]
    const __nv_bfloat16 *q, *k, *b, *g, *v, *w;
    float *dq, *dk, *db, *dg, *dv, *dw;
    int T, H, nch, n_cache;
    int* err;
    // packed sequences: token offsets [N + 1] and first global chunk of each sequence
    // (T, nch and n_cache unused), or null; the grid may hold items past the last chunk
    const int* cu;
    const int* chunk_base;
    int N, total;
    // items in the grid, and the item distance to the one that runs on this SM next
    // (the resident CTAs: one per SM); 0 turns the L2 prefetch of that item off
    int items, pf_stride;
    // head sizes (up to 128): token rows are kdim or vdim wide, the states S0 and Sc
    // are [kdim][vdim]; inside, every operand is zero-padded to 128 channels
    int kdim, vdim;
};

// Item `it` = (global chunk gc, head h): its sequence, chunk within the sequence,
// token rows inside the sequence and first token row; false past the last chunk.
struct CgItem {
    int h, seq, c, nvalid;
    int64_t row0;
};
__device__ __forceinline__ bool cg_locate(const Params& prm, int it, CgItem& x) {
    const int gc = it / prm.H;
    x.h = it - gc * prm.H;
    if (prm.cu) {
        // packed sequences: the last sequence whose first global chunk is at or before gc
        // (offsets clamped as in the forward kernels)
        const int* cbs = prm.chunk_base;
        if (gc >= cbs[prm.N]) return false;
        int lo = 0, hi = prm.N;
        while (hi - lo > 1) {
            const int mid = (lo + hi) >> 1;
            if (cbs[mid] <= gc) lo = mid; else hi = mid;
        }
        x.seq = lo;
        x.c = gc - cbs[lo];
        const int a = min(max(prm.cu[lo], 0), prm.total);
        const int e = min(max(prm.cu[lo + 1], a), prm.total);
        x.nvalid = min(e - a - x.c * kC, kC);
        x.row0 = static_cast<int64_t>(a) + static_cast<int64_t>(x.c) * kC;
    } else {
        x.seq = gc / prm.nch;
        x.c = gc - x.seq * prm.nch;
        x.nvalid = min(prm.T - x.c * kC, kC);
        x.row0 = static_cast<int64_t>(x.seq) * prm.T + static_cast<int64_t>(x.c) * kC;
    }
    return true;
}
// The item's start state ([d_k][d_v], st = d_k d_v floats; null: zero), as the load
// phase reads it.
__device__ __forceinline__ const float* cg_start_state(const Params& prm, int it, const CgItem& x, int64_t st) {
    const int64_t bh = static_cast<int64_t>(x.seq) * prm.H + x.h;
    return x.c == 0  ? (prm.S0 ? prm.S0 + bh * st : nullptr)
           : prm.cu ? prm.Sc + (static_cast<int64_t>(it) - prm.H) * st   // global chunk gc - 1
                    : prm.Sc + (bh * prm.n_cache + (x.c - 1)) * st;
}

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, uint32_t src_bytes) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(src_bytes) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }
__device__ __forceinline__ float bf(uint16_t x) { return __uint_as_float(static_cast<uint32_t>(x) << 16); }

// 16 values as two 16-byte pieces of row `row`, columns k0 .. k0 + 15, of an fp16 image
__device__ __forceinline__ void put16(uint8_t* img, uint32_t kblk, uint32_t row, uint32_t k0, const float (&v)[16]) {
    uint32_t w[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) w[e] = pack_h2(v[2 * e], v[2 * e + 1]);
    *reinterpret_cast<uint4*>(img + k_off16(kblk, row, k0)) = make_uint4(w[0], w[1], w[2], w[3]);
    *reinterpret_cast<uint4*>(img + k_off16(kblk, row, k0 + 8u)) = make_uint4(w[4], w[5], w[6], w[7]);
}

// Lane l of a warp holds one key / value channel (a0 + l) at 16 tokens r0 .. r0 + 15;
// the warp writes them to its 2 KB buffer and reads them back as 4 channels of one
// token, so that each global store moves 16 bytes (8 lanes: one token's 32 channels)
// instead of 4.  Rows at or past `nvalid` and channels at or past `width` (the row
// width of `out`, a multiple of 32) are not stored.
__device__ __forceinline__ void store_tokens(float* buf, const float (&v)[16], float* out, int64_t row0, int H,
                                             int h, int a0, int r0, int nvalid, int lane, int width) {
#pragma unroll
    for (int t = 0; t < 16; ++t) buf[t * 32 + lane] = v[t];
    __syncwarp();
#pragma unroll
    for (int s4 = 0; s4 < 4; ++s4) {
        const int t = 4 * s4 + (lane >> 3), c4 = 4 * (lane & 7);
        const float4 x = *reinterpret_cast<const float4*>(buf + t * 32 + c4);
        if (r0 + t < nvalid && a0 < width)
            *reinterpret_cast<float4*>(out + ((row0 + r0 + t) * H + h) * width + a0 + c4) = x;
    }
    __syncwarp();
}

// 16 values as an fp16 pair x = hi + lo (about 22 significant bits) in two images
__device__ __forceinline__ void put16_pair(uint8_t* hi, uint8_t* lo, uint32_t kblk, uint32_t row, uint32_t k0,
                                           const float (&v)[16]) {
    float h[16], l[16];
#pragma unroll
    for (int e = 0; e < 16; ++e) {
        h[e] = __half2float(__float2half_rn(v[e]));
        l[e] = v[e] - h[e];
    }
    put16(hi, kblk, row, k0, h);
    put16(lo, kblk, row, k0, l);
}

// kPad: head sizes below 128 (zero-padded channels); the d_k = d_v = 128 instantiation
// keeps compile-time row strides and no channel guards.
template <bool kPad>
__global__ void __launch_bounds__(kThreads, 1) cgrad_kernel(const Params prm) {
    const int kdim = kPad ? prm.kdim : 128, vdim = kPad ? prm.vdim : 128;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t base = (smem_u32(smem_raw) + 1023u) & ~1023u;
    uint8_t* sgen = smem_raw + (base - smem_u32(smem_raw));
    auto bar = [&](uint32_t i) { return base + kMisc + 8u * i; };
    volatile uint32_t* tmem_slot = reinterpret_cast<volatile uint32_t*>(sgen + kTmemSlot);
    float* const gsum = reinterpret_cast<float*>(sgen + kGsum);
    float* const scr = reinterpret_cast<float*>(sgen + kScr);
    const float* const Gt = reinterpret_cast<const float*>(sgen + kG);
    const uint16_t* const raw = reinterpret_cast<const uint16_t*>(sgen + kRaw);   // [4][64][128]
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, quarter = warp & 3, cb = warp >> 2;
    const uint32_t lane_base = static_cast<uint32_t>(quarter * 32) << 16;
    const int a = 32 * quarter + lane;   // M = 128 accumulator row (key channel or d_v column)

    const int it = static_cast<int>(blockIdx.x);
    CgItem item;
    if (!cg_locate(prm, it, item)) return;   // packed: past the last chunk (the grid is a bound)
    const int h = item.h, seq = item.seq, c = item.c, nvalid = item.nvalid;
    const int64_t row0 = item.row0;   // first token row of the chunk
    const int bh = seq * prm.H + h;
    // element index of channel ch of token r in a key-side (dk wide) or value-side row
    auto kidx = [&](int r, int ch) { return ((row0 + r) * prm.H + h) * kdim + ch; };
    auto vidx = [&](int r, int ch) { return ((row0 + r) * prm.H + h) * vdim + ch; };

    if (tid == 0) {
        for (uint32_t i = 0; i < kNumBars; ++i) mbar_init(bar(i), 1);
        fence_mbar_init();
    }
    if (warp == 0) tmem_alloc<kTmCols>(base + kTmemSlot);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    if (tid == 0) {
        mbar_expect_tx(bar(kBarLd), kWyBytes);
        bulk_g2s(base, prm.wy + static_cast<int64_t>(it) * kWyBytes, kWyBytes, bar(kBarLd));
    }
    bool ok = true;
    uint32_t ph = 0;
    auto wait_mma = [&]() {
        ok = mbar_wait(bar(kBarMma), ph) && ok;
        ph ^= 1u;
        tc_fence_after();
    };
    auto operands_done = [&]() {
        fence_async_smem();
        tc_fence_before();
        __syncthreads();
        tc_fence_after();
    };

    // ---- S, dS' -> fp16 images [d_k][d_v]; rowsum(dS' * S) ----------------------------------
    {
        const float* Sp = cg_start_state(prm, it, item, static_cast<int64_t>(kdim) * vdim);
        const float* dSp = prm.dsn + static_cast<int64_t>(it) * 16384;   // global chunk gc, head h
        const int r = tid >> 2, e0 = 32 * (tid & 3);
        float part = 0.f;
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
            const int e = e0 + 16 * hh;
            float sv[16], dv[16];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const float4 x = Sp && r < kdim && e < vdim
                                     ? __ldg(reinterpret_cast<const float4*>(Sp + r * vdim + e) + u)
                                     : make_float4(0.f, 0.f, 0.f, 0.f);
                const float4 y = __ldg(reinterpret_cast<const float4*>(dSp + r * 128 + e) + u);
                sv[4 * u] = x.x; sv[4 * u + 1] = x.y; sv[4 * u + 2] = x.z; sv[4 * u + 3] = x.w;
                dv[4 * u] = y.x; dv[4 * u + 1] = y.y; dv[4 * u + 2] = y.z; dv[4 * u + 3] = y.w;
            }
#pragma unroll
            for (int jj = 0; jj < 16; ++jj) part = fmaf(sv[jj], dv[jj], part);
            put16(sgen + kS, 16384u, static_cast<uint32_t>(r), static_cast<uint32_t>(e), sv);
            put16_pair(sgen + kdS, sgen + kdSL, 16384u, static_cast<uint32_t>(r), static_cast<uint32_t>(e), dv);
        }
        part += __shfl_xor_sync(0xffffffffu, part, 1);
        part += __shfl_xor_sync(0xffffffffu, part, 2);
        if ((tid & 3) == 0) gsum[r] = part;
    }
    // ---- dO and u = w v -> fp16 images [token][d_v] (tokens past the sequence end: 0) --------
    {
        const int r = tid >> 3, e = 16 * (tid & 7);
        const bool valid = r < nvalid && e < vdim;   // value columns past d_v: zero
        float ov[16], uv[16];
        if (valid) {
            const int64_t gi = vidx(r, e);
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const float4 x = __ldg(reinterpret_cast<const float4*>(prm.dO + gi) + u);
                ov[4 * u] = x.x; ov[4 * u + 1] = x.y; ov[4 * u + 2] = x.z; ov[4 * u + 3] = x.w;
            }
            const uint4* pv = reinterpret_cast<const uint4*>(prm.v + gi);
            const uint4* pw = reinterpret_cast<const uint4*>(prm.w + gi);
#pragma unroll
            for (int u = 0; u < 2; ++u) {
                const uint4 xv = __ldg(pv + u), xw = __ldg(pw + u);
                const uint32_t wv[4] = {xv.x, xv.y, xv.z, xv.w}, ww[4] = {xw.x, xw.y, xw.z, xw.w};
#pragma unroll
                for (int e2 = 0; e2 < 4; ++e2) {
                    uv[8 * u + 2 * e2] = __uint_as_float(wv[e2] << 16) * __uint_as_float(ww[e2] << 16);
                    uv[8 * u + 2 * e2 + 1] = __uint_as_float(wv[e2] & 0xFFFF0000u) * __uint_as_float(ww[e2] & 0xFFFF0000u);
                }
            }
        } else {
#pragma unroll
            for (int jj = 0; jj < 16; ++jj) ov[jj] = uv[jj] = 0.f;
        }
        put16_pair(sgen + kdO, sgen + kdOL, 8192u, static_cast<uint32_t>(r), static_cast<uint32_t>(e), ov);
        put16_pair(sgen + kU, sgen + kUL, 8192u, static_cast<uint32_t>(r), static_cast<uint32_t>(e), uv);
    }
    operands_done();

    // The item the next CTA on this SM will take is not in flight yet: one thread asks L2
    // for its three contiguous inputs (backward record, start state, end-state gradient:
    // 176 of its 320 KB) now, while this item's products and epilogues leave DRAM idle, so
    // that its load phase finds them in L2 instead of every SM loading from DRAM at once.
    // (The token rows, 64 strided 256- and 512-byte pieces each, are left to the load
    // phase: prefetching them too, as bulk or as line prefetches, measured slower.)
    if (tid == 32 && prm.pf_stride > 0 && it + prm.pf_stride < prm.items) {
        const int nit = it + prm.pf_stride;
        CgItem nx;
        if (cg_locate(prm, nit, nx)) {
            bulk_prefetch_l2(prm.wy + static_cast<int64_t>(nit) * kWyBytes, kWyBytes);
            if (const float* ns = cg_start_state(prm, nit, nx, static_cast<int64_t>(kdim) * vdim))
                bulk_prefetch_l2(ns, static_cast<uint32_t>(kdim * vdim * 4));
            bulk_prefetch_l2(prm.dsn + static_cast<int64_t>(nit) * 16384, 65536u);
        }
    }

    // ---- 1. E^T = u^T T^T - S^T W^T  [d_v][token] ---------------------------------------------
    if (tid == 0) {
        ok = mbar_wait(bar(kBarLd), 0u) && ok;
        tc_fence_after();
        const uint64_t dUm = umma_desc2(base + kU, 8192u, 1024u), dTk = umma_desc2(base + kT, 16u, 1024u);
        const uint64_t dULm = umma_desc2(base + kUL, 8192u, 1024u);
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
            mma_ss_f16(tmem + kTmEa, dUm + 128u * kk, dTk + 2u * kk, idesc_f16x(128, 64, 0, 1, 0), kk > 0);
            mma_ss_f16(tmem + kTmEa, dULm + 128u * kk, dTk + 2u * kk, idesc_f16x(128, 64, 0, 1, 0), 1u);
        }
        const uint64_t dSm = umma_desc2(base + kS, 16384u, 1024u), dWm = umma_desc2(base + kWt, 8192u, 1024u);
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) mma_ss_f16(tmem + kTmEb, dSm + 128u * kk, dWm + 128u * kk, idesc_f16x(128, 64, 0, 1, 1), kk > 0);
        mma_commit(bar(kBarMma));
    }
    wait_mma();
    {
        float ea[16], eb[16];
        tmem_ld16(tmem + lane_base + kTmEa + 16u * cb, ea);
        tmem_ld16(tmem + lane_base + kTmEb + 16u * cb, eb);
#pragma unroll
        for (int jj = 0; jj < 16; ++jj) ea[jj] -= eb[jj];
        put16_pair(sgen + kEt, sgen + kEtL, 0u, static_cast<uint32_t>(a), 16u * cb, ea);
    }
    operands_done();

    // ---- 2. dA_qk = dO E^T, dKb^T = dS' E^T, dE^T = dO^T A_qk + dS'^T Kb^T, dQb0^T = S dO^T ------
    if (tid == 0) {
        // dO, dS' and E as hi + lo pairs: each product runs once per half of dO / dS',
        // plus once with E's low half and the high half of dO / dS'
        const uint64_t dEm = umma_desc2(base + kEt, 8192u, 1024u), dSk0 = umma_desc2(base + kS, 16u, 1024u);
        {
            const uint64_t dELm = umma_desc2(base + kEtL, 8192u, 1024u);
            const uint64_t dOk = umma_desc2(base + kdO, 16u, 1024u), dSk = umma_desc2(base + kdS, 16u, 1024u);
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) {
                const uint32_t ko = kk < 4 ? 2u * kk : (8192u >> 4) + 2u * (kk - 4);
                const uint32_t ks = kk < 4 ? 2u * kk : (16384u >> 4) + 2u * (kk - 4);
                mma_ss_f16(tmem + kTmAqk, dOk + ko, dELm + 128u * kk, idesc_f16x(64, 64, 0, 0, 1), kk > 0);
                mma_ss_f16(tmem + kTmKb, dSk + ks, dELm + 128u * kk, idesc_f16x(128, 64, 0, 0, 1), kk > 0);
            }
        }
        const uint64_t dKk = umma_desc2(base + kKb, 16u, 1024u), dAm = umma_desc2(base + kAq, 8192u, 1024u);
#pragma unroll
        for (int half = 0; half < 2; ++half) {
            const uint64_t dOk = umma_desc2(base + (half ? kdOL : kdO), 16u, 1024u);
            const uint64_t dSk = umma_desc2(base + (half ? kdSL : kdS), 16u, 1024u);
            const uint64_t dOm = umma_desc2(base + (half ? kdOL : kdO), 8192u, 1024u);
            const uint64_t dSm = umma_desc2(base + (half ? kdSL : kdS), 16384u, 1024u);
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) {
                const uint32_t ko = kk < 4 ? 2u * kk : (8192u >> 4) + 2u * (kk - 4);
                const uint32_t ks = kk < 4 ? 2u * kk : (16384u >> 4) + 2u * (kk - 4);
                const uint32_t acc = half > 0 || kk > 0;
                mma_ss_f16(tmem + kTmAqk, dOk + ko, dEm + 128u * kk, idesc_f16x(64, 64, 0, 0, 1), 1u);
                mma_ss_f16(tmem + kTmKb, dSk + ks, dEm + 128u * kk, idesc_f16x(128, 64, 0, 0, 1), 1u);
                mma_ss_f16(tmem + kTmQb, dSk0 + ks, dOk + ko, idesc_f16x(128, 64, 0, 0, 0), acc);
            }
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
                mma_ss_f16(tmem + kTmdE, dOm + 128u * kk, dAm + 128u * kk, idesc_f16x(128, 64, 0, 1, 1), half > 0 || kk > 0);
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) {
                const uint32_t ko = kk < 4 ? 2u * kk : (8192u >> 4) + 2u * (kk - 4);
                mma_ss_f16(tmem + kTmdE, dSm + 128u * kk, dKk + ko, idesc_f16x(128, 64, 0, 1, 0), 1u);
            }
        }
        mma_commit(bar(kBarMma));
    }
    wait_mma();
    {
        float v[16];
        tmem_ld16(tmem + lane_base + kTmAqk + 16u * cb, v);
        if (lane < 16) {
            const int r = 16 * quarter + lane;
            float t[16];
#pragma unroll
            for (int jj = 0; jj < 16; ++jj) t[jj] = 16 * cb + jj <= r ? tf32r(v[jj]) : 0.f;
#pragma unroll
            for (int u = 0; u < 4; ++u)
                *reinterpret_cast<float4*>(sgen + kAqk + sw(8192u, r, 16u * cb + 4u * u)) =
                    make_float4(t[4 * u], t[4 * u + 1], t[4 * u + 2], t[4 * u + 3]);
#pragma unroll
            for (int jj = 0; jj < 16; ++jj)
                *reinterpret_cast<float*>(sgen + kAqkT + sw(8192u, 16u * cb + jj, static_cast<uint32_t>(r))) = t[jj];
        }
        tmem_ld16(tmem + lane_base + kTmdE + 16u * cb, v);
        put16_pair(sgen + kdEt, sgen + kdEtL, 0u, static_cast<uint32_t>(a), 16u * cb, v);
    }
    operands_done();

    // ---- 3. -dW^T = S dE^T, du^T = dE^T T  ------------------------------------------------------
    if (tid == 0) {
        const uint64_t dSk0 = umma_desc2(base + kS, 16u, 1024u), dTm = umma_desc2(base + kT, 8192u, 1024u);
#pragma unroll
        for (int half = 0; half < 2; ++half) {   // dE^T as hi + lo
            const uint64_t dEm = umma_desc2(base + (half ? kdEtL : kdEt), 8192u, 1024u);
            const uint64_t dEk = umma_desc2(base + (half ? kdEtL : kdEt), 16u, 1024u);
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) {
                const uint32_t ks = kk < 4 ? 2u * kk : (16384u >> 4) + 2u * (kk - 4);
                mma_ss_f16(tmem + kTmdW, dSk0 + ks, dEm + 128u * kk, idesc_f16x(128, 64, 0, 0, 1), half > 0 || kk > 0);
            }
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
                mma_ss_f16(tmem + kTmdu, dEk + 2u * kk, dTm + 128u * kk, idesc_f16x(128, 64, 0, 0, 1), half > 0 || kk > 0);
        }
        mma_commit(bar(kBarMma));
    }
    {
        // v, w of this thread's d_v column, fetched while the products run
        uint16_t vb[16], wb[16];
#pragma unroll
        for (int jj = 0; jj < 16; ++jj) {
            const int r = 16 * cb + jj;
            const bool valid = r < nvalid && a < vdim;
            const int64_t gi = valid ? vidx(r, a) : 0;
            vb[jj] = valid ? __ldg(reinterpret_cast<const unsigned short*>(prm.v) + gi) : 0;
            wb[jj] = valid ? __ldg(reinterpret_cast<const unsigned short*>(prm.w) + gi) : 0;
        }
        wait_mma();
        float v[16];
        tmem_ld16(tmem + lane_base + kTmdW + 16u * cb, v);
#pragma unroll
        for (int jj = 0; jj < 16; ++jj) v[jj] = -v[jj];
        put16(sgen + kdWt, 0u, static_cast<uint32_t>(a), 16u * cb, v);
        tmem_ld16(tmem + lane_base + kTmdu + 16u * cb, v);
        {
            float* xb = reinterpret_cast<float*>(sgen + kXpA) + warp * 512;
            float t[16];
#pragma unroll
            for (int jj = 0; jj < 16; ++jj) t[jj] = v[jj] * bf(wb[jj]);
            store_tokens(xb, t, prm.dv, row0, prm.H, h, 32 * quarter, 16 * cb, nvalid, lane, vdim);
#pragma unroll
            for (int jj = 0; jj < 16; ++jj) t[jj] = v[jj] * bf(vb[jj]);
            store_tokens(xb, t, prm.dw, row0, prm.H, h, 32 * quarter, 16 * cb, nvalid, lane, vdim);
        }
        put16_pair(sgen + kdUt, sgen + kdUtL, 0u, static_cast<uint32_t>(a), 16u * cb, v);
    }
    // raw q, k, b, log decay rows of the chunk -> [4][64][128] bf16 (S and dS' are consumed);
    // rows past the sequence end read as zero
    {
        const __nv_bfloat16* src[4] = {prm.q, prm.k, prm.b, prm.g};
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int p = tid + kThreads * i;
            const int tsel = p >> 10, r = (p >> 4) & 63, piece = p & 15;
            const bool valid = r < nvalid && 8 * piece < kdim;   // key channels past d_k: zero
            const __nv_bfloat16* s = src[tsel] + (valid ? kidx(r, 8 * piece) : kidx(0, 0));
            cp_async16(base + kRaw + static_cast<uint32_t>(tsel) * 16384u + static_cast<uint32_t>(r) * 256u + 16u * piece, s,
                       valid ? 16u : 0u);
        }
        cp_async_commit();
    }
    operands_done();

    // ---- 4. du E^T (dA_kk = -du E^T below the diagonal) and (T^T dW)^T = dW^T T -------------------
    if (tid == 0) {
        // du and E as hi + lo pairs: du_hi E_hi + du_hi E_lo + du_lo E_hi
        const uint64_t dUm = umma_desc2(base + kdUt, 8192u, 1024u), dEm = umma_desc2(base + kEt, 8192u, 1024u);
        const uint64_t dULm = umma_desc2(base + kdUtL, 8192u, 1024u), dELm = umma_desc2(base + kEtL, 8192u, 1024u);
        const uint64_t dWk = umma_desc2(base + kdWt, 16u, 1024u), dTm = umma_desc2(base + kT, 8192u, 1024u);
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
            mma_ss_f16(tmem + kTmAkk, dUm + 128u * kk, dEm + 128u * kk, idesc_f16x(64, 64, 0, 1, 1), kk > 0);
            mma_ss_f16(tmem + kTmAkk, dUm + 128u * kk, dELm + 128u * kk, idesc_f16x(64, 64, 0, 1, 1), 1u);
            mma_ss_f16(tmem + kTmAkk, dULm + 128u * kk, dEm + 128u * kk, idesc_f16x(64, 64, 0, 1, 1), 1u);
        }
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) mma_ss_f16(tmem + kTmCb0, dWk + 2u * kk, dTm + 128u * kk, idesc_f16x(128, 64, 0, 0, 1), kk > 0);
        mma_commit(bar(kBarMma));
    }
    // G[r][j] = sum_{t <= r} max(g_t, floor) per key channel (tokens past the end: 0), fp32
    cp_async_wait_all();
    __syncthreads();
    {
        const int ch = tid & 127, s = tid >> 7;
        const uint16_t* gr = raw + 3 * 8192;
        float run = 0.f, loc[16];
#pragma unroll
        for (int jj = 0; jj < 16; ++jj) {
            const int r = 16 * s + jj;
            run += r < nvalid ? fmaxf(bf(gr[r * 128 + ch]), kMinLogDecay) : 0.f;
            loc[jj] = run;
        }
        scr[s * 128 + ch] = run;
        __syncthreads();
        float off = 0.f;
        for (int s2 = 0; s2 < s; ++s2) off += scr[s2 * 128 + ch];
        float* G = reinterpret_cast<float*>(sgen + kG);
#pragma unroll
        for (int jj = 0; jj < 16; ++jj) G[(16 * s + jj) * 128 + ch] = loc[jj] + off;
    }
    __syncthreads();
    // K-groups (tf32, lane = key channel): group R holds k_i e^{G_m(R) - G_i} for tokens
    // i < 16 (R + 1); chunks of 16 tokens (R, ic) spread over the quarter's four warps
#pragma unroll 1
    for (int f = cb; f < 10; f += 4) {
        const int R = f == 0 ? 0 : f < 3 ? 1 : f < 6 ? 2 : 3;
        const int ic = f - R * (R + 1) / 2;
        const float gm = Gt[(16 * R + 7) * 128 + a];
        float x[16];
#pragma unroll
        for (int jj = 0; jj < 16; ++jj) {
            const int i = 16 * ic + jj;
            x[jj] = tf32r(bf(raw[8192 + i * 128 + a]) * __expf(gm - Gt[i * 128 + a]));
        }
        tmem_st16(tmem + lane_base + col_kg(R) + 16u * ic, x);
    }
    tmem_st_wait();
    wait_mma();
    {
        float v[16];
        tmem_ld16(tmem + lane_base + kTmAkk + 16u * cb, v);
        if (lane < 16) {
            const int i = 16 * quarter + lane;   // row of dA_kk (the later token)
            float t[16];
#pragma unroll
            for (int jj = 0; jj < 16; ++jj) t[jj] = 16 * cb + jj < i ? tf32r(-v[jj]) : 0.f;
#pragma unroll
            for (int u = 0; u < 4; ++u)
                *reinterpret_cast<float4*>(sgen + kAkk + sw(8192u, i, 16u * cb + 4u * u)) =
                    make_float4(t[4 * u], t[4 * u + 1], t[4 * u + 2], t[4 * u + 3]);
#pragma unroll
            for (int jj = 0; jj < 16; ++jj)
                *reinterpret_cast<float*>(sgen + kAkkT + sw(8192u, 16u * cb + jj, static_cast<uint32_t>(i))) = t[jj];
        }
    }
    operands_done();

    // ---- 5. X1 = K-groups x dA_kk^T, X2 = K-groups x dA_qk^T (per row stripe R, N = 16) ----------
    if (tid == 0) {
#pragma unroll
        for (int R = 0; R < 4; ++R) {
            const uint32_t rk = base + kAkk + 2048u * R, rq = base + kAqk + 2048u * R;
            for (int s = 0; s < 2 * (R + 1); ++s) {
                const uint32_t acol = tmem + col_kg(R) + 8u * s;
                mma_ts(tmem + kTmX1 + 16u * R, acol, umma_desc(kstep(rk, 8192u, s)), idesc_tf32(128, 16), s > 0);
                mma_ts(tmem + kTmX2 + 16u * R, acol, umma_desc(kstep(rq, 8192u, s)), idesc_tf32(128, 16), s > 0);
            }
        }
        mma_commit(bar(kBarMma));
    }
    wait_mma();
    // this thread: key channel a, tokens r = 16 cb + jj (stripe cb)
    const float gC = Gt[63 * 128 + a], gM = Gt[(16 * cb + 7) * 128 + a];
    float dkp[16], dgp[16];
    {
        // two halves of 8 tokens, so that the accumulators read out stay few in registers
        float zk = 0.f;
        float dqv[16], dbv[16];
#pragma unroll
        for (int hf = 0; hf < 2; ++hf) {
        const uint32_t col = 16u * cb + 8u * hf;
        uint32_t x1[8], x2[8], kb[8], qb[8], c0[8];
        tmem_ld8_nw(tmem + lane_base + kTmX1 + col, x1);
        tmem_ld8_nw(tmem + lane_base + kTmX2 + col, x2);
        tmem_ld8_nw(tmem + lane_base + kTmKb + col, kb);
        tmem_ld8_nw(tmem + lane_base + kTmQb + col, qb);
        tmem_ld8_nw(tmem + lane_base + kTmCb0 + col, c0);
        tmem_ld_wait();
#pragma unroll
        for (int j8 = 0; j8 < 8; ++j8) {
            const int jj = 8 * hf + j8;
            const int r = 16 * cb + jj;
            const float gr = Gt[r * 128 + a];
            const float eg = __expf(gr), ed = __expf(gr - gM), ec = __expf(gC - gr);
            const float qv = bf(raw[r * 128 + a]), kv = bf(raw[8192 + r * 128 + a]), bv = bf(raw[16384 + r * 128 + a]);
            const float x1v = __uint_as_float(x1[j8]), x2v = __uint_as_float(x2[j8]);
            const float c0v = __uint_as_float(c0[j8]), qbv = __uint_as_float(qb[j8]);
            const float dc = eg * c0v + ed * x1v;
            const float dq = eg * qbv + ed * x2v;
            const float z1 = __uint_as_float(kb[j8]) * ec;
            // dG's pair terms take the C- and Q-group factors as rounded for Y1, so that
            // a pair within a stripe enters dG_r and dG_i as the same product
            const float cgr = tf32r(bv * kv * ed), qgr = tf32r(qv * ed);
            dqv[jj] = dq;
            dbv[jj] = dc * kv;
            dkp[jj] = z1 + dc * bv;
            dgp[jj] = (eg * c0v) * (bv * kv) + x1v * cgr + (eg * qbv) * qv + x2v * qgr - z1 * kv;
            zk = fmaf(z1, kv, zk);
        }
        }
        scr[cb * 128 + a] = zk;
        float* xb = reinterpret_cast<float*>(sgen + kXpB) + warp * 512;
        store_tokens(xb, dqv, prm.dq, row0, prm.H, h, 32 * quarter, 16 * cb, nvalid, lane, kdim);
        store_tokens(xb, dbv, prm.db, row0, prm.H, h, 32 * quarter, 16 * cb, nvalid, lane, kdim);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    // C- and Q-groups (tf32, lane = key channel): group s holds c_r e^{G_r - G_m(s)} and
    // q_r e^{G_r - G_m(s)} for tokens r >= 16 s
#pragma unroll 1
    for (int f = cb; f < 10; f += 4) {
        const int s = f < 4 ? 0 : f < 7 ? 1 : f < 9 ? 2 : 3;
        const int jc = f - (s == 0 ? 0 : s == 1 ? 4 : s == 2 ? 7 : 9);
        const float gm = Gt[(16 * s + 7) * 128 + a];
        float xc[16], xq[16];
#pragma unroll
        for (int jj = 0; jj < 16; ++jj) {
            const int r = 16 * (s + jc) + jj;
            const float ex = __expf(Gt[r * 128 + a] - gm);
            xc[jj] = tf32r(bf(raw[16384 + r * 128 + a]) * bf(raw[8192 + r * 128 + a]) * ex);
            xq[jj] = tf32r(bf(raw[r * 128 + a]) * ex);
        }
        tmem_st16(tmem + lane_base + col_cg(s) + 16u * jc, xc);
        tmem_st16(tmem + lane_base + kQgOff + col_cg(s) + 16u * jc, xq);
    }
    tmem_st_wait();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();

    // ---- 6. Y1 = C-groups x dA_kk + Q-groups x dA_qk (per column stripe s, N = 16) ------------------
    if (tid == 0) {
#pragma unroll
        for (int s = 0; s < 4; ++s) {
            const uint32_t rk = base + kAkkT + 2048u * s, rq = base + kAqkT + 2048u * s;
            for (int t = 0; t < 8 - 2 * s; ++t)
                mma_ts(tmem + kTmY + 16u * s, tmem + col_cg(s) + 8u * t, umma_desc(kstep(rk, 8192u, 2 * s + t)),
                       idesc_tf32(128, 16), t > 0);
            for (int t = 0; t < 8 - 2 * s; ++t)
                mma_ts(tmem + kTmY + 16u * s, tmem + kQgOff + col_cg(s) + 8u * t, umma_desc(kstep(rq, 8192u, 2 * s + t)),
                       idesc_tf32(128, 16), 1u);
        }
        mma_commit(bar(kBarMma));
    }
    wait_mma();
    {
        float y[16];
        tmem_ld16(tmem + lane_base + kTmY + 16u * cb, y);
        float tot = 0.f;
#pragma unroll
        for (int jj = 0; jj < 16; ++jj) {
            const int r = 16 * cb + jj;
            const float gr = Gt[r * 128 + a];
            const float kv = bf(raw[8192 + r * 128 + a]);
            const float fi = __expf(gM - gr);
            const float y1 = y[jj] * fi;
            dkp[jj] += y1;
            dgp[jj] -= y[jj] * tf32r(kv * fi);   // the K-group factor as rounded for X
        }
        float* xb = reinterpret_cast<float*>(sgen + kXpB) + warp * 512;
        store_tokens(xb, dkp, prm.dk, row0, prm.H, h, 32 * quarter, 16 * cb, nvalid, lane, kdim);
        if (cb == 3) {
            // G_C's own terms land on the chunk's last token row
            float zk = 0.f;
#pragma unroll
            for (int s = 0; s < 4; ++s) zk += scr[s * 128 + a];
            dgp[15] += zk + __expf(gC) * gsum[a];
        }
#pragma unroll
        for (int jj = 0; jj < 16; ++jj) tot += dgp[jj];
        scr[512 + cb * 128 + a] = tot;
        __syncthreads();
        float run = 0.f;
        for (int s = cb + 1; s < 4; ++s) run += scr[512 + s * 128 + a];
#pragma unroll
        for (int jj = 15; jj >= 0; --jj) {
            run += dgp[jj];
            dgp[jj] = run;
        }
        store_tokens(xb, dgp, prm.dg, row0, prm.H, h, 32 * quarter, 16 * cb, nvalid, lane, kdim);
    }
    if (!ok && tid == 0) atomicExch(prm.err, kDevTimeout);
    if (tid == 0) {
        // every product issued has completed before the TMEM is freed (after a timeout too)
        mma_commit(bar(kBarDrain));
        mbar_wait(bar(kBarDrain), 0u);
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc<kTmCols>(tmem);
    }
}
}  // namespace cgr

}  // namespace

namespace {
// The item distance between this CTA and the one that follows it on the same SM: one
// CTA per SM is resident, so the SM count (0 if it cannot be read: no prefetch).
int cgrad_prefetch_stride() {
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) !=
                                                    cudaSuccess)
        return 0;
    return sms > 0 ? sms : 0;
}

// Chunks of the call (packed sequences: an upper bound, every sequence adding at most
// one partial chunk) and the workspace regions, in order: the context that the forward
// part leaves for the backward part (forward slots, backward records, start states --
// the chain's cached states -- and, packed, the first global chunk of each sequence),
// then the end-state gradients and the recomputed forward's o.
struct ChunkedLayout {
    int64_t chunks, n_cache;
    size_t slots, wy, sc, cb, ctx, dsn, o, total;
};
ChunkedLayout chunked_layout(int64_t B, int64_t T, int64_t H, bool packed, int64_t total_rows) {
    auto r256 = [](size_t x) { return (x + 255) / 256 * 256; };
    ChunkedLayout l{};
    const int64_t rows = packed ? total_rows : B * T;
    l.chunks = packed ? (total_rows + kC - 1) / kC + B : B * ((T + kC - 1) / kC);
    l.n_cache = packed ? 0 : T / kC;
    const size_t items = static_cast<size_t>(l.chunks * H);
    l.slots = r256(items * kSlot2Bytes);
    l.wy = r256(items * kWyBytes);
    l.sc = r256((packed ? items : static_cast<size_t>(B * H * l.n_cache)) * 16384 * 4);
    l.cb = packed ? r256(static_cast<size_t>(B + 1) * 4) : 0;
    l.ctx = l.slots + l.wy + l.sc + l.cb;
    l.dsn = r256(items * 16384 * 4);
    l.o = r256(static_cast<size_t>(rows * H) * 128 * 2);
    l.total = l.ctx + l.dsn + l.o;
    return l;
}

struct ChunkedCtx {
    uint8_t* slots;
    uint8_t* wy;
    float* Sc;
    int* cb;
};
ChunkedCtx chunked_ctx(uint8_t* base, const ChunkedLayout& l, bool packed) {
    return ChunkedCtx{base, base + l.slots, reinterpret_cast<float*>(base + l.slots + l.wy),
                      packed ? reinterpret_cast<int*>(base + l.slots + l.wy + l.sc) : nullptr};
}

// bf16 inputs, head sizes in {32, 64, 128} (below 128 on channels zero-padded to 128,
// as in the forward), at least one token; the grid limits of the kernels.
int chunked_check(const BackwardArgs& a, const ChunkedLayout& l) {
    const bool packed = a.cu != nullptr;
    auto dim_ok = [](int64_t d) { return d == 32 || d == 64 || d == 128; };
    if (a.in_dtype != GDR2_BF16 || !dim_ok(a.dk) || !dim_ok(a.dv) || (packed ? a.total <= 0 : a.T <= 0))
        return GDR2_ERR_UNSUPPORTED;
    if (l.chunks * a.H >= (1ll << 31) || a.B * a.H >= 65536ll * 32768ll || (packed && a.total >= (1ll << 31)))
        return GDR2_ERR_SHAPE;
    return GDR2_OK;
}

// The forward part: every chunk's maps and backward record, and its start state (the
// chain's cached state after each chunk) into the context; o (out_dtype) and S_T (or
// null) as gdr2_forward writes them.
int chunked_forward_part(const BackwardArgs& a, const ChunkedLayout& l, const ChunkedCtx& c, void* o, int out_dtype,
                         float* S_T, cudaStream_t stream, int* err) {
    const bool packed = a.cu != nullptr;
    ForwardArgs f{a.q, a.k, a.v, a.b, a.w, a.g, a.S0, o, S_T, a.B, packed ? 0 : a.T, a.H, a.dk, a.dv,
                  a.cu, packed ? a.total : a.B * a.T, GDR2_BF16, out_dtype};
    if (packed || l.n_cache > 0) {
        f.S_cache = c.Sc;
        f.cache_chunks = 1;
    }
    int rc = packed ? launch_chunk_base(a.cu, a.B, a.total, c.cb, stream) : GDR2_OK;
    if (rc == GDR2_OK) rc = launch_prep2(f, c.slots, c.cb, l.chunks, stream, err, 0, 0, c.wy);
    if (rc == GDR2_OK) rc = launch_chain(f, c.slots, c.cb, stream, err);
    return rc;
}

// The backward part, from the context: dS from the last chunk to the first (end-state
// gradients into dsn), then every chunk's token gradients.
int chunked_backward_part(const BackwardArgs& a, const ChunkedLayout& l, const ChunkedCtx& c, float* dsn,
                          cudaStream_t stream, int* err) {
    const bool packed = a.cu != nullptr;
    const int64_t items = l.chunks * a.H, nch = packed ? 0 : (a.T + kC - 1) / kC;
    static std::once_flag attr_once;
    static cudaError_t attr_err = cudaSuccess;
    std::call_once(attr_once, [] {
        attr_err = cudaFuncSetAttribute(rch::rchain_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                        static_cast<int>(rch::kSmemAlloc));
        if (attr_err == cudaSuccess)
            attr_err = cudaFuncSetAttribute(cgr::cgrad_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                            static_cast<int>(cgr::kSmemAlloc));
        if (attr_err == cudaSuccess)
            attr_err = cudaFuncSetAttribute(cgr::cgrad_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                            static_cast<int>(cgr::kSmemAlloc));
    });
    if (attr_err != cudaSuccess) return GDR2_ERR_CUDA;
    rch::Params rp{c.slots, a.dST, a.dO, dsn, a.d_S0, err, static_cast<int>(a.T), static_cast<int>(a.H),
                   static_cast<int>(nch), kWaitCycles, a.cu, c.cb, static_cast<int>(packed ? a.total : 0),
                   static_cast<int>(a.dk), static_cast<int>(a.dv)};
    rch::rchain_kernel<<<dim3(static_cast<unsigned>(a.B * a.H), 2), rch::kThreads, rch::kSmemAlloc, stream>>>(rp);
    if (cudaPeekAtLastError() != cudaSuccess) return GDR2_ERR_CUDA;
    cgr::Params gp{c.wy, c.Sc, a.S0, dsn, a.dO,
                   static_cast<const __nv_bfloat16*>(a.q), static_cast<const __nv_bfloat16*>(a.k),
                   static_cast<const __nv_bfloat16*>(a.b), static_cast<const __nv_bfloat16*>(a.g),
                   static_cast<const __nv_bfloat16*>(a.v), static_cast<const __nv_bfloat16*>(a.w),
                   a.d_q, a.d_k, a.d_b, a.d_g, a.d_v, a.d_w,
                   static_cast<int>(a.T), static_cast<int>(a.H), static_cast<int>(nch), static_cast<int>(l.n_cache), err,
                   a.cu, c.cb, static_cast<int>(a.B), static_cast<int>(packed ? a.total : 0),
                   static_cast<int>(items), cgrad_prefetch_stride(), static_cast<int>(a.dk), static_cast<int>(a.dv)};
    if (a.dk == 128 && a.dv == 128)
        cgr::cgrad_kernel<false><<<static_cast<unsigned>(items), cgr::kThreads, cgr::kSmemAlloc, stream>>>(gp);
    else
        cgr::cgrad_kernel<true><<<static_cast<unsigned>(items), cgr::kThreads, cgr::kSmemAlloc, stream>>>(gp);
    return cudaPeekAtLastError() == cudaSuccess ? GDR2_OK : GDR2_ERR_CUDA;
}
}  // namespace

size_t backward_chunked_workspace_bytes(int64_t B, int64_t T, int64_t H, bool packed, int64_t total) {
    return chunked_layout(B, T, H, packed, total).total;
}

size_t chunked_context_bytes(int64_t B, int64_t T, int64_t H, bool packed, int64_t total) {
    return chunked_layout(B, T, H, packed, total).ctx;
}

int launch_backward_chunked(const BackwardArgs& a, void* ws, cudaStream_t stream, int* err) {
    const bool packed = a.cu != nullptr;
    const ChunkedLayout l = chunked_layout(a.B, a.T, a.H, packed, a.total);
    int rc = chunked_check(a, l);
    if (rc != GDR2_OK) return rc;
    uint8_t* base = static_cast<uint8_t*>(ws);
    const ChunkedCtx c = chunked_ctx(base, l, packed);
    float* dsn = reinterpret_cast<float*>(base + l.ctx);
    void* o_scratch = base + l.ctx + l.dsn;
    rc = chunked_forward_part(a, l, c, o_scratch, GDR2_BF16, nullptr, stream, err);
    if (rc == GDR2_OK) rc = chunked_backward_part(a, l, c, dsn, stream, err);
    return rc;
}

int launch_forward_train(const BackwardArgs& a, void* o, int out_dtype, float* S_T, void* ctx, cudaStream_t stream,
                         int* err) {
    const bool packed = a.cu != nullptr;
    const ChunkedLayout l = chunked_layout(a.B, a.T, a.H, packed, a.total);
    const int rc = chunked_check(a, l);
    if (rc != GDR2_OK) return rc;
    return chunked_forward_part(a, l, chunked_ctx(static_cast<uint8_t*>(ctx), l, packed), o, out_dtype, S_T, stream,
                                err);
}

size_t backward_from_context_workspace_bytes(int64_t B, int64_t T, int64_t H, bool packed, int64_t total) {
    return chunked_layout(B, T, H, packed, total).dsn;
}

int launch_backward_from_context(const BackwardArgs& a, const void* ctx, void* ws, cudaStream_t stream, int* err) {
    const bool packed = a.cu != nullptr;
    const ChunkedLayout l = chunked_layout(a.B, a.T, a.H, packed, a.total);
    const int rc = chunked_check(a, l);
    if (rc != GDR2_OK) return rc;
    // the kernels only read the context
    const ChunkedCtx c = chunked_ctx(static_cast<uint8_t*>(const_cast<void*>(ctx)), l, packed);
    return chunked_backward_part(a, l, c, static_cast<float*>(ws), stream, err);
}

}  // namespace gdr2
