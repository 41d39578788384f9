// Chunked Gated Delta Rule-2 prefill, part 1 of 2: the state-independent
// preparation of every 64-token chunk, all chunks in parallel.
//
// Method ("Gated DeltaNet-2: Decoupling Erase and Write in Linear Attention"
// page: update equation, and the "efficient implementation" section's WY form
// with decay absorption and chunkwise algorithm).  For one chunk of C = 64
// tokens r = 0..63 with cumulative log decay G_r = sum_{t<=r} g_t (per key
// channel), c_r = b_r * k_r and chunk-initial state S, the recurrence unrolls to
//     [E; O] = [T; A_qk T] U + [-W; P] S,     S <- diag(e^{G_C}) S + Kb^T E
// with A_kk[r,i] = sum_j c_r[j] k_i[j] e^{G_r[j]-G_i[j]} (i < r),
// A_qk[r,i] = sum_j q_r[j] k_i[j] e^{G_r[j]-G_i[j]} (i <= r),
// T = (I + A_kk)^-1 (the UT transform), Cb = c e^{G}, Qb = q e^{G},
// Kb = k e^{G_C - G}, W = T Cb, P = Qb - A_qk W and U = w * v.  Everything but
// U and S depends on q, k, b and g of the chunk alone; this kernel computes
// it for every (chunk, head) at once and writes one workspace slot:
//     [T; A_qk T], -Cb^T, Kb^T, Qb (fp16), e^{G_C} (fp32).
// The state kernel forms [-W; P] = [T; A_qk T](-Cb) + [0; Qb] on the tensor
// core and runs the chunk-to-chunk chain.
//
// Overflow-free decay factors: e^{G_r - G_i} is formed about a reference m, the
// 8th token of the 16-token stripe holding r: e^{G_r - G_m} * e^{G_m - G_i}.
// Row r carries e^{G_r - G_m}; column i is scaled once per stripe R >= stripe(i)
// ("K-group" R).  For i in an earlier stripe both factors are <= 1; inside the
// stripe each spans at most 8 tokens, and with per-token log decays floored at
// -10 it stays within e^{+-80}.
//
// Precision: the intra-chunk products take tf32 operands (rounded to nearest)
// with fp32 accumulation; the triangular solve is fp32 on CUDA cores.  -Cb, Qb
// and Kb are bounded by |b k| and |q|, |k| and are later used at tf32
// precision, so fp16 (the same 11 significant bits) carries them.
//
// Work split: one persistent CTA (640 threads) per SM.  In pass 1 thread
// (jp = tid % 64, hs = tid / 64) of the first 512 owns key channels 2jp, 2jp + 1
// over the 8 tokens of half-stripe hs; in the accumulator phases thread
// (j = tid % 128, R = tid / 128) owns TMEM lane j, columns 16R..16R+15.  One
// thread of the last warpgroup issues the TMA loads and tcgen05 MMAs.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_fp16.h>

#include <mutex>

#include "gdr2.h"
#include "gdr2_internal.cuh"
#include "gdr2_tc.cuh"

namespace gdr2 {
namespace {

using namespace tc;

constexpr int kC = kPrepC;
constexpr int kDK = kPrepDK;
constexpr int kSimt = 512;              // 16 elementwise / accumulator warps
constexpr int kThreads = kSimt + 128;   // + the TMA / MMA warpgroup
// Registers: 640 x 96 at launch; the MMA warpgroup drops to 32 and the
// elementwise warps rise to 112 (512 x 112 + 128 x 32 = 61440).
constexpr int kRegsSimt = 112, kRegsMma = 32;
static_assert(kSimt * kRegsSimt + (kThreads - kSimt) * kRegsMma <= kThreads * 96, "register pool");

// ---- shared memory (bytes from a 1024-aligned base) ------------------------------
// MMA operands are K-major with the 128-byte swizzle (K-blocks of 32 tf32).
constexpr uint32_t kRawQ = 0, kRawK = 16384, kRawB = 32768, kRawG = 49152;  // bf16 [2 kblk][64][64]
// K-groups [G3 (64 rows) | G1 (32) | G2 (48) | G0 (16)]: one 160-row operand (K-blocks
// 20 KB apart), written over the raw tiles once pass 1 has read them
constexpr uint32_t kKG = 0, kKGStride = 20480;
constexpr uint32_t kOpA = 81920;       // [Ct; Qt]: 128 rows x 128 K (64 KB)
constexpr uint32_t kIA = 147456;       // [I; A_qk]: 128 rows x 64 K (32 KB)
constexpr uint32_t kTT = 180224;       // T^T: 64 rows x 64 K (16 KB)
constexpr uint32_t kMisc = 196608;     // mbarriers, TMEM slot
constexpr uint32_t kSmemBytes = kMisc + 128;
constexpr uint32_t kSmemAlloc = kSmemBytes + 1024;
constexpr uint32_t kXTot = kOpA;   // per-half-stripe decay sums, 8 x 128 fp32 (before [Ct; Qt])
// solve scratch inside the [Ct; Qt] area (dead once the intra-chunk products are done)
constexpr int kLd = 65;                   // A_kk staging row (floats)
constexpr int kLt = 68;                   // T staging row (floats; rows 16-byte aligned)
constexpr uint32_t kSL = kOpA;            // A_kk staging  [64][65] fp32
constexpr uint32_t kSTs = kOpA + 16640;   // T staging     [64][68] fp32
constexpr uint32_t kSP = kOpA + 34048;    // M_{RJ} blocks, 6 x 16 x 17 fp32
static_assert(kSTs + 64 * kLt * 4 <= kSP && kSP + 6 * 16 * 17 * 4 <= kOpA + 65536, "solve scratch");
static_assert(kKG + 4 * kKGStride <= kOpA && kRawG + 16384 <= kOpA, "K-groups over the raw tiles");
static_assert(kSmemAlloc <= 232448, "shared memory");
enum : uint32_t { kBarTma = 0, kRdyAP, kRdyA0, kDoneP1, kDoneP2, kNumBars };
constexpr uint32_t kTmemSlot = kMisc + 8 * kNumBars;

// ---- TMEM columns ---------------------------------------------------------------
constexpr uint32_t kTmA0 = 0;     // [T; A_qk T]: 128 lanes x 64 columns
constexpr uint32_t kTmAP = 64;    // intra-chunk products [Ct; Qt] x [G3|G1|G2|G0]^T: columns 64..223
constexpr int kTmCols = 256;

constexpr float kMinLogDecay = -10.f;

__device__ __forceinline__ void simt_sync() { team_sync<kSimt>(); }
__device__ __forceinline__ bool simt_any(bool p) { return team_any<kSimt>(p); }
__device__ __forceinline__ uint32_t group_col(int R) {
    return kTmAP + (R == 3 ? 0u : R == 1 ? 64u : R == 2 ? 96u : 144u);
}

struct PrepParams {
    PrepSlots s;
    const int* cu;        // packed sequences: [N + 1] token offsets, or null
    int N, T, H, total;   // T: common length when cu is null
    int nchunks;          // chunks per sequence in this launch when cu is null
    int c0;               // first chunk of each sequence in this launch (cu null)
    int nitems;           // work items = global chunk bound x H; item = slot index
    int* err;
};

// Work item `it` = (global chunk it / H, head it % H), its slot index.  False for
// items past the last real chunk (packed sequences: the chunk count is a bound).
struct Item {
    int tok0, T, tp, h;
};
__device__ __forceinline__ bool locate(const PrepParams& prm, int it, Item& x) {
    const int gc = it / prm.H;
    x.h = it - gc * prm.H;
    if (prm.cu) {
        const int* cb = prm.s.chunk_base;
        if (gc >= cb[prm.N]) return false;
        int lo = 0, hi = prm.N;   // last sequence with cb[seq] <= gc
        while (hi - lo > 1) {
            const int mid = (lo + hi) >> 1;
            if (cb[mid] <= gc) lo = mid; else hi = mid;
        }
        const int a = min(max(prm.cu[lo], 0), prm.total);
        const int e = min(max(prm.cu[lo + 1], a), prm.total);
        x.tok0 = a;
        x.T = e - a;
        x.tp = (gc - cb[lo]) * kC;
    } else {
        // chunks c0 .. c0 + nchunks - 1 of every sequence: token offsets relative to
        // the first of them
        const int seq = gc / prm.nchunks;
        x.tok0 = seq * prm.T + prm.c0 * kC;
        x.T = prm.T - prm.c0 * kC;
        x.tp = (gc - seq * prm.nchunks) * kC;
    }
    return true;
}

// Persistent: CTA b handles items b, b + gridDim.x, ...  The next item's tiles load
// while this item's solve runs, its [T; A_qk T] is written out while the next
// item's intra-chunk products run, and the next item's pass 1 overlaps this
// item's [T; A_qk T] product.
__global__ void __launch_bounds__(kThreads, 1)
prep_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
            const __grid_constant__ CUtensorMap tm_b, const __grid_constant__ CUtensorMap tm_g,
            const PrepParams prm) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t base = (smem_u32(smem_raw) + 1023u) & ~1023u;
    uint8_t* sgen = smem_raw + (base - smem_u32(smem_raw));
    float* const F = reinterpret_cast<float*>(sgen);
    const unsigned short* const H16 = reinterpret_cast<const unsigned short*>(sgen);
    auto bar = [&](uint32_t i) { return base + kMisc + 8u * i; };
    volatile uint32_t* tmem_slot = reinterpret_cast<volatile uint32_t*>(sgen + kTmemSlot);

    const int tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;
    const int j = tid & 127;
    const int R = (tid >> 7) & 3;
    const int quarter = warp & 3;
    // next real item after `it` (or nitems)
    auto next_item = [&](int it, Item& x) {
        for (it += gridDim.x; it < prm.nitems; it += gridDim.x)
            if (locate(prm, it, x)) return it;
        return prm.nitems;
    };

    if (tid == 0) {
        for (uint32_t i = 0; i < kNumBars; ++i) mbar_init(bar(i), 1);
        fence_mbar_init();
        fence_async_smem();
    }
    if (warp == 0) tmem_alloc<kTmCols>(base + kTmemSlot);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    Item first;
    const int it0 = (static_cast<int>(blockIdx.x) < prm.nitems && locate(prm, blockIdx.x, first))
                        ? static_cast<int>(blockIdx.x)
                        : next_item(blockIdx.x, first);

    if (warp >= kSimt / 32) {
        // ================= TMA / MMA warpgroup: one elected thread =================
        asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kRegsMma));
        if (warp == kSimt / 32 && lane == 0) {
            auto load = [&](const Item& x) {
                mbar_expect_tx(bar(kBarTma), 65536u);
                const int row = x.tok0 + x.tp;
                tma_load_4d(base + kRawQ, &tm_q, 0, x.h, row, 0, bar(kBarTma));
                tma_load_4d(base + kRawQ + 8192, &tm_q, 64, x.h, row, 0, bar(kBarTma));
                tma_load_4d(base + kRawK, &tm_k, 0, x.h, row, 0, bar(kBarTma));
                tma_load_4d(base + kRawK + 8192, &tm_k, 64, x.h, row, 0, bar(kBarTma));
                tma_load_4d(base + kRawB, &tm_b, 0, x.h, row, 0, bar(kBarTma));
                tma_load_4d(base + kRawB + 8192, &tm_b, 64, x.h, row, 0, bar(kBarTma));
                tma_load_4d(base + kRawG, &tm_g, 0, x.h, row, 0, bar(kBarTma));
                tma_load_4d(base + kRawG + 8192, &tm_g, 64, x.h, row, 0, bar(kBarTma));
            };
            bool ok = true;
            uint32_t ph = 0;      // phase of this item's barriers
            int loads = 0;        // tile loads issued
            if (it0 < prm.nitems) { load(first); ++loads; }
#pragma unroll 1
            for (int it = it0; it < prm.nitems && ok; ph ^= 1u) {
                // intra-chunk products [Ct; Qt] x [G3|G1|G2|G0]^T
                if (!(ok = mbar_wait(bar(kRdyAP), ph))) break;
                tc_fence_after();
#pragma unroll 1
                for (int s = 0; s < 16; ++s)
                    mma_ss(tmem + kTmAP, umma_desc(kstep(base + kOpA, 16384, s)),
                           umma_desc(kstep(base + kKG, kKGStride, s)), idesc_tf32(128, 160), s > 0 ? 1u : 0u);
                mma_commit(bar(kDoneP1));
                // the products have read the K-groups over the raw tiles: next item's tiles
                if (!(ok = mbar_wait(bar(kDoneP1), ph))) break;
                Item nx;
                const int nit = next_item(it, nx);
                if (nit < prm.nitems) { load(nx); ++loads; }
                // [T; A_qk T] = [I; A_qk] T
                if (!(ok = mbar_wait(bar(kRdyA0), ph))) break;
                tc_fence_after();
#pragma unroll 1
                for (int s = 0; s < 8; ++s)
                    mma_ss(tmem + kTmA0, umma_desc(kstep(base + kIA, 16384, s)),
                           umma_desc(kstep(base + kTT, 8192, s)), idesc_tf32(128, 64), s > 0 ? 1u : 0u);
                mma_commit(bar(kDoneP2));
                it = nit;
            }
            if (!ok) {
                atomicExch(prm.err, kDevTimeout);
                // the last tile load may still be in flight (bounded wait)
                if (loads > 0) mbar_wait(bar(kBarTma), static_cast<uint32_t>((loads - 1) & 1));
            }
        }
        __syncwarp();
    } else {
        // ================= 16 elementwise / accumulator warps =====================
        asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kRegsSimt));
        const uint32_t lane_base = static_cast<uint32_t>(quarter * 32) << 16;
        bool failed = false;
        auto wait_done = [&](uint32_t b, uint32_t ph) -> bool {
            const bool ok = mbar_wait(bar(b), ph);
            const bool bad = simt_any(!ok);
            tc_fence_after();
            return !bad;
        };
        auto signal = [&](uint32_t b) {
            fence_async_smem();
            tc_fence_before();
            simt_sync();
            if (tid == 0) mbar_arrive(bar(b));
        };
        // [T; A_qk T] of a finished item -> its slot as fp16 (the 11 significant bits of
        // the tf32 operand it becomes)
        auto write_a0 = [&](int64_t slot) {
            float v[16];
            tmem_ld16(tmem + lane_base + kTmA0 + static_cast<uint32_t>(16 * R), v);
            uint4 pk[2];
            __half2* ph = reinterpret_cast<__half2*>(pk);
#pragma unroll
            for (int e = 0; e < 16; e += 2) ph[e / 2] = __floats2half2_rn(v[e], v[e + 1]);
            uint4* dst = reinterpret_cast<uint4*>(prm.s.a0 + slot * (128 * kC) + (R * 128 + j) * 16);
            dst[0] = pk[0];
            dst[1] = pk[1];
        };

        uint32_t ph = 0;
        int prev = -1;
        Item cur = first;
#pragma unroll 1
        for (int it = it0; it < prm.nitems && !failed; ph ^= 1u) {
            const int T = cur.T, tp = cur.tp;
            const int64_t slot = it;
            // ---- pass 1: raw tiles -> decay factors, [Ct; Qt], K-groups, -Cb, Qb, Kb --------
            // Thread (jp = tid % 64, hs = tid / 64) owns key channels 2jp and 2jp + 1 over tokens
            // 8hs .. 8hs + 7 (half hs % 2 of stripe hs / 2): 32-bit raw loads and 64-bit
            // operand stores carry both channels.
            {
                const int jp = tid & 63, hs = tid >> 6, Rs = hs >> 1, hf = hs & 1;
                const uint32_t ch = 2u * static_cast<uint32_t>(jp);
                float cr[2][8], qr[2][8], kr[2][8];   // [channel][token]: c*rho, q*rho, k/rho
                if (!wait_done(kBarTma, ph)) { failed = true; break; }
                // element (token 8hs + s, channels ch, ch + 1) of a bf16 tile: one 32-bit word
                const uint32_t cbase = (ch >> 6) * 8192u + static_cast<uint32_t>(8 * hs) * 128u + ((ch & 7u) << 1);
                const uint32_t c8 = (ch & 63u) >> 3;
                float Gl[2][8];
                float acc0 = 0.f, acc1 = 0.f;
                // tokens past the sequence end enter as q = k = b = log_decay = 0
                const int nvalid = T - tp - 8 * hs;
#pragma unroll
                for (int s = 0; s < 8; ++s) {
                    const uint32_t off = cbase + static_cast<uint32_t>(s) * 128u + ((c8 ^ static_cast<uint32_t>(s)) << 4);
                    const uint32_t live = s < nvalid ? 0xFFFFFFFFu : 0u;
                    const uint32_t g2 = *reinterpret_cast<const uint32_t*>(sgen + kRawG + off) & live;
                    const uint32_t k2 = *reinterpret_cast<const uint32_t*>(sgen + kRawK + off) & live;
                    const uint32_t b2 = *reinterpret_cast<const uint32_t*>(sgen + kRawB + off);
                    const uint32_t q2 = *reinterpret_cast<const uint32_t*>(sgen + kRawQ + off) & live;
                    acc0 += fmaxf(__uint_as_float(g2 << 16), kMinLogDecay);
                    acc1 += fmaxf(__uint_as_float(g2 & 0xFFFF0000u), kMinLogDecay);
                    Gl[0][s] = acc0;
                    Gl[1][s] = acc1;
                    const float k0 = __uint_as_float(k2 << 16), k1 = __uint_as_float(k2 & 0xFFFF0000u);
                    cr[0][s] = __uint_as_float(b2 << 16) * k0;
                    cr[1][s] = __uint_as_float(b2 & 0xFFFF0000u) * k1;
                    qr[0][s] = __uint_as_float(q2 << 16);
                    qr[1][s] = __uint_as_float(q2 & 0xFFFF0000u);
                    kr[0][s] = k0;
                    kr[1][s] = k1;
                }
                // half-stripe totals -> every thread: G at each stripe's reference token (the
                // last token of its first half) and G_C, per channel
                float* const xt = F + (kXTot >> 2);
                xt[hs * 128 + ch] = acc0;
                xt[hs * 128 + ch + 1] = acc1;
                simt_sync();   // raw tiles fully read; totals visible
                float gmid0[4], gmid1[4], gC0 = 0.f, gC1 = 0.f;
#pragma unroll
                for (int h2 = 0; h2 < 8; ++h2) {
                    gC0 += xt[h2 * 128 + ch];
                    gC1 += xt[h2 * 128 + ch + 1];
                    if (!(h2 & 1)) {
                        gmid0[h2 >> 1] = gC0;
                        gmid1[h2 >> 1] = gC1;
                    }
                }
                const float gm0 = gmid0[Rs], gm1 = gmid1[Rs];
                const float em0 = __expf(gm0), em1 = __expf(gm1);                  // e^{G_m}        (<= 1)
                const float ecm0 = __expf(gC0 - gm0), ecm1 = __expf(gC1 - gm1);    // e^{G_C - G_m}  (<= 1)
                // G_r - G_m within the stripe: the first half ends at m, the second starts after it
#pragma unroll
                for (int s = 0; s < 8; ++s) {
                    const float d0 = hf ? Gl[0][s] : Gl[0][s] - Gl[0][7];
                    const float d1 = hf ? Gl[1][s] : Gl[1][s] - Gl[1][7];
                    const float rho0 = __expf(fminf(d0, 80.f)), irho0 = __expf(fminf(-d0, 80.f));
                    const float rho1 = __expf(fminf(d1, 80.f)), irho1 = __expf(fminf(-d1, 80.f));
                    cr[0][s] *= rho0; qr[0][s] *= rho0; kr[0][s] *= irho0;
                    cr[1][s] *= rho1; qr[1][s] *= rho1; kr[1][s] *= irho1;
                }
                simt_sync();   // exchange reads done before [Ct; Qt] overwrites it
                const uint32_t row0 = static_cast<uint32_t>(8 * hs);   // this half-stripe's first token row
#pragma unroll
                for (int s = 0; s < 8; ++s) {
                    const uint32_t r = row0 + static_cast<uint32_t>(s);
                    *reinterpret_cast<float2*>(sgen + kOpA + sw(16384, r, ch)) =
                        make_float2(tf32r(cr[0][s]), tf32r(cr[1][s]));
                    *reinterpret_cast<float2*>(sgen + kOpA + sw(16384, 64u + r, ch)) =
                        make_float2(tf32r(qr[0][s]), tf32r(qr[1][s]));
                }
                // K-groups: this half-stripe's tokens scaled to each later stripe's reference
#pragma unroll
                for (int g = 0; g < 4; ++g) {
                    if (g < Rs) continue;
                    const float sc0 = g == Rs ? 1.f : __expf(gmid0[g] - gm0);
                    const float sc1 = g == Rs ? 1.f : __expf(gmid1[g] - gm1);
                    const uint32_t r0 = g == 3 ? 0u : g == 1 ? 64u : g == 2 ? 96u : 144u;   // = group_col(g) - kTmAP
#pragma unroll
                    for (int s = 0; s < 8; ++s)
                        *reinterpret_cast<float2*>(sgen + kKG + sw(kKGStride, r0 + row0 + static_cast<uint32_t>(s), ch)) =
                            make_float2(tf32r(kr[0][s] * sc0), tf32r(kr[1][s] * sc1));
                }
                // -Cb, Kb as fp16 [token / 8][channel][token % 8] (this half-stripe is token group
                // hs), Qb as [channel / 8][token][channel % 8], e^{G_C}: into the slot
                {
                    uint4 cb[2], kb[2];
                    __half2* pc = reinterpret_cast<__half2*>(cb);
                    __half2* pk = reinterpret_cast<__half2*>(kb);
#pragma unroll
                    for (int s = 0; s < 8; s += 2) {
                        pc[s / 2] = __floats2half2_rn(-cr[0][s] * em0, -cr[0][s + 1] * em0);
                        pc[4 + s / 2] = __floats2half2_rn(-cr[1][s] * em1, -cr[1][s + 1] * em1);
                        pk[s / 2] = __floats2half2_rn(kr[0][s] * ecm0, kr[0][s + 1] * ecm0);
                        pk[4 + s / 2] = __floats2half2_rn(kr[1][s] * ecm1, kr[1][s + 1] * ecm1);
                    }
                    const int64_t o = slot * (kDK * kC) + (static_cast<int64_t>(hs) * kDK + ch) * 8;
                    uint4* dc = reinterpret_cast<uint4*>(prm.s.cbt + o);
                    uint4* dk = reinterpret_cast<uint4*>(prm.s.kbt + o);
                    dc[0] = cb[0]; dc[1] = cb[1];
                    dk[0] = kb[0]; dk[1] = kb[1];
                    __half2* dq = reinterpret_cast<__half2*>(reinterpret_cast<__half*>(prm.s.qb) + slot * (kC * kDK) +
                                                             ((ch >> 3) * kC + 8 * hs) * 8 + (ch & 7u));
#pragma unroll
                    for (int s = 0; s < 8; ++s) dq[s * 4] = __floats2half2_rn(qr[0][s] * em0, qr[1][s] * em1);
                    if (hs == 0) {
                        prm.s.gam[slot * kDK + ch] = __expf(gC0);
                        prm.s.gam[slot * kDK + ch + 1] = __expf(gC1);
                    }
                }
                signal(kRdyAP);
            }
            // ---- the previous item's [T; A_qk T] out (overlaps this item's products) -------
            if (prev >= 0) {
                if (!wait_done(kDoneP2, ph ^ 1u)) { failed = true; break; }
                write_a0(prev);
            }
            // ---- A_kk, A_qk out of TMEM; T = (I + A_kk)^-1; [I; A_qk] and T^T operands -------
            if (!wait_done(kDoneP1, ph)) { failed = true; break; }
            {
                const int m = j;                          // TMEM lane = product row
                const int r = m & 63;                     // token row within the chunk
                const int s0 = 2 * (quarter & 1);         // the two stripes of this quarter
                uint32_t ra[16], rb[16];
                if (R <= s0) tmem_ld16_nw(tmem + lane_base + group_col(s0) + 16u * R, ra);
                if (R <= s0 + 1) tmem_ld16_nw(tmem + lane_base + group_col(s0 + 1) + 16u * R, rb);
                tmem_ld_wait();
                const int rs = r >> 4;
                const bool have = R <= rs;
                float out[16];
#pragma unroll
                for (int e = 0; e < 16; ++e) out[e] = have ? __uint_as_float(rs == s0 ? ra[e] : rb[e]) : 0.f;
                if (m < 64) {
#pragma unroll
                    for (int e = 0; e < 16; ++e) {
                        const int i = 16 * R + e;
                        if (i < r) F[(kSL >> 2) + r * kLd + i] = out[e];
                    }
#pragma unroll
                    for (int e = 0; e < 16; e += 4) {
                        const int i = 16 * R + e;
                        *reinterpret_cast<float4*>(sgen + kIA + sw(16384, r, i)) =
                            make_float4(i == r ? 1.f : 0.f, i + 1 == r ? 1.f : 0.f, i + 2 == r ? 1.f : 0.f,
                                        i + 3 == r ? 1.f : 0.f);
                    }
                } else {
#pragma unroll
                    for (int e = 0; e < 16; e += 4) {
                        const int i = 16 * R + e;
                        *reinterpret_cast<float4*>(sgen + kIA + sw(16384, m, i)) =
                            make_float4(i <= r ? tf32r(out[e]) : 0.f, i + 1 <= r ? tf32r(out[e + 1]) : 0.f,
                                        i + 2 <= r ? tf32r(out[e + 2]) : 0.f, i + 3 <= r ? tf32r(out[e + 3]) : 0.f);
                    }
                }
            }
            // T above the diagonal blocks is zero
            for (int e = tid; e < 6 * 256; e += kSimt) {
                const int blk = e >> 8, rr = (e >> 4) & 15, cc = e & 15;
                const int Rb = blk < 3 ? 0 : blk < 5 ? 1 : 2;
                const int Ib = blk < 3 ? blk + 1 : blk < 5 ? blk - 1 : 3;
                F[(kSTs >> 2) + (16 * Rb + rr) * kLt + 16 * Ib + cc] = 0.f;
            }
            simt_sync();

            // 16x16 diagonal blocks by column forward substitution
            const float* L = F + (kSL >> 2);
            float* Ts = F + (kSTs >> 2);
            float* SP = F + (kSP >> 2);
            if (tid < 64) {
                const int o16 = 16 * (tid >> 4), col = tid & 15;
                float tcol[16];
#pragma unroll
                for (int r = 0; r < 16; ++r) tcol[r] = r == col ? 1.f : 0.f;
#pragma unroll
                for (int r = 1; r < 16; ++r) {
                    float s0 = 0.f, s1 = 0.f;
#pragma unroll
                    for (int i = 0; i < r; ++i) {
                        const float a = L[(o16 + r) * kLd + o16 + i];
                        if (i & 1) s1 = fmaf(a, tcol[i], s1); else s0 = fmaf(a, tcol[i], s0);
                    }
                    if (r > col) tcol[r] = -(s0 + s1);
                }
#pragma unroll
                for (int r = 0; r < 16; ++r) Ts[(o16 + r) * kLt + o16 + col] = tcol[r];
            }
            simt_sync();
            // off-diagonal blocks: with M_{RJ} = T_{RR} A_{RJ} (R > J),
            //   T_{RI} = -sum_{J=I}^{R-1} M_{RJ} T_{JI}, level by level (R - I = 1, 2, 3).
            if (tid < 6 * 64) {
                const int p = tid >> 6, rr = (tid >> 2) & 15, c4 = 4 * (tid & 3);
                const int Rb = p == 0 ? 1 : p < 3 ? 2 : 3, Jb = p - Rb * (Rb - 1) / 2;
                float a0 = 0.f, a1 = 0.f, a2 = 0.f, a3 = 0.f;
#pragma unroll
                for (int x = 0; x < 16; ++x) {
                    const float t = Ts[(16 * Rb + rr) * kLt + 16 * Rb + x];
                    const float* lr = L + (16 * Rb + x) * kLd + 16 * Jb + c4;
                    a0 = fmaf(t, lr[0], a0); a1 = fmaf(t, lr[1], a1);
                    a2 = fmaf(t, lr[2], a2); a3 = fmaf(t, lr[3], a3);
                }
                float* mp = SP + p * 272 + rr * 17 + c4;
                mp[0] = a0; mp[1] = a1; mp[2] = a2; mp[3] = a3;
            }
            simt_sync();
#pragma unroll
            for (int d = 1; d < 4; ++d) {
                if (tid < (4 - d) * 64) {
                    const int Ib = tid >> 6, Rb = Ib + d, rr = (tid >> 2) & 15, c4 = 4 * (tid & 3);
                    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
                    for (int Jd = 0; Jd < d; ++Jd) {
                        const int Jb = Ib + Jd, p = Rb * (Rb - 1) / 2 + Jb;
#pragma unroll
                        for (int x = 0; x < 16; ++x) {
                            const float m = SP[p * 272 + rr * 17 + x];
                            const float4 tv = *reinterpret_cast<const float4*>(Ts + (16 * Jb + x) * kLt + 16 * Ib + c4);
                            acc.x = fmaf(m, tv.x, acc.x); acc.y = fmaf(m, tv.y, acc.y);
                            acc.z = fmaf(m, tv.z, acc.z); acc.w = fmaf(m, tv.w, acc.w);
                        }
                    }
                    *reinterpret_cast<float4*>(Ts + (16 * Rb + rr) * kLt + 16 * Ib + c4) =
                        make_float4(-acc.x, -acc.y, -acc.z, -acc.w);
                }
                simt_sync();
            }
            // T^T operand: row n (column of T), K = k (row of T)
            {
                const int n = tid & 63, k0 = (tid >> 6) * 8;
                float t8[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) t8[e] = tf32r(Ts[(k0 + e) * kLt + n]);
                *reinterpret_cast<float4*>(sgen + kTT + sw(8192, n, k0)) = make_float4(t8[0], t8[1], t8[2], t8[3]);
                *reinterpret_cast<float4*>(sgen + kTT + sw(8192, n, k0 + 4)) =
                    make_float4(t8[4], t8[5], t8[6], t8[7]);
            }
            signal(kRdyA0);
            prev = it;
            Item nx;
            it = next_item(it, nx);
            cur = nx;
        }
        if (!failed && prev >= 0) {
            if (wait_done(kDoneP2, ph ^ 1u)) write_a0(prev);
            else failed = true;
        }
        if (failed && tid == 0) atomicExch(prm.err, kDevTimeout);
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc<kTmCols>(tmem);
    }
}

// First global chunk of each packed sequence: cb[s] = sum_{s' < s} ceil(len_s' / 64),
// with the same offset clamping the kernels use.  One CTA.
__global__ void chunk_base_kernel(const int* cu, int N, int total, int* cb) {
    __shared__ int part[1024];
    const int tid = threadIdx.x;
    const int per = (N + blockDim.x - 1) / blockDim.x;
    const int s0 = tid * per, s1 = min(N, s0 + per);
    auto nch = [&](int s) {
        const int a = min(max(cu[s], 0), total);
        const int e = min(max(cu[s + 1], a), total);
        return (e - a + kC - 1) / kC;
    };
    int sum = 0;
    for (int s = s0; s < s1; ++s) sum += nch(s);
    part[tid] = sum;
    __syncthreads();
    if (tid == 0) {   // exclusive scan of the partial sums
        int run = 0;
        for (int i = 0; i < static_cast<int>(blockDim.x); ++i) {
            const int x = part[i];
            part[i] = run;
            run += x;
        }
    }
    __syncthreads();
    int run = part[tid];
    for (int s = s0; s < s1; ++s) {
        cb[s] = run;
        run += nch(s);
    }
    if (s0 < N && s1 == N) cb[N] = run;
    if (N == 0 && tid == 0) cb[0] = 0;
}

PFN_cuTensorMapEncodeTiled_v12000 get_encode() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

// Packed [1, total, H, d] bf16 tokens as a 4-D map (d, H, total, 1); box
// (64, 1, 64, 1), 128-byte swizzle; rows past the tensor read as zeros.
bool make_token_map(CUtensorMap* m, const void* ptr, int64_t total, int64_t H, int64_t d) {
    auto enc = get_encode();
    if (!enc) return false;
    const cuuint64_t dims[4] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(H),
                                static_cast<cuuint64_t>(total), 1};
    const cuuint64_t strides[3] = {static_cast<cuuint64_t>(d * 2), static_cast<cuuint64_t>(H * d * 2),
                                   static_cast<cuuint64_t>(total * H * d * 2)};
    const cuuint32_t box[4] = {64, 1, 64, 1};
    const cuuint32_t estr[4] = {1, 1, 1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(ptr), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

bool two_kernel_supports(const ForwardArgs& a) {
    const int64_t total = a.cu ? a.total : a.B * a.T;
    return a.in_dtype == GDR2_BF16 && a.dk == kDK && (a.dv == 64 || a.dv == 128) && total > 0 &&
           total < (1ll << 31) && a.B * a.H < (1ll << 31) && a.H <= 65535 && get_encode() != nullptr;
}

int launch_chunk_base(const int* cu, int64_t N, int64_t total, int* chunk_base, cudaStream_t stream) {
    chunk_base_kernel<<<1, 1024, 0, stream>>>(cu, static_cast<int>(N), static_cast<int>(total), chunk_base);
    return cudaPeekAtLastError() == cudaSuccess ? GDR2_OK : GDR2_ERR_CUDA;
}

int64_t prep_chunk_bound(const ForwardArgs& a) {
    if (!a.cu) return a.B * ((a.T + kC - 1) / kC);
    return (a.total + kC - 1) / kC + a.B;
}

size_t prep_workspace_bytes(int64_t chunks, int64_t H, int64_t N) {
    return static_cast<size_t>(chunks) * static_cast<size_t>(H) * kSlotBytes + static_cast<size_t>(N + 1) * 4 +
           6 * 256;
}

PrepSlots prep_carve(void* ws, int64_t chunks, int64_t H) {
    const size_t n = static_cast<size_t>(chunks) * static_cast<size_t>(H);
    uintptr_t p = (reinterpret_cast<uintptr_t>(ws) + 255u) & ~static_cast<uintptr_t>(255u);
    auto take = [&](size_t bytes) {
        const uintptr_t r = p;
        p = (p + bytes + 255u) & ~static_cast<uintptr_t>(255u);
        return r;
    };
    PrepSlots s;
    s.a0 = reinterpret_cast<uint16_t*>(take(n * 64 * 128 * 2));
    s.cbt = reinterpret_cast<uint16_t*>(take(n * 64 * 128 * 2));
    s.kbt = reinterpret_cast<uint16_t*>(take(n * 64 * 128 * 2));
    s.qb = reinterpret_cast<uint16_t*>(take(n * 64 * 128 * 2));
    s.gam = reinterpret_cast<float*>(take(n * 128 * 4));
    s.chunk_base = reinterpret_cast<int*>(take(4));
    return s;
}

int launch_prep(const ForwardArgs& a, const PrepSlots& s, int64_t chunks, int c0, int cpiece, cudaStream_t stream,
                int* err) {
    const int64_t total = a.cu ? a.total : a.B * a.T;
    if (chunks <= 0) return GDR2_OK;
    if (chunks >= (1ll << 31)) return GDR2_ERR_SHAPE;
    CUtensorMap mq, mk, mb, mg;
    if (!make_token_map(&mq, a.q, total, a.H, a.dk) || !make_token_map(&mk, a.k, total, a.H, a.dk) ||
        !make_token_map(&mb, a.b, total, a.H, a.dk) || !make_token_map(&mg, a.g, total, a.H, a.dk))
        return GDR2_ERR_CUDA;
    static std::once_flag attr_once;
    static cudaError_t attr_err = cudaSuccess;
    std::call_once(attr_once, [] {
        attr_err = cudaFuncSetAttribute(prep_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                        static_cast<int>(kSmemAlloc));
    });
    if (attr_err != cudaSuccess) return GDR2_ERR_CUDA;
    if (a.cu && launch_chunk_base(a.cu, a.B, total, s.chunk_base, stream) != GDR2_OK) return GDR2_ERR_CUDA;
    const int64_t nitems = chunks * a.H;
    if (nitems >= (1ll << 31)) return GDR2_ERR_SHAPE;
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms <= 0)
        return GDR2_ERR_CUDA;
    PrepParams prm{s, a.cu, static_cast<int>(a.B), static_cast<int>(a.T), static_cast<int>(a.H),
                   static_cast<int>(total), a.cu ? 0 : cpiece, a.cu ? 0 : c0, static_cast<int>(nitems), err};
    // persistent: one CTA per SM, each looping over its items
    const unsigned grid = static_cast<unsigned>(nitems < sms ? nitems : sms);
    prep_kernel<<<grid, kThreads, kSmemAlloc, stream>>>(mq, mk, mb, mg, prm);
    return cudaPeekAtLastError() == cudaSuccess ? GDR2_OK : GDR2_ERR_CUDA;
}

}  // namespace gdr2
