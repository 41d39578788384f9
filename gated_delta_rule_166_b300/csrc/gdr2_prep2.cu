// Chunked Gated Delta Rule-2 prefill in affine form, part 1 of 2: the
// state-independent operands of every 64-token chunk, all chunks in parallel.
//
// Method ("Gated DeltaNet-2: Decoupling Erase and Write in Linear Attention"
// page: update equation, and the "efficient implementation" section's WY form
// with decay absorption and chunkwise algorithm).  For one chunk of C = 64
// tokens with cumulative log decay G_r = sum_{t<=r} g_t (per key channel),
// c = b * k, u = w * v, A_kk[r,i] = sum_j c_r k_i e^{G_r - G_i} (i < r),
// A_qk[r,i] = sum_j q_r k_i e^{G_r - G_i} (i <= r), T = (I + A_kk)^-1,
// Cb = c e^{G}, Qb = q e^{G}, Kb = k e^{G_C - G}, W = T Cb, the chunk maps its
// start state S to
//     S' = diag(e^{G_C}) S + M' S + Y U,      O = P S + X U
// with M' = -Kb^T W, Y = Kb^T T, P = Qb - A_qk W and X = A_qk T (the WY form
// with E = T U - W S folded into the state update: S' = e^{G_C} S + Kb^T E).
// Everything but U and S depends on q, k, b and g of the chunk alone.  This
// kernel computes M', Y, P, X and e^{G_C} for every (chunk, head) and writes
// them to one workspace slot as fp16 images that the chain kernel copies to
// shared memory unchanged (K-major, 128-byte swizzle).
//
// Decay factors are formed about the middle token m of each 16-token stripe:
// e^{G_r - G_i} = e^{G_r - G_m} e^{G_m - G_i} stays within e^{+-80} because
// per-token log decays are floored at -10; products of earlier stripes go
// through per-channel factors e^{G_m(R) - G_m(s)} <= 1 ("K-groups").  The
// offsets d_r = G_r - G_m come from one tensor-core product of the floored
// log decays with a constant +-1 matrix.
//
// Work split: one persistent CTA (640 threads) per SM, one (chunk, head) item
// at a time.  The 16 elementwise warps own TMEM lane quarters (warp % 4) and
// column blocks (warp / 4); thread-per-row passes write the intra-chunk product
// operands straight into TMEM (A = [Ct; Qt]) and shared memory, and elementwise
// thread 0 issues the tcgen05 MMAs once all threads have written their operands.
// One thread of the last warpgroup issues the TMA loads: the next item's tiles
// load while the current item's products, solve and slot write-out run.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>
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
constexpr int kSimt = 512;
constexpr int kThreads = kSimt + 128;
constexpr int kRegsSimt = 104, kRegsMma = 56;
static_assert(kSimt * kRegsSimt + (kThreads - kSimt) * kRegsMma <= kThreads * 96, "register pool");

// ---- shared memory (bytes from a 1024-aligned base) ------------------------------
// raw bf16 tiles, each [2 channel blocks][64 tokens][128 B] (TMA, 128-byte swizzle)
constexpr uint32_t kRawQ = 0, kRawK = 16384, kRawB = 32768, kRawG = 49152;
// K-groups [G3 (64 rows) | G1 (32) | G2 (48) | G0 (16)] x 128 channels, tf32,
// K-major: 4 K-blocks of 32 channels, each 160 rows x 128 B
constexpr uint32_t kKG = 65536, kKGStride = 20480;
// after the intra-chunk products the K-group area holds the solve and the
// operands of the affine-form products
constexpr uint32_t kB1 = kKG;              // [T^T; W^T] fp16 K-major, 192 rows x 64 K
constexpr uint32_t kAq = kKG + 24576;      // A_qk fp16 K-major, 64 rows x 64 K
constexpr uint32_t kTo = kKG + 32768;      // T fp16 K-major, 64 rows x 64 K
constexpr int kLd = 65, kLt = 68;
constexpr uint32_t kSL = kKG + 40960;      // A_kk staging [64][65] fp32
constexpr uint32_t kSTs = kSL + 64 * kLd * 4;   // T staging [64][68] fp32
constexpr uint32_t kSP = kSTs + 64 * kLt * 4;   // M_{RJ} blocks 6 x 16 x 17 fp32
static_assert(kSP + 6 * 16 * 17 * 4 <= kKG + 4 * kKGStride, "solve area");
static_assert((kSTs & 15u) == 0, "T staging alignment");
constexpr uint32_t kAG = 147456;   // constant stripe matrix, bf16 K-major 128 rows x 64 K
constexpr uint32_t kCB = 163840;   // Cb fp16 MN-major image [2][64 tokens][64 channels]
constexpr uint32_t kKB = 180224;   // Kb, same layout
constexpr uint32_t kQB = 196608;   // Qb, same layout
// per-channel decay tables, [row][128] fp32, two buffers (items alternate): e^{G_m(s)},
// e^{G_C - G_m(s)}, e^{G_m(R) - G_m(s)} (R > s, row R (R - 1) / 2 + s) and e^{G_C}
constexpr uint32_t kTab = 212992;
enum : uint32_t { kTEm = 0, kTEc = 4, kTEg = 8, kTGam = 14, kTRows = 16 };
constexpr uint32_t kTabBuf = kTRows * 512;
constexpr uint32_t kMisc = kTab + 2 * kTabBuf;
enum : uint32_t { kBarRaw = 0, kOpsRdy, kTabRdy, kGDone, kProdDone, kWDone, kDDone, kPDrain, kNumBars };
constexpr uint32_t kTmemSlot = kMisc + 8 * kNumBars;
constexpr uint32_t kSmemBytes = kMisc + 128;
constexpr uint32_t kSmemAlloc = kSmemBytes + 1024;
static_assert(kTmemSlot + 4 <= kSmemBytes, "misc area");
static_assert(kSmemAlloc <= 232448, "shared memory");
static_assert(kSlot2Bytes <= 4 * kKGStride, "slot staging in the K-group area");
// the backward record copies [W^T | A_qk | T] from the K-group area as it lies, then Kb
static_assert(kB1 + 8192u + kWyWt == kKG + 8192u && kAq == kB1 + 8192u + (kWyAq - kWyWt) &&
                  kTo == kB1 + 8192u + (kWyT - kWyWt) && kWyKb - kWyWt == 32768u && kWyBytes - kWyKb == 16384u,
              "backward record layout");

// ---- TMEM columns ---------------------------------------------------------------
// The next item's d offsets land in kTmA while this item's map products (D1, D2)
// are still in use, so those stay clear of columns 0-127.
constexpr uint32_t kTmA = 0;      // d offsets, then the A operand [Ct; Qt] (tf32), 128 columns
constexpr uint32_t kTmP = 128;    // intra-chunk products [Ct; Qt] x [G3|G1|G2|G0]^T, 160 columns
constexpr uint32_t kTmW = 320;    // W^T, 64 columns
constexpr uint32_t kTmD1 = 320;   // [Y | Kb^T W], 192 columns (after W^T is read out)
constexpr uint32_t kTmD2 = 128;   // [X | A_qk W] (M = 64), 192 columns (after the products are read out)
constexpr int kTmCols = 512;

constexpr float kMinLogDecay = -10.f;

// Slot image offsets (bytes); the chain kernel reads the same constants.
static_assert(kSlotM == 0 && kSlotY == 32768 && kSlotP == 49152 && kSlotX == 65536 && kSlotGam == 73728,
              "slot layout");

__device__ __forceinline__ void simt_sync() { team_sync<kSimt>(); }
// the table team: warps 17-19 (named barrier 2)
constexpr int kTeam = 96;
__device__ __forceinline__ void team2_sync() { asm volatile("bar.sync 2, %0;" ::"n"(kTeam) : "memory"); }
__device__ __forceinline__ bool team2_all(bool pred) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.u32 p, %1, 0;\n\t"
        "bar.red.and.pred q, 2, %2, p;\n\t"
        "selp.u32 %0, 1, 0, q;\n\t}"
        : "=r"(r)
        : "r"(pred ? 1u : 0u), "n"(kTeam)
        : "memory");
    return r != 0;
}
__device__ __forceinline__ bool simt_any(bool p) { return team_any<kSimt>(p); }
// first row of K-group R within the merged [G3 | G1 | G2 | G0] operand
__device__ __forceinline__ uint32_t group_row(int R) {
    return R == 3 ? 0u : R == 1 ? 64u : R == 2 ? 96u : 144u;
}
// Token of row m of the [Ct; Qt] operand: lane quarters hold Ct tokens 0-31, Qt
// tokens 0-31, Ct tokens 32-63, Qt tokens 32-63 (so that every SM sub-partition
// gets Ct and Qt rows alike).
__device__ __forceinline__ int row_token(int m) { return (m & 31) + 32 * (m >> 6); }

struct Prep2Params {
    uint8_t* slots;       // [items][kSlot2Bytes]
    const int* chunk_base;   // packed sequences: [N + 1] first global chunk of each sequence
    const int* cu;        // packed sequences: [N + 1] token offsets, or null
    int N, T, H, total;
    int nitems;           // global chunk bound x H; item = slot index
    int* err;
    int c0, cpiece;       // fixed-length: chunks c0 .. c0 + cpiece - 1 of every sequence
    uint8_t* wy;          // backward records [items][kWyBytes], or null (prep2_kernel<true> only)
};

struct Item {
    int tok0, T, tp, h;
};
__device__ __forceinline__ bool locate(const Prep2Params& prm, int it, Item& x) {
    const int gc = it / prm.H;
    x.h = it - gc * prm.H;
    if (prm.cu) {
        const int* cb = prm.chunk_base;
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
        const int seq = gc / prm.cpiece;
        x.tok0 = seq * prm.T;
        x.T = prm.T;
        x.tp = (prm.c0 + gc - seq * prm.cpiece) * kC;
    }
    return true;
}

// kWY: also write each item's W^T, A_qk, T and Kb images to its backward record
// (the operands of the chunk gradients, gdr2_bwd_chunk.cu).
template <bool kWY>
__global__ void __launch_bounds__(kThreads, 1)
prep2_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
             const __grid_constant__ CUtensorMap tm_b, const __grid_constant__ CUtensorMap tm_g,
             const Prep2Params prm) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t base = (smem_u32(smem_raw) + 1023u) & ~1023u;
    uint8_t* sgen = smem_raw + (base - smem_u32(smem_raw));
    float* const F = reinterpret_cast<float*>(sgen);
    auto bar = [&](uint32_t i) { return base + kMisc + 8u * i; };
    volatile uint32_t* tmem_slot = reinterpret_cast<volatile uint32_t*>(sgen + kTmemSlot);

    const int tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;
    const int quarter = warp & 3;
    auto next_item = [&](int it, Item& x) {
        for (it += gridDim.x; it < prm.nitems; it += gridDim.x)
            if (locate(prm, it, x)) return it;
        return prm.nitems;
    };

    if (tid == 0) {
        for (uint32_t i = 0; i < kNumBars; ++i) mbar_init(bar(i), 1);
        fence_mbar_init();
    }
    if (tid < kSimt) {
        // constant stripe matrix: row m (token t = row_token(m), stripe middle mid)
        // has +-1 where sum_t' A[m][t'] g_t' = G_t - G_mid
        const int m = tid >> 2, k0 = (tid & 3) * 16;
        const int t = row_token(m), mid = 16 * (t >> 4) + 7;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            uint32_t wv[4];
#pragma unroll
            for (int e = 0; e < 8; e += 2) {
                uint32_t pr = 0;
#pragma unroll
                for (int f = 0; f < 2; ++f) {
                    const int tp = k0 + 8 * h + e + f;
                    const int a = (tp <= t ? 1 : 0) - (tp <= mid ? 1 : 0);
                    const uint32_t bits = a > 0 ? 0x3F80u : a < 0 ? 0xBF80u : 0u;
                    pr |= bits << (16 * f);
                }
                wv[e / 2] = pr;
            }
            *reinterpret_cast<uint4*>(sgen + kAG + k_off16(0, static_cast<uint32_t>(m), static_cast<uint32_t>(k0 + 8 * h))) =
                make_uint4(wv[0], wv[1], wv[2], wv[3]);
        }
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
                mbar_expect_tx(bar(kBarRaw), 65536u);
                const int row = x.tok0 + x.tp;
                tma_load_4d(base + kRawQ, &tm_q, 0, x.h, row, 0, bar(kBarRaw));
                tma_load_4d(base + kRawQ + 8192, &tm_q, 64, x.h, row, 0, bar(kBarRaw));
                tma_load_4d(base + kRawK, &tm_k, 0, x.h, row, 0, bar(kBarRaw));
                tma_load_4d(base + kRawK + 8192, &tm_k, 64, x.h, row, 0, bar(kBarRaw));
                tma_load_4d(base + kRawB, &tm_b, 0, x.h, row, 0, bar(kBarRaw));
                tma_load_4d(base + kRawB + 8192, &tm_b, 64, x.h, row, 0, bar(kBarRaw));
                tma_load_4d(base + kRawG, &tm_g, 0, x.h, row, 0, bar(kBarRaw));
                tma_load_4d(base + kRawG + 8192, &tm_g, 64, x.h, row, 0, bar(kBarRaw));
            };
            bool ok = true;
            uint32_t ph = 0;
            int loads = 0;
            if (it0 < prm.nitems) { load(first); ++loads; }
#pragma unroll 1
            for (int it = it0; it < prm.nitems && ok; ph ^= 1u) {
                // pass 1 has read the raw tiles: next item's tiles
                if (!(ok = mbar_wait(bar(kOpsRdy), ph))) break;
                Item nx;
                const int nit = next_item(it, nx);
                if (nit < prm.nitems) { load(nx); ++loads; }
                it = nit;
            }
            if (!ok) {
                atomicExch(prm.err, kDevTimeout);
                if (loads > 0) mbar_wait(bar(kBarRaw), static_cast<uint32_t>((loads - 1) & 1));
            }
        } else if (warp > kSimt / 32) {
            // ---- table team (warps 17-19): per item, once its raw tiles are in, the
            // floored log decays (tokens past the sequence end: 0), the decay tables into
            // buffer (item & 1), and the d-offset product into kTmA once the previous
            // item's intra-chunk products have read that region; then kTabRdy.  The
            // elementwise warps meanwhile finish the previous item.
            const int pt = tid - (kSimt + 32);
            bool ok = true, issued = false;
            uint32_t ph = 0;
            Item cur = first;
#pragma unroll 1
            for (int it = it0, k = 0; it < prm.nitems; ph ^= 1u, ++k) {
                const int nvalid = min(cur.T - cur.tp, kC);
                if (!(ok = team2_all(mbar_wait(bar(kBarRaw), ph)))) break;
                const __nv_bfloat162 lo2 = __float2bfloat162_rn(kMinLogDecay);
#pragma unroll 1
                for (uint32_t ui = static_cast<uint32_t>(pt); ui < 1024u; ui += kTeam) {   // 16-byte units
                    const int r = static_cast<int>((ui >> 3) & 63u);
                    uint4 x = *reinterpret_cast<const uint4*>(sgen + kRawG + 16u * ui);
                    __nv_bfloat162* p2 = reinterpret_cast<__nv_bfloat162*>(&x);
#pragma unroll
                    for (int e = 0; e < 4; ++e) p2[e] = __hmax2(p2[e], lo2);
                    if (r >= nvalid) x = make_uint4(0u, 0u, 0u, 0u);
                    *reinterpret_cast<uint4*>(sgen + kRawG + 16u * ui) = x;
                }
                fence_async_smem();   // the floored tile is the B operand of the d-offset product
                team2_sync();
                float* const tb = F + ((kTab + kTabBuf * ph) >> 2);
                if (pt < kDK / 2) {
                    // channels j, j + 1 (one 32-bit word of the MN-major tile per token); the
                    // swizzled offset of token 8 q + e is e * 128 + ((c8 ^ e) << 4) + q * 1024
                    const uint32_t j = 2u * static_cast<uint32_t>(pt);
                    const uint8_t* const gt = sgen + kRawG + (j >> 6) * 8192u + ((j & 7u) << 1);
                    const uint32_t c8 = (j & 63u) >> 3;
                    float gm0[4], gm1[4], run0 = 0.f, run1 = 0.f;
#pragma unroll
                    for (int sx = 0; sx < 4; ++sx) {
                        float a0 = 0.f, a1 = 0.f, h0 = 0.f, h1 = 0.f;
#pragma unroll
                        for (int q = 0; q < 2; ++q) {
#pragma unroll
                            for (int e = 0; e < 8; ++e) {
                                const uint32_t w = *reinterpret_cast<const uint32_t*>(
                                    gt + static_cast<uint32_t>(e) * 128u + ((c8 ^ static_cast<uint32_t>(e)) << 4) +
                                    static_cast<uint32_t>(2 * sx + q) * 1024u);
                                a0 += __uint_as_float(w << 16);
                                a1 += __uint_as_float(w & 0xFFFF0000u);
                            }
                            if (q == 0) { h0 = a0; h1 = a1; }
                        }
                        gm0[sx] = run0 + h0;   // G at the stripe's middle token 16 s + 7
                        gm1[sx] = run1 + h1;
                        run0 += a0;
                        run1 += a1;
                    }
                    auto put = [&](uint32_t c, const float (&gm)[4], float gC) {
#pragma unroll
                        for (int sx = 0; sx < 4; ++sx) {
                            tb[(kTEm + sx) * 128 + c] = __expf(gm[sx]);         // e^{G_m(s)}        (<= 1)
                            tb[(kTEc + sx) * 128 + c] = __expf(gC - gm[sx]);    // e^{G_C - G_m(s)}  (<= 1)
#pragma unroll
                            for (int R = sx + 1; R < 4; ++R) tb[(kTEg + R * (R - 1) / 2 + sx) * 128 + c] = __expf(gm[R] - gm[sx]);
                        }
                        tb[kTGam * 128 + c] = __expf(gC);
                    };
                    put(j, gm0, run0);
                    put(j + 1u, gm1, run1);
                }
                team2_sync();
                bool ok0 = true;
                if (pt == 0) {
                    // the previous item's intra-chunk products have read kTmA
                    ok0 = k == 0 || mbar_wait(bar(kProdDone), ph ^ 1u);
                    if (ok0) {
                        tc_fence_after();
                        // d offsets: [A_G] (128 x 64, K-major bf16) x floored log decays (MN-major)
                        const uint64_t dAG = umma_desc2(base + kAG, 16u, 1024u), dG = umma_desc2(base + kRawG, 8192u, 1024u);
#pragma unroll
                        for (int sx = 0; sx < 4; ++sx)
                            mma_ss_f16(tmem + kTmA, dAG + 2u * sx, dG + 128u * sx, idesc_f16x(128, 128, 1, 0, 1),
                                       sx > 0 ? 1u : 0u);
                        mma_commit(bar(kGDone));
                        issued = true;
                        mbar_arrive(bar(kTabRdy));   // tables (ordered by the team barrier) and floor done
                    }
                }
                if (!(ok = team2_all(ok0))) break;
                Item nx;
                it = next_item(it, nx);
                cur = nx;
            }
            if (!ok && pt == 0) atomicExch(prm.err, kDevTimeout);
            if (pt == 0 && issued) {
                // a d-offset product still in flight completes before the TMEM is freed
                mma_commit(bar(kPDrain));
                mbar_wait(bar(kPDrain), 0u);
            }
        }
        __syncwarp();
    } else {
        // ================= 16 elementwise / accumulator warps =====================
        asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kRegsSimt));
        const uint32_t lane_base = static_cast<uint32_t>(quarter * 32) << 16;
        const int cg = warp >> 2;   // column block of this warp
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
        // Operands written by all elementwise threads -> visible to the tensor core; then
        // thread 0 issues the products (and commits them to `b`) itself.
        auto operands_done = [&]() {
            fence_async_smem();
            tc_fence_before();
            simt_sync();
            tc_fence_after();
        };

        uint32_t ph = 0;
        Item cur = first;
#pragma unroll 1
        for (int it = it0; it < prm.nitems && !failed; ph ^= 1u) {
            const int nvalid = min(cur.T - cur.tp, kC);   // tokens of this chunk inside the sequence
            uint8_t* const slot = prm.slots + static_cast<int64_t>(it) * kSlot2Bytes;
            float* const tab = F + ((kTab + kTabBuf * ph) >> 2);   // this item's decay tables
            // the table team has floored the log decays, written the tables and issued the
            // d-offset product (the raw tiles are in)
            if (!wait_done(kTabRdy, ph)) { failed = true; break; }
            if (tid == 0) bulk_wait_read();   // the previous item's slot copy has left the K-group area
            simt_sync();
            // ---- pass 1, one token row per thread: [Ct; Qt] -> TMEM, K-groups, Cb, Kb, Qb ----
            if (!wait_done(kGDone, ph)) { failed = true; break; }
            {
                const int L = 32 * quarter + lane;
                const bool is_q = quarter & 1;
                const int r = row_token(L), s = r >> 4;
                const bool valid = r < nvalid;
                const uint32_t rr = static_cast<uint32_t>(r);
                const uint32_t cb = static_cast<uint32_t>(cg >> 1);
#pragma unroll 1
                for (int h = 0; h < 2; ++h) {
                    const int c0 = 32 * cg + 16 * h;   // first channel of these 16
                    uint32_t dr[16];
                    tmem_ld16_nw(tmem + lane_base + kTmA + static_cast<uint32_t>(c0), dr);
                    // raw rows: 16 channels = two 16-byte chunks of each tile
                    uint4 xa[2], xk[2];
                    const uint32_t ua = static_cast<uint32_t>(4 * (cg & 1) + 2 * h);
#pragma unroll
                    for (int u = 0; u < 2; ++u) {
                        const uint32_t off = cb * 8192u + rr * 128u + (((ua + u) ^ (rr & 7u)) << 4);
                        xa[u] = *reinterpret_cast<const uint4*>(sgen + (is_q ? kRawQ : kRawB) + off);
                        xk[u] = *reinterpret_cast<const uint4*>(sgen + kRawK + off);
                        if (!valid) { xa[u] = make_uint4(0u, 0u, 0u, 0u); xk[u] = xa[u]; }
                    }
                    tmem_ld_wait();
                    const uint32_t* wa = reinterpret_cast<const uint32_t*>(xa);
                    const uint32_t* wk = reinterpret_cast<const uint32_t*>(xk);
                    float kk[16], ro[16], rop[16], rin[16];
#pragma unroll
                    for (int e = 0; e < 16; e += 2) {
                        const uint32_t a2 = wa[e / 2], k2 = wk[e / 2];
                        const float a0 = __uint_as_float(a2 << 16), a1 = __uint_as_float(a2 & 0xFFFF0000u);
                        kk[e] = __uint_as_float(k2 << 16);
                        kk[e + 1] = __uint_as_float(k2 & 0xFFFF0000u);
                        const float d0 = __uint_as_float(dr[e]), d1 = __uint_as_float(dr[e + 1]);
                        const float p0 = __expf(d0), p1 = __expf(d1);          // e^{G_r - G_m}
                        rin[e] = __expf(-d0);                                  // e^{G_m - G_r}
                        rin[e + 1] = __expf(-d1);
                        // Ct = b k e^{d} (Ct rows) or Qt = q e^{d} (Qt rows)
                        rop[e] = (is_q ? a0 : a0 * kk[e]) * p0;
                        rop[e + 1] = (is_q ? a1 : a1 * kk[e + 1]) * p1;
                        ro[e] = tf32r(rop[e]);
                        ro[e + 1] = tf32r(rop[e + 1]);
                    }
                    tmem_st16(tmem + lane_base + kTmA + static_cast<uint32_t>(c0), ro);
                    // Cb = c e^{G} (Ct rows) or Qb = q e^{G} (Qt rows), fp16, token-major image
                    {
                        const float* em = tab + (kTEm + s) * 128 + c0;
                        uint32_t pw[8];
#pragma unroll
                        for (int e = 0; e < 16; e += 2) pw[e / 2] = pack_h2(rop[e] * em[e], rop[e + 1] * em[e + 1]);
                        const uint32_t img = is_q ? kQB : kCB;
#pragma unroll
                        for (int u = 0; u < 2; ++u)
                            *reinterpret_cast<uint4*>(sgen + img + cb * 8192u + rr * 128u + (((ua + u) ^ (rr & 7u)) << 4)) =
                                make_uint4(pw[4 * u], pw[4 * u + 1], pw[4 * u + 2], pw[4 * u + 3]);
                    }
                    // key rows k e^{G_m(R) - G_r} of the K-groups R >= s: Ct rows write G3 and
                    // (s <= 1) G2; Qt rows write G1 (s <= 1), G0 (s = 0) and G2 (s = 2)
                    auto put_group = [&](int R) {
                        const float* eg = R == s ? nullptr : tab + (kTEg + R * (R - 1) / 2 + s) * 128 + c0;
                        float v[16];
#pragma unroll
                        for (int e = 0; e < 16; ++e) v[e] = tf32r(kk[e] * rin[e] * (eg ? eg[e] : 1.f));
                        const uint32_t row = group_row(R) + rr;
                        const uint32_t kb = static_cast<uint32_t>(c0 >> 5), c4 = static_cast<uint32_t>((c0 & 31) >> 2);
#pragma unroll
                        for (int u = 0; u < 4; ++u)
                            *reinterpret_cast<float4*>(sgen + kKG + kb * kKGStride + row * 128u + (((c4 + u) ^ (row & 7u)) << 4)) =
                                make_float4(v[4 * u], v[4 * u + 1], v[4 * u + 2], v[4 * u + 3]);
                    };
                    if (!is_q) {
                        put_group(3);
                        if (s <= 1) put_group(2);
                        // Kb = k e^{G_C - G_r}, fp16, token-major image
                        const float* ec = tab + (kTEc + s) * 128 + c0;
                        uint32_t pw[8];
#pragma unroll
                        for (int e = 0; e < 16; e += 2)
                            pw[e / 2] = pack_h2(kk[e] * rin[e] * ec[e], kk[e + 1] * rin[e + 1] * ec[e + 1]);
#pragma unroll
                        for (int u = 0; u < 2; ++u)
                            *reinterpret_cast<uint4*>(sgen + kKB + cb * 8192u + rr * 128u + (((ua + u) ^ (rr & 7u)) << 4)) =
                                make_uint4(pw[4 * u], pw[4 * u + 1], pw[4 * u + 2], pw[4 * u + 3]);
                    } else {
                        if (s <= 1) put_group(1);
                        if (s == 0) put_group(0);
                        if (s == 2) put_group(2);
                    }
                }
                tmem_st_wait();
            }
            signal(kOpsRdy);   // raw tiles read (next item's tiles may load); operands visible
            if (tid == 0) {
                tc_fence_after();
                // intra-chunk products [Ct; Qt] (TMEM, tf32) x K-groups^T
                const uint64_t dKG = umma_desc(base + kKG);
#pragma unroll
                for (int s = 0; s < 16; ++s)
                    mma_ts(tmem + kTmP, tmem + kTmA + 8u * s, dKG + (kKGStride >> 4) * (s >> 2) + 2u * (s & 3),
                           idesc_tf32(128, 160), s > 0 ? 1u : 0u);
                mma_commit(bar(kProdDone));
            }
            // ---- A_kk, A_qk out of TMEM; T = (I + A_kk)^-1 --------------------------------------
            if (!wait_done(kProdDone, ph)) { failed = true; break; }
            {
                const int L = 32 * quarter + lane;
                const bool is_q = quarter & 1;
                const int r = row_token(L), rs = r >> 4;
                const int s0 = 2 * (quarter >> 1);   // the two stripes of this quarter
                const int Rb = warp >> 2;            // 16-column block of the K-group
                float ra[16], rb[16];
                if (Rb <= s0) tmem_ld16(tmem + lane_base + kTmP + group_row(s0) + 16u * Rb, ra);
                if (Rb <= s0 + 1) tmem_ld16(tmem + lane_base + kTmP + group_row(s0 + 1) + 16u * Rb, rb);
                const bool have = Rb <= rs;
                float out[16];
#pragma unroll
                for (int e = 0; e < 16; ++e) out[e] = have ? (rs == s0 ? ra[e] : rb[e]) : 0.f;
                if (!is_q) {
#pragma unroll
                    for (int e = 0; e < 16; ++e) {
                        const int i = 16 * Rb + e;
                        if (i < r) F[(kSL >> 2) + r * kLd + i] = out[e];
                    }
                } else {
                    uint32_t pw[8];
#pragma unroll
                    for (int e = 0; e < 16; e += 2) {
                        const int i = 16 * Rb + e;
                        pw[e / 2] = pack_h2(i <= r ? out[e] : 0.f, i + 1 <= r ? out[e + 1] : 0.f);
                    }
#pragma unroll
                    for (int u = 0; u < 2; ++u)
                        *reinterpret_cast<uint4*>(sgen + kAq + k_off16(0, static_cast<uint32_t>(r), static_cast<uint32_t>(16 * Rb + 8 * u))) =
                            make_uint4(pw[4 * u], pw[4 * u + 1], pw[4 * u + 2], pw[4 * u + 3]);
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
            const float* Lm = F + (kSL >> 2);
            float* Ts = F + (kSTs >> 2);
            float* SP = F + (kSP >> 2);
            // 16x16 diagonal blocks by column forward substitution
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
                        const float a = Lm[(o16 + r) * kLd + o16 + i];
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
                    const float* lr = Lm + (16 * Rb + x) * kLd + 16 * Jb + c4;
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
            // T (rows r, K = i) and T^T (rows 0..63 of [T^T; W^T]) as fp16 operands
            {
                const int n = tid & 63, k0 = (tid >> 6) * 8;
                uint32_t pr[4], pc[4];
#pragma unroll
                for (int e = 0; e < 8; e += 2) {
                    pr[e / 2] = pack_h2(Ts[n * kLt + k0 + e], Ts[n * kLt + k0 + e + 1]);
                    pc[e / 2] = pack_h2(Ts[(k0 + e) * kLt + n], Ts[(k0 + e + 1) * kLt + n]);
                }
                *reinterpret_cast<uint4*>(sgen + kTo + k_off16(0, static_cast<uint32_t>(n), static_cast<uint32_t>(k0))) =
                    make_uint4(pr[0], pr[1], pr[2], pr[3]);
                *reinterpret_cast<uint4*>(sgen + kB1 + k_off16(0, static_cast<uint32_t>(n), static_cast<uint32_t>(k0))) =
                    make_uint4(pc[0], pc[1], pc[2], pc[3]);
            }
            operands_done();
            if (tid == 0) {
                // W^T = Cb^T T^T  (A: Cb, MN-major; B: T, K-major)
                const uint64_t dCB = umma_desc2(base + kCB, 8192u, 1024u), dTo = umma_desc2(base + kTo, 16u, 1024u);
#pragma unroll
                for (int s = 0; s < 4; ++s)
                    mma_ss_f16(tmem + kTmW, dCB + 128u * s, dTo + 2u * s, idesc_f16x(128, 64, 0, 1, 0), s > 0 ? 1u : 0u);
                mma_commit(bar(kWDone));
            }
            // ---- W^T out of TMEM -> rows 64 .. 191 of [T^T; W^T] ----------------------------
            if (!wait_done(kWDone, ph)) { failed = true; break; }
            {
                const int j = 32 * quarter + lane;
                float v[16];
                tmem_ld16(tmem + lane_base + kTmW + 16u * static_cast<uint32_t>(cg), v);
                uint32_t pw[8];
#pragma unroll
                for (int e = 0; e < 16; e += 2) pw[e / 2] = pack_h2(v[e], v[e + 1]);
#pragma unroll
                for (int u = 0; u < 2; ++u)
                    *reinterpret_cast<uint4*>(sgen + kB1 + k_off16(0, static_cast<uint32_t>(64 + j), static_cast<uint32_t>(16 * cg + 8 * u))) =
                        make_uint4(pw[4 * u], pw[4 * u + 1], pw[4 * u + 2], pw[4 * u + 3]);
            }
            operands_done();
            if (tid == 0) {
                // [Y | Kb^T W] = Kb^T [T^T; W^T]^T and [X | A_qk W] = A_qk [T^T; W^T]^T
                const uint64_t dKB = umma_desc2(base + kKB, 8192u, 1024u), dB1 = umma_desc2(base + kB1, 16u, 1024u);
                const uint64_t dAq = umma_desc2(base + kAq, 16u, 1024u);
#pragma unroll
                for (int s = 0; s < 4; ++s) {
                    mma_ss_f16(tmem + kTmD1, dKB + 128u * s, dB1 + 2u * s, idesc_f16x(128, 192, 0, 1, 0), s > 0 ? 1u : 0u);
                    mma_ss_f16(tmem + kTmD2, dAq + 2u * s, dB1 + 2u * s, idesc_f16x(64, 192, 0, 0, 0), s > 0 ? 1u : 0u);
                }
                mma_commit(bar(kDDone));
                if (kWY) {
                    // backward record: [W^T | A_qk | T] (contiguous in the K-group area) and Kb
                    uint8_t* const rec = prm.wy + static_cast<int64_t>(it) * kWyBytes;
                    bulk_s2g(rec + kWyWt, base + kB1 + 8192u, kWyKb - kWyWt);
                    bulk_s2g(rec + kWyKb, base + kKB, kWyBytes - kWyKb);
                    bulk_commit();
                }
            }
            // ---- slot images: Y, M' = -Kb^T W (rows d_k), X, P = Qb - A_qk W (rows tokens) ----
            // K-major fp16 images staged in the K-group area (its operands are consumed),
            // then one bulk copy to the workspace slot
            if (!wait_done(kDDone, ph)) { failed = true; break; }
            if (kWY) {
                if (tid == 0) bulk_wait_read();   // the record copy has read the K-group area
                simt_sync();
            }
            uint8_t* const stage = sgen + kKG;
            {
                auto put_row = [&](uint32_t img, uint32_t kblk, uint32_t row, uint32_t k0, const float (&v)[16], bool neg) {
                    uint32_t w[8];
#pragma unroll
                    for (int e = 0; e < 16; e += 2) w[e / 2] = neg ? pack_h2(-v[e], -v[e + 1]) : pack_h2(v[e], v[e + 1]);
                    *reinterpret_cast<uint4*>(stage + img + k_off16(kblk, row, k0)) = make_uint4(w[0], w[1], w[2], w[3]);
                    *reinterpret_cast<uint4*>(stage + img + k_off16(kblk, row, k0 + 8u)) = make_uint4(w[4], w[5], w[6], w[7]);
                };
                const uint32_t j = static_cast<uint32_t>(32 * quarter + lane);   // D1 lane: key channel (row of Y and M')
                float v[16];
#pragma unroll 1
                for (int t3 = 0; t3 < 3; ++t3) {
                    const uint32_t col = static_cast<uint32_t>(48 * cg + 16 * t3);
                    tmem_ld16(tmem + lane_base + kTmD1 + col, v);
                    if (col < 64) put_row(kSlotY, 0u, j, col, v, false);
                    else put_row(kSlotM, 16384u, j, col - 64u, v, true);
                }
                // M' and Y leave while X and P are staged
                fence_async_smem();
                simt_sync();
                if (tid == 0) bulk_s2g(slot, base + kKG, kSlotP);
                // D2 (M = 64): row r at lanes 32 (r / 16) + r % 16
                const uint32_t r = static_cast<uint32_t>(16 * quarter + (lane & 15));
                const bool active = lane < 16;
#pragma unroll 1
                for (int t3 = 0; t3 < 3; ++t3) {
                    const uint32_t col = static_cast<uint32_t>(48 * cg + 16 * t3);
                    tmem_ld16(tmem + lane_base + kTmD2 + col, v);
                    if (!active) continue;
                    if (col < 64) {
                        put_row(kSlotX, 0u, r, col, v, false);
                    } else {
                        const uint32_t j0 = col - 64u;
#pragma unroll
                        for (int u = 0; u < 2; ++u) {
                            const uint32_t jj = j0 + 8u * u;
                            const uint4 x = *reinterpret_cast<const uint4*>(
                                sgen + kQB + (jj >> 6) * 8192u + r * 128u + ((((jj & 63u) >> 3) ^ (r & 7u)) << 4));
                            const __half2* h2 = reinterpret_cast<const __half2*>(&x);
#pragma unroll
                            for (int e = 0; e < 8; e += 2) {
                                const float2 qf = __half22float2(h2[e / 2]);
                                v[8 * u + e] = qf.x - v[8 * u + e];
                                v[8 * u + e + 1] = qf.y - v[8 * u + e + 1];
                            }
                        }
                        put_row(kSlotP, 8192u, r, j0, v, false);
                    }
                }
                if (tid < kDK) reinterpret_cast<float*>(stage + kSlotGam)[tid] = tab[kTGam * 128 + tid];
            }
            fence_async_smem();
            tc_fence_before();
            simt_sync();   // D2, the Qb image and the staged slot are complete
            if (tid == 0) {
                bulk_s2g(slot + kSlotP, base + kKG + kSlotP, static_cast<uint32_t>(kSlot2Bytes) - kSlotP);
                bulk_commit();
            }
            Item nx;
            it = next_item(it, nx);
            cur = nx;
        }
        if (tid == 0) bulk_wait_all();   // the last slot copy completes before the CTA exits
        if (failed && tid == 0) atomicExch(prm.err, kDevTimeout);
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc<kTmCols>(tmem);
    }
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

// First global chunk of each packed sequence: cb[s] = sum_{s' < s} ceil(len_s' / 64),
// with the same offset clamping the kernels use, capped at the workspace's chunk bound
// ceil(total / 64) + N.  Valid offsets never reach the cap (each sequence adds at most
// one partial chunk); overlapping malformed ones can, and then the sequences past the
// cap get fewer chunks (cb[s + 1] - cb[s]) than their length, so that no kernel indexes
// a chunk beyond the workspace.  One CTA.
__global__ void chunk_base_kernel(const int* cu, int N, int total, int* cb) {
    __shared__ long long part[1024];
    const int tid = threadIdx.x;
    const int per = (N + blockDim.x - 1) / blockDim.x;
    const int s0 = tid * per, s1 = min(N, s0 + per);
    const long long cap = min(static_cast<long long>((total + kC - 1) / kC) + N, 0x7fffffffLL);
    auto nch = [&](int s) {
        const int a = min(max(cu[s], 0), total);
        const int e = min(max(cu[s + 1], a), total);
        return static_cast<long long>((e - a + kC - 1) / kC);
    };
    long long sum = 0;
    for (int s = s0; s < s1; ++s) sum += nch(s);
    part[tid] = sum;
    __syncthreads();
    if (tid == 0) {   // exclusive scan of the partial sums
        long long run = 0;
        for (int i = 0; i < static_cast<int>(blockDim.x); ++i) {
            const long long x = part[i];
            part[i] = run;
            run += x;
        }
    }
    __syncthreads();
    long long run = part[tid];
    for (int s = s0; s < s1; ++s) {
        cb[s] = static_cast<int>(min(run, cap));
        run += nch(s);
    }
    if (s1 == N && s0 < s1) cb[N] = static_cast<int>(min(run, cap));
    if (N == 0 && tid == 0) cb[0] = 0;
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

int launch_prep2(const ForwardArgs& a, uint8_t* slots, const int* chunk_base, int64_t chunks, cudaStream_t stream,
                 int* err, int c0, int cpiece, uint8_t* wy) {
    const int64_t total = a.cu ? a.total : a.B * a.T;
    if (chunks <= 0) return GDR2_OK;
    const int64_t nitems = chunks * a.H;
    if (nitems >= (1ll << 31)) return GDR2_ERR_SHAPE;
    CUtensorMap mq, mk, mb, mg;
    if (!make_token_map(&mq, a.q, total, a.H, a.dk) || !make_token_map(&mk, a.k, total, a.H, a.dk) ||
        !make_token_map(&mb, a.b, total, a.H, a.dk) || !make_token_map(&mg, a.g, total, a.H, a.dk))
        return GDR2_ERR_CUDA;
    static std::once_flag attr_once;
    static cudaError_t attr_err = cudaSuccess;
    std::call_once(attr_once, [] {
        attr_err = cudaFuncSetAttribute(prep2_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                        static_cast<int>(kSmemAlloc));
        if (attr_err == cudaSuccess)
            attr_err = cudaFuncSetAttribute(prep2_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                            static_cast<int>(kSmemAlloc));
    });
    if (attr_err != cudaSuccess) return GDR2_ERR_CUDA;
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms <= 0)
        return GDR2_ERR_CUDA;
    const int nch = static_cast<int>((a.T + kC - 1) / kC);
    if (!a.cu && (c0 < 0 || cpiece < 0 || c0 + cpiece > nch)) return GDR2_ERR_ARG;
    Prep2Params prm{slots, chunk_base, a.cu, static_cast<int>(a.B), static_cast<int>(a.T), static_cast<int>(a.H),
                    static_cast<int>(total), static_cast<int>(nitems), err, c0, cpiece > 0 ? cpiece : nch, wy};
    const unsigned grid = static_cast<unsigned>(nitems < sms ? nitems : sms);
    if (wy)
        prep2_kernel<true><<<grid, kThreads, kSmemAlloc, stream>>>(mq, mk, mb, mg, prm);
    else
        prep2_kernel<false><<<grid, kThreads, kSmemAlloc, stream>>>(mq, mk, mb, mg, prm);
    return cudaPeekAtLastError() == cudaSuccess ? GDR2_OK : GDR2_ERR_CUDA;
}

}  // namespace gdr2
