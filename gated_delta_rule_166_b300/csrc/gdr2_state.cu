// Chunked Gated Delta Rule-2 prefill, part 2 of 2: the chunk-to-chunk state
// pass, one CTA per (sequence*head, 64-column d_v tile).
//
// Method ("Gated DeltaNet-2: Decoupling Erase and Write in Linear Attention"
// page, "efficient implementation" section: chunkwise algorithm).  With the
// state-independent operands of each chunk read from its workspace slot
// (written by the preparation kernel), the chunk with initial state S is
//     A1 = [T; A_qk T] (-Cb) + [0; Qb] = [-W; P]
//     [E; O] = [T; A_qk T] U + A1 S,            U = w * v
//     S <- diag(e^{G_C}) S + Kb^T E
// The products run on tcgen05 tensor cores (kind::tf32, fp32 accumulators in
// TMEM); U and E enter as tf32 pairs x = x_hi + x_lo.  Every thread keeps its
// 16 entries of the fp32 state in registers for the whole sequence.
//
// Only A1 S, the E read-out, Kb^T E and the state update are on the
// chunk-to-chunk chain.  [T; A_qk T] U of the next chunk is issued while the
// state update runs and A1 of the next chunk while E is read out, so the
// state-independent products overlap the chain.
//
// Operands: [T; A_qk T], A1 and Kb^T are TMEM-resident A operands (so every
// product reads one operand from shared memory); S^T, U^T, E^T and -Cb^T are
// shared-memory B operands; the v, w tiles (two buffers) arrive by TMA and O
// leaves through a shared-memory tile and a TMA store.
//
// Work split: 640 threads.  One thread of the last warpgroup issues the TMA
// loads and all MMAs.  Warp w < 16 owns TMEM lane quarter q = w % 4 (lanes
// 32q..32q+31) and column block R = w / 4; thread j = tid % 128 is TMEM lane j
// and key channel j.  Warps of quarters 0-1 read E out (token rows 0..63),
// warps of quarters 2-3 write O and complete P.  Warps signal the MMA thread
// through mbarriers (one arrival per warp), so no CTA-wide barrier sits on the
// chain.
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
constexpr int kDVT = 64;                // value columns per CTA
constexpr int kSimt = 512;
constexpr int kThreads = kSimt + 128;
constexpr int kRegsSimt = 112, kRegsMma = 32;
static_assert(kSimt * kRegsSimt + (kThreads - kSimt) * kRegsMma <= kThreads * 96, "register pool");

// ---- shared memory (bytes from a 1024-aligned base); K-major, 128-byte swizzle ----
constexpr uint32_t kVW = 0;            // two buffers of {v, w} bf16 tiles [64 tokens][64 d_v] (16 KB each)
constexpr uint32_t kCbT = 32768;       // -Cb^T fp16: 128 rows (channels) x 64 K (tokens), one 128 B K-block
constexpr uint32_t kSt = 49152;        // S^T tf32: 64 rows (d_v) x 128 K (channels)
constexpr uint32_t kU = 81920;         // [U_hi^T; U_lo^T] fp16: 128 rows x 64 K (tokens)
constexpr uint32_t kE = 98304;         // [E_hi^T; E_lo^T] tf32: 128 rows x 64 K (tokens)
constexpr uint32_t kO = 131072;        // O tile for the TMA store: [64 tokens][64 d_v] (16 KB)
constexpr uint32_t kMisc = 147456;
enum : uint32_t {
    kBarVW = 0, kBarVWb,                                    // TMA completions
    kRdyA1, kRdyA0, kRdyU, kRdyChain, kRdyMma2,             // elementwise warps -> MMA thread
    kOFull, kOFree,                                         // O tile: written / stored
    kDoneC1, kDoneC2, kDoneP3,                     // MMA commits
    kNumBars
};
constexpr uint32_t kTmemSlot = kMisc + 8 * kNumBars;
constexpr uint32_t kAbort = kTmemSlot + 4;
constexpr uint32_t kSmemBytes = kMisc + 128;
constexpr uint32_t kSmemAlloc = kSmemBytes + 1024;
static_assert(kAbort + 4 <= kSmemBytes, "misc area");
static_assert(kSmemAlloc <= 232448, "shared memory");

// ---- TMEM columns ------------------------------------------------------------------
constexpr uint32_t kTmA1 = 0;      // [-W; P] (A operand, K = 128 channels)
constexpr uint32_t kTmA2 = 128;    // Kb^T (A operand: lanes = channels, K = 64 tokens)
constexpr uint32_t kTmEO = 192;    // [E; O] as two 64-column halves (hi | lo products)
constexpr uint32_t kTmD2 = 320;    // Kb^T E as two 64-column halves
constexpr uint32_t kTmA0 = 448;    // [T; A_qk T] fp16 pairs (A operand, K = 64 tokens in 32 columns)
constexpr int kTmCols = 512;

struct StateParams {
    PrepSlots s;
    const float* S0;
    void* o;
    float* ST;
    int* err;
    const int* cu;
    int T, H, dv, total, nchunks;   // nchunks: chunks per sequence in this launch when cu is null
    int c0;                         // first chunk of each sequence in this launch (cu null)
    int chunk_bound;                // global chunks with a workspace slot
    int out_bf16;
    // Segmented pass (fixed-length sequences, G > 1): blockIdx.x = (sequence * G + g) * H
    // + head runs chunks g*L .. g*L + L - 1.  Value tiles of segment 0 start from S0
    // and write o; those of later segments start from zero and write fp32 rows to
    // o32.  Transfer tiles (blockIdx.y >= dv / 64, segments g >= 1) start from the
    // identity columns j0.. of d_k with U = 0 and write r_t = M_t^T q_t to r.  Every
    // tile leaves its end state in seg_state ([sequence][head][g][d_k][dv], value) or
    // seg_m ([sequence][head][g][d_k][d_k], transfer).
    int G, L;
    int Tr;                         // rows per sequence of o32 and r: T - L * 64
    float* seg_state;
    float* seg_m;
    float* o32;                     // [N * Tr][H][dv] fp32
    float* r;                       // [N * Tr][H][d_k] fp32
    // the state after every cache_chunks chunks: [N][H][n_cache][d_k][dv] (null: not kept)
    float* cache;
    int cache_chunks, n_cache;
};

// Element (token t, column n) of a TMA-loaded bf16 [64][64] tile (128-byte rows, swizzled).
__device__ __forceinline__ uint32_t vw_off(int t, int n) {
    return static_cast<uint32_t>(t) * 128u + ((static_cast<uint32_t>(n >> 3) ^ (static_cast<uint32_t>(t) & 7u)) << 4) +
           (static_cast<uint32_t>(n & 7) << 1);
}

// One CTA of the state pass; kTransfer: a transfer tile (identity start, U = 0).
// The two kinds are separate instantiations so that value tiles carry no test of
// the tile kind on their chain.
template <bool kTransfer, bool kCache>
__device__ __forceinline__ void state_cta(const CUtensorMap& tm_v, const CUtensorMap& tm_w, const CUtensorMap& tm_o,
                                          const CUtensorMap& tm_o32, const CUtensorMap& tm_r,
                                          const StateParams& prm) {
    constexpr bool mtile = kTransfer;
    // segment and output routing (uniform over the CTA)
    const int ntv = prm.dv / kDVT;
    const int h = static_cast<int>(blockIdx.x) % prm.H;
    const int sg = static_cast<int>(blockIdx.x) / prm.H;
    const int seq = sg / prm.G, g = sg % prm.G;
    if (mtile && g == 0) return;   // segment 0 starts from S0 itself: no transfer needed
    const int bh = seq * prm.H + h;
    const int j0 = (mtile ? static_cast<int>(blockIdx.y) - ntv : static_cast<int>(blockIdx.y)) * kDVT;

    extern __shared__ uint8_t smem_raw[];
    const uint32_t base = (smem_u32(smem_raw) + 1023u) & ~1023u;
    uint8_t* sgen = smem_raw + (base - smem_u32(smem_raw));
    float* const F = reinterpret_cast<float*>(sgen);
    auto bar = [&](uint32_t i) { return base + kMisc + 8u * i; };
    volatile uint32_t* tmem_slot = reinterpret_cast<volatile uint32_t*>(sgen + kTmemSlot);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(sgen + kAbort);

    const int tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;
    const int j = tid & 127;
    const int R = (tid >> 7) & 3;
    const int quarter = warp & 3;
    int tok0, T, cb0;
    if (prm.cu) {
        const int a = min(max(prm.cu[seq], 0), prm.total);
        const int e = min(max(prm.cu[seq + 1], a), prm.total);
        tok0 = a;
        T = e - a;
        cb0 = prm.s.chunk_base[seq];
    } else {
        // chunks c0 + g L .. c0 + nchunks - 1: token offsets relative to the first of them
        tok0 = seq * prm.T + (prm.c0 + g * prm.L) * kC;
        T = prm.T - (prm.c0 + g * prm.L) * kC;
        cb0 = seq * prm.nchunks + g * prm.L;
    }
    // Well-formed offsets never reach the slot bound; overlapping malformed ones
    // can, and their chunks past it are not run (the sequence is truncated).
    int n = min((T + kC - 1) / kC, max(prm.chunk_bound - cb0, 0));
    if (!prm.cu) n = min(n, min(prm.nchunks - g * prm.L, prm.L));
    // o rows: the caller's o (whole sequence, or segment 0), else fp32 scratch rows
    const bool to_o = prm.G == 1 || (!mtile && g == 0);
    const CUtensorMap* const om = to_o ? &tm_o : (mtile ? &tm_r : &tm_o32);
    const bool obf16 = to_o && prm.out_bf16;
    const int ow = mtile ? kDK : prm.dv;
    const int orow0 = to_o ? tok0 : seq * prm.Tr + (g - 1) * prm.L * kC;
    auto slot = [&](int c) { return static_cast<int64_t>(cb0 + c) * prm.H + h; };

    if (tid == 0) {
        for (uint32_t i = 0; i < kNumBars; ++i) {
            // one arrival per warp: 8 E warps (the Kb^T E operand), 8 O warps (A1, U
            // operands, O tile), all 16 ([T; A_qk T] and the chain)
            const uint32_t cnt = (i == kRdyChain || i == kRdyA0) ? 16u
                                 : (i == kRdyA1 || i == kRdyU || i == kRdyMma2 || i == kOFull) ? 8u
                                                                                                             : 1u;
            mbar_init(bar(i), cnt);
        }
        *abort_flag = 0;
        fence_mbar_init();
        fence_async_smem();
    }
    if (warp == 0) tmem_alloc<kTmCols>(base + kTmemSlot);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp >= kSimt / 32) {
        // ================= TMA / MMA warpgroup: one elected thread =================
        asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kRegsMma));
        if (warp == kSimt / 32 && lane == 0) {
            // TMA batches issued per barrier kBarVW + i (i = 0, 1): any (bit i of iss_any) and
            // the parity of their count (bit i of iss_par); bit-packed to stay in registers
            uint32_t iss_any = 0, iss_par = 0;
            auto load_vw = [&](int c) {
                if (mtile) return;   // U = 0: no v, w tiles
                const uint32_t b = bar(kBarVW + (c & 1));
                const uint32_t dst = base + kVW + static_cast<uint32_t>(c & 1) * 16384u;
                const int row = tok0 + c * kC;
                mbar_expect_tx(b, 16384u);
                tma_load_4d(dst, &tm_v, j0, h, row, 0, b);
                tma_load_4d(dst + 8192u, &tm_w, j0, h, row, 0, b);
                iss_any |= 1u << (c & 1);
                iss_par ^= 1u << (c & 1);
            };
            auto wait = [&](uint32_t b, uint32_t& ph) {
                const bool ok = mbar_wait_ab(bar(b), ph, abort_flag);
                ph ^= 1u;
                return ok;
            };
            uint32_t ph_a0 = 0, ph_a1 = 0, ph_u = 0, ph_chain = 0, ph_mma2 = 0, ph_c1 = 0;
            // A1(c) = [T; A_qk T](c) (-Cb^T)(c)
            auto issue_a1 = [&]() {
                if (!wait(kRdyA1, ph_a1) || !wait(kRdyA0, ph_a0)) return false;
                tc_fence_after();
#pragma unroll 1
                for (int s = 0; s < 4; ++s)   // kind::f16, K = 16 per step
                    mma_ts_f16(tmem + kTmA1, tmem + kTmA0 + 8u * s, umma_desc(base + kCbT + 32u * s),
                               idesc_f16(128, 128), s > 0 ? 1u : 0u);
                mma_commit(bar(kDoneP3));
                return true;
            };
            // [E; O](c) halves := [T; A_qk T](c) [U_hi^T; U_lo^T](c)
            auto issue_u = [&]() {
                // the E warps finished reading [E; O] before Kb^T E was issued; the O
                // warps signal U after reading their half
                if (!wait(kRdyU, ph_u)) return false;
                tc_fence_after();
#pragma unroll 1
                for (int s = 0; s < 4; ++s)   // kind::f16, K = 16 per step
                    mma_ts_f16(tmem + kTmEO, tmem + kTmA0 + 8u * s, umma_desc(base + kU + 32u * s),
                               idesc_f16(128, 128), s > 0 ? 1u : 0u);
                return true;
            };
            bool ok = true;
            if (n > 0) {
                load_vw(0);
                if (n > 1) load_vw(1);
                ok = issue_a1() && issue_u();
                if (ok && n > 2) load_vw(2);
            }
#pragma unroll 1
            for (int c = 0; c < n && ok; ++c) {
                // chain: [E; O] += A1 S^T, the d_k sum split over both halves
                if (!(ok = wait(kRdyChain, ph_chain))) break;
                tc_fence_after();
#pragma unroll 1
                for (int s = 0; s < 8; ++s) {
                    mma_ts(tmem + kTmEO, tmem + kTmA1 + 8u * s, umma_desc(kstep(base + kSt, 8192, s)),
                           idesc_tf32(128, kDVT), 1u);
                    mma_ts(tmem + kTmEO + 64u, tmem + kTmA1 + 8u * (s + 8), umma_desc(kstep(base + kSt, 8192, s + 8)),
                           idesc_tf32(128, kDVT), 1u);
                }
                mma_commit(bar(kDoneC1));
                if (c + 1 < n) {
                    // A1 of the next chunk once this pass has read A1 (runs during the E read-out)
                    if (!(ok = wait(kDoneC1, ph_c1))) break;
                    if (!(ok = issue_a1())) break;
                }
                // chain: Kb^T [E_hi^T; E_lo^T]
                if (!(ok = wait(kRdyMma2, ph_mma2))) break;
                tc_fence_after();
#pragma unroll 1
                for (int s = 0; s < 8; ++s)
                    mma_ts(tmem + kTmD2, tmem + kTmA2 + 8u * s, umma_desc(kstep(base + kE, 16384, s)),
                           idesc_tf32(128, 128), s > 0 ? 1u : 0u);
                mma_commit(bar(kDoneC2));
                if (c + 1 < n) {
                    // next chunk's U product (runs during the state update); the v, w
                    // buffer it was computed from takes chunk c + 3
                    if (!(ok = issue_u())) break;
                    if (c + 3 < n) load_vw(c + 3);
                }
            }
            if (!ok) {
                *abort_flag = 1;
                atomicExch(prm.err, kDevTimeout);
                // tile loads may still be in flight: wait for them (bounded) before exiting
                for (int b = 0; b < 2; ++b)
                    if ((iss_any >> b) & 1u) mbar_wait(bar(kBarVW + b), ((iss_par >> b) & 1u) ^ 1u);
            }
        } else if (warp == kSimt / 32 + 1 && lane == 0) {
            // O tile stores: one per chunk that lies wholly inside the sequence
            uint32_t ph_full = 0;
            mbar_arrive(bar(kOFree));   // the tile starts free
#pragma unroll 1
            for (int c = 0; (c + 1) * kC <= T && c < n; ++c) {
                if (!mbar_wait_ab(bar(kOFull), ph_full, abort_flag)) break;
                ph_full ^= 1u;
                const int row = orow0 + c * kC;
                tma_store_4d(om, base + kO, j0, h, row, 0);
                if (!obf16) tma_store_4d(om, base + kO + 8192u, j0 + 32, h, row, 0);
                bulk_commit();
                bulk_wait_read();           // the tile has been read: it may take the next chunk
                mbar_arrive(bar(kOFree));
            }
            bulk_wait_all();
        }
        __syncwarp();
    } else {
        // ================= 16 elementwise / accumulator warps ====================
        asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kRegsSimt));
        const uint32_t lane_base = static_cast<uint32_t>(quarter * 32) << 16;
        // Quarters 0-1 ("E warps", lanes 0..63 = token rows of E) read E out, the chain's
        // critical step; quarters 2-3 ("O warps") write O, complete P and build the next
        // chunks' U^T and -Cb^T operands while Kb^T E runs.  All warps update their state
        // slice, Kb^T and [T; A_qk T].
        const bool e_warp = quarter < 2;
        const int et = ((warp >> 2) * 2 + (warp & 1)) * 32 + lane;   // 0..255 within each group
        // Shared-memory byte offset of element (row, k) of an operand with K-blocks `kstride`
        // apart, for this thread's k (its TMEM lane) and rows row0 + jj: the swizzle term
        // depends on jj % 8 only, so it is (xk ^ (jj % 8)) << 4 with xk = (k % 32) / 4.
        auto lane_col = [&](uint32_t kstride, uint32_t k) {
            return (k >> 5) * kstride + ((k & 3u) << 2);
        };
        const uint32_t xk4 = ((static_cast<uint32_t>(j) & 31u) >> 2) << 4;
        // fp32 state S[j][j0 + 16R + jj] in registers; the S^T operand in shared memory
        float S[16];
        const uint32_t st_base = kSt + lane_col(8192, static_cast<uint32_t>(j)) + static_cast<uint32_t>(16 * R) * 128u;
        auto put_st = [&]() {
#pragma unroll
            for (int jj = 0; jj < 16; ++jj)
                *reinterpret_cast<float*>(sgen + st_base + jj * 128 + (xk4 ^ ((jj & 7) << 4))) = tf32r(S[jj]);
        };
        {
            // S0 for the whole sequence or segment 0, zero for later segments' value
            // tiles, identity columns for transfer tiles
            const float* s0 = prm.S0 && !mtile && g == 0
                                  ? prm.S0 + (static_cast<int64_t>(bh) * kDK + j) * prm.dv + j0 + 16 * R
                                  : nullptr;
#pragma unroll
            for (int jj = 0; jj < 16; jj += 4) {
                const float4 x = s0 ? *reinterpret_cast<const float4*>(s0 + jj) : make_float4(0.f, 0.f, 0.f, 0.f);
                S[jj] = x.x; S[jj + 1] = x.y; S[jj + 2] = x.z; S[jj + 3] = x.w;
            }
            if (mtile) {
#pragma unroll
                for (int jj = 0; jj < 16; ++jj) S[jj] = j == j0 + 16 * R + jj ? 1.f : 0.f;
            }
            put_st();
        }
        bool failed = false;
        uint32_t ph_c1 = 0, ph_c2 = 0, ph_p3 = 0, ph_vw0 = 0, ph_vw1 = 0, ph_of = 0;
        auto wait = [&](uint32_t b, uint32_t& ph) {
            const bool ok = mbar_wait_ab(bar(b), ph, abort_flag);
            ph ^= 1u;
            tc_fence_after();
            return ok;
        };
        // Publish this warp's shared-memory / TMEM writes, then one arrival.
        auto arrive = [&](uint32_t b) {
            fence_async_smem();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(b));
        };
        // x = hi + lo with hi = x truncated to tf32 and lo = x - hi exactly; the tensor
        // core then reads lo truncated, which keeps about 21 significant bits of x.
        auto split = [](float x, float& hi, float& lo) {
            hi = __uint_as_float(__float_as_uint(x) & 0xFFFFE000u);
            lo = x - hi;
        };
        // O warps: -Cb^T rows (channels) ej, tokens 32*eh .. 32*eh + 31
        const int ej = et & 127, eh = et >> 7;
        auto ld_cb = [&](int c, uint4 (&x)[4]) {
            if (c < n && !e_warp) {
                const uint4* p =
                    reinterpret_cast<const uint4*>(prm.s.cbt + slot(c) * (kDK * kC) + ((4 * eh) * kDK + ej) * 8);
#pragma unroll
                for (int g = 0; g < 4; ++g) x[g] = p[g * kDK];
            }
        };
        // the fp16 operand row holds all 64 tokens in 128 bytes: 16-byte chunk = 8 tokens
        auto put_cb = [&](const uint4 (&x)[4]) {
            const uint32_t rb = kCbT + static_cast<uint32_t>(ej) * 128u;
#pragma unroll
            for (int g = 0; g < 4; ++g)
                *reinterpret_cast<uint4*>(sgen + rb + (((static_cast<uint32_t>(4 * eh + g)) ^ (static_cast<uint32_t>(ej) & 7u)) << 4)) = x[g];
        };
        // O warps: U^T of chunk c from its v, w tile: d_v column un, tokens 16*ut .. 16*ut + 15
        const int un = et & 63, ut = et >> 6;
        // u = hi + lo as an fp16 pair (22 significant bits); the fp16 operand row holds all
        // 64 tokens in 128 bytes, 8 tokens per 16-byte chunk
        auto put_u = [&](int c) {
            const uint8_t* tv = sgen + kVW + static_cast<uint32_t>(c & 1) * 16384u;
            const int tvalid = T - c * kC - 16 * ut;   // tokens past the sequence end give U = 0
            const uint32_t rb = kU + static_cast<uint32_t>(un) * 128u;
#pragma unroll
            for (int q8 = 0; q8 < 2; ++q8) {
                uint4 hk, lk;
                __half2* hh = reinterpret_cast<__half2*>(&hk);
                __half2* lh = reinterpret_cast<__half2*>(&lk);
#pragma unroll
                for (int e = 0; e < 8; e += 2) {
                    float u[2];
#pragma unroll
                    for (int f = 0; f < 2; ++f) {
                        const int t = 16 * ut + 8 * q8 + e + f;
                        const uint32_t off = vw_off(t, un);
                        const float vv =
                            __uint_as_float(static_cast<uint32_t>(*reinterpret_cast<const uint16_t*>(tv + off)) << 16);
                        const float ww = __uint_as_float(
                            static_cast<uint32_t>(*reinterpret_cast<const uint16_t*>(tv + 8192 + off)) << 16);
                        u[f] = !mtile && 8 * q8 + e + f < tvalid ? vv * ww : 0.f;
                    }
                    const __half2 h2 = __floats2half2_rn(u[0], u[1]);
                    const float2 hf = __half22float2(h2);
                    hh[e / 2] = h2;
                    lh[e / 2] = __floats2half2_rn(u[0] - hf.x, u[1] - hf.y);
                }
                const uint32_t cofs = (static_cast<uint32_t>(2 * ut + q8) ^ (static_cast<uint32_t>(un) & 7u)) << 4;
                *reinterpret_cast<uint4*>(sgen + rb + cofs) = hk;
                *reinterpret_cast<uint4*>(sgen + rb + 64u * 128u + cofs) = lk;
            }
        };
        // all warps: Kb (channel j, tokens 16R..16R+15) -> TMEM Kb^T
        auto ld_kb = [&](int c, uint4 (&x)[2]) {
            if (c < n) {
                const uint4* p = reinterpret_cast<const uint4*>(prm.s.kbt + slot(c) * (kDK * kC) + ((2 * R) * kDK + j) * 8);
                x[0] = p[0];
                x[1] = p[kDK];
            }
        };
        auto put_kb = [&](const uint4 (&x)[2]) {
            const __half2* hk = reinterpret_cast<const __half2*>(x);
            float kb[16];
#pragma unroll
            for (int s = 0; s < 16; s += 2) {
                const float2 f = __half22float2(hk[s / 2]);
                kb[s] = f.x;
                kb[s + 1] = f.y;
            }
            tmem_st16(tmem + lane_base + kTmA2 + static_cast<uint32_t>(16 * R), kb);
            tmem_st_wait();
        };
        // O warps: P = Qb - A_qk W on lanes 64..127 of A1 (token j - 64, columns 32R .. 32R + 31)
        auto ld_qb = [&](int c, uint4 (&x)[4]) {
            if (c < n && !e_warp) {
                const uint4* p = reinterpret_cast<const uint4*>(prm.s.qb + slot(c) * (kC * kDK) +
                                                                ((4 * R) * kC + (j - 64)) * 8);
#pragma unroll
                for (int k = 0; k < 4; ++k) x[k] = p[k * kC];
            }
        };
        auto add_qb = [&](const uint4 (&x)[4]) {
            const __half2* hq = reinterpret_cast<const __half2*>(x);
#pragma unroll
            for (int half = 0; half < 2; ++half) {
                const uint32_t col = static_cast<uint32_t>(32 * R + 16 * half);
                float v[16];
                tmem_ld16(tmem + lane_base + kTmA1 + col, v);
#pragma unroll
                for (int e = 0; e < 16; e += 2) {
                    const float2 q2 = __half22float2(hq[(16 * half + e) / 2]);
                    v[e] += q2.x;
                    v[e + 1] += q2.y;
                }
                tmem_st16(tmem + lane_base + kTmA1 + col, v);
            }
            tmem_st_wait();
        };

        // all warps: [T; A_qk T] row j, columns 16R..16R+15 -> TMEM
        // fp16 pairs: column 8R + e holds tokens 16R + 2e (low half) and 16R + 2e + 1
        auto ld_a0 = [&](int c, uint32_t (&x)[8]) {
            if (c < n) {
                const uint4* p = reinterpret_cast<const uint4*>(prm.s.a0 + slot(c) * (128 * kC) + (R * 128 + j) * 16);
                const uint4 a = p[0], b = p[1];
                x[0] = a.x; x[1] = a.y; x[2] = a.z; x[3] = a.w;
                x[4] = b.x; x[5] = b.y; x[6] = b.z; x[7] = b.w;
            }
        };
        auto put_a0 = [&](const uint32_t (&x)[8]) {
            tmem_st8(tmem + lane_base + kTmA0 + static_cast<uint32_t>(8 * R), x);
            tmem_st_wait();
        };

        uint4 cbr[4], kbr[2], qbr[4];
        uint32_t a0r[8];
        float gam = 1.f;
        if (n > 0) {
            // ---- prologue: operands of chunk 0, and -Cb^T of chunk 1 ----------------------
            ld_a0(0, a0r);
            put_a0(a0r);
            arrive(kRdyA0);
            ld_cb(0, cbr);
            ld_kb(0, kbr);
            ld_qb(0, qbr);
            if (!e_warp) {
                put_cb(cbr);
                arrive(kRdyA1);                                   // A1(0)
                ld_cb(1, cbr);
                if (!mtile && !wait(kBarVW, ph_vw0)) failed = true;
                if (!failed) {
                    put_u(0);
                    arrive(kRdyU);                                // [T; A_qk T] U (0)
                }
                if (!failed && !wait(kDoneP3, ph_p3)) failed = true;
                if (!failed) {
                    add_qb(qbr);
                    if (n > 1) {
                        put_cb(cbr);
                        arrive(kRdyA1);                           // A1(1)
                    }
                }
            }
            if (!failed) {
                put_kb(kbr);
                arrive(kRdyChain);                                // chain of chunk 0
            }
        }

        for (int c = 0; c < n && !failed; ++c) {
            const int tc = c * kC;
            // workspace operands used later in this iteration
            ld_cb(c + 2, cbr);
            ld_kb(c + 1, kbr);
            ld_qb(c + 1, qbr);
            ld_a0(c + 1, a0r);
            gam = prm.s.gam[slot(c) * kDK + j];

            if (!wait(kDoneC1, ph_c1)) { failed = true; break; }
            // the products that read [T; A_qk T](c) are done: next chunk's into TMEM
            if (c + 1 < n) {
                put_a0(a0r);
                arrive(kRdyA0);
            }
            if (e_warp) {
                // ---- chain: E -> [E_hi^T; E_lo^T] --------------------------------------------
                float v[16];
                tmem_ld16_pair(tmem + lane_base + kTmEO + static_cast<uint32_t>(16 * R), v);
                const uint32_t rb = kE + lane_col(16384, static_cast<uint32_t>(j)) + static_cast<uint32_t>(16 * R) * 128u;
#pragma unroll
                for (int jj = 0; jj < 16; ++jj) {
                    float eh, el;
                    split(v[jj], eh, el);
                    const uint32_t a = rb + jj * 128 + (xk4 ^ ((jj & 7) << 4));
                    *reinterpret_cast<float*>(sgen + a) = eh;
                    *reinterpret_cast<float*>(sgen + a + 8192u) = el;
                }
                arrive(kRdyMma2);
            } else {
                // ---- O -> global ---------------------------------------------------------------
                float v[16];
                tmem_ld16_pair(tmem + lane_base + kTmEO + static_cast<uint32_t>(16 * R), v);
                const int r = j - 64;
                if (tc + kC <= T) {
                    // whole chunk inside the sequence: O tile -> shared memory -> one TMA store
                    if (!wait(kOFree, ph_of)) { failed = true; break; }
                    if (obf16) {
                        uint4 pk[2];
                        uint32_t* pw = reinterpret_cast<uint32_t*>(pk);
#pragma unroll
                        for (int jj = 0; jj < 16; jj += 2) {
                            __nv_bfloat162 x2 = __floats2bfloat162_rn(v[jj], v[jj + 1]);
                            pw[jj / 2] = *reinterpret_cast<uint32_t*>(&x2);
                        }
#pragma unroll
                        for (int q = 0; q < 2; ++q)
                            *reinterpret_cast<uint4*>(sgen + kO + r * 128 + ((((2 * R + q) ^ (r & 7)) & 7) << 4)) = pk[q];
                    } else {
                        const uint32_t tb = kO + static_cast<uint32_t>(R >> 1) * 8192u + static_cast<uint32_t>(r) * 128u;
#pragma unroll
                        for (int q = 0; q < 4; ++q)
                            *reinterpret_cast<float4*>(sgen + tb + ((((4 * (R & 1) + q) ^ (r & 7)) & 7) << 4)) =
                                make_float4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
                    }
                    arrive(kOFull);
                } else if (tc + r < T) {   // the sequence's last, partial chunk: row by row
                    const int64_t off = ((static_cast<int64_t>(orow0) + tc + r) * prm.H + h) * ow + j0 + 16 * R;
                    if (obf16) {
                        __nv_bfloat16* op = static_cast<__nv_bfloat16*>(prm.o) + off;
                        uint4 pk[2];
                        uint32_t* pw = reinterpret_cast<uint32_t*>(pk);
#pragma unroll
                        for (int jj = 0; jj < 16; jj += 2) {
                            __nv_bfloat162 x2 = __floats2bfloat162_rn(v[jj], v[jj + 1]);
                            pw[jj / 2] = *reinterpret_cast<uint32_t*>(&x2);
                        }
                        reinterpret_cast<uint4*>(op)[0] = pk[0];
                        reinterpret_cast<uint4*>(op)[1] = pk[1];
                    } else {
                        float* const ob = to_o ? static_cast<float*>(prm.o) : (mtile ? prm.r : prm.o32);
                        float4* op = reinterpret_cast<float4*>(ob + off);
#pragma unroll
                        for (int jj = 0; jj < 16; jj += 4)
                            op[jj / 4] = make_float4(v[jj], v[jj + 1], v[jj + 2], v[jj + 3]);
                    }
                }
                if (c + 1 < n) {
                    // ---- next chunk: U^T operand (its product overwrites [E; O] after this) -----
                    const bool odd = (c + 1) & 1;
                    if (!mtile && !wait(odd ? kBarVWb : kBarVW, odd ? ph_vw1 : ph_vw0)) { failed = true; break; }
                    put_u(c + 1);
                    arrive(kRdyU);
                    // ---- next chunk: P on A1, then -Cb^T of chunk c + 2 into the freed buffer -----
                    if (!wait(kDoneP3, ph_p3)) { failed = true; break; }
                    add_qb(qbr);
                    if (c + 2 < n) {
                        put_cb(cbr);
                        arrive(kRdyA1);
                    }
                }
            }
            // ---- chain: S <- gamma S + Kb^T E; S^T operand; next chunk's Kb^T ----------------
            if (!wait(kDoneC2, ph_c2)) { failed = true; break; }
            {
                uint32_t a[16], b[16];
                tmem_ld16_nw(tmem + lane_base + kTmD2 + static_cast<uint32_t>(16 * R), a);
                tmem_ld16_nw(tmem + lane_base + kTmD2 + 64u + static_cast<uint32_t>(16 * R), b);
                tmem_ld_wait();
#pragma unroll
                for (int jj = 0; jj < 16; ++jj) S[jj] = fmaf(gam, S[jj], __uint_as_float(a[jj]) + __uint_as_float(b[jj]));
                put_st();
                // the state at a cache point (the end of every cache_chunks chunks)
                if (kCache && (c + 1) % prm.cache_chunks == 0 && (c + 1) / prm.cache_chunks <= prm.n_cache) {
                    float* cs = prm.cache +
                                ((static_cast<int64_t>(bh) * prm.n_cache + (c + 1) / prm.cache_chunks - 1) * kDK + j) * prm.dv +
                                j0 + 16 * R;
#pragma unroll
                    for (int jj = 0; jj < 16; jj += 4)
                        *reinterpret_cast<float4*>(cs + jj) = make_float4(S[jj], S[jj + 1], S[jj + 2], S[jj + 3]);
                }
            }
            if (c + 1 < n) {
                put_kb(kbr);
                arrive(kRdyChain);
            }
        }

        if (failed) {
            *abort_flag = 1;
            if (lane == 0) atomicExch(prm.err, kDevTimeout);
        } else if (prm.G > 1 || prm.ST) {
            // S_T, else the segment's end-state slot [blockIdx.x][d_k][width]
            float* st = prm.G == 1 ? prm.ST + (static_cast<int64_t>(bh) * kDK + j) * prm.dv + j0 + 16 * R
                                   : (mtile ? prm.seg_m : prm.seg_state) +
                                         (static_cast<int64_t>(bh * prm.G + g) * kDK + j) * (mtile ? kDK : prm.dv) +
                                         j0 + 16 * R;
#pragma unroll
            for (int jj = 0; jj < 16; jj += 4)
                *reinterpret_cast<float4*>(st + jj) = make_float4(S[jj], S[jj + 1], S[jj + 2], S[jj + 3]);
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc<kTmCols>(tmem);
    }
}

__global__ void __launch_bounds__(kThreads, 1)
state_kernel(const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_w,
             const __grid_constant__ CUtensorMap tm_o, const __grid_constant__ CUtensorMap tm_o32,
             const __grid_constant__ CUtensorMap tm_r, const StateParams prm) {
    if (static_cast<int>(blockIdx.y) >= prm.dv / kDVT)
        state_cta<true, false>(tm_v, tm_w, tm_o, tm_o32, tm_r, prm);
    else
        state_cta<false, false>(tm_v, tm_w, tm_o, tm_o32, tm_r, prm);
}

// The sequential state pass that also keeps the state at every cache point: a kernel
// of its own, so that the pass above is compiled without the extra stores.
__global__ void __launch_bounds__(kThreads, 1)
state_kernel_cached(const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_w,
                    const __grid_constant__ CUtensorMap tm_o, const StateParams prm) {
    state_cta<false, true>(tm_v, tm_w, tm_o, tm_o, tm_o, prm);
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

// Packed [1, total, H, dv] token rows (bf16 or fp32) as a 4-D map (dv, H, total, 1);
// box (128 bytes of d_v, 1, 64 tokens, 1) with the 128-byte swizzle.  Loads past
// the tensor read zeros; stores past it are dropped.
bool make_row_map(CUtensorMap* m, const void* ptr, int64_t total, int64_t H, int64_t dv, bool f32) {
    auto enc = get_encode();
    if (!enc) return false;
    const cuuint64_t esz = f32 ? 4 : 2;
    const cuuint64_t dims[4] = {static_cast<cuuint64_t>(dv), static_cast<cuuint64_t>(H),
                                static_cast<cuuint64_t>(total), 1};
    const cuuint64_t strides[3] = {static_cast<cuuint64_t>(dv) * esz, static_cast<cuuint64_t>(H * dv) * esz,
                                   static_cast<cuuint64_t>(total * H * dv) * esz};
    const cuuint32_t box[4] = {static_cast<cuuint32_t>(128 / esz), 1, 64, 1};
    const cuuint32_t estr[4] = {1, 1, 1, 1};
    return enc(m, f32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4,
               const_cast<void*>(ptr), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
               CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

int launch_state(const ForwardArgs& a, const PrepSlots& s, int64_t chunks, int c0, int cpiece, cudaStream_t stream,
                 int* err, const SegArgs& seg) {
    const int64_t total = a.cu ? a.total : a.B * a.T;
    const int64_t slots = chunks * a.H;
    if (slots * 128 >= (1ll << 31) || chunks >= (1ll << 31)) return GDR2_ERR_SHAPE;
    const bool segmented = seg.G > 1;
    if (a.S_cache && (segmented || a.cu || c0 != 0 || a.cache_chunks < 1)) return GDR2_ERR_ARG;
    if (segmented && (a.cu || c0 != 0 || seg.L < 1 || static_cast<int64_t>(seg.G - 1) * seg.L * kC >= a.T ||
                      !seg.seg_state || !seg.seg_m || !seg.o32 || !seg.r))
        return GDR2_ERR_ARG;
    CUtensorMap mv, mw, mo, mo32, mr;
    if (!make_row_map(&mv, a.v, total, a.H, a.dv, false) || !make_row_map(&mw, a.w, total, a.H, a.dv, false) ||
        !make_row_map(&mo, a.o, total, a.H, a.dv, a.out_dtype != GDR2_BF16))
        return GDR2_ERR_CUDA;
    if (segmented) {
        if (!make_row_map(&mo32, seg.o32, a.B * seg.Tr, a.H, a.dv, true) ||
            !make_row_map(&mr, seg.r, a.B * seg.Tr, a.H, kDK, true))
            return GDR2_ERR_CUDA;
    } else {
        mo32 = mo;   // not read
        mr = mo;
    }
    static std::once_flag attr_once;
    static cudaError_t attr_err = cudaSuccess;
    std::call_once(attr_once, [] {
        attr_err = cudaFuncSetAttribute(state_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                        static_cast<int>(kSmemAlloc));
        if (attr_err == cudaSuccess)
            attr_err = cudaFuncSetAttribute(state_kernel_cached, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                            static_cast<int>(kSmemAlloc));
    });
    if (attr_err != cudaSuccess) return GDR2_ERR_CUDA;
    StateParams prm{s, a.S0, a.o, a.ST, err, a.cu, static_cast<int>(a.T), static_cast<int>(a.H),
                    static_cast<int>(a.dv), static_cast<int>(total),
                    a.cu ? 0 : cpiece, a.cu ? 0 : c0, static_cast<int>(chunks),
                    a.out_dtype == GDR2_BF16 ? 1 : 0,
                    segmented ? seg.G : 1, segmented ? seg.L : cpiece, segmented ? static_cast<int>(seg.Tr) : 0,
                    seg.seg_state, seg.seg_m, seg.o32, seg.r,
                    a.S_cache, static_cast<int>(a.cache_chunks),
                    a.S_cache ? static_cast<int>(a.T / (a.cache_chunks * kC)) : 0};
    // value tiles, then (segmented) the d_k / 64 transfer tiles of each (sequence, segment, head)
    const int ytiles = static_cast<int>(a.dv / kDVT) + (segmented ? kDK / kDVT : 0);
    const dim3 grid(static_cast<unsigned>(a.B * (segmented ? seg.G : 1) * a.H), static_cast<unsigned>(ytiles));
    if (a.S_cache)
        state_kernel_cached<<<grid, kThreads, kSmemAlloc, stream>>>(mv, mw, mo, prm);
    else
        state_kernel<<<grid, kThreads, kSmemAlloc, stream>>>(mv, mw, mo, mo32, mr, prm);
    return cudaPeekAtLastError() == cudaSuccess ? GDR2_OK : GDR2_ERR_CUDA;
}

}  // namespace gdr2
