// Chunked Gated Delta Rule-2 prefill for bf16 inputs on sm_103a:
// TMA-staged input tiles, tcgen05 tensor-core products with TMEM
// accumulators and TMEM-resident operands, an fp32 state carried on chip
// across chunks, and the state-independent work of chunk n+1 overlapped
// with the state pass of chunk n.
//
// Method ("Gated DeltaNet-2: Decoupling Erase and Write in Linear Attention"
// page: update equation, and the "efficient implementation" section's WY form
// with decay absorption and chunkwise algorithm).  For one chunk of C = 64
// tokens r = 0..63 with chunk-initial state S (d_k x d_v), cumulative log
// decay G_r = sum_{t<=r} g_t (per key channel), c_r = b_r * k_r,
// u_r = w_r * v_r, the recurrence unrolls to
//     e_r = u_r - (c_r * e^{G_r})^T S - sum_{i<r} A_kk[r,i] e_i
//     o_r = (q_r * e^{G_r})^T S + sum_{i<=r} A_qk[r,i] e_i
//     S_C = diag(e^{G_C}) S + sum_i diag(e^{G_C - G_i}) k_i e_i^T
// with A_kk[r,i] = sum_j c_r[j] k_i[j] e^{G_r[j]-G_i[j]} (i < r) and
// A_qk[r,i] = sum_j q_r[j] k_i[j] e^{G_r[j]-G_i[j]} (i <= r): the cumulative
// channel decay sits inside the rank-1 erase factors.  With T = (I + A_kk)^-1
// (UT transform), Cb = c*e^{G}, Qb = q*e^{G}, Kb = k*e^{G_C - G},
// W = T Cb and P = Qb - A_qk W, the chunk is
//     [E; O] = [T; A_qk T] U + [-W; P] S,     S <- diag(e^{G_C}) S + Kb^T E.
// Everything left of S is independent of the state, so the only products on
// the chunk-to-chunk chain are [-W; P] S and Kb^T E.
//
// Overflow-free decay factors: e^{G_r - G_i} is formed as a product of two
// factors about a reference m, the 8th token of the 16-token sub-chunk
// ("stripe") holding r: e^{G_r - G_m} * e^{G_m - G_i}.  Row r carries
// e^{G_r - G_m}; column i is scaled once per stripe R >= stripe(i)
// ("K-group" R).  For i in an earlier stripe both factors are <= 1; inside
// the stripe each spans at most 8 tokens, and with per-token log decays
// floored at -10 it stays within e^{+-80}.
//
// Precision: tensor-core operands are tf32 (kind::tf32, fp32 accumulators);
// U and E, whose rounding the later products amplify most, enter as a tf32
// pair x = x_hi + x_lo (two products each).  Operands the tensor core reads
// from TMEM (T, A_qk T, -W, P, Kb^T) are fp32 accumulator values taken as
// tf32.  The triangular solve, decay factors and state update are fp32 on
// CUDA cores.
//
// Work split: one CTA (512 threads, one per SM) per (batch*head, 64-column
// d_v tile).  Thread (j = tid % 128, R = tid / 128) owns key channel j of
// stripe R in the elementwise phases and TMEM lane j, columns 16R..16R+15 in
// the accumulator phases (warp w may only touch TMEM lanes 32*(w%4)..+31,
// and j = 32*(w%4) + lane).  Loop iteration `it` runs the state pass of chunk
// it-1 and the state-independent preparation of chunk it:
//   (a) chain MMAs [E;O] = A0 U + A1 S          (A0 = [T; A_qk T], A1 = [-W; P])
//   (b) prep pass 1: raw tiles -> registers, decay factors, [Ct; Qt] and the
//       K-groups in shared memory
//   (c) chain epilogue: E -> E^T operand, O -> global; MMA2 Kb^T E; prep
//       intra-chunk products [Ct; Qt] K-groups^T
//   (e) chain: S <- gamma S + Kb^T E, S^T operand refreshed
//   (f) prep: A_kk, A_qk out of TMEM, triangular solve, A0 = [I; A_qk] T,
//       pass 2 (-Cb^T, Kb^T -> TMEM, U^T), A1 = A0 (-Cb^T), P += Qb.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <cuda_fp16.h>

#include <mutex>

#include "gdr2.h"
#include "gdr2_internal.cuh"

namespace gdr2 {
namespace {

constexpr int kC = 64;         // chunk length
constexpr int kDK = 128;       // key channels
constexpr int kDVT = 64;       // value columns per CTA
constexpr int kSimt = 512;     // 16 warps: elementwise and accumulator phases
constexpr int kThreads = kSimt + 128;  // + one warpgroup whose first thread issues TMA loads and MMAs
// Registers: launched at 96 per thread (640 x 96 = 61440 in the CTA's pool); the
// MMA warpgroup drops to 32 and the 16 elementwise warps rise to 112:
// 512 x 112 + 128 x 32 = 61440 <= 61440, and per SM sub-partition (4 elementwise
// warps + 1 MMA-group warp) 4 x 112 x 32 + 32 x 32 = 15360 <= 16384.
constexpr int kRegsSimt = 112, kRegsMma = 32;
static_assert(kSimt * kRegsSimt + (kThreads - kSimt) * kRegsMma <= kThreads * 96, "register pool");

// ---- shared-memory map (bytes from a 1024-aligned base) ------------------------
// Every MMA operand is K-major with the 128-byte swizzle: K-blocks of 32 tf32,
// each K-block `rows` x 128 B, 16-byte chunk index XOR (row % 8).
constexpr uint32_t kRawQ = 0, kRawK = 16384, kRawB = 32768, kRawG = 49152;  // bf16 [2 kblk][64][64]
constexpr uint32_t kG31 = 0;           // K-groups [G3 (64 rows) | G1 (32 rows)], 96 x 128 K (48 KB)
constexpr uint32_t kOpA = 65536;       // [Ct; Qt]: 128 rows x 128 K (64 KB)
constexpr uint32_t kG20 = 131072;      // K-groups [G2 (48 rows) | G0 (16 rows)], 64 x 128 K (32 KB)
constexpr uint32_t kSt = 163840;       // S^T: 64 rows (d_v) x 128 K (d_k) (32 KB)
constexpr uint32_t kEU = 196608;       // [U_hi^T; U_lo^T], later [E_hi^T; E_lo^T]: 128 rows x 64 K (32 KB)
constexpr uint32_t kMisc = 229376;     // mbarriers, TMEM base
constexpr uint32_t kSmemBytes = kMisc + 128;
constexpr uint32_t kSmemAlloc = kSmemBytes + 1024;
// pass-1 exchange of per-stripe decay sums (inside [Ct; Qt] before it is written)
constexpr uint32_t kXTot = kOpA, kXMid = kOpA + 2048;
// phase (f) scratch inside kOpA .. kOpA + 96 KB (the intra-chunk product operands are dead)
constexpr int kLd = 65;                              // A_kk staging row (floats)
constexpr int kLt = 68;                              // T staging row (floats; rows 16-byte aligned)
constexpr uint32_t kSL = kOpA;                       // A_kk staging  [64][65] fp32
constexpr uint32_t kSTs = kOpA + 16640;              // T staging     [64][68] fp32
constexpr uint32_t kSP = kOpA + 34048;               // solve: 6 blocks M_{RJ} of 16 x 17 fp32
constexpr uint32_t kIA = kOpA + 40960;               // [I; A_qk]: 128 rows x 64 K (32 KB)
constexpr uint32_t kTT = kIA + 32768;                // T^T: 64 rows x 64 K (16 KB)
constexpr uint32_t kCbT = kOpA;                      // -Cb^T: 128 rows x 64 K (32 KB), after the solve
constexpr int kLq = 132;                             // padded Qb row (floats)
constexpr uint32_t kQb = kOpA + 40960;               // Qb [64][132] fp32, after the A0 product
static_assert(kSTs + 64 * kLt * 4 <= kSP && kSP + 6 * 16 * 17 * 4 <= kIA, "solve scratch");
static_assert(kTT + 16384 <= kSt && kQb + 64 * kLq * 4 <= kSt, "phase (f) scratch");
static_assert(kCbT + 32768 <= kIA, "-Cb^T below [I; A_qk]");
static_assert(kG31 + 3 * 12288 + 12288 <= kOpA, "K-groups in the raw area");
static_assert(kSmemAlloc <= 232448, "shared memory");
// mbarriers (8 bytes each) inside kMisc
enum : uint32_t { kBarTma = 0, kRdyChain, kRdyMma2, kRdyAP, kRdyA0, kRdyA1, kDoneC1, kDoneC2, kDoneP1,
                  kDoneP2, kDoneP3, kNumBars };
constexpr uint32_t kTmemSlot = kMisc + 8 * kNumBars;

// ---- TMEM columns ------------------------------------------------------------------
constexpr uint32_t kTmA0 = 0;      // [T; A_qk T]   (A operand, K = 64 tokens)
constexpr uint32_t kTmA1 = 64;     // [-W; P]       (A operand, K = 128 channels)
constexpr uint32_t kTmAP = 64;     // intra-chunk products while A1 is free: [G3|G1] 64..159, [G2|G0] 160..223
constexpr uint32_t kTmA2 = 224;    // Kb^T          (A operand, lanes = channels, K = 64 tokens)
constexpr uint32_t kTmEO = 288;    // [E; O] as hi | lo halves (128 columns), then Kb^T E likewise
constexpr uint32_t kTmS = 416;     // fp32 state S[j][j0 + c], lanes = key channels, 64 columns
constexpr uint32_t kTmCols = 512;

constexpr long long kWaitCycles = 4ll * 1000 * 1000 * 1000;   // ~2 s at 2 GHz
// Per-token log decays below this are taken as this value: a factor spanning the
// 8 tokens either side of a stripe's reference then stays within e^{+-80}.  The
// decay factor e^{-10} = 4.5e-5 instead of a smaller one changes the state carried
// across such a token by at most 4.5e-5 of itself.
constexpr float kMinLogDecay = -10.f;

// ---- PTX helpers ---------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ float tf32r(float x) {   // round to nearest tf32
    uint32_t r;
    asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(r) : "f"(x));
    return __uint_as_float(r);
}
// Byte offset of element (row, k) of a K-major 128B-swizzled tf32 operand
// whose K-blocks are `kstride` bytes apart.
__device__ __forceinline__ uint32_t sw(uint32_t kstride, uint32_t row, uint32_t k) {
    return (k >> 5) * kstride + row * 128u + ((((k & 31u) >> 2) ^ (row & 7u)) << 4) + ((k & 3u) << 2);
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ bool mbar_try(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}
// Bounded wait on an mbarrier phase; false when it gave up.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity) {
    if (mbar_try(bar, parity)) return true;
    const long long t0 = clock64();
    while (!mbar_try(bar, parity))
        if (clock64() - t0 > kWaitCycles) return false;
    return true;
}
__device__ __forceinline__ void fence_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
// Barrier over the 16 elementwise warps only (the MMA warp never joins it).
__device__ __forceinline__ void simt_sync() { asm volatile("bar.sync 1, 512;" ::: "memory"); }
__device__ __forceinline__ bool simt_any(bool pred) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.u32 p, %1, 0;\n\t"
        "bar.red.or.pred q, 1, 512, p;\n\t"
        "selp.u32 %0, 1, 0, q;\n\t}"
        : "=r"(r)
        : "r"(static_cast<uint32_t>(pred))
        : "memory");
    return r != 0;
}
__device__ __forceinline__ void tma_load_4d(uint32_t dst, const CUtensorMap* map, int c0, int c1, int c2,
                                            int c3, uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3, %4, %5}], [%6];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(bar)
        : "memory");
}

// tcgen05 shared-memory matrix descriptor: K-major, 128-byte swizzle,
// 8-row groups 1024 B apart.
__device__ __forceinline__ uint64_t umma_desc(uint32_t saddr) {
    uint64_t d = static_cast<uint64_t>((saddr >> 4) & 0x3FFFu);
    d |= static_cast<uint64_t>(1) << 16;             // leading byte offset (unused for this layout)
    d |= static_cast<uint64_t>(1024 >> 4) << 32;     // stride byte offset
    d |= static_cast<uint64_t>(1) << 46;             // descriptor version
    d |= static_cast<uint64_t>(2) << 61;             // 128-byte swizzle
    return d;
}
// Instruction descriptor, kind::tf32: fp32 accumulate, A and B tf32, K-major.
__host__ __device__ constexpr uint32_t idesc_tf32(uint32_t M, uint32_t N) {
    return (1u << 4) | (2u << 7) | (2u << 10) | ((N >> 3) << 17) | ((M >> 4) << 24);
}
__device__ __forceinline__ void mma_ss(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc,
                                       uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::tf32 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a), "l"(b), "r"(idesc), "r"(accumulate)
        : "memory");
}
__device__ __forceinline__ void mma_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b, uint32_t idesc,
                                       uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::tf32 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
        "r"(a_tmem), "l"(b), "r"(idesc), "r"(accumulate)
        : "memory");
}
__device__ __forceinline__ void mma_commit(uint32_t bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
                 : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
// 32 lanes x 32 bit, 16 consecutive columns per thread (no wait).
__device__ __forceinline__ void tmem_ld16_nw(uint32_t taddr, uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
          "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
}
__device__ __forceinline__ void tmem_ld_wait() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float (&v)[16]) {
    uint32_t r[16];
    tmem_ld16_nw(taddr, r);
    tmem_ld_wait();
#pragma unroll
    for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}
// Sum of the two 64-column halves (hi and lo products) at columns c and c + 64.
__device__ __forceinline__ void tmem_ld16_pair(uint32_t taddr, float (&v)[16]) {
    uint32_t a[16], b[16];
    tmem_ld16_nw(taddr, a);
    tmem_ld16_nw(taddr + 64u, b);
    tmem_ld_wait();
#pragma unroll
    for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(a[i]) + __uint_as_float(b[i]);
}
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const float (&v)[16]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
        "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16};" ::"r"(taddr),
        "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])), "r"(__float_as_uint(v[2])),
        "r"(__float_as_uint(v[3])), "r"(__float_as_uint(v[4])), "r"(__float_as_uint(v[5])),
        "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7])), "r"(__float_as_uint(v[8])),
        "r"(__float_as_uint(v[9])), "r"(__float_as_uint(v[10])), "r"(__float_as_uint(v[11])),
        "r"(__float_as_uint(v[12])), "r"(__float_as_uint(v[13])), "r"(__float_as_uint(v[14])),
        "r"(__float_as_uint(v[15]))
        : "memory");
}
__device__ __forceinline__ void tmem_st_wait() {
    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ uint32_t kstep(uint32_t base, uint32_t kstride, int s) {   // tf32 K-step s
    return base + (static_cast<uint32_t>(s) >> 2) * kstride + (static_cast<uint32_t>(s) & 3u) * 32u;
}

struct ChunkParams {
    const void* v;
    const void* w;
    const float* S0;
    void* o;
    float* ST;
    int* err;
    const int* cu;      // sequence start offsets [N + 1] (packed sequences), or null: all of length T
    int T, H, dv;       // T: the common length when cu is null
    int total;          // token rows in the packed [total, H, d] tensors
    int out_bf16;
};

// First TMEM column of K-group R in the intra-chunk product block.
__device__ __forceinline__ uint32_t group_col(int R) {
    return kTmAP + (R == 3 ? 0u : R == 1 ? 64u : R == 2 ? 96u : 144u);
}

__global__ void __launch_bounds__(kThreads, 1)
chunk_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
             const __grid_constant__ CUtensorMap tm_b, const __grid_constant__ CUtensorMap tm_g,
             const ChunkParams prm) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t base = (smem_u32(smem_raw) + 1023u) & ~1023u;
    uint8_t* sgen = smem_raw + (base - smem_u32(smem_raw));   // generic pointer to the same base
    float* const F = reinterpret_cast<float*>(sgen);
    const unsigned short* const H16 = reinterpret_cast<const unsigned short*>(sgen);
    auto bar = [&](uint32_t i) { return base + kMisc + 8u * i; };
    volatile uint32_t* tmem_slot = reinterpret_cast<volatile uint32_t*>(sgen + kTmemSlot);

    const int tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;
    const int j = tid & 127;          // key channel (elementwise) / TMEM lane (accumulator phases)
    const int R = (tid >> 7) & 3;     // stripe (elementwise) / 16-column block (accumulator phases)
    const int quarter = warp & 3;     // TMEM lane quarter this warp may access
    const int bh = blockIdx.x;
    const int seq = bh / prm.H, h = bh % prm.H;
    const int j0 = blockIdx.y * kDVT;
    // This sequence's token rows [tok0, tok0 + T) of the packed [total, H, d] tensors.
    int tok0, T;
    if (prm.cu) {   // offsets clamped to [0, total] and made non-decreasing
        const int a = min(max(prm.cu[seq], 0), prm.total);
        const int e = min(max(prm.cu[seq + 1], a), prm.total);
        tok0 = a;
        T = e - a;
    } else {
        tok0 = seq * prm.T;
        T = prm.T;
    }
    const int nchunks = (T + kC - 1) / kC;

    if (tid == 0) {
        for (uint32_t i = 0; i < kNumBars; ++i) mbar_init(bar(i), 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        fence_async_smem();
    }
    if (warp == 0) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(base + kTmemSlot),
                     "r"(kTmCols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp >= kSimt / 32) {
        // ================= MMA / TMA warpgroup: one elected thread ================
        asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kRegsMma));
        if (warp == kSimt / 32 && lane == 0) {
            auto issue_loads = [&](int n) {
                const int t0 = n * kC;
                mbar_expect_tx(bar(kBarTma), 65536u);
                tma_load_4d(base + kRawQ, &tm_q, 0, h, tok0 + t0, 0, bar(kBarTma));
                tma_load_4d(base + kRawQ + 8192, &tm_q, 64, h, tok0 + t0, 0, bar(kBarTma));
                tma_load_4d(base + kRawK, &tm_k, 0, h, tok0 + t0, 0, bar(kBarTma));
                tma_load_4d(base + kRawK + 8192, &tm_k, 64, h, tok0 + t0, 0, bar(kBarTma));
                tma_load_4d(base + kRawB, &tm_b, 0, h, tok0 + t0, 0, bar(kBarTma));
                tma_load_4d(base + kRawB + 8192, &tm_b, 64, h, tok0 + t0, 0, bar(kBarTma));
                tma_load_4d(base + kRawG, &tm_g, 0, h, tok0 + t0, 0, bar(kBarTma));
                tma_load_4d(base + kRawG + 8192, &tm_g, 64, h, tok0 + t0, 0, bar(kBarTma));
            };
            uint32_t ph_chain = 0, ph_mma2 = 0, ph_ap = 0, ph_a0 = 0, ph_a1 = 0, ph_c1 = 0;
            int issued = 0;
            bool ok = true;
            if (nchunks > 0) { issue_loads(0); issued = 1; }
#pragma unroll 1
            for (int it = 0; it <= nchunks && ok; ++it) {
                const bool has_prep = it < nchunks, has_chain = it > 0;
                if (has_chain) {
                    // [E; O] (hi | lo halves) = A0 [U_hi^T; U_lo^T] + A1 S^T, the d_k sum split over both halves
                    ok = mbar_wait(bar(kRdyChain), ph_chain); ph_chain ^= 1u;
                    if (!ok) break;
                    tc_fence_after();
#pragma unroll 1
                    for (int s = 0; s < 8; ++s)
                        mma_ts(tmem + kTmEO, tmem + kTmA0 + 8u * s, umma_desc(kstep(base + kEU, 16384, s)),
                               idesc_tf32(128, 128), s > 0 ? 1u : 0u);
#pragma unroll 1
                    for (int s = 0; s < 8; ++s) {
                        mma_ts(tmem + kTmEO, tmem + kTmA1 + 8u * s, umma_desc(kstep(base + kSt, 8192, s)),
                               idesc_tf32(128, kDVT), 1u);
                        mma_ts(tmem + kTmEO + 64u, tmem + kTmA1 + 8u * (s + 8),
                               umma_desc(kstep(base + kSt, 8192, s + 8)), idesc_tf32(128, kDVT), 1u);
                    }
                    mma_commit(bar(kDoneC1));
                }
                if (has_prep) {
                    // intra-chunk products [Ct; Qt] x [G3|G1]^T and x [G2|G0]^T, interleaved.
                    // Their accumulator overlaps A1, which the state pass above reads: wait
                    // for that pass to complete first.
                    ok = mbar_wait(bar(kRdyAP), ph_ap); ph_ap ^= 1u;
                    if (ok && has_chain) ok = mbar_wait(bar(kDoneC1), ph_c1);
                    if (has_chain) ph_c1 ^= 1u;
                    if (!ok) break;
                    tc_fence_after();
#pragma unroll 1
                    for (int s = 0; s < 16; ++s) {
                        const uint64_t a = umma_desc(kstep(base + kOpA, 16384, s));
                        mma_ss(tmem + kTmAP, a, umma_desc(kstep(base + kG31, 12288, s)), idesc_tf32(128, 96),
                               s > 0 ? 1u : 0u);
                        mma_ss(tmem + kTmAP + 96u, a, umma_desc(kstep(base + kG20, 8192, s)), idesc_tf32(128, 64),
                               s > 0 ? 1u : 0u);
                    }
                    mma_commit(bar(kDoneP1));
                }
                if (has_chain) {
                    // Kb^T [E_hi^T; E_lo^T] -> the same 128 columns
                    ok = mbar_wait(bar(kRdyMma2), ph_mma2); ph_mma2 ^= 1u;
                    if (!ok) break;
                    tc_fence_after();
#pragma unroll 1
                    for (int s = 0; s < 8; ++s)
                        mma_ts(tmem + kTmEO, tmem + kTmA2 + 8u * s, umma_desc(kstep(base + kEU, 16384, s)),
                               idesc_tf32(128, 128), s > 0 ? 1u : 0u);
                    mma_commit(bar(kDoneC2));
                }
                if (has_prep) {
                    // A0 = [I; A_qk] T = [T; A_qk T].  By this signal the elementwise warps
                    // have read the K-group 3 tile (for Kb^T) and the products are done: the
                    // raw area may take the next chunk's tiles.
                    ok = mbar_wait(bar(kRdyA0), ph_a0); ph_a0 ^= 1u;
                    if (!ok) break;
                    tc_fence_after();
                    if (it + 1 < nchunks) { issue_loads(it + 1); ++issued; }
#pragma unroll 1
                    for (int s = 0; s < 8; ++s)
                        mma_ss(tmem + kTmA0, umma_desc(kstep(base + kIA, 16384, s)),
                               umma_desc(kstep(base + kTT, 8192, s)), idesc_tf32(128, 64), s > 0 ? 1u : 0u);
                    mma_commit(bar(kDoneP2));
                    // A1 = A0 (-Cb^T) = [-W; -A_qk W]
                    ok = mbar_wait(bar(kRdyA1), ph_a1); ph_a1 ^= 1u;
                    if (!ok) break;
                    tc_fence_after();
#pragma unroll 1
                    for (int s = 0; s < 8; ++s)
                        mma_ts(tmem + kTmA1, tmem + kTmA0 + 8u * s, umma_desc(kstep(base + kCbT, 16384, s)),
                               idesc_tf32(128, 128), s > 0 ? 1u : 0u);
                    mma_commit(bar(kDoneP3));
                }
            }
            if (!ok) {
                atomicExch(prm.err, kDevTimeout);
                // a tile load may still be in flight: wait for it (bounded) before exiting
                if (issued > 0) mbar_wait(bar(kBarTma), static_cast<uint32_t>((issued - 1) & 1));
            }
        }
        __syncwarp();
    } else {
        // ================= 16 elementwise / accumulator warps ====================
        asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kRegsSimt));
        const uint32_t lane_base = static_cast<uint32_t>(quarter * 32) << 16;
        // fp32 state slice S[j][j0 + 16R + jj], jj = 0..15, held in registers; S^T operand.
        {
            const float* s0 = prm.S0 ? prm.S0 + (static_cast<int64_t>(bh) * kDK + j) * prm.dv + j0 + 16 * R
                                     : nullptr;
            float S[16];
#pragma unroll
            for (int jj = 0; jj < 16; ++jj) {
                S[jj] = s0 ? s0[jj] : 0.f;
                F[(kSt + sw(8192, 16 * R + jj, j)) >> 2] = tf32r(S[jj]);
            }
            tmem_st16(tmem + lane_base + kTmS + static_cast<uint32_t>(16 * R), S);
            tmem_st_wait();
        }
        uint32_t ph_tma = 0, ph_c1 = 0, ph_c2 = 0, ph_p1 = 0, ph_p2 = 0, ph_p3 = 0;
        bool failed = false;
        float gamma_prev = 1.f;   // e^{G_C} of the chunk whose state pass comes next, channel j
        auto wait_done = [&](uint32_t b, uint32_t& ph) -> bool {
            const bool ok = mbar_wait(bar(b), ph);
            ph ^= 1u;
            const bool bad = simt_any(!ok);
            tc_fence_after();
            return !bad;
        };
        // Publish smem / TMEM writes of all 16 warps, then signal the MMA warp.
        auto signal = [&](uint32_t b) {
            fence_async_smem();
            tc_fence_before();
            simt_sync();
            if (tid == 0) mbar_arrive(bar(b));
        };

        for (int it = 0; it <= nchunks && !failed; ++it) {
            const bool has_prep = it < nchunks;
            const bool has_chain = it > 0;
            const int tp = it * kC;                  // first token of the prepared chunk
            const int tc = (it - 1) * kC;            // first token of the chained chunk

            // ---- (b) prep pass 1 -------------------------------------------------------
            // This chunk's -Cb, Qb and Kb for the stripe's 16 tokens, kept until their
            // buffers are free.  All three are bounded by 2 in magnitude and later rounded
            // to tf32 (11 significant bits), so fp16 pairs carry them exactly enough.
            __half2 cbp[8], qbp[8], kbp[8];
            float gam = 1.f;
            if (has_prep) {
                float cr[16], qr[16], kr[16];     // c*rho, q*rho, k/rho
                {
                    const bool ok = mbar_wait(bar(kBarTma), ph_tma);
                    ph_tma ^= 1u;
                    if (simt_any(!ok)) { failed = true; break; }
                }
                // raw loads: element (token 16R+s, channel j) of a bf16 tile
                const uint32_t cbase = (static_cast<uint32_t>(j) >> 6) * 8192u +
                                       static_cast<uint32_t>(16 * R) * 128u + ((static_cast<uint32_t>(j) & 7u) << 1);
                const uint32_t c8 = (static_cast<uint32_t>(j) & 63u) >> 3;
                float Gl[16];
                float acc = 0.f;
                // tokens past the sequence end (the next sequence's rows, or the zero fill
                // past the tensor) enter as q = k = b = log_decay = 0
                const int nvalid = T - tp - 16 * R;
#pragma unroll
                for (int s = 0; s < 16; ++s) {
                    const uint32_t off =
                        cbase + static_cast<uint32_t>(s) * 128u + ((c8 ^ (static_cast<uint32_t>(s) & 7u)) << 4);
                    const uint32_t live = s < nvalid ? 0xFFFFFFFFu : 0u;
                    acc += fmaxf(__uint_as_float((static_cast<uint32_t>(H16[(kRawG + off) >> 1]) << 16) & live),
                                 kMinLogDecay);
                    Gl[s] = acc;
                    const float kv = __uint_as_float((static_cast<uint32_t>(H16[(kRawK + off) >> 1]) << 16) & live);
                    cr[s] = __uint_as_float(static_cast<uint32_t>(H16[(kRawB + off) >> 1]) << 16) * kv;
                    qr[s] = __uint_as_float((static_cast<uint32_t>(H16[(kRawQ + off) >> 1]) << 16) & live);
                    kr[s] = kv;
                }
                F[(kXTot >> 2) + R * 128 + j] = acc;
                F[(kXMid >> 2) + R * 128 + j] = Gl[7];
                simt_sync();   // raw tiles fully read; stripe sums visible
                float gmid[4];
                float gC = 0.f;
#pragma unroll
                for (int r2 = 0; r2 < 4; ++r2) {
                    gmid[r2] = gC + F[(kXMid >> 2) + r2 * 128 + j];
                    gC += F[(kXTot >> 2) + r2 * 128 + j];
                }
                const float gm = gmid[R];
                const float em = __expf(gm);          // e^{G_m}        (<= 1)
                const float ecm = __expf(gC - gm);    // e^{G_C - G_m}  (<= 1)
                gam = __expf(gC);                     // e^{G_C}
#pragma unroll
                for (int s = 0; s < 16; ++s) {
                    const float d = Gl[s] - Gl[7];
                    const float rho = __expf(fminf(d, 80.f)), irho = __expf(fminf(-d, 80.f));
                    cr[s] *= rho;
                    qr[s] *= rho;
                    kr[s] *= irho;
                }
                simt_sync();   // exchange reads done before [Ct; Qt] overwrites it
#pragma unroll
                for (int s = 0; s < 16; ++s) {
                    const uint32_t r = static_cast<uint32_t>(16 * R + s);
                    F[(kOpA + sw(16384, r, j)) >> 2] = tf32r(cr[s]);
                    F[(kOpA + sw(16384, 64u + r, j)) >> 2] = tf32r(qr[s]);
                }
                // K-groups: this stripe's tokens scaled to each later stripe's reference
#pragma unroll
                for (int g = 0; g < 4; ++g) {
                    if (g < R) continue;
                    const float sc = g == R ? 1.f : __expf(gmid[g] - gm);
                    const uint32_t gb = g == 3 ? kG31 : g == 1 ? kG31 : kG20;
                    const uint32_t ks = g == 3 || g == 1 ? 12288u : 8192u;
                    const uint32_t r0 = g == 1 ? 64u : g == 0 ? 48u : 0u;
#pragma unroll
                    for (int s = 0; s < 16; ++s)
                        F[(gb + sw(ks, r0 + static_cast<uint32_t>(16 * R + s), j)) >> 2] = tf32r(kr[s] * sc);
                }
#pragma unroll
                for (int s = 0; s < 16; s += 2) {
                    cbp[s / 2] = __floats2half2_rn(-cr[s] * em, -cr[s + 1] * em);
                    qbp[s / 2] = __floats2half2_rn(qr[s] * em, qr[s + 1] * em);
                    kbp[s / 2] = __floats2half2_rn(kr[s] * ecm, kr[s + 1] * ecm);
                }
                signal(kRdyAP);
            }

            // w, v of the prepared chunk (consumed after the state pass) for U = w * v: token tu, d_v columns 8*cu .. +7
            const int tu = tid & 63, cu = tid >> 6;
            uint4 vraw = make_uint4(0, 0, 0, 0), wraw = vraw;
            if (has_prep && tp + tu < T) {
                const int64_t off = ((static_cast<int64_t>(tok0) + tp + tu) * prm.H + h) * prm.dv + j0 + 8 * cu;
                vraw = *reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(prm.v) + off);
                wraw = *reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(prm.w) + off);
            }

            // ---- (c) chain: E -> [E_hi^T; E_lo^T], O -> global ---------------------------
            if (has_chain) {
                if (!wait_done(kDoneC1, ph_c1)) { failed = true; break; }
                float v[16];
                tmem_ld16_pair(tmem + lane_base + kTmEO + static_cast<uint32_t>(16 * R), v);
                if (quarter < 2) {
                    const uint32_t r = static_cast<uint32_t>(j);       // token of the chained chunk
#pragma unroll
                    for (int jj = 0; jj < 16; ++jj) {
                        const uint32_t n = static_cast<uint32_t>(16 * R + jj);
                        const float eh = tf32r(v[jj]);
                        F[(kEU + sw(16384, n, r)) >> 2] = eh;
                        F[(kEU + sw(16384, 64u + n, r)) >> 2] = tf32r(v[jj] - eh);
                    }
                } else {
                    const int r = j - 64;
                    if (tc + r < T) {
                        const int64_t off =
                            ((static_cast<int64_t>(tok0) + tc + r) * prm.H + h) * prm.dv + j0 + 16 * R;
                        if (prm.out_bf16) {
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
                            float4* op = reinterpret_cast<float4*>(static_cast<float*>(prm.o) + off);
#pragma unroll
                            for (int jj = 0; jj < 16; jj += 4)
                                op[jj / 4] = make_float4(v[jj], v[jj + 1], v[jj + 2], v[jj + 3]);
                        }
                    }
                }
                signal(kRdyMma2);
            }

            // ---- (e) chain: S <- gamma S + Kb^T E; then this chunk's Kb^T and U operands ---
            if (has_chain) {
                if (!wait_done(kDoneC2, ph_c2)) { failed = true; break; }
                uint32_t a[16], b[16], c[16];
                tmem_ld16_nw(tmem + lane_base + kTmEO + static_cast<uint32_t>(16 * R), a);
                tmem_ld16_nw(tmem + lane_base + kTmEO + 64u + static_cast<uint32_t>(16 * R), b);
                tmem_ld16_nw(tmem + lane_base + kTmS + static_cast<uint32_t>(16 * R), c);
                tmem_ld_wait();
                float S[16];
#pragma unroll
                for (int jj = 0; jj < 16; ++jj) {
                    S[jj] = fmaf(gamma_prev, __uint_as_float(c[jj]), __uint_as_float(a[jj]) + __uint_as_float(b[jj]));
                    F[(kSt + sw(8192, static_cast<uint32_t>(16 * R + jj), j)) >> 2] = tf32r(S[jj]);
                }
                tmem_st16(tmem + lane_base + kTmS + static_cast<uint32_t>(16 * R), S);
                tmem_st_wait();
            }
            if (has_prep) {
                float kb[16];
#pragma unroll
                for (int s = 0; s < 16; s += 2) {
                    const float2 f = __half22float2(kbp[s / 2]);
                    kb[s] = f.x;
                    kb[s + 1] = f.y;
                }
                tmem_st16(tmem + lane_base + kTmA2 + static_cast<uint32_t>(16 * R), kb);
                const __nv_bfloat16* vb = reinterpret_cast<const __nv_bfloat16*>(&vraw);
                const __nv_bfloat16* wb = reinterpret_cast<const __nv_bfloat16*>(&wraw);
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    const float u = __bfloat162float(vb[e]) * __bfloat162float(wb[e]);
                    const float uh = tf32r(u);
                    const uint32_t n = static_cast<uint32_t>(8 * cu + e);
                    F[(kEU + sw(16384, n, static_cast<uint32_t>(tu))) >> 2] = uh;
                    F[(kEU + sw(16384, 64u + n, static_cast<uint32_t>(tu))) >> 2] = tf32r(u - uh);
                }
                tmem_st_wait();
            }

            // ---- (f) prep: A_kk, A_qk; solve; A0; -Cb^T; A1; P ---------------------------
            if (has_prep) {
                if (!wait_done(kDoneP1, ph_p1)) { failed = true; break; }
                // A_kk -> fp32 staging (strictly lower part), A_qk -> rows 64..127 of [I; A_qk]
                // (tf32, zero above the diagonal), identity -> rows 0..63.  Warp: TMEM lane
                // quarter, K range [16R, 16R + 16).
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
                    for (int e = 0; e < 16; ++e)
                        out[e] = have ? __uint_as_float(rs == s0 ? ra[e] : rb[e]) : 0.f;
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
                tc_fence_before();
                simt_sync();

                // ---- T = (I + A_kk)^-1: 16x16 diagonal blocks by column forward substitution
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
                // M_{RJ} is stored as block p = R(R-1)/2 + J (16 x 17 floats each).  Each
                // thread computes 4 adjacent columns of one row.
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
                // -Cb^T operand (overlaps the A0 product; the solve staging is dead)
#pragma unroll
                for (int s = 0; s < 16; s += 4) {
                    const uint32_t r = static_cast<uint32_t>(16 * R + s);
                    const float2 a = __half22float2(cbp[s / 2]), b2 = __half22float2(cbp[s / 2 + 1]);
                    *reinterpret_cast<float4*>(sgen + kCbT + sw(16384, static_cast<uint32_t>(j), r)) =
                        make_float4(a.x, a.y, b2.x, b2.y);
                }
                if (!wait_done(kDoneP2, ph_p2)) { failed = true; break; }   // A0 ready; [I; A_qk], T^T free
                signal(kRdyA1);
                // Qb staging (overlaps the A1 product)
#pragma unroll
                for (int s = 0; s < 16; s += 2) {
                    const float2 f = __half22float2(qbp[s / 2]);
                    F[(kQb >> 2) + (16 * R + s) * kLq + j] = f.x;
                    F[(kQb >> 2) + (16 * R + s + 1) * kLq + j] = f.y;
                }
                gamma_prev = gam;
                if (!wait_done(kDoneP3, ph_p3)) { failed = true; break; }
                // P = Qb - A_qk W on lanes 64..127 of A1 (columns 32R .. 32R + 31)
                if (quarter >= 2) {
                    const int r = j - 64;
#pragma unroll
                    for (int half = 0; half < 2; ++half) {
                        const uint32_t col = static_cast<uint32_t>(32 * R + 16 * half);
                        float v[16];
                        tmem_ld16(tmem + lane_base + kTmA1 + col, v);
#pragma unroll
                        for (int e = 0; e < 16; e += 4) {
                            const float4 qb = *reinterpret_cast<const float4*>(sgen + kQb + (r * kLq + col + e) * 4);
                            v[e] += qb.x; v[e + 1] += qb.y; v[e + 2] += qb.z; v[e + 3] += qb.w;
                        }
                        tmem_st16(tmem + lane_base + kTmA1 + col, v);
                    }
                    tmem_st_wait();
                }
                signal(kRdyChain);   // A0, A1, A2, [U_hi^T; U_lo^T] and S^T ready for the next state pass
            }
        }

        if (failed) {
            if (tid == 0) atomicExch(prm.err, kDevTimeout);
        } else if (prm.ST) {
            float* st = prm.ST + (static_cast<int64_t>(bh) * kDK + j) * prm.dv + j0 + 16 * R;
            float S[16];
            tmem_ld16(tmem + lane_base + kTmS + static_cast<uint32_t>(16 * R), S);
#pragma unroll
            for (int jj = 0; jj < 16; jj += 4)
                *reinterpret_cast<float4*>(st + jj) = make_float4(S[jj], S[jj + 1], S[jj + 2], S[jj + 3]);
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmCols)
                     : "memory");
    }
}

// ---- host side ------------------------------------------------------------------
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

// Tensor [B, T, H, d] bf16 as a 4-D map (d, H, T, B); box (64, 1, 64, 1),
// 128-byte swizzle; tokens past T read as zeros.
bool make_map(CUtensorMap* m, const void* ptr, int64_t B, int64_t T, int64_t H, int64_t d) {
    auto enc = get_encode();
    if (!enc) return false;
    const cuuint64_t dims[4] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(H),
                                static_cast<cuuint64_t>(T), static_cast<cuuint64_t>(B)};
    const cuuint64_t strides[3] = {static_cast<cuuint64_t>(d * 2), static_cast<cuuint64_t>(H * d * 2),
                                   static_cast<cuuint64_t>(T * H * d * 2)};
    const cuuint32_t box[4] = {64, 1, 64, 1};
    const cuuint32_t estr[4] = {1, 1, 1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(ptr), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

bool chunked_bf16_supports(const ForwardArgs& a) {
    const int64_t total = a.cu ? a.total : a.B * a.T;
    return a.in_dtype == GDR2_BF16 && a.dk == kDK && (a.dv == 64 || a.dv == 128) && total > 0 &&
           total < (1ll << 31) && a.B * a.H < (1ll << 31) && get_encode() != nullptr;
}

int launch_chunked_bf16(const ForwardArgs& a, cudaStream_t stream, int* err) {
    // token tensors as one packed [1, total, H, d] sequence; each CTA reads its own rows
    const int64_t total = a.cu ? a.total : a.B * a.T;
    CUtensorMap mq, mk, mb, mg;
    if (!make_map(&mq, a.q, 1, total, a.H, a.dk) || !make_map(&mk, a.k, 1, total, a.H, a.dk) ||
        !make_map(&mb, a.b, 1, total, a.H, a.dk) || !make_map(&mg, a.g, 1, total, a.H, a.dk))
        return GDR2_ERR_CUDA;
    static std::once_flag attr_once;
    static cudaError_t attr_err = cudaSuccess;
    std::call_once(attr_once, [] {
        attr_err = cudaFuncSetAttribute(chunk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                        static_cast<int>(kSmemAlloc));
    });
    if (attr_err != cudaSuccess) return GDR2_ERR_CUDA;
    ChunkParams prm{a.v, a.w, a.S0, a.o, a.ST, err, a.cu, static_cast<int>(a.T), static_cast<int>(a.H),
                    static_cast<int>(a.dv), static_cast<int>(total), a.out_dtype == GDR2_BF16 ? 1 : 0};
    const dim3 grid(static_cast<unsigned>(a.B * a.H), static_cast<unsigned>(a.dv / kDVT));
    chunk_kernel<<<grid, kThreads, kSmemAlloc, stream>>>(mq, mk, mb, mg, prm);
    return cudaPeekAtLastError() == cudaSuccess ? GDR2_OK : GDR2_ERR_CUDA;
}

}  // namespace gdr2
