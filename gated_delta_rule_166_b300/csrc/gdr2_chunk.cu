// Chunked Gated Delta Rule-2 prefill for bf16 inputs on sm_103a:
// TMA-staged input tiles, tcgen05 tensor-core contractions with TMEM
// accumulators, fp32 state carried on chip across chunks.
//
// Method ("Gated DeltaNet-2: Decoupling Erase and Write in Linear Attention"
// page: update equation, and the "efficient implementation" section's WY form
// with decay absorption and chunkwise algorithm).  For one chunk of C = 64
// tokens r = 0..63 with chunk-initial state S (d_k x d_v), cumulative log
// decay G_r = sum_{t<=r} g_t (per key channel), c_r = b_r * k_r,
// u_r = w_r * v_r, the recurrence unrolls to
//     S_r = diag(e^{G_r}) S + sum_{i<=r} diag(e^{G_r - G_i}) k_i e_i^T
//     e_r = u_r - (c_r * e^{G_r})^T S - sum_{i<r} A_kk[r,i] e_i
//     o_r = (q_r * e^{G_r})^T S + sum_{i<=r} A_qk[r,i] e_i
// with A_kk[r,i] = sum_j c_r[j] k_i[j] e^{G_r[j]-G_i[j]} (i < r) and
// A_qk[r,i] = sum_j q_r[j] k_i[j] e^{G_r[j]-G_i[j]} (i <= r): the cumulative
// channel decay sits inside the rank-1 erase factors.  With T = (I + A_kk)^-1
// (UT transform), Cb = c*e^{G}, Qb = q*e^{G}, Kb = k*e^{G_C - G}:
//     X = U - Cb S,   E = T X,   O = Qb S + A_qk E,   S <- diag(e^{G_C}) S + Kb^T E.
//
// Overflow-free decay factors: e^{G_r - G_i} is formed as a product of two
// factors about a reference m of the 16-token sub-chunk holding r (its 8th
// token): e^{G_r - G_m} * e^{G_m - G_i}.  For i in an earlier sub-chunk both
// factors are <= 1; inside the sub-chunk each spans at most 8 tokens of decay.
//
// Precision: every tensor-core operand is an fp32 value rounded to nearest
// tf32 (10-bit mantissa) and multiplied with kind::tf32 into fp32 TMEM
// accumulators; bf16 operands (8-bit mantissa) are too coarse for the
// max|err|/RMS <= 2e-2 bar (the output is a small residual of O(1) terms).
// X and E, whose rounding the later products amplify most, enter as a tf32
// pair x = x_hi + x_lo (two MMAs each, x_lo = tf32(x - x_hi)).  The triangular
// solve (16x16 diagonal blocks by forward substitution, then the off-diagonal
// blocks level by level), decay factors and the state carry are fp32 on CUDA
// cores.
//
// Work split: one CTA (512 threads, one per SM) per (batch*head, 64-column
// d_v tile); the CTA walks the chunks of its sequence in order.  Thread
// (c = tid % 128, R = tid / 128) owns key channel c of sub-chunk R in the
// elementwise phases and TMEM lane c (or token row), columns 16R..16R+15 in
// the epilogues.  Every operand lives in shared memory in the K-major
// 128-byte-swizzled layout the tensor core reads.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <mutex>

#include "gdr2.h"
#include "gdr2_internal.cuh"

namespace gdr2 {
namespace {

constexpr int kC = 64;        // chunk length
constexpr int kDK = 128;      // key channels
constexpr int kDVT = 64;      // value columns per CTA
constexpr int kThreads = 512;

// ---- shared-memory map (bytes from a 1024-aligned base) -------------------
constexpr uint32_t kRawQ = 0, kRawK = 16384, kRawB = 32768, kRawG = 49152;  // bf16 [2 kblk][64][64]
constexpr uint32_t kRawV = 65536, kRawW = 73728;                            // bf16 [64][64]
constexpr uint32_t kRawBytes = 81920;
constexpr uint32_t kOpA = 81920;      // 64 KB: [Ct;Qt] -> solve staging -> [Cb;Qb] -> Kb^T
constexpr uint32_t kOpB = 147456;     // 32 KB: K~ group columns -> [T; A_qk]
constexpr uint32_t kSt = 180224;      // 32 KB: S^T operand  (64 rows j x 128 K)
constexpr uint32_t kXE = 212992;      // 16 KB: K~ group 1 -> X^T / E^T operand (64 rows j x 64 K)
constexpr uint32_t kLo = kOpA + 32768; // 16 KB: tf32 remainder of X^T / E^T (second half of kOpA)
constexpr uint32_t kMisc = 229376;    // mbarriers, TMEM base, abort flag
constexpr uint32_t kSmemBytes = kMisc + 64;
constexpr uint32_t kSmemAlloc = kSmemBytes + 1024;
// solve staging inside the kOpA area (padded fp32 rows)
constexpr int kLd = 65;
constexpr uint32_t kStAkk = kOpA, kStT = kOpA + 64 * kLd * 4;
constexpr uint32_t kStP = kOpA + 2 * 64 * kLd * 4;   // 3 blocks of 16 x 17 floats
// P1 scratch inside the g tile once every g value is in registers
constexpr uint32_t kTot = kRawG, kMid = kRawG + 2048;

// ---- TMEM columns ------------------------------------------------------------
constexpr uint32_t kTmA = 0;      // A_kk / A_qk raw products: 160 columns
constexpr uint32_t kTmD1 = 160;   // [Cb S ; Qb S], then rows 64..127 += A_qk E (= O)
constexpr uint32_t kTmD2 = 224;   // [E ; A_qk X (unused)]  128 lanes x 64
constexpr uint32_t kTmD3 = 288;   // Kb^T E                 128 lanes (key channel) x 64
constexpr uint32_t kTmCols = 512;

constexpr long long kWaitCycles = 4ll * 1000 * 1000 * 1000;   // ~2 s at 2 GHz

// ---- PTX helpers ---------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ float tf32r(float x) {   // round to nearest tf32
    uint32_t r;
    asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(r) : "f"(x));
    return __uint_as_float(r);
}
__device__ __forceinline__ void st_f32(uint32_t addr, float v) {
    asm volatile("st.shared.f32 [%0], %1;" ::"r"(addr), "f"(v) : "memory");
}
__device__ __forceinline__ float ld_f32(uint32_t addr) {
    float v;
    asm volatile("ld.shared.f32 %0, [%1];" : "=f"(v) : "r"(addr) : "memory");
    return v;
}
__device__ __forceinline__ float ld_bf16(uint32_t addr) {
    unsigned short h;
    asm volatile("ld.shared.u16 %0, [%1];" : "=h"(h) : "r"(addr) : "memory");
    return __uint_as_float(static_cast<uint32_t>(h) << 16);
}
// 128-byte swizzled K-major layout, 4-byte elements: K-blocks of 32 elements,
// each K-block `rows` x 128 B; 16-byte chunk index XOR (row % 8).
__device__ __forceinline__ uint32_t sw_f32(uint32_t base, uint32_t rows, uint32_t row, uint32_t k) {
    const uint32_t kb = k >> 5, kk = k & 31;
    return base + kb * rows * 128u + row * 128u + ((((kk >> 2) ^ (row & 7u)) << 4) | ((kk & 3u) << 2));
}
// The same swizzle for the bf16 tiles TMA writes (64 elements per 128-B row).
__device__ __forceinline__ uint32_t sw_bf16(uint32_t base, uint32_t rows, uint32_t row, uint32_t c) {
    const uint32_t kb = c >> 6, cc = c & 63;
    return base + kb * rows * 128u + row * 128u + ((((cc >> 3) ^ (row & 7u)) << 4) | ((cc & 7u) << 1));
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
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
__device__ __forceinline__ void mma_tf32(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc,
                                         uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::tf32 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a), "l"(b), "r"(idesc), "r"(accumulate)
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
// 32 lanes x 32 bit, 16 consecutive columns per thread.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float (&v)[16]) {
    uint32_t r[16];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
          "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

// One full-K tile product: D (+)= A[M x K] * B[N x K]^T, both K-major
// swizzled tiles in shared memory.  Issued by a single thread.
__device__ __forceinline__ void mma_tile(uint32_t d_tmem, uint32_t a_base, uint32_t a_rows,
                                         uint32_t b_base, uint32_t b_rows, int k_elems,
                                         uint32_t idesc, bool accumulate = false) {
    const int steps = k_elems / 8;   // tf32: 8 elements (32 bytes) per instruction
    for (int s = 0; s < steps; ++s) {
        const uint32_t kb = static_cast<uint32_t>(s) >> 2, kin = (static_cast<uint32_t>(s) & 3u) * 32u;
        mma_tf32(d_tmem, umma_desc(a_base + kb * a_rows * 128u + kin),
                 umma_desc(b_base + kb * b_rows * 128u + kin), idesc, (s > 0 || accumulate) ? 1u : 0u);
    }
}

struct ChunkParams {
    const float* S0;
    void* o;
    float* ST;
    int* err;
    int T, H, dv;
    int out_bf16;
};

// Column of the raw-product TMEM block holding A[r, i] for a row of
// sub-chunk R: group 3 at 0, group 2 at 64, group 0 at 112, group 1 at 128.
__device__ __forceinline__ int group_of_col(int col, int* i) {
    if (col < 64) { *i = col; return 3; }
    if (col < 112) { *i = col - 64; return 2; }
    if (col < 128) { *i = col - 112; return 0; }
    *i = col - 128;
    return 1;
}

__global__ void __launch_bounds__(kThreads, 1)
chunk_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
             const __grid_constant__ CUtensorMap tm_b, const __grid_constant__ CUtensorMap tm_g,
             const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_w,
             const ChunkParams prm) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t base = (smem_u32(smem_raw) + 1023u) & ~1023u;
    uint8_t* sgen = smem_raw + (base - smem_u32(smem_raw));   // generic pointer to the same base
    const uint32_t bar_tma = base + kMisc, bar_mma = base + kMisc + 8;
    volatile uint32_t* tmem_slot = reinterpret_cast<volatile uint32_t*>(sgen + kMisc + 16);

    const int tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;
    const int c = tid & 127;          // key channel (elementwise phases) / TMEM lane
    const int R = tid >> 7;           // sub-chunk (elementwise) / 16-column piece (epilogues)
    const int quarter = warp & 3;     // TMEM lane quarter this warp may access
    const int bh = blockIdx.x;
    const int bi = bh / prm.H, h = bh % prm.H;
    const int j0 = blockIdx.y * kDVT;
    const int T = prm.T;
    const int nchunks = (T + kC - 1) / kC;

    if (tid == 0) {
        mbar_init(bar_tma, 1);
        mbar_init(bar_mma, 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        fence_async_smem();
    }
    if (warp == 0) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         base + kMisc + 16),
                     "r"(kTmCols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const uint32_t lane_base = static_cast<uint32_t>(quarter * 32) << 16;

    auto issue_loads = [&](int n) {
        const int t0 = n * kC;
        mbar_expect_tx(bar_tma, kRawBytes);
        tma_load_4d(base + kRawQ, &tm_q, 0, h, t0, bi, bar_tma);
        tma_load_4d(base + kRawQ + 8192, &tm_q, 64, h, t0, bi, bar_tma);
        tma_load_4d(base + kRawK, &tm_k, 0, h, t0, bi, bar_tma);
        tma_load_4d(base + kRawK + 8192, &tm_k, 64, h, t0, bi, bar_tma);
        tma_load_4d(base + kRawB, &tm_b, 0, h, t0, bi, bar_tma);
        tma_load_4d(base + kRawB + 8192, &tm_b, 64, h, t0, bi, bar_tma);
        tma_load_4d(base + kRawG, &tm_g, 0, h, t0, bi, bar_tma);
        tma_load_4d(base + kRawG + 8192, &tm_g, 64, h, t0, bi, bar_tma);
        tma_load_4d(base + kRawV, &tm_v, j0, h, t0, bi, bar_tma);
        tma_load_4d(base + kRawW, &tm_w, j0, h, t0, bi, bar_tma);
    };
    if (tid == 0 && nchunks > 0) issue_loads(0);

    // fp32 state: S[c][j0 + 16R + jj], jj = 0..15, kept in registers.
    float S[16];
    {
        const float* s0 = prm.S0 ? prm.S0 + (static_cast<int64_t>(bh) * kDK + c) * prm.dv + j0 + 16 * R
                                 : nullptr;
#pragma unroll
        for (int jj = 0; jj < 16; ++jj) {
            S[jj] = s0 ? s0[jj] : 0.f;
            st_f32(sw_f32(base + kSt, 64, 16 * R + jj, c), tf32r(S[jj]));
        }
    }

    uint32_t mma_phase = 0;
    int loads_done = 0;               // chunks whose raw tiles have arrived
    bool failed = false;
    auto mma_wait = [&]() -> bool {
        const bool ok = mbar_wait(bar_mma, mma_phase);
        mma_phase ^= 1u;
        const bool bad = __syncthreads_or(!ok);
        tc_fence_after();
        return !bad;
    };
    // Make generic-proxy smem writes visible to the tensor core, then issue.
    auto sync_for_mma = [&]() {
        fence_async_smem();
        tc_fence_before();
        __syncthreads();
        tc_fence_after();
    };

    for (int n = 0; n < nchunks && !failed; ++n) {
        const int t0 = n * kC;
        const int nv = min(kC, T - t0);
        {
            const bool ok = mbar_wait(bar_tma, static_cast<uint32_t>(n & 1));
            if (__syncthreads_or(!ok)) { failed = true; break; }
            loads_done = n + 1;
        }

        // ---- P1: cumulative decay and the decay factors about each sub-chunk's reference
        float rho[16], irho[16];
        float gmu, emu, eCmu, gamma;
        {
            float Gm[16];
            float acc = 0.f;
#pragma unroll
            for (int s = 0; s < 16; ++s) {
                acc += ld_bf16(sw_bf16(base + kRawG, 64, 16 * R + s, c));
                Gm[s] = acc;
            }
            __syncthreads();   // every g value is in registers: the g tile becomes scratch
            st_f32(base + kTot + (R * 128 + c) * 4, acc);
            __syncthreads();
            float pre = 0.f, gC = 0.f;
#pragma unroll
            for (int r2 = 0; r2 < 4; ++r2) {
                const float t = ld_f32(base + kTot + (r2 * 128 + c) * 4);
                gC += t;
                if (r2 < R) pre += t;
            }
            gmu = Gm[7] + pre;
            st_f32(base + kMid + (R * 128 + c) * 4, gmu);
#pragma unroll
            for (int s = 0; s < 16; ++s) {
                const float d = Gm[s] + pre - gmu;
                rho[s] = __expf(fminf(d, 80.f));
                irho[s] = __expf(fminf(-d, 80.f));
            }
            emu = __expf(gmu);           // e^{G_m}       (<= 1)
            eCmu = __expf(gC - gmu);     // e^{G_C - G_m} (<= 1)
            gamma = __expf(gC);          // e^{G_C}
        }
        // [Ct; Qt]: rows scaled by e^{G_r - G_m(r)}
#pragma unroll
        for (int s = 0; s < 16; ++s) {
            const int r = 16 * R + s;
            const float kv = ld_bf16(sw_bf16(base + kRawK, 64, r, c));
            const float bv = ld_bf16(sw_bf16(base + kRawB, 64, r, c));
            const float qv = ld_bf16(sw_bf16(base + kRawQ, 64, r, c));
            st_f32(sw_f32(base + kOpA, 128, r, c), tf32r(bv * kv * rho[s]));
            st_f32(sw_f32(base + kOpA, 128, 64 + r, c), tf32r(qv * rho[s]));
        }
        __syncthreads();   // kMid visible to all

        // ---- intra-chunk products.  Key-column group g holds k_i * e^{G_m(g) - G_i}
        // for i < 16(g+1).  Pass 0: group 3 (kOpB) -> TMEM columns 0..63 and
        // group 1 (kXE) -> 128..159; pass 1: groups 2 and 0 (kOpB) -> 64..127.
        auto put_group = [&](int grp, uint32_t buf, uint32_t rows, int row0) {
            if (grp < R) return;
            const float sc = grp == R ? 1.f : __expf(ld_f32(base + kMid + (grp * 128 + c) * 4) - gmu);
#pragma unroll
            for (int s = 0; s < 16; ++s) {
                const int i = 16 * R + s;
                const float kv = ld_bf16(sw_bf16(base + kRawK, 64, i, c));
                st_f32(sw_f32(buf, rows, row0 + i, c), tf32r(kv * irho[s] * sc));
            }
        };
        put_group(3, base + kOpB, 64, 0);
        put_group(1, base + kXE, 32, 0);
        sync_for_mma();
        if (tid == 0) {
            mma_tile(tmem + kTmA, base + kOpA, 128, base + kOpB, 64, kDK, idesc_tf32(128, 64));
            mma_tile(tmem + kTmA + 128, base + kOpA, 128, base + kXE, 32, kDK, idesc_tf32(128, 32));
            mma_commit(bar_mma);
        }
        if (!mma_wait()) { failed = true; break; }
        put_group(2, base + kOpB, 64, 0);
        put_group(0, base + kOpB, 64, 48);
        sync_for_mma();
        if (tid == 0) {
            mma_tile(tmem + kTmA + 64, base + kOpA, 128, base + kOpB, 64, kDK, idesc_tf32(128, 64));
            mma_commit(bar_mma);
        }
        if (!mma_wait()) { failed = true; break; }

        // ---- A_kk -> padded fp32 staging (solve input); A_qk -> rows 64..127 of the
        // [T; A_qk] operand (tf32, zero above the diagonal).  T staging zeroed.
        for (int e = tid; e < 1024; e += kThreads) {   // operand rows 64..127, both K-blocks
            const uint32_t kb = static_cast<uint32_t>(e >> 9), rw = 64u + ((e >> 3) & 63), ch = e & 7;
            asm volatile("st.shared.v4.f32 [%0], {%1, %1, %1, %1};" ::"r"(base + kOpB + kb * 16384u + rw * 128u + ch * 16u), "f"(0.f) : "memory");
        }
        for (int e = tid; e < 64 * kLd; e += kThreads) st_f32(base + kStT + e * 4, 0.f);
        __syncthreads();
        {
            const int q2 = quarter & 1;                 // lanes 0-15: group 2*q2, 16-31: group 2*q2+1
            const int rr = q2 * 32 + lane;              // row of A_kk (quarters 0,1) or A_qk (2,3)
            const int Rr = rr >> 4;
            const bool is_q = quarter >= 2;
            int pieces[2], np = 0;
            if (q2 == 0) { if (R < 3) pieces[np++] = 7 + R; }
            else { pieces[np++] = R; if (R + 4 < 7) pieces[np++] = R + 4; }
            for (int pi = 0; pi < np; ++pi) {
                float v[16];
                tmem_ld16(tmem + lane_base + kTmA + static_cast<uint32_t>(pieces[pi]) * 16u, v);
#pragma unroll
                for (int e = 0; e < 16; ++e) {
                    int i;
                    const int g = group_of_col(pieces[pi] * 16 + e, &i);
                    if (g != Rr) continue;
                    if (!is_q) {
                        if (i < rr) st_f32(base + kStAkk + (rr * kLd + i) * 4, v[e]);
                    } else if (i <= rr) {
                        st_f32(sw_f32(base + kOpB, 128, 64 + rr, i), tf32r(v[e]));
                    }
                }
            }
        }
        tc_fence_before();
        __syncthreads();

        // ---- T = (I + A_kk)^-1.  16x16 diagonal blocks by column forward substitution
        if (tid < 64) {
            const int o16 = 16 * (tid >> 4), col = tid & 15;
            float tcol[16];
#pragma unroll
            for (int r = 0; r < 16; ++r) tcol[r] = r == col ? 1.f : 0.f;
#pragma unroll
            for (int r = 1; r < 16; ++r) {
                float sum = 0.f;
#pragma unroll
                for (int i = 0; i < r; ++i)
                    sum = fmaf(ld_f32(base + kStAkk + ((o16 + r) * kLd + o16 + i) * 4), tcol[i], sum);
                if (r > col) tcol[r] = -sum;
            }
#pragma unroll
            for (int r = 0; r < 16; ++r) st_f32(base + kStT + ((o16 + r) * kLd + o16 + col) * 4, tcol[r]);
        }
        __syncthreads();
        // off-diagonal blocks, level d = Rb - I:  T_{Rb,I} = -T_{Rb,Rb} sum_{J=I}^{Rb-1} A_{Rb,J} T_{J,I}
        // one warp per block; lane -> row lane/2, columns 8*(lane&1) .. +7
#pragma unroll 1
        for (int d = 1; d < 4; ++d) {
            const int rr = lane >> 1, c8 = 8 * (lane & 1);
            const int bI = warp, Rb = d + warp;
            if (warp < 4 - d) {
                float p[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) p[e] = 0.f;
#pragma unroll 1
                for (int J = bI; J < Rb; ++J) {
#pragma unroll
                    for (int k16 = 0; k16 < 16; ++k16) {
                        const int kk = 16 * J + k16;
                        const float a = ld_f32(base + kStAkk + ((16 * Rb + rr) * kLd + kk) * 4);
#pragma unroll
                        for (int e = 0; e < 8; ++e)
                            p[e] = fmaf(a, ld_f32(base + kStT + (kk * kLd + 16 * bI + c8 + e) * 4), p[e]);
                    }
                }
#pragma unroll
                for (int e = 0; e < 8; ++e) st_f32(base + kStP + (bI * 16 * 17 + rr * 17 + c8 + e) * 4, p[e]);
            }
            __syncthreads();
            if (warp < 4 - d) {
                float t[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) t[e] = 0.f;
#pragma unroll
                for (int kk = 0; kk < 16; ++kk) {
                    const float a = ld_f32(base + kStT + ((16 * Rb + rr) * kLd + 16 * Rb + kk) * 4);
#pragma unroll
                    for (int e = 0; e < 8; ++e)
                        t[e] = fmaf(a, ld_f32(base + kStP + (bI * 16 * 17 + kk * 17 + c8 + e) * 4), t[e]);
                }
#pragma unroll
                for (int e = 0; e < 8; ++e) st_f32(base + kStT + ((16 * Rb + rr) * kLd + 16 * bI + c8 + e) * 4, -t[e]);
            }
            __syncthreads();
        }
        // T -> rows 0..63 of the [T; A_qk] operand
        {
            const int cc = tid & 63;
#pragma unroll
            for (int m = 0; m < 8; ++m) {
                const int r = (tid >> 6) + 8 * m;
                st_f32(sw_f32(base + kOpB, 128, r, cc), tf32r(ld_f32(base + kStT + (r * kLd + cc) * 4)));
            }
        }
        __syncthreads();   // staging reads done before [Cb; Qb] overwrites the area

        // ---- [Cb; Qb] = [c * e^{G}; q * e^{G}] rows, then MMA1: [Cb S ; Qb S]
#pragma unroll
        for (int s = 0; s < 16; ++s) {
            const int r = 16 * R + s;
            const float eg = rho[s] * emu;
            const float kv = ld_bf16(sw_bf16(base + kRawK, 64, r, c));
            const float bv = ld_bf16(sw_bf16(base + kRawB, 64, r, c));
            const float qv = ld_bf16(sw_bf16(base + kRawQ, 64, r, c));
            st_f32(sw_f32(base + kOpA, 128, r, c), tf32r(bv * kv * eg));
            st_f32(sw_f32(base + kOpA, 128, 64 + r, c), tf32r(qv * eg));
        }
        sync_for_mma();
        if (tid == 0) {
            mma_tile(tmem + kTmD1, base + kOpA, 128, base + kSt, 64, kDK, idesc_tf32(128, kDVT));
            mma_commit(bar_mma);
        }
        if (!mma_wait()) { failed = true; break; }

        // ---- X = U - Cb S (rows 0..63) -> X^T operand as a tf32 pair; Kb^T operand
        if (quarter < 2) {
            float v[16];
            tmem_ld16(tmem + lane_base + kTmD1 + static_cast<uint32_t>(R) * 16u, v);
            const int r = quarter * 32 + lane;
#pragma unroll
            for (int jj = 0; jj < 16; ++jj) {
                const int j = 16 * R + jj;
                const float u = ld_bf16(sw_bf16(base + kRawW, 64, r, j)) * ld_bf16(sw_bf16(base + kRawV, 64, r, j));
                const float x = u - v[jj], xh = tf32r(x);
                st_f32(sw_f32(base + kXE, 64, j, r), xh);
                st_f32(sw_f32(base + kLo, 64, j, r), tf32r(x - xh));
            }
        }
#pragma unroll
        for (int s = 0; s < 16; ++s) {
            const int r = 16 * R + s;
            const float kv = ld_bf16(sw_bf16(base + kRawK, 64, r, c));
            st_f32(sw_f32(base + kOpA, 128, c, r), tf32r(kv * eCmu * irho[s]));
        }
        sync_for_mma();
        if (tid == 0) {   // MMA2: [T; A_qk] (X_hi + X_lo) -> rows 0..63 = E
            mma_tile(tmem + kTmD2, base + kOpB, 128, base + kXE, 64, kC, idesc_tf32(128, kDVT));
            mma_tile(tmem + kTmD2, base + kOpB, 128, base + kLo, 64, kC, idesc_tf32(128, kDVT), true);
            mma_commit(bar_mma);
            if (n + 1 < nchunks) issue_loads(n + 1);   // every read of the raw tiles is done
        }
        if (!mma_wait()) { failed = true; break; }

        // ---- E (rows 0..63) -> E^T operand as a tf32 pair
        if (quarter < 2) {
            float v[16];
            tmem_ld16(tmem + lane_base + kTmD2 + static_cast<uint32_t>(R) * 16u, v);
            const int r = quarter * 32 + lane;
#pragma unroll
            for (int jj = 0; jj < 16; ++jj) {
                const float eh = tf32r(v[jj]);
                st_f32(sw_f32(base + kXE, 64, 16 * R + jj, r), eh);
                st_f32(sw_f32(base + kLo, 64, 16 * R + jj, r), tf32r(v[jj] - eh));
            }
        }
        sync_for_mma();
        if (tid == 0) {
            // MMA3: Kb^T E -> D3.  MMA_O: [T; A_qk] E accumulated onto [Cb S; Qb S]:
            // rows 64..127 become O = Qb S + A_qk E (rows 0..63 are not used).
            mma_tile(tmem + kTmD3, base + kOpA, 128, base + kXE, 64, kC, idesc_tf32(128, kDVT));
            mma_tile(tmem + kTmD3, base + kOpA, 128, base + kLo, 64, kC, idesc_tf32(128, kDVT), true);
            mma_tile(tmem + kTmD1, base + kOpB, 128, base + kXE, 64, kC, idesc_tf32(128, kDVT), true);
            mma_tile(tmem + kTmD1, base + kOpB, 128, base + kLo, 64, kC, idesc_tf32(128, kDVT), true);
            mma_commit(bar_mma);
        }
        if (!mma_wait()) { failed = true; break; }

        // ---- S <- diag(e^{G_C}) S + Kb^T E; refresh the S^T operand; store O
        {
            float v[16];
            tmem_ld16(tmem + lane_base + kTmD3 + static_cast<uint32_t>(R) * 16u, v);
#pragma unroll
            for (int jj = 0; jj < 16; ++jj) {
                S[jj] = fmaf(gamma, S[jj], v[jj]);
                st_f32(sw_f32(base + kSt, 64, 16 * R + jj, c), tf32r(S[jj]));
            }
        }
        if (quarter >= 2) {
            float v[16];
            tmem_ld16(tmem + lane_base + kTmD1 + static_cast<uint32_t>(R) * 16u, v);
            const int r = quarter * 32 + lane - 64;
            if (r < nv) {
                const int64_t off = ((static_cast<int64_t>(bi) * T + t0 + r) * prm.H + h) * prm.dv + j0 + 16 * R;
                if (prm.out_bf16) {
                    __nv_bfloat16* op = static_cast<__nv_bfloat16*>(prm.o) + off;
#pragma unroll
                    for (int jj = 0; jj < 16; jj += 2)
                        *reinterpret_cast<__nv_bfloat162*>(op + jj) = __floats2bfloat162_rn(v[jj], v[jj + 1]);
                } else {
                    float4* op = reinterpret_cast<float4*>(static_cast<float*>(prm.o) + off);
#pragma unroll
                    for (int jj = 0; jj < 16; jj += 4) op[jj / 4] = make_float4(v[jj], v[jj + 1], v[jj + 2], v[jj + 3]);
                }
            }
        }
        tc_fence_before();
        __syncthreads();
    }

    if (failed) {
        if (tid == 0) {
            atomicExch(prm.err, kDevTimeout);
            // a tile load may still be in flight: wait for it (bounded) before exiting
            if (loads_done < nchunks) mbar_wait(bar_tma, static_cast<uint32_t>(loads_done & 1));
        }
    } else if (prm.ST) {
        float* st = prm.ST + (static_cast<int64_t>(bh) * kDK + c) * prm.dv + j0 + 16 * R;
#pragma unroll
        for (int jj = 0; jj < 16; jj += 4)
            *reinterpret_cast<float4*>(st + jj) = make_float4(S[jj], S[jj + 1], S[jj + 2], S[jj + 3]);
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
    return a.in_dtype == GDR2_BF16 && a.dk == kDK && (a.dv == 64 || a.dv == 128) && a.T > 0 &&
           a.T < (1ll << 31) && a.B < (1ll << 31) && a.B * a.H < (1ll << 31) && get_encode() != nullptr;
}

int launch_chunked_bf16(const ForwardArgs& a, cudaStream_t stream, int* err) {
    CUtensorMap mq, mk, mb, mg, mv, mw;
    if (!make_map(&mq, a.q, a.B, a.T, a.H, a.dk) || !make_map(&mk, a.k, a.B, a.T, a.H, a.dk) ||
        !make_map(&mb, a.b, a.B, a.T, a.H, a.dk) || !make_map(&mg, a.g, a.B, a.T, a.H, a.dk) ||
        !make_map(&mv, a.v, a.B, a.T, a.H, a.dv) || !make_map(&mw, a.w, a.B, a.T, a.H, a.dv))
        return GDR2_ERR_CUDA;
    static std::once_flag attr_once;
    static cudaError_t attr_err = cudaSuccess;
    std::call_once(attr_once, [] {
        attr_err = cudaFuncSetAttribute(chunk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                        static_cast<int>(kSmemAlloc));
    });
    if (attr_err != cudaSuccess) return GDR2_ERR_CUDA;
    ChunkParams prm{a.S0, a.o, a.ST, err, static_cast<int>(a.T), static_cast<int>(a.H),
                    static_cast<int>(a.dv), a.out_dtype == GDR2_BF16 ? 1 : 0};
    const dim3 grid(static_cast<unsigned>(a.B * a.H), static_cast<unsigned>(a.dv / kDVT));
    chunk_kernel<<<grid, kThreads, kSmemAlloc, stream>>>(mq, mk, mb, mg, mv, mw, prm);
    return cudaPeekAtLastError() == cudaSuccess ? GDR2_OK : GDR2_ERR_CUDA;
}

}  // namespace gdr2
