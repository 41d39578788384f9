// Chunk-parallel scan over sequence segments for the chunked prefill.
//
// Method ("Gated DeltaNet-2: Decoupling Erase and Write in Linear Attention"
// page, "efficient implementation" section: the state recurrence is a product
// of affine maps).  Every chunk maps its start state S to diag(e^{G_C}) S + Kb^T E
// with E linear in S, so a run of chunks (a segment) maps its start state by
//     S_end = M S_start + N,          o_t = o_t^0 + S_start^T r_t,
// where N and o^0 come from the segment run from a zero state and M, r_t (= M_t^T
// q_t, M_t the map up to token t) from the segment run from the identity with
// U = 0.  The state kernel produces those for all segments at once; here
//     S_start(1) = end state of segment 0 (run from S0),
//     S_start(g + 1) = M_g S_start(g) + N_g,      S_T = S_start(G),
// then o_t = o_t^0 + S_start(g)^T r_t for the tokens of every segment g >= 1.
// The scan (G - 1 products of 128 x 128 by 128 x d_v per (sequence, head)) is fp32
// FMA on CUDA cores; the correction is a dense contraction over the 128 key channels
// per token and runs on tcgen05 tensor cores while streaming r, o^0 and o once.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <mutex>

#include "gdr2.h"
#include "gdr2_internal.cuh"
#include "gdr2_tc.cuh"

namespace gdr2 {
namespace {

constexpr int kDK = kPrepDK;

PFN_cuTensorMapEncodeTiled_v12000 encoder() {
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

// [N][rows][H][width] token rows (fp32, or bf16) as a 4-D map (width, H, rows, N) with a
// box of (box_cols, 1, 128 rows, 1) and the 128-byte swizzle: rows past a sequence's
// end are outside the map (loads read zeros, stores are dropped).
bool make_seq_map(CUtensorMap* m, const void* ptr, int64_t N, int64_t rows, int64_t H, int64_t width, bool f32,
                  uint32_t box_cols) {
    auto enc = encoder();
    if (!enc) return false;
    const cuuint64_t esz = f32 ? 4 : 2;
    const cuuint64_t dims[4] = {static_cast<cuuint64_t>(width), static_cast<cuuint64_t>(H),
                                static_cast<cuuint64_t>(rows), static_cast<cuuint64_t>(N)};
    const cuuint64_t strides[3] = {static_cast<cuuint64_t>(width) * esz, static_cast<cuuint64_t>(H * width) * esz,
                                   static_cast<cuuint64_t>(rows * H * width) * esz};
    const cuuint32_t box[4] = {box_cols, 1, 128, 1};
    const cuuint32_t estr[4] = {1, 1, 1, 1};
    return enc(m, f32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4,
               const_cast<void*>(ptr), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
               CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// fp32 matrix of `rows` rows of 128 as a 2-D map, box (32, 64 rows), 128-byte swizzle.
bool make_rows_map(CUtensorMap* m, const float* ptr, int64_t rows) {
    auto enc = encoder();
    if (!enc) return false;
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(kDK), static_cast<cuuint64_t>(rows)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(kDK) * 4};
    const cuuint32_t box[2] = {32, 64};
    const cuuint32_t estr[2] = {1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<float*>(ptr), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// One CTA per (sequence * head, 64-column tile of d_v): the segments' start states in
// order, each written over the segment's own end-state slot (slot g then holds
// S_start(g + 1)) and, transposed ([d_v][d_k], the correction's K-major operand), to
// slot g of sT; the last is S_T.
constexpr int kScanThreads = 256;
constexpr int kSpPitch = 68;   // row pitch (floats) of the state tile: 16-byte rows, 4-way column reads
__global__ void __launch_bounds__(kScanThreads)
scan_kernel(float* seg_state, const float* seg_m, float* sT, float* ST, int G, int H, int dv) {
    __shared__ __align__(16) float sp[kDK][kSpPitch];   // S_start(g), this tile's 64 columns
    const int seq = blockIdx.x / H, h = blockIdx.x % H;
    const int c0 = blockIdx.y * 64;
    const int tid = threadIdx.x;
    const int i = tid >> 1, cb = (tid & 1) * 32;   // row i, columns cb .. cb + 31 of the tile
    auto slot = [&](int g) { return static_cast<int64_t>(blockIdx.x) * G + g; };   // (seq * H + h) * G + g
    {
        const float* s = seg_state + slot(0) * kDK * dv + c0;
        for (int e = tid; e < kDK * 16; e += kScanThreads) {
            const int row = e >> 4, q = e & 15;
            *reinterpret_cast<float4*>(&sp[row][4 * q]) = *reinterpret_cast<const float4*>(s + row * dv + 4 * q);
        }
    }
    __syncthreads();
    for (int g = 1; g < G; ++g) {
        {
            float* d = sT + (slot(g) * dv + c0) * kDK;
            for (int e = tid; e < kDK * 64; e += kScanThreads) d[e] = sp[e & (kDK - 1)][e >> 7];
        }
        float* n = seg_state + (slot(g) * kDK + i) * dv + c0 + cb;
        const float4* m = reinterpret_cast<const float4*>(seg_m + (slot(g) * kDK + i) * kDK);
        float acc[32];
#pragma unroll
        for (int e = 0; e < 32; e += 4) {
            const float4 x = *reinterpret_cast<const float4*>(n + e);
            acc[e] = x.x; acc[e + 1] = x.y; acc[e + 2] = x.z; acc[e + 3] = x.w;
        }
#pragma unroll 2
        for (int k4 = 0; k4 < kDK / 4; ++k4) {
            const float4 mv = m[k4];
            const float mk[4] = {mv.x, mv.y, mv.z, mv.w};
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const float* srow = &sp[4 * k4 + u][cb];
#pragma unroll
                for (int e = 0; e < 32; e += 4) {
                    const float4 s4 = *reinterpret_cast<const float4*>(srow + e);
                    acc[e] = fmaf(mk[u], s4.x, acc[e]);
                    acc[e + 1] = fmaf(mk[u], s4.y, acc[e + 1]);
                    acc[e + 2] = fmaf(mk[u], s4.z, acc[e + 2]);
                    acc[e + 3] = fmaf(mk[u], s4.w, acc[e + 3]);
                }
            }
        }
        __syncthreads();   // every thread has read S_start(g)
#pragma unroll
        for (int e = 0; e < 32; e += 4) {
            const float4 x = make_float4(acc[e], acc[e + 1], acc[e + 2], acc[e + 3]);
            *reinterpret_cast<float4*>(&sp[i][cb + e]) = x;
            *reinterpret_cast<float4*>(n + e) = x;
        }
        __syncthreads();
    }
    if (ST) {
        float* d = ST + (static_cast<int64_t>(seq) * H + h) * kDK * dv + c0;
        for (int e = tid; e < kDK * 16; e += kScanThreads) {
            const int row = e >> 4, q = e & 15;
            *reinterpret_cast<float4*>(d + row * dv + 4 * q) = *reinterpret_cast<const float4*>(&sp[row][4 * q]);
        }
    }
}

// o rows of segments g >= 1: o_t = o32_t + S_start(g)^T r_t on tcgen05 (kind::tf32,
// fp32 accumulate).  One CTA of 128 threads per (128-row tile of one sequence's
// later-segment rows, 64 output columns, head, sequence): TMA brings the r tile (A,
// 128 rows x 128 channels) and 64 rows of S_start(g)^T (B, 64 columns x 128
// channels), one thread issues the 16 K-steps into a 64-column TMEM accumulator, the
// o32 tile then arrives by TMA in A's buffer, each warp adds its 32 accumulator rows
// to it and one TMA store writes the tile to o (rows past the sequence are dropped).
// Segments hold an even number of chunks, so no tile straddles two of them.
constexpr int kCorrThreads = 128;
constexpr int kCorrRows = 128;
constexpr uint32_t kCA = 0;          // r tile: 4 K-blocks of [128 rows][32 fp32], 128-byte swizzle
constexpr uint32_t kCB = 65536;      // S_start^T rows: 4 K-blocks of [64 rows][32 fp32]
constexpr uint32_t kCBar = 98304;    // mbarriers: operands, MMA done, o32 tile
constexpr uint32_t kCSlot = kCBar + 32;
constexpr uint32_t kCSmem = kCBar + 64 + 1024;

// Packed sequences: the 128-row correction tiles of segment g of sequence s start at
// tile_base[s (G - 1) + g - 1] (segments g >= 1; each segment's rows tiled from its
// first row, so that no tile straddles two segments), the total at tile_base[N (G - 1)].
// One CTA.
__global__ void seg_plan_kernel(const int* cu, const int* cb, int N, int G, int total, int* tile_base) {
    __shared__ int part[1024];
    const int tid = threadIdx.x;
    const int per = (N + blockDim.x - 1) / blockDim.x;
    const int s0 = tid * per, s1 = min(N, s0 + per);
    auto tiles = [&](int s, int g) {
        const PackedSegment ps = packed_segment(cu, cb, total, s, G, g);
        const int r0 = ps.cs * kPrepC, r1 = min(min(ps.cs + ps.Lc, ps.given) * kPrepC, ps.Ts);
        return r1 > r0 ? (r1 - r0 + kCorrRows - 1) / kCorrRows : 0;
    };
    int sum = 0;
    for (int s = s0; s < s1; ++s)
        for (int g = 1; g < G; ++g) sum += tiles(s, g);
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
    for (int s = s0; s < s1; ++s)
        for (int g = 1; g < G; ++g) {
            tile_base[s * (G - 1) + g - 1] = run;
            run += tiles(s, g);
        }
    if (s1 == N && s0 < s1) tile_base[N * (G - 1)] = run;
    if (N == 0 && tid == 0) tile_base[0] = 0;
}

// kPacked: packed sequences.  blockIdx.x / (dv / 64) numbers the tiles of all
// (sequence, segment g >= 1) in turn (tile_base, from seg_plan_kernel; the grid is an
// upper bound and later CTAs exit), r and o32 are indexed by global row (one-sequence
// 4-D maps over all rows), and each thread stores its row of o itself, rows past the
// segment's end left alone.
struct PackedCorr {
    const int* cu;
    const int* cb;
    const int* tile_base;
    int N, total;
};

template <bool kBf16Out, bool kPacked>
__global__ void __launch_bounds__(kCorrThreads)
correct_kernel(const __grid_constant__ CUtensorMap tm_r, const __grid_constant__ CUtensorMap tm_st,
               const __grid_constant__ CUtensorMap tm_o32, const __grid_constant__ CUtensorMap tm_o, int G, int L,
               int H, int dv, int* err, const PackedCorr pk, void* o) {
    extern __shared__ uint8_t csm_raw[];
    using namespace tc;
    const uint32_t base = (smem_u32(csm_raw) + 1023u) & ~1023u;
    uint8_t* sgen = csm_raw + (base - smem_u32(csm_raw));
    const uint32_t bar_ab = base + kCBar, bar_mma = bar_ab + 8, bar_o = bar_ab + 16;
    volatile uint32_t* tslot = reinterpret_cast<volatile uint32_t*>(sgen + kCSlot);
    const int nh = dv / 64;
    const int tile = blockIdx.x / nh, j0 = (blockIdx.x % nh) * 64;
    const int h = blockIdx.y;
    int seq, g, t0, nrows;   // t0: the tile's first row (within the sequence's later-segment rows;
                             // packed: global); nrows: rows of the tile inside the segment
    if constexpr (kPacked) {
        const int nsg = pk.N * (G - 1);
        if (tile >= pk.tile_base[nsg]) return;   // past the last tile (the grid is a bound)
        int lo = 0, hi = nsg;                    // the last (sequence, segment) starting at or before it
        while (hi - lo > 1) {
            const int mid = (lo + hi) >> 1;
            if (pk.tile_base[mid] <= tile) lo = mid; else hi = mid;
        }
        seq = lo / (G - 1);
        g = 1 + lo % (G - 1);
        const PackedSegment ps = packed_segment(pk.cu, pk.cb, pk.total, seq, G, g);
        const int r0 = ps.cs * kPrepC, r1 = min(min(ps.cs + ps.Lc, ps.given) * kPrepC, ps.Ts);
        t0 = ps.a + r0 + (tile - pk.tile_base[lo]) * kCorrRows;
        nrows = min(kCorrRows, ps.a + r1 - t0);
    } else {
        seq = blockIdx.z;
        t0 = tile * kCorrRows;
        g = 1 + t0 / (L * kPrepC);
        nrows = kCorrRows;
    }
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    if (tid == 0) {
        mbar_init(bar_ab, 1);
        mbar_init(bar_mma, 1);
        mbar_init(bar_o, 1);
        fence_mbar_init();
    }
    if (warp == 0) tmem_alloc<64>(base + kCSlot);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tslot;
    bool ok = true;
    if (tid == 0) {
        mbar_expect_tx(bar_ab, 4u * 16384u + 4u * 8192u);
        const int srow = ((seq * H + h) * G + g) * dv + j0;   // S_start(g)^T rows j0 .. j0 + 63
        const int mseq = kPacked ? 0 : seq;   // packed: one map over every row
        for (int kb = 0; kb < 4; ++kb) {
            tma_load_4d(base + kCA + kb * 16384u, &tm_r, 32 * kb, h, t0, mseq, bar_ab);
            tma_load_2d(base + kCB + kb * 8192u, &tm_st, 32 * kb, srow, bar_ab);
        }
        ok = mbar_wait(bar_ab, 0);
        if (ok) {
            tc_fence_after();
#pragma unroll 1
            for (int s = 0; s < 16; ++s)
                mma_ss(tmem, umma_desc(kstep(base + kCA, 16384u, s)), umma_desc(kstep(base + kCB, 8192u, s)),
                       idesc_tf32(128, 64), s > 0 ? 1u : 0u);
            mma_commit(bar_mma);
            // A is free once the products have read it: the o32 tile takes its place
            ok = mbar_wait(bar_mma, 0);
            if (ok) {
                mbar_expect_tx(bar_o, 2u * 16384u);
                tma_load_4d(base + kCA, &tm_o32, j0, h, t0, mseq, bar_o);
                tma_load_4d(base + kCA + 16384u, &tm_o32, j0 + 32, h, t0, mseq, bar_o);
            }
        }
        if (!ok) {
            atomicExch(err, kDevTimeout);
            mbar_arrive(bar_o);   // release the other threads (no copy in flight on this barrier)
        }
    }
    // every thread: the accumulator and the o32 tile
    ok = mbar_wait(bar_o, 0) && ok;
    if (ok) ok = mbar_wait(bar_mma, 0);
    tc_fence_after();
    if (ok) {
        const int row = warp * 32 + lane;
        const uint32_t taddr = tmem + (static_cast<uint32_t>(warp * 32) << 16);
#pragma unroll
        for (int c16 = 0; c16 < 4; ++c16) {
            uint32_t acc[16];
            tmem_ld16_nw(taddr + 16u * c16, acc);
            tmem_ld_wait();
            // o32 box c16 / 2, columns 16 (c16 % 2) .. + 15: four 16-byte chunks of the swizzled row
            const uint32_t rb = kCA + static_cast<uint32_t>(c16 >> 1) * 16384u + static_cast<uint32_t>(row) * 128u;
            float y[16];
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const uint32_t a = rb + ((((4 * (c16 & 1) + q) ^ (row & 7)) & 7) << 4);
                const float4 x = *reinterpret_cast<const float4*>(sgen + a);
                y[4 * q] = x.x + __uint_as_float(acc[4 * q]);
                y[4 * q + 1] = x.y + __uint_as_float(acc[4 * q + 1]);
                y[4 * q + 2] = x.z + __uint_as_float(acc[4 * q + 2]);
                y[4 * q + 3] = x.w + __uint_as_float(acc[4 * q + 3]);
            }
            if constexpr (kPacked) {
                // this thread's row of o, columns j0 + 16 c16 .. + 15, if inside the segment
                if (row < nrows) {
                    const int64_t off = (static_cast<int64_t>(t0 + row) * H + h) * dv + j0 + 16 * c16;
                    if constexpr (kBf16Out) {
                        uint4 pk4[2];
                        uint32_t* pw = reinterpret_cast<uint32_t*>(pk4);
#pragma unroll
                        for (int e = 0; e < 8; ++e) {
                            __nv_bfloat162 b2 = __floats2bfloat162_rn(y[2 * e], y[2 * e + 1]);
                            pw[e] = *reinterpret_cast<uint32_t*>(&b2);
                        }
                        uint4* op = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(o) + off);
                        op[0] = pk4[0];
                        op[1] = pk4[1];
                    } else {
                        float4* op = reinterpret_cast<float4*>(static_cast<float*>(o) + off);
#pragma unroll
                        for (int q = 0; q < 4; ++q) op[q] = make_float4(y[4 * q], y[4 * q + 1], y[4 * q + 2], y[4 * q + 3]);
                    }
                }
            } else if constexpr (!kBf16Out) {
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const uint32_t a = rb + ((((4 * (c16 & 1) + q) ^ (row & 7)) & 7) << 4);
                    *reinterpret_cast<float4*>(sgen + a) =
                        make_float4(y[4 * q], y[4 * q + 1], y[4 * q + 2], y[4 * q + 3]);
                }
            } else {
                // bf16 tile [128 rows][64 columns] (128-byte rows, swizzled) after the o32 tile
                const uint32_t ob = kCA + 32768u + static_cast<uint32_t>(row) * 128u;
#pragma unroll
                for (int q = 0; q < 2; ++q) {
                    uint4 pk;
                    uint32_t* pw = reinterpret_cast<uint32_t*>(&pk);
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        __nv_bfloat162 b2 = __floats2bfloat162_rn(y[8 * q + 2 * e], y[8 * q + 2 * e + 1]);
                        pw[e] = *reinterpret_cast<uint32_t*>(&b2);
                    }
                    *reinterpret_cast<uint4*>(sgen + ob + ((((2 * c16 + q) ^ (row & 7)) & 7) << 4)) = pk;
                }
            }
        }
    }
    fence_async_smem();
    tc_fence_before();
    __syncthreads();
    if (!kPacked && tid == 0 && ok) {
        const int orow = L * kPrepC + t0;   // row of o within the sequence
        if constexpr (kBf16Out) {
            tma_store_4d(&tm_o, base + kCA + 32768u, j0, h, orow, seq);
        } else {
            tma_store_4d(&tm_o, base + kCA, j0, h, orow, seq);
            tma_store_4d(&tm_o, base + kCA + 16384u, j0 + 32, h, orow, seq);
        }
        bulk_commit();
        bulk_wait_all();
    }
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc<64>(tmem);
    }
}

}  // namespace

int launch_scan(const ForwardArgs& a, const SegArgs& seg, cudaStream_t stream) {
    if (seg.G < 2 || a.dk != kDK || (a.dv != 64 && a.dv != 128) || !seg.sT) return GDR2_ERR_ARG;
    const dim3 grid(static_cast<unsigned>(a.B * a.H), static_cast<unsigned>(a.dv / 64));
    scan_kernel<<<grid, kScanThreads, 0, stream>>>(seg.seg_state, seg.seg_m, seg.sT, a.ST, seg.G,
                                                   static_cast<int>(a.H), static_cast<int>(a.dv));
    return cudaPeekAtLastError() == cudaSuccess ? GDR2_OK : GDR2_ERR_CUDA;
}

int launch_seg_plan(const ForwardArgs& a, const SegArgs& seg, cudaStream_t stream) {
    if (!a.cu || seg.G < 2 || !seg.chunk_base || !seg.tile_base) return GDR2_ERR_ARG;
    seg_plan_kernel<<<1, 1024, 0, stream>>>(a.cu, seg.chunk_base, static_cast<int>(a.B), seg.G,
                                            static_cast<int>(a.total), seg.tile_base);
    return cudaPeekAtLastError() == cudaSuccess ? GDR2_OK : GDR2_ERR_CUDA;
}

int launch_correct(const ForwardArgs& a, const SegArgs& seg, cudaStream_t stream, int* err) {
    const bool packed = a.cu != nullptr;
    if (seg.G < 2 || !seg.sT || (packed ? !seg.chunk_base || !seg.tile_base : seg.Tr <= 0 || (seg.L & 1)))
        return GDR2_ERR_ARG;
    if (a.B > 65535 || a.H > 65535) return GDR2_ERR_SHAPE;   // grid z and y
    const bool bf = a.out_dtype == GDR2_BF16;
    CUtensorMap mr, mst, mo32, mo;
    if (packed) {   // one map over every row; o is stored row by row
        if (!make_seq_map(&mr, seg.r, 1, a.total, a.H, kDK, true, 32) ||
            !make_seq_map(&mo32, seg.o32, 1, a.total, a.H, a.dv, true, 32) ||
            !make_rows_map(&mst, seg.sT, a.B * a.H * seg.G * a.dv))
            return GDR2_ERR_CUDA;
        mo = mo32;   // not read
    } else if (!make_seq_map(&mr, seg.r, a.B, seg.Tr, a.H, kDK, true, 32) ||
               !make_seq_map(&mo32, seg.o32, a.B, seg.Tr, a.H, a.dv, true, 32) ||
               !make_seq_map(&mo, a.o, a.B, a.T, a.H, a.dv, !bf, bf ? 64 : 32) ||
               !make_rows_map(&mst, seg.sT, a.B * a.H * seg.G * a.dv)) {
        return GDR2_ERR_CUDA;
    }
    static std::once_flag once;
    static cudaError_t attr = cudaSuccess;
    std::call_once(once, [] {
        const void* kernels[4] = {reinterpret_cast<const void*>(correct_kernel<false, false>),
                                  reinterpret_cast<const void*>(correct_kernel<true, false>),
                                  reinterpret_cast<const void*>(correct_kernel<false, true>),
                                  reinterpret_cast<const void*>(correct_kernel<true, true>)};
        for (const void* k : kernels)
            if (attr == cudaSuccess)
                attr = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(kCSmem));
    });
    if (attr != cudaSuccess) return GDR2_ERR_CUDA;
    const PackedCorr pk{a.cu, seg.chunk_base, seg.tile_base, static_cast<int>(a.B), static_cast<int>(a.total)};
    const int nh = static_cast<int>(a.dv / 64);
    // packed: at most total / 128 + N (G - 1) tiles (each segment adds at most one partial tile)
    const int64_t tiles = packed ? a.total / kCorrRows + a.B * (seg.G - 1) + 1 : (seg.Tr + kCorrRows - 1) / kCorrRows;
    if (tiles * nh >= (1ll << 31)) return GDR2_ERR_SHAPE;
    const dim3 grid(static_cast<unsigned>(tiles * nh), static_cast<unsigned>(a.H),
                    static_cast<unsigned>(packed ? 1 : a.B));
    const int G = seg.G, L = seg.L, H = static_cast<int>(a.H), dv = static_cast<int>(a.dv);
    if (packed) {
        if (bf) correct_kernel<true, true><<<grid, kCorrThreads, kCSmem, stream>>>(mr, mst, mo32, mo, G, L, H, dv, err, pk, a.o);
        else correct_kernel<false, true><<<grid, kCorrThreads, kCSmem, stream>>>(mr, mst, mo32, mo, G, L, H, dv, err, pk, a.o);
    } else {
        if (bf) correct_kernel<true, false><<<grid, kCorrThreads, kCSmem, stream>>>(mr, mst, mo32, mo, G, L, H, dv, err, pk, a.o);
        else correct_kernel<false, false><<<grid, kCorrThreads, kCSmem, stream>>>(mr, mst, mo32, mo, G, L, H, dv, err, pk, a.o);
    }
    return cudaPeekAtLastError() == cudaSuccess ? GDR2_OK : GDR2_ERR_CUDA;
}

}  // namespace gdr2
