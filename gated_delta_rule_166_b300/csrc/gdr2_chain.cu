// Chunked Gated Delta Rule-2 prefill in affine form, part 2 of 2: the
// chunk-to-chunk state pass, one CTA per (sequence * head, 64-column d_v tile).
//
// Method ("Gated DeltaNet-2: Decoupling Erase and Write in Linear Attention"
// page, "efficient implementation" section: chunkwise algorithm).  Each 64-token
// chunk maps its start state S (d_k x d_v, fp32) to
//     S' = diag(gamma) S + M' S + Y U,      O = P S + X U,      U = w * v
// with M', Y, P, X and gamma = e^{G_C} written per (chunk, head) by the
// preparation kernel (gdr2_prep2.cu, which derives them).  Only M' S and the
// state update sit on the chunk-to-chunk chain: Y U and X U of the next chunk
// are issued while the chain runs, P S after it.
//
// Products on tcgen05 (kind::f16, fp32 accumulators in TMEM): M', Y, P, X are
// K-major fp16 A operands copied from the workspace slot unchanged; S (fp16,
// MN-major) and U^T (an fp16 pair u = u_hi + u_lo, 22 significant bits,
// K-major) are the B operands written by the elementwise warps.  The fp32 state stays in registers
// (16 entries per thread); only its fp16 image is an operand.
//
// Work split: 640 threads.  One thread of the last warpgroup issues the bulk
// copies of the slots and all MMAs (v and w are plain loads of the elementwise
// warps, one chunk ahead); a second one issues the TMA stores of
// O.  Warp w < 16 owns TMEM lane quarter w % 4 (d_k rows of the state, token
// rows of O) and 16 columns 16 (w / 4) .. of the d_v tile.  Warps signal the MMA
// thread through mbarriers with one arrival per warp; every wait is bounded.
#include <cuda.h>
#include <cudaTypedefs.h>
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
constexpr int kDVT = 64;
constexpr int kSimt = 512;
constexpr int kThreads = kSimt + 128;
constexpr int kRegsSimt = 104, kRegsMma = 56;
static_assert(kSimt * kRegsSimt + (kThreads - kSimt) * kRegsMma <= kThreads * 96, "register pool");

// ---- shared memory (bytes from a 1024-aligned base) ------------------------------
// two slot buffers, each the chunk's images copied unchanged: M' (32 KB), P (16 KB),
// Y (16 KB), X (8 KB)
constexpr uint32_t kSlotBuf = 73728;
constexpr uint32_t kBM = kSlotM, kBY = kSlotY, kBP = kSlotP, kBX = kSlotX;   // offsets within a slot buffer
constexpr uint32_t kSB = 2 * kSlotBuf;   // two S operands, fp16 MN-major [128 K rows][64] (16 KB each)
constexpr uint32_t kUB = kSB + 32768;    // two [U_hi^T | U_lo^T] operands, fp16 K-major [64][64] x 2 (16 KB each)
constexpr uint32_t kO = kUB + 32768;     // O tile for the TMA store (16 KB)
constexpr uint32_t kMisc = kO + 16384;
enum : uint32_t {
    kBarSlot0 = 0, kBarSlot1,                          // slot copies
    kSRdy, kURdy0, kURdy1, kORead0, kORead1, kOFull,   // elementwise warps -> issuing threads
    kOFree,                                            // O tile stored
    kDS0, kDS1, kDO0, kDO1,                            // MMA commits
    kDrain,                                            // every product issued has completed
    kNumBars
};
constexpr uint32_t kTmemSlot = kMisc + 8 * kNumBars;
constexpr uint32_t kAbort = kTmemSlot + 4;
constexpr uint32_t kSmemBytes = kMisc + 256;
constexpr uint32_t kSmemAlloc = kSmemBytes + 1024;
static_assert(kAbort + 4 <= kSmemBytes, "misc area");
static_assert(kSmemAlloc <= 232448, "shared memory");
constexpr uint32_t kSlotCopyBytes = kSlotGam;   // M', Y, P, X (gamma is read from global memory)
static_assert(kSlotCopyBytes <= kSlotBuf && (kSlotCopyBytes & 15u) == 0, "slot copy");

// ---- TMEM columns ------------------------------------------------------------------
// Products that accumulate into one TMEM accumulator run one after another (each
// waits for the previous one), so every product is split over two accumulators
// (K steps alternating, or u_hi / u_lo) whose instructions interleave; the read-out
// adds the two halves.  Per chunk buffer b: S' - gamma S in columns 128 b + [0, 128),
// O (M = 64) in 256 + 128 b + [0, 128).
constexpr uint32_t kTmDS = 0;
constexpr uint32_t kTmDO = 256;
constexpr int kTmCols = 512;

struct ChainParams {
    const uint8_t* slots;
    const float* S0;
    const __nv_bfloat16 *v, *w;
    void* o;
    float* ST;
    int* err;
    const int* cu;           // packed sequences: [N + 1] token offsets, or null
    const int* chunk_base;   // packed sequences: [N + 1] first global chunk of each sequence
    int T, H, dk, dv, nch, total;   // dk, dv <= 128 / 64 per tile; channels past them are zero padding
    int out_bf16;
    long long wait_cycles;   // limit of each handshake wait (copy drains keep the default)
    // Segments (G > 1): blockIdx.x = (sequence * G + g) * H + head runs chunks g L ..
    // g L + L - 1 (packed sequences: L = ceil(chunks / G) per sequence, o32 and r by
    // global row, Tr unused).  Value tiles of segment 0 start from S0 and write o;
    // those of later segments start from zero and write fp32 rows to o32.  Transfer tiles
    // (blockIdx.y >= the value tiles, segments g >= 1) start from identity columns j0 ..
    // of d_k with U = 0: their O rows are r_t = M_t^T q_t (M_t the map from the segment
    // start to token t), written to r.  End states go to seg_state [sequence][head][g]
    // [d_k][dv] (value) or seg_m [sequence][head][g][d_k][d_k] (transfer).
    int G, L, Tr;            // G = 1: one pass, L = the chunks of a sequence
    float *seg_state, *seg_m, *o32, *r;
    // fixed-length: this launch covers chunks c0 .. c0 + nch - 1 of every sequence (its
    // slots numbered from 0 per sequence); S0 is the state before chunk c0
    int c0;
    // the state after every cache_chunks chunks: [N][H][n_cache][d_k][dv] (null: not kept);
    // packed sequences (cache_chunks = 1): after every chunk, [global chunk][H][d_k][dv]
    float* cache;
    int cache_chunks, n_cache;
};

// One CTA; kTransfer: a transfer tile (identity start, U = 0), a separate
// instantiation so that value tiles carry no test of the tile kind on their chain.
template <bool kTransfer>
__device__ __forceinline__ void chain_cta(const CUtensorMap& tm_o, const CUtensorMap& tm_o32, const CUtensorMap& tm_r,
                                          const ChainParams& prm) {
    const int ntv = (prm.dv + kDVT - 1) / kDVT;
    const int h = static_cast<int>(blockIdx.x) % prm.H;
    const int sg = static_cast<int>(blockIdx.x) / prm.H;
    const int seq = sg / prm.G, g = sg - seq * prm.G;
    if (kTransfer && g == 0) return;   // segment 0 starts from S0 itself: no transfer map
    const int bh = seq * prm.H + h;
    const int j0 = (kTransfer ? static_cast<int>(blockIdx.y) - ntv : static_cast<int>(blockIdx.y)) * kDVT;

    extern __shared__ uint8_t smem_raw[];
    const uint32_t base = (smem_u32(smem_raw) + 1023u) & ~1023u;
    uint8_t* sgen = smem_raw + (base - smem_u32(smem_raw));
    auto bar = [&](uint32_t i) { return base + kMisc + 8u * i; };
    volatile uint32_t* tmem_slot = reinterpret_cast<volatile uint32_t*>(sgen + kTmemSlot);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(sgen + kAbort);

    const int tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;
    const int quarter = warp & 3;
    // this sequence's token rows and its first global chunk (offsets clamped as in prep2)
    int T, tok0, Lc = prm.L;   // Lc: chunks per segment of this sequence
    int64_t chunk0;
    if (prm.cu) {
        // only the chunks this sequence was given slots for (fewer than its length only
        // for overlapping malformed offsets, see chunk_base_kernel); with segments,
        // segment g's run of them
        const PackedSegment ps = packed_segment(prm.cu, prm.chunk_base, prm.total, seq, prm.G, g);
        if (prm.G > 1) Lc = ps.Lc;
        tok0 = ps.a + ps.cs * kC;
        T = max(ps.Ts - ps.cs * kC, 0);
        chunk0 = prm.chunk_base[seq] + ps.cs;
    } else {
        // chunks c0 + g L .. of the sequence: tokens counted from the first of them
        T = prm.T - (prm.c0 + g * prm.L) * kC;
        tok0 = seq * prm.T + (prm.c0 + g * prm.L) * kC;
        chunk0 = static_cast<int64_t>(seq) * prm.nch + static_cast<int64_t>(g) * prm.L;
    }
    const int n = min((T + kC - 1) / kC, Lc);
    // o rows: the caller's o (one pass, or segment 0), else fp32 scratch rows
    const bool to_o = prm.G == 1 || (!kTransfer && g == 0);
    const CUtensorMap* const om = to_o ? &tm_o : (kTransfer ? &tm_r : &tm_o32);
    const bool obf16 = to_o && prm.out_bf16;
    const int ow = kTransfer ? kPrepDK : prm.dv;   // width of an output row
    // o32 and r rows: per sequence after its first segment, or (packed) the global row
    const int orow0 = to_o || prm.cu ? tok0 : seq * prm.Tr + (g - 1) * prm.L * kC;
    void* const obase = to_o ? prm.o : (kTransfer ? static_cast<void*>(prm.r) : static_cast<void*>(prm.o32));
    auto slot_of = [&](int c) {
        return prm.slots + ((chunk0 + c) * prm.H + h) * static_cast<int64_t>(kSlot2Bytes);
    };

    if (tid == 0) {
        for (uint32_t i = 0; i < kNumBars; ++i) {
            // one arrival per warp; a barrier never runs more than one phase ahead of its
            // waiter (U of chunk c arrives on kURdy0 + c % 2, two chunks ahead of its use)
            const bool per_warp = i == kSRdy || i == kURdy0 || i == kURdy1 || i == kORead0 || i == kORead1 ||
                                  i == kOFull;
            mbar_init(bar(i), per_warp ? 16u : 1u);
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
        // ================= copies / MMAs / O stores ===================================
        asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kRegsMma));
        if (warp == kSimt / 32 && lane == 0) {
            // Per chunk c (buffer b = c & 1): the chain products of c as soon as its S^T is
            // written; then Y U and X U of chunk c + 1 (the first products in its
            // accumulators); then, once chunk c's products are done, the copy of chunk
            // c + 2's slot into buffer b.  Counters give each wait's parity.  Descriptors
            // are formed once; a K step adds its byte offset / 16 to the start address
            // field (every operand lies below 256 KB, so the field never carries).
            uint32_t c_slot0 = 0, c_slot1 = 0, c_s = 0, c_u0 = 0, c_u1 = 0, c_do0 = 0, c_do1 = 0, c_or0 = 0, c_or1 = 0;
            uint32_t iss_slot0 = 0, iss_slot1 = 0;   // copies issued per buffer (at most one in flight)
            // a wait that gave up does not count the phase as seen, so that the copy drain
            // below still waits for a copy whose completion was not observed
            auto wait = [&](uint32_t b, uint32_t& cnt) {
                const bool ok = mbar_wait_ab(bar(b), cnt & 1u, abort_flag, prm.wait_cycles);
                if (ok) ++cnt;
                return ok;
            };
            auto load_slot = [&](int c) {
                const uint32_t b = static_cast<uint32_t>(c & 1);
                mbar_expect_tx(bar(kBarSlot0 + b), kSlotCopyBytes);
                bulk_g2s(base + kSlotBuf * b, slot_of(c), kSlotCopyBytes, bar(kBarSlot0 + b));
                if (b) ++iss_slot1; else ++iss_slot0;
            };
            // A operands and U^T are K-major: a K step of 16 elements is 32 bytes within a
            // 128-byte row; M' (K = 128) has its two K blocks 16 KB apart, P 8 KB apart.  The
            // state S is MN-major (one 64-column block): a K step is 16 rows = 2048 bytes
            const uint64_t dM0 = umma_desc2(base + kBM, 16u, 1024u), dP0 = umma_desc2(base + kBP, 16u, 1024u);
            const uint64_t dY0 = umma_desc2(base + kBY, 16u, 1024u), dX0 = umma_desc2(base + kBX, 16u, 1024u);
            const uint64_t dS0 = umma_desc2(base + kSB, 16384u, 1024u), dU0 = umma_desc2(base + kUB, 16u, 1024u);
            constexpr uint32_t idS = idesc_f16x(128, 64, 0, 0, 1), idO = idesc_f16x(64, 64, 0, 0, 1);
            // Y U and X U of chunk c into accumulator buffer c & 1 (the first products
            // there): [U_hi^T; U_lo^T] is one 128-row B operand, so each product writes
            // u_hi terms to the first 64 columns of its accumulator pair and u_lo terms to
            // the second
            constexpr uint32_t idSU = idesc_f16x(128, 128, 0, 0, 0), idOU = idesc_f16x(64, 128, 0, 0, 0);
            auto issue_u = [&](int c) {
                const uint32_t b = static_cast<uint32_t>(c & 1);
                const uint64_t dY = dY0 + (kSlotBuf >> 4) * b, dX = dX0 + (kSlotBuf >> 4) * b;
                const uint64_t dU = dU0 + (16384u >> 4) * b;
                const uint32_t tS = tmem + kTmDS + 128u * b, tO = tmem + kTmDO + 128u * b;
                tc_fence_after();
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    const uint32_t acc = k > 0 ? 1u : 0u;
                    mma_ss_f16(tS, dY + 2u * k, dU + 2u * k, idSU, acc);
                    mma_ss_f16(tO, dX + 2u * k, dU + 2u * k, idOU, acc);
                }
            };
            bool ok = true;   // an empty sequence issues nothing
            bool issued = false;
            if (n > 0) {
                load_slot(0);
                if (n > 1) load_slot(1);
                ok = wait(kURdy0, c_u0) && wait(kBarSlot0, c_slot0);
                if (ok) {
                    issue_u(0);
                    issued = true;
                }
            }
#pragma unroll 1
            for (int c = 0; c < n && ok; ++c) {
                const uint32_t b = static_cast<uint32_t>(c & 1);
                const uint64_t dM = dM0 + (kSlotBuf >> 4) * b, dP = dP0 + (kSlotBuf >> 4) * b;
                const uint64_t dS = dS0 + (16384u >> 4) * b;
                // ---- chain: S' - gamma S += M' S;  O += P S ------------------------------
                if (!(ok = wait(kSRdy, c_s))) break;
                tc_fence_after();
                {
                    // K steps 0-3 (key channels 0-63) into the first accumulator of each
                    // pair, 4-7 into the second
                    const uint32_t tS = tmem + kTmDS + 128u * b, tO = tmem + kTmDO + 128u * b;
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        mma_ss_f16(tS, dM + 2u * k, dS + 128u * k, idS, 1u);
                        mma_ss_f16(tS + 64u, dM + (16384u >> 4) + 2u * k, dS + 512u + 128u * k, idS, 1u);
                    }
                    mma_commit(bar(kDS0 + b));
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        mma_ss_f16(tO, dP + 2u * k, dS + 128u * k, idO, 1u);
                        mma_ss_f16(tO + 64u, dP + (8192u >> 4) + 2u * k, dS + 512u + 128u * k, idO, 1u);
                    }
                    mma_commit(bar(kDO0 + b));
                }
                if (c + 1 < n) {
                    // ---- next chunk's Y U and X U (its accumulators were read out) --------
                    if (c >= 1 && !(ok = b ? wait(kORead0, c_or0) : wait(kORead1, c_or1))) break;
                    if (!(ok = b ? (wait(kURdy0, c_u0) && wait(kBarSlot0, c_slot0))
                                 : (wait(kURdy1, c_u1) && wait(kBarSlot1, c_slot1))))
                        break;
                    issue_u(c + 1);
                }
                if (c + 2 < n) {
                    // ---- chunk c's products done: its slot buffer takes chunk c + 2 --------
                    if (!(ok = b ? wait(kDO1, c_do1) : wait(kDO0, c_do0))) break;
                    load_slot(c + 2);
                }
            }
            if (!ok) {
                *abort_flag = 1;
                atomicExch(prm.err, kDevTimeout);
            }
            // copies still in flight land before the CTA exits (bounded waits; the last
            // copy of each buffer completes the phase of parity (issued - 1) & 1)
            if (iss_slot0 > c_slot0) mbar_wait(bar(kBarSlot0), (iss_slot0 - 1u) & 1u);
            if (iss_slot1 > c_slot1) mbar_wait(bar(kBarSlot1), (iss_slot1 - 1u) & 1u);
            // and every product issued completes before the TMEM is freed (after an abort
            // some may still be running)
            if (issued) {
                mma_commit(bar(kDrain));
                mbar_wait(bar(kDrain), 0u);
            }
        } else if (warp == kSimt / 32 + 1 && lane == 0) {
            // O tile stores: one per chunk that lies wholly inside the sequence
            uint32_t ph_full = 0;
            mbar_arrive(bar(kOFree));   // the tile starts free
#pragma unroll 1
            for (int c = 0; (c + 1) * kC <= T && c < n; ++c) {
                if (!mbar_wait_ab(bar(kOFull), ph_full, abort_flag, prm.wait_cycles)) break;
                ph_full ^= 1u;
                const int row = orow0 + c * kC;
                tma_store_4d(om, base + kO, j0, h, row, 0);
                if (!obf16 && j0 + 32 < ow) tma_store_4d(om, base + kO + 8192u, j0 + 32, h, row, 0);
                bulk_commit();
                bulk_wait_read();
                mbar_arrive(bar(kOFree));
            }
            bulk_wait_all();
        }
        __syncwarp();
    } else {
        // ================= 16 elementwise / accumulator warps ====================
        asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kRegsSimt));
        const uint32_t lane_base = static_cast<uint32_t>(quarter * 32) << 16;
        const int R = warp >> 2;                 // column block: d_v columns 16R .. 16R + 15 of the tile
        const int j = 32 * quarter + lane;       // state row (key channel)
        bool failed = false;
        uint32_t c_ds0 = 0, c_ds1 = 0, c_do0 = 0, c_do1 = 0, c_of = 0;
        auto wait = [&](uint32_t b, uint32_t& cnt) {
            const bool ok = mbar_wait_ab(bar(b), cnt & 1u, abort_flag, prm.wait_cycles);
            ++cnt;
            tc_fence_after();
            return ok;
        };
        auto arrive = [&](uint32_t b) {
            fence_async_smem();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(b));
        };
        // S operand (fp16, MN-major: 128 K rows j of 64 n-values, 128-byte swizzle): the
        // thread's 16 columns n = 16R .. 16R + 15 of row j are two 16-byte pieces
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
        // v, w of chunk c for d_v column un, tokens 8 ug .. 8 ug + 7 (raw bf16 bits; tokens past
        // the sequence end read as 0), fetched a chunk before they are used.  The loaded
        // values stay unpacked until put_u, so the loads overlap the rest of the chunk.
        const int un = tid & 63, ug = tid >> 6;
        struct VW {
            uint32_t v[8], w[8];   // raw bf16 bits, zero-extended by the load itself
        };
        // Consecutive tokens are H * d_v elements apart: one base address per chunk, and
        // rows past the sequence end (masked in put_u) read the last row instead.  Columns
        // past d_v (a 32-column value dim in a 64-column tile) read column d_v - 1: they
        // only feed state columns that are never stored.
        const int64_t row_stride = static_cast<int64_t>(prm.H) * prm.dv;
        const unsigned short* const vcol = reinterpret_cast<const unsigned short*>(prm.v) +
                                           static_cast<int64_t>(tok0) * row_stride + static_cast<int64_t>(h) * prm.dv +
                                           min(j0 + un, prm.dv - 1);
        const unsigned short* const wcol = reinterpret_cast<const unsigned short*>(prm.w) + (vcol - reinterpret_cast<const unsigned short*>(prm.v));
        auto fetch_vw = [&](int c, VW& x) {
            if (kTransfer) return;   // U = 0
            const int t0 = c * kC + 8 * ug;
            if (t0 + 7 < T) {
                const unsigned short* pv = vcol + static_cast<int64_t>(t0) * row_stride;
                const unsigned short* pw = wcol + static_cast<int64_t>(t0) * row_stride;
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    x.v[e] = __ldg(pv + e * row_stride);
                    x.w[e] = __ldg(pw + e * row_stride);
                }
            } else {
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    const int64_t t = min(t0 + e, T - 1);
                    x.v[e] = __ldg(vcol + t * row_stride);
                    x.w[e] = __ldg(wcol + t * row_stride);
                }
            }
        };
        // U^T of chunk c (fp16 pair u = u_hi + u_lo) into buffer c & 1: row un, tokens 8 ug ..
        auto put_u = [&](int c, const VW& x) {
            if (kTransfer) {   // U = 0
                uint8_t* ub = sgen + kUB + 16384u * static_cast<uint32_t>(c & 1);
                const uint32_t off = static_cast<uint32_t>(un) * 128u + ((static_cast<uint32_t>(ug) ^ (static_cast<uint32_t>(un) & 7u)) << 4);
                *reinterpret_cast<uint4*>(ub + off) = make_uint4(0u, 0u, 0u, 0u);
                *reinterpret_cast<uint4*>(ub + 8192u + off) = make_uint4(0u, 0u, 0u, 0u);
                return;
            }
            const int tvalid = T - c * kC - 8 * ug;   // tokens past the sequence end give U = 0
            uint4 hk, lk;
            __half2* hh = reinterpret_cast<__half2*>(&hk);
            __half2* lh = reinterpret_cast<__half2*>(&lk);
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const float u0 = 2 * e < tvalid ? __uint_as_float(x.v[2 * e] << 16) * __uint_as_float(x.w[2 * e] << 16) : 0.f;
                const float u1 = 2 * e + 1 < tvalid
                                     ? __uint_as_float(x.v[2 * e + 1] << 16) * __uint_as_float(x.w[2 * e + 1] << 16)
                                     : 0.f;
                const __half2 h2 = __floats2half2_rn(u0, u1);
                const float2 hf = __half22float2(h2);
                hh[e] = h2;
                lh[e] = __floats2half2_rn(u0 - hf.x, u1 - hf.y);
            }
            uint8_t* ub = sgen + kUB + 16384u * static_cast<uint32_t>(c & 1);
            const uint32_t off = static_cast<uint32_t>(un) * 128u + ((static_cast<uint32_t>(ug) ^ (static_cast<uint32_t>(un) & 7u)) << 4);
            *reinterpret_cast<uint4*>(ub + off) = hk;
            *reinterpret_cast<uint4*>(ub + 8192u + off) = lk;
        };

        float S[16];
        if (kTransfer) {
#pragma unroll
            for (int jj = 0; jj < 16; ++jj) S[jj] = j == j0 + 16 * R + jj ? 1.f : 0.f;   // identity columns
        } else {
            // state rows past d_k and columns past d_v are zero padding; segments after the
            // first start from zero
            const bool live = j < prm.dk && j0 + 16 * R < prm.dv && g == 0;
            const float* s0 = prm.S0 && live ? prm.S0 + (static_cast<int64_t>(bh) * prm.dk + j) * prm.dv + j0 + 16 * R : nullptr;
#pragma unroll
            for (int jj = 0; jj < 16; jj += 4) {
                const float4 x = s0 ? *reinterpret_cast<const float4*>(s0 + jj) : make_float4(0.f, 0.f, 0.f, 0.f);
                S[jj] = x.x; S[jj + 1] = x.y; S[jj + 2] = x.z; S[jj + 3] = x.w;
            }
        }
        // gamma of the next chunk, read from its slot one chunk ahead
        float gam_next = n > 0 ? __ldg(reinterpret_cast<const float*>(slot_of(0) + kSlotGam) + j) : 1.f;
        VW vpre;   // v, w of chunk c + 2
        if (n > 0) {
            put_st(0, S);
            arrive(kSRdy);
            fetch_vw(0, vpre);
            put_u(0, vpre);
            arrive(kURdy0);
            if (n > 1) {
                fetch_vw(1, vpre);
                put_u(1, vpre);
                arrive(kURdy1);
            }
            if (n > 2) fetch_vw(2, vpre);
        }
#pragma unroll 1
        for (int c = 0; c < n && !failed; ++c) {
            const uint32_t b = static_cast<uint32_t>(c & 1);
            const int tc = c * kC;
            // ---- chain: S <- gamma S + (M' S + Y U); S^T operand of the next chunk ------------
            const float gam = gam_next;
            if (c + 1 < n) gam_next = __ldg(reinterpret_cast<const float*>(slot_of(c + 1) + kSlotGam) + j);
            if (!(b ? wait(kDS1, c_ds1) : wait(kDS0, c_ds0))) { failed = true; break; }
            {
                float v[16];
                tmem_ld16_pair(tmem + lane_base + kTmDS + 128u * b + static_cast<uint32_t>(16 * R), v);
#pragma unroll
                for (int jj = 0; jj < 16; ++jj) S[jj] = fmaf(gam, S[jj], v[jj]);
            }
            if (c + 1 < n) {
                // the other S^T buffer was read by chunk c - 1's products, which completed
                // before that chunk's O was read out
                put_st(b ^ 1u, S);
                arrive(kSRdy);
            }
            if (!kTransfer && prm.cache) {
                // the state after chunk cc of the sequence, every cache_chunks chunks (stored
                // after the next chunk's operand is released: off the chain's critical path)
                if (prm.cu) {
                    if (j < prm.dk && j0 + 16 * R < prm.dv) {
                        float* cp = prm.cache + (((chunk0 + c) * prm.H + h) * prm.dk + j) * prm.dv + j0 + 16 * R;
#pragma unroll
                        for (int jj = 0; jj < 16; jj += 4)
                            *reinterpret_cast<float4*>(cp + jj) = make_float4(S[jj], S[jj + 1], S[jj + 2], S[jj + 3]);
                    }
                } else {
                    const int cc = prm.c0 + c;
                    const int ci = (cc + 1) / prm.cache_chunks - 1;
                    if ((cc + 1) % prm.cache_chunks == 0 && ci < prm.n_cache && j < prm.dk && j0 + 16 * R < prm.dv) {
                        float* cp = prm.cache + ((static_cast<int64_t>(bh) * prm.n_cache + ci) * prm.dk + j) * prm.dv + j0 + 16 * R;
#pragma unroll
                        for (int jj = 0; jj < 16; jj += 4)
                            *reinterpret_cast<float4*>(cp + jj) = make_float4(S[jj], S[jj + 1], S[jj + 2], S[jj + 3]);
                    }
                }
            }
            if (c + 2 < n) {
                // ---- U^T of chunk c + 2 into the buffer chunk c's products have read ----
                put_u(c + 2, vpre);
                arrive(kURdy0 + b);
                if (c + 3 < n) fetch_vw(c + 3, vpre);
            }
            // ---- O -> global ----------------------------------------------------------------
            if (!(b ? wait(kDO1, c_do1) : wait(kDO0, c_do0))) { failed = true; break; }
            {
                float v[16];
                tmem_ld16_pair(tmem + lane_base + kTmDO + 128u * b + static_cast<uint32_t>(16 * R), v);
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(bar(kORead0 + b));   // the accumulator may take chunk c + 2
                const int r = 16 * quarter + (lane & 15);          // M = 64: token row r at lane 32 (r / 16) + r % 16
                const bool active = lane < 16;
                if (tc + kC <= T) {
                    if (!wait(kOFree, c_of)) { failed = true; break; }
                    if (active) {
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
                    }
                    arrive(kOFull);
                } else if (active && tc + r < T && j0 + 16 * R < ow) {   // the last, partial chunk: row by row
                    const int64_t off = ((static_cast<int64_t>(orow0) + tc + r) * prm.H + h) * ow + j0 + 16 * R;
                    if (obf16) {
                        __nv_bfloat16* op = static_cast<__nv_bfloat16*>(obase) + off;
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
                        float4* op = reinterpret_cast<float4*>(static_cast<float*>(obase) + off);
#pragma unroll
                        for (int jj = 0; jj < 16; jj += 4)
                            op[jj / 4] = make_float4(v[jj], v[jj + 1], v[jj + 2], v[jj + 3]);
                    }
                }
            }
        }
        if (failed) {
            *abort_flag = 1;
            if (lane == 0) atomicExch(prm.err, kDevTimeout);
        } else if (prm.G > 1) {
            // the segment's end state (d_k = 128 on this path)
            float* st = (kTransfer ? prm.seg_m : prm.seg_state) +
                        (static_cast<int64_t>(bh * prm.G + g) * kPrepDK + j) * ow + j0 + 16 * R;
#pragma unroll
            for (int jj = 0; jj < 16; jj += 4)
                *reinterpret_cast<float4*>(st + jj) = make_float4(S[jj], S[jj + 1], S[jj + 2], S[jj + 3]);
        } else if (prm.ST && j < prm.dk && j0 + 16 * R < prm.dv) {
            float* st = prm.ST + (static_cast<int64_t>(bh) * prm.dk + j) * prm.dv + j0 + 16 * R;
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
chain_kernel(const __grid_constant__ CUtensorMap tm_o, const __grid_constant__ CUtensorMap tm_o32,
             const __grid_constant__ CUtensorMap tm_r, const ChainParams prm) {
    if (static_cast<int>(blockIdx.y) >= (prm.dv + kDVT - 1) / kDVT)
        chain_cta<true>(tm_o, tm_o32, tm_r, prm);
    else
        chain_cta<false>(tm_o, tm_o32, tm_r, prm);
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

namespace {
std::atomic<int64_t> g_wait_limit{0};
}  // namespace

int64_t set_chain_wait_limit(int64_t cycles) { return g_wait_limit.exchange(cycles); }

int launch_chain(const ForwardArgs& a, const uint8_t* slots, const int* chunk_base, cudaStream_t stream, int* err,
                 const SegArgs& seg, int c0, int cpiece) {
    if (a.cu && !chunk_base) return GDR2_ERR_ARG;
    const bool segmented = seg.G > 1;
    const int64_t nch = cpiece > 0 ? cpiece : (a.T + kC - 1) / kC;   // chunks per sequence in this launch
    if ((segmented || a.cu) && (c0 != 0 || cpiece > 0)) return GDR2_ERR_ARG;
    if (a.cu && a.S_cache && a.cache_chunks != 1) return GDR2_ERR_ARG;   // packed: every chunk's state
    if (segmented && (a.dk != kPrepDK || !seg.seg_state || !seg.seg_m || !seg.o32 || !seg.r ||
                      (!a.cu && (seg.L < 1 || static_cast<int64_t>(seg.G - 1) * seg.L >= nch)) ||
                      (a.cu && a.S_cache)))
        return GDR2_ERR_ARG;
    const int64_t total = a.cu ? a.total : a.B * a.T;
    CUtensorMap mo, mo32, mr;
    if (!make_row_map(&mo, a.o, total, a.H, a.dv, a.out_dtype != GDR2_BF16)) return GDR2_ERR_CUDA;
    if (segmented) {
        const int64_t srows = a.cu ? total : a.B * seg.Tr;   // rows of o32 and r
        if (!make_row_map(&mo32, seg.o32, srows, a.H, a.dv, true) ||
            !make_row_map(&mr, seg.r, srows, a.H, kPrepDK, true))
            return GDR2_ERR_CUDA;
    } else {
        mo32 = mo;   // not read
        mr = mo;
    }
    static std::once_flag attr_once;
    static cudaError_t attr_err = cudaSuccess;
    std::call_once(attr_once, [] {
        attr_err = cudaFuncSetAttribute(chain_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                        static_cast<int>(kSmemAlloc));
    });
    if (attr_err != cudaSuccess) return GDR2_ERR_CUDA;
    ChainParams prm{slots, a.S0, static_cast<const __nv_bfloat16*>(a.v), static_cast<const __nv_bfloat16*>(a.w),
                    a.o, a.ST, err, a.cu, chunk_base, static_cast<int>(a.T), static_cast<int>(a.H),
                    static_cast<int>(a.dk), static_cast<int>(a.dv), static_cast<int>(nch),
                    static_cast<int>(total),
                    a.out_dtype == GDR2_BF16 ? 1 : 0, 0,
                    segmented ? seg.G : 1,
                    segmented && !a.cu ? seg.L : (a.cu ? 0x7fffffff : static_cast<int>(nch)),
                    segmented ? static_cast<int>(seg.Tr) : 0,
                    seg.seg_state, seg.seg_m, seg.o32, seg.r, c0, a.S_cache,
                    a.S_cache ? static_cast<int>(a.cache_chunks) : 1,
                    a.S_cache ? static_cast<int>(a.T / (a.cache_chunks * kC)) : 0};
    const int64_t lim = g_wait_limit.load();
    prm.wait_cycles = lim > 0 ? static_cast<long long>(lim) : kWaitCycles;
    const int ntv = static_cast<int>((a.dv + kDVT - 1) / kDVT);
    const dim3 grid(static_cast<unsigned>(a.B * (segmented ? seg.G : 1) * a.H),
                    static_cast<unsigned>(ntv + (segmented ? kPrepDK / kDVT : 0)));
    chain_kernel<<<grid, kThreads, kSmemAlloc, stream>>>(mo, mo32, mr, prm);
    return cudaPeekAtLastError() == cudaSuccess ? GDR2_OK : GDR2_ERR_CUDA;
}

}  // namespace gdr2
