// fr_attn_sw.cu -- the decode attention for few query rows with the KV tile
// on the MMA's M side: S^T = K Q^T and O^T = V^T P^T on tcgen05.
//
// FlashRT PR #185, commits "FLASH_ATTN_EXT with q_tokens <= 16 over a single
// padded f16 KV head ..." (QK^T with the K operand shared by every GQA head,
// masked fp32-accurate softmax, PV into [hd, n_head, n_tok]) and "The GQA query
// heads share the one KV head, so the per-head batched QK^T and PV GEMMs
// collapse into single GEMMs over all n_head*n_tok query rows". For decode
// shapes a 128-row query tile (the MMA's M) would be mostly padding; here 128
// keys are the MMA's M and a slice of NQ query rows its N (16, 32 or 64), so
// the tensor work follows the real rows.
//
// One CTA = one KV split x one slice of NQ of the M <= 128 query rows (one CTA
// per SM; when M is cut into several slices, the slices' CTAs of a split read
// the same K/V tiles, the later reads served by L2); W softmax warps (8 for 16
// rows, 16 for 32 or 64 rows) and two more:
//   warps 0..W-1  softmax, one thread per (key of the tile, W/4-th of the
//              slice's rows): warps w, w + 4, ... share TMEM lane quadrant
//              w % 4 (keys 32(w%4)..+31 of S^T), each owning at most 16 rows.
//              kq_scale and the mask; the per-row reference maxima are only
//              recomputed when some score exceeds its row's reference by more
//              than 2^8 (one barrier-OR vote per tile; the row maxima then come
//              from warp shuffles and the four lane quadrants through shared
//              memory, and O and the partial sums are rescaled); P = 2^(s - m)
//              as two f16 terms P_hi + P_lo, written MN-major (one 128-byte row
//              per key) as the B operand of the PV MMA; partial row sums per
//              thread. After the loop the same threads own the TMEM lanes of
//              O^T (lane = head dim) for the epilogue, where O = O_hi + O_lo.
//   warp W     TMA producer: one ring of 32 KiB stages (128 keys x 128 dims of
//              K or of V, two 64-dim boxes) filled in exactly the order the
//              MMAs consume them, a ring of mask tiles, and in the fused call
//              the slice's f32 Q rows (one bulk copy per token) for the
//              in-kernel RoPE.
//   warp W+1   MMA issuer: S^T_j = K_j Q^T (A = K stage, K-major; B = the Q
//              rows), O^T += V_j^T [P_hi; P_lo]^T (A = V stage and B = P^T, both
//              read MN-major; the P_lo product accumulates in its own columns).
//              S_{j+1} is issued before PV_j, so the softmax of tile j+1
//              overlaps PV_j.
// In the fused call the kernel ropes its rows itself with qkv_post's
// arithmetic (fr_qkv_post's device routines), so one call is one launch.
// Each split writes its unnormalised O rows with its row maxima (log2 units)
// and sums to the workspace (part_o[s][r][hd] over all M rows: a split's rows
// are contiguous); after a bounded grid barrier (cooperative launch) the
// softmax warps of every CTA merge a share of the output rows. A single split
// normalises and writes the output rows itself.
// Every mbarrier wait is bounded; a wait that gives up sets the status word,
// and the CTA still drains its copies and MMAs and frees its TMEM.
#include <math.h>
#include <string.h>

#include <cudaTypedefs.h>

#include "fr_attn.h"
#include "fr_common.cuh"
#include "fr_sm100.cuh"
#include "fr_split_merge.cuh"
#include "fr_trace.cuh"

namespace fr {
namespace sw {

using namespace sm100;

constexpr int kKeys = 128;               // keys per KV tile = the MMA's M
constexpr float kTau = 8.0f;
constexpr float kLog2e = 1.4426950408889634f;
constexpr int kBox = 16384;              // 128 rows x 128 bytes (64 f16), 128-byte swizzle
constexpr int kStage = 2 * kBox;         // 128 keys x 128 dims of K or V
constexpr int kPrefetchPieces = 2;       // ring pieces prefetched to L2 before the launch wait
constexpr int kSmemLimit = 232448;

template <int HD, int NQ>
struct Cfg {
    static_assert(HD == 128 || HD == 256, "head dims");
    static_assert(NQ == 16 || NQ == 32 || NQ == 64, "query rows");
    static constexpr int HALVES = HD / 128;          // K (and V) stages per tile
    // softmax warps: 8 (two per TMEM lane quadrant) for 16 rows, 16 (four per
    // quadrant) for 32 or 64 rows, so that a thread owns at most 16 rows
    static constexpr int SMW = NQ >= 32 ? 16 : 8;
    static constexpr int SMT = SMW * 32;             // softmax threads
    static constexpr int PROD_WARP = SMW, MMA_WARP = SMW + 1;
    static constexpr int THREADS = (SMW + 2) * 32;
    static constexpr int RH = NQ / (SMW / 4);        // rows per softmax thread
    static constexpr int N2 = 2 * NQ < 64 ? 64 : 2 * NQ;   // PV MMA N: [P_hi | P_lo | zeros]
    static constexpr int Q_BOX = NQ * 128;           // 64 dims of the NQ rows (K-major)
    static constexpr int Q_BYTES = (HD / 64) * Q_BOX;
    static constexpr int P_BYTES = (N2 / 64) * kBox; // P^T: 128 keys x N2 (MN-major, 64 columns per box)
    static constexpr int MASK_BOX = kMaskWin * 128;  // <= 16 token rows x 64 keys, unswizzled
    static constexpr int MASK_BYTES = 2 * MASK_BOX;
    static constexpr int MS = 3;                     // mask slots
    static constexpr int AUX = 4096;
    static constexpr int FIXED = Q_BYTES + 2 * P_BYTES + MS * MASK_BYTES + AUX + 1024;
    static constexpr int R = (kSmemLimit - 1024 - FIXED) / kStage;     // ring stages
    static_assert(R >= 2, "ring depth");
    static constexpr int RING_OFF = 0;
    static constexpr int Q_OFF = R * kStage;
    static constexpr int P_OFF = Q_OFF + Q_BYTES;
    static constexpr int M_OFF = P_OFF + 2 * P_BYTES;
    static constexpr int AUX_OFF = M_OFF + MS * MASK_BYTES;
    static constexpr int BAR_OFF = AUX_OFF + AUX;
    static constexpr int SMEM = BAR_OFF + 1024 + 1024;   // barriers + TMEM word, + alignment slack
    static_assert(SMEM <= kSmemLimit, "shared memory budget");
    static_assert(Q_BYTES % 1024 == 0 && MASK_BOX % 1024 == 0, "1024-B alignment of swizzled tiles");
    // the f32 Q rows of the fused call land in the P buffers (free until the
    // first P tile, which comes after QFULL)
    static_assert(NQ * HD * 4 <= 2 * P_BYTES, "f32 Q rows in the P buffers");
    // aux: [4][NQ] per-quadrant partial maxima / sums, [NQ] row max m, [NQ]
    // rescale factors, [NQ] row sums l, a flag; then the RoPE table
    static constexpr int AUX_RED = 0;
    static constexpr int AUX_M = 4 * NQ * 4;
    static constexpr int AUX_A = AUX_M + NQ * 4;
    static constexpr int AUX_L = AUX_A + NQ * 4;
    static constexpr int AUX_FLAG = AUX_L + NQ * 4;
    static constexpr int AUX_POS = AUX_FLAG + 16;    // [kMaskWin] token positions (fused call)
    static constexpr int AUX_TB = (AUX_POS + kMaskWin * 4 + 15) / 16 * 16;
    static_assert(AUX_TB + (int)sizeof(RopeTable) <= AUX, "aux");
    static_assert(RH % 8 == 0, "P rows per thread: whole 16-byte chunks");
    static constexpr int B_FULL = 0, B_EMPTY = R, B_MFULL = 2 * R, B_MEMPTY = 2 * R + MS,
                         B_SFULL = 2 * (R + MS), B_PFULL = B_SFULL + 2, B_ODONE = B_SFULL + 4,
                         B_QFULL = B_SFULL + 5, B_MMADONE = B_SFULL + 6, B_PROBE = B_SFULL + 7,
                         B_QF32 = B_SFULL + 8, N_BARS = B_SFULL + 9;
    static constexpr int TMEM_SLOT = 120 * 8;
    static_assert(N_BARS <= 120, "barrier slots");
    // TMEM columns: S^T double buffer (NQ each), then O^T per 128-dim half
    // (N2: O_hi^T in [0, NQ), O_lo^T in [NQ, 2NQ))
    static constexpr int TM_S = 0;
    static constexpr int TM_O = 2 * NQ;
    static constexpr int TM_USED = TM_O + HALVES * N2;
    static constexpr uint32_t TM_COLS = TM_USED <= 32 ? 32u : TM_USED <= 64 ? 64u : TM_USED <= 128 ? 128u
                                        : TM_USED <= 256 ? 256u : 512u;
};

// Reduce-scatter across the 32 lanes of a warp (maximum or sum) of CH values
// per lane (CH = 8, 16 or 32): at each step the lanes with bit S set keep the
// upper half of the values and their partners the lower half, so that after
// log2(CH) steps a lane holds one value, reduced over the lanes that differ
// in the bits used so far; the remaining steps reduce over the other bits.
// Lane L then holds row rs_row(L) of the chunk.
template <int S, int CNT, int CH, bool MAX>
struct ReduceScatter {
    __device__ static __forceinline__ void run(float (&v)[CH], int lane) {
        if constexpr (CNT >= 2) {
            constexpr int H = CNT / 2;
            const bool up = (lane & S) != 0;
#pragma unroll
            for (int i = 0; i < H; ++i) {
                const float send = up ? v[i] : v[i + H];
                const float keep = up ? v[i + H] : v[i];
                const float got = __shfl_xor_sync(0xffffffffu, send, S);
                v[i] = MAX ? fmaxf(keep, got) : keep + got;
            }
            if constexpr (S > 1) ReduceScatter<S / 2, H, CH, MAX>::run(v, lane);
        } else {
            const float got = __shfl_xor_sync(0xffffffffu, v[0], S);
            v[0] = MAX ? fmaxf(v[0], got) : v[0] + got;
            if constexpr (S > 1) ReduceScatter<S / 2, 1, CH, MAX>::run(v, lane);
        }
    }
};

// Row (within a chunk of CH rows) that lane L holds after ReduceScatter.
template <int CH>
__device__ __forceinline__ int rs_row(int lane) {
    int base = 0, cnt = CH;
#pragma unroll
    for (int s = 16; s >= 1; s >>= 1) {
        if (cnt >= 2) {
            cnt >>= 1;
            if (lane & s) base += cnt;
        }
    }
    return base;
}

__device__ __forceinline__ void record_timeout(unsigned* status, unsigned bit) { atomicOr(status, bit); }
// Barrier over the N softmax threads (named barrier 1).
template <int N>
__device__ __forceinline__ void softmax_bar_sync() {
    asm volatile("bar.sync 1, %0;" :: "n"(N) : "memory");
}
// The same barrier, returning whether any softmax thread passed a true vote.
template <int N>
__device__ __forceinline__ bool softmax_bar_any(bool vote) {
    uint32_t r;
    asm volatile("{ .reg .pred p, q; setp.ne.u32 q, %1, 0; bar.red.or.pred p, 1, %2, q; selp.u32 %0, 1, 0, p; }"
                 : "=r"(r) : "r"((uint32_t)vote), "n"(N) : "memory");
    return r != 0;
}

template <int N>
__device__ __forceinline__ void tmem_ld_cols(uint32_t taddr, float* x) {
    if constexpr (N == 8) {
        tmem_ld_x8(taddr, reinterpret_cast<uint32_t*>(x));
    } else if constexpr (N == 16) {
        tmem_ld_x16(taddr, reinterpret_cast<uint32_t*>(x));
    } else {
#pragma unroll
        for (int c = 0; c < N; c += 32) tmem_ld_x32(taddr + c, reinterpret_cast<uint32_t*>(x) + c);
    }
}
template <int N>
__device__ __forceinline__ void tmem_st_cols(uint32_t taddr, const float* x) {
    if constexpr (N == 8) {
        tmem_st_x8(taddr, reinterpret_cast<const uint32_t*>(x));
    } else if constexpr (N == 16) {
        tmem_st_x16(taddr, reinterpret_cast<const uint32_t*>(x));
    } else {
#pragma unroll
        for (int c = 0; c < N; c += 32) tmem_st_x32(taddr + c, reinterpret_cast<const uint32_t*>(x) + c);
    }
}

template <int HD, int NQ>
__global__ void __launch_bounds__(Cfg<HD, NQ>::THREADS, 1)
attn_sw_kernel(const __grid_constant__ SwArgs a, const __grid_constant__ SwMaps mp,
               const __grid_constant__ RopeTable tb) {
    using C = Cfg<HD, NQ>;
    constexpr int RH = C::RH;
    constexpr int kSmaxWarps = C::SMW, kSmaxThreads = C::SMT;
    constexpr int kProdWarp = C::PROD_WARP, kMmaWarp = C::MMA_WARP;
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    unsigned char* sm = reinterpret_cast<unsigned char*>(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    uint64_t* bars = reinterpret_cast<uint64_t*>(sm + C::BAR_OFF);
    uint32_t* sTmemBase = reinterpret_cast<uint32_t*>(sm + C::BAR_OFF + C::TMEM_SLOT);
    float* sRed = reinterpret_cast<float*>(sm + C::AUX_OFF + C::AUX_RED);     // [4][NQ]
    float* sM = reinterpret_cast<float*>(sm + C::AUX_OFF + C::AUX_M);         // [NQ] row max (log2 units)
    float* sA = reinterpret_cast<float*>(sm + C::AUX_OFF + C::AUX_A);         // [NQ] rescale factors
    float* sL = reinterpret_cast<float*>(sm + C::AUX_OFF + C::AUX_L);         // [NQ] row sums
    int* sFlag = reinterpret_cast<int*>(sm + C::AUX_OFF + C::AUX_FLAG);       // some row's reference grew

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int split = blockIdx.x / a.slices;                        // KV split
    const int r_lo = (blockIdx.x - split * a.slices) * NQ;          // this CTA's query rows [r_lo, r_lo + r_n)
    const int r_n = min(NQ, a.M - r_lo);
    const int k_begin = split * a.keys_per_split;                   // this split's keys
    const int k_end = min(a.n_kv, k_begin + a.keys_per_split);
    const int n_my = k_end > k_begin ? (k_end - k_begin + kKeys - 1) / kKeys : 0;   // tiles (the last may be short)
    const uint64_t limit = a.wait_limit_ns;
    bool failed = false;                 // after a first timeout, later waits give up at once
    auto wait = [&](uint32_t b, uint32_t parity) {
        if (mbar_wait(b, parity, failed ? 0ull : limit)) return true;
        failed = true;
        record_timeout(a.status, 1u);
        return false;
    };
    auto bar = [&](int i) { return smem_addr(&bars[i]); };

    // ---- set-up ------------------------------------------------------------
    if (tid == 0) {
        for (int s = 0; s < C::R; ++s) {
            mbar_init(bar(C::B_FULL + s), 1);
            mbar_init(bar(C::B_EMPTY + s), 1);
        }
        for (int s = 0; s < C::MS; ++s) {
            mbar_init(bar(C::B_MFULL + s), 1);
            mbar_init(bar(C::B_MEMPTY + s), kSmaxWarps);     // one arrival per softmax warp
        }
        mbar_init(bar(C::B_SFULL + 0), 1);
        mbar_init(bar(C::B_SFULL + 1), 1);
        mbar_init(bar(C::B_PFULL + 0), kSmaxThreads);
        mbar_init(bar(C::B_PFULL + 1), kSmaxThreads);
        mbar_init(bar(C::B_ODONE), 1);
        mbar_init(bar(C::B_QFULL), a.rope_in_kernel ? kSmaxThreads : 1);
        mbar_init(bar(C::B_MMADONE), 1);
        mbar_init(bar(C::B_PROBE), 1);
        mbar_init(bar(C::B_QF32), 1);
        mbar_fence_init();
        prefetch_tmap(&mp.k);
        prefetch_tmap(&mp.v);
        if (!a.rope_in_kernel) prefetch_tmap(&mp.q16);
    }
    if (tid < NQ) {
        sM[tid] = -INFINITY;
        sA[tid] = 1.f;
        sL[tid] = 0.f;
    }
    if (tid == 0) sFlag[0] = 0;
    if (warp == kMmaWarp) tmem_alloc(smem_addr(sTmemBase), C::TM_COLS);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tbase = *sTmemBase;
    if (tid == 0) FR_STAMP(0);                   // set-up done
    if (tid == 0) FR_STAMP_SMID();
    // a dependent grid (the merge kernel, or the next call) may be scheduled
    // now; it waits for this grid's completion before reading what this grid
    // writes. Only when this grid is one wave.
    if (a.early_dep) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

    const int n_units = 2 * n_my;                        // K_0, K_1, V_0, K_2, V_1, ..., V_{n-1}
    const int n_pieces = n_units * C::HALVES;

    if (warp == kProdWarp) {
        if (lane == 0) {
            const int mask_rows = min(a.n_tok, kMaskWin);
            const uint32_t mask_tx = 2u * 128u * (uint32_t)mask_rows;
            const int n_masks = a.has_mask ? n_my : 0;
            // piece p: 128-dim half h of unit u, in the order the MMAs consume them
            auto load_piece = [&](int p) {
                const int u = p / C::HALVES, h = p - u * C::HALVES;
                bool is_v;
                int tile;
                if (u == 0) {
                    is_v = false;
                    tile = 0;
                } else if (u == n_units - 1) {
                    is_v = true;
                    tile = n_my - 1;
                } else if (u & 1) {
                    is_v = false;
                    tile = (u + 1) >> 1;
                } else {
                    is_v = true;
                    tile = (u >> 1) - 1;
                }
                const int st = p % C::R;
                const uint32_t dst = smem_addr(sm + C::RING_OFF + st * kStage);
                const CUtensorMap* m = is_v ? &mp.v : &mp.k;
                const int y = k_begin + tile * kKeys;
                mbar_expect_tx(bar(C::B_FULL + st), (uint32_t)kStage);
                tma_load_2d(dst, m, (2 * h) * 64, y, bar(C::B_FULL + st));
                tma_load_2d(dst + kBox, m, (2 * h + 1) * 64, y, bar(C::B_FULL + st));
            };
            auto load_mask = [&](int i) {
                const int st = i % C::MS;
                const uint32_t dst = smem_addr(sm + C::M_OFF + st * C::MASK_BYTES);
                mbar_expect_tx(bar(C::B_MFULL + st), mask_tx);
                tma_load_2d(dst, &mp.mask, k_begin + i * kKeys, 0, bar(C::B_MFULL + st));
                tma_load_2d(dst + C::MASK_BOX, &mp.mask, k_begin + i * kKeys + 64, 0, bar(C::B_MFULL + st));
            };
            // While the grid ahead finishes, the first inputs are prefetched into
            // L2 (a prefetch returns no data, so it may precede the wait below):
            // the Q rows, the first mask tiles and the first K tile (more K/V
            // prefetches from every CTA would queue ahead of the Q rows).
            // this slice's rows of token t: heads [max(0, r_lo - t*n_head), min(n_head, r_lo + r_n - t*n_head))
            const int t_lo = r_lo / a.n_head, t_hi = (r_lo + r_n - 1) / a.n_head;
            auto q_run = [&](int t, int& h_a, int& h_b) {
                h_a = max(0, r_lo - t * a.n_head);
                h_b = min(a.n_head, r_lo + r_n - t * a.n_head);
            };
            if (a.rope_in_kernel)
                for (int t = t_lo; t <= t_hi; ++t) {
                    int h_a, h_b;
                    q_run(t, h_a, h_b);
                    bulk_prefetch_l2(a.q + (int64_t)t * a.q_tok_stride + (int64_t)h_a * HD, (uint32_t)((h_b - h_a) * HD * 4));
                }
            for (int i = 0; i < min(C::MS, n_masks); ++i) {
                tma_prefetch_2d(&mp.mask, k_begin + i * kKeys, 0);
                tma_prefetch_2d(&mp.mask, k_begin + i * kKeys + 64, 0);
            }
            for (int p = 0; p < min(kPrefetchPieces, n_pieces); ++p) {
                const int u = p / C::HALVES, h = p - u * C::HALVES;
                const bool is_v = u == n_units - 1 || (u > 0 && !(u & 1));
                const int tile = u == 0 ? 0 : (u == n_units - 1 ? n_my - 1 : ((u & 1) ? (u + 1) >> 1 : (u >> 1) - 1));
                const CUtensorMap* m = is_v ? &mp.v : &mp.k;
                tma_prefetch_2d(m, (2 * h) * 64, k_begin + tile * kKeys);
                tma_prefetch_2d(m, (2 * h + 1) * 64, k_begin + tile * kKeys);
            }
            // launched as a programmatic dependent: no input is read before the
            // grids ahead of this one on the stream are complete (one of them
            // may have written the KV rows or the Q rows)
            asm volatile("griddepcontrol.wait;" ::: "memory");
            FR_STAMP(4);                         // the grids ahead are complete
            if (a.rope_in_kernel) {
                // this slice's f32 Q rows, one bulk copy per token (a token's
                // heads are contiguous), staged as rows [0, r_n)
                mbar_expect_tx(bar(C::B_QF32), (uint32_t)(r_n * HD * 4));
                for (int t = t_lo; t <= t_hi; ++t) {
                    int h_a, h_b;
                    q_run(t, h_a, h_b);
                    bulk_load(smem_addr(sm + C::P_OFF + (t * a.n_head + h_a - r_lo) * HD * 4),
                              a.q + (int64_t)t * a.q_tok_stride + (int64_t)h_a * HD, (uint32_t)((h_b - h_a) * HD * 4),
                              bar(C::B_QF32));
                }
            } else {
                // rows [r_lo, r_lo + NQ) of the f16 rows: past M the copy reads
                // zeros; rows of the next slice are masked out below
                mbar_expect_tx(bar(C::B_QFULL), (uint32_t)C::Q_BYTES);
                for (int b = 0; b < HD / 64; ++b)
                    tma_load_2d(smem_addr(sm + C::Q_OFF + b * C::Q_BOX), &mp.q16, b * 64, r_lo, bar(C::B_QFULL));
            }
            // the Q rows and the first mask tiles first (ahead of every K/V
            // request in the queues), then the whole ring at once: its first fill
            // overlaps the Q rows' latency and their RoPE
            int np = 0, nm = 0;
            for (; nm < min(C::MS, n_masks); ++nm) load_mask(nm);
            for (; np < min(C::R, n_pieces); ++np) load_piece(np);
            uint64_t t_last = global_ns();
            while (np < n_pieces || nm < n_masks) {
                bool moved = false;
                if (np < n_pieces && mbar_ready(bar(C::B_EMPTY + np % C::R), ((np / C::R) - 1) & 1)) {
                    load_piece(np++);
                    moved = true;
                }
                if (nm < n_masks && mbar_ready(bar(C::B_MEMPTY + nm % C::MS), ((nm / C::MS) - 1) & 1)) {
                    load_mask(nm++);
                    moved = true;
                }
                if (moved) {
                    t_last = global_ns();
                } else {
                    if (global_ns() - t_last > limit) {
                        record_timeout(a.status, 1u);
                        break;
                    }
                    __nanosleep(32);
                }
            }
            // drain: every issued copy has landed before the CTA exits (full
            // time limit even after a failure)
            for (int i = max(0, np - C::R); i < np; ++i)
                if (!mbar_wait(bar(C::B_FULL + i % C::R), (i / C::R) & 1, limit)) record_timeout(a.status, 1u);
            for (int i = max(0, nm - C::MS); i < nm; ++i)
                if (!mbar_wait(bar(C::B_MFULL + i % C::MS), (i / C::MS) & 1, limit)) record_timeout(a.status, 1u);
            if (!mbar_wait(bar(a.rope_in_kernel ? C::B_QF32 : C::B_QFULL), 0, limit)) record_timeout(a.status, 1u);
        }
        if (a.probe_iters && lane == 1) {
            // test hook: a bounded wait on a barrier nothing ever signals
            if (!mbar_wait_polls(bar(C::B_PROBE), 0, a.probe_iters)) record_timeout(a.status, 2u);
        }
    } else if (warp == kMmaWarp) {
        if (lane == 0) {
            if (!mbar_wait(bar(C::B_QFULL), 0, limit)) record_timeout(a.status, 1u);
            FR_STAMP(3);                         // the Q tile is in place
            tc_fence_after();
            constexpr uint32_t idS = idesc_f16_f32(kKeys, NQ, 0, 0);
            constexpr uint32_t idO = idesc_f16_f32(128, C::N2, 1, 1);
            const uint32_t q_base = smem_addr(sm + C::Q_OFF);
            int piece = 0;
            auto issue_s = [&](int i) {
                const uint32_t d = tbase + C::TM_S + (i & 1) * NQ;
                for (int h = 0; h < C::HALVES; ++h) {
                    const int st = piece % C::R;
                    wait(bar(C::B_FULL + st), (piece / C::R) & 1);
                    tc_fence_after();
                    const uint32_t kb = smem_addr(sm + C::RING_OFF + st * kStage);
#pragma unroll
                    for (int kk = 0; kk < 8; ++kk) {            // 16 head dims per MMA
                        const int b = kk >> 2, off = (kk & 3) * 32;
                        mma_ss(d, sdesc_sw128(kb + b * kBox + off, 16, 1024),
                               sdesc_sw128(q_base + (2 * h + b) * C::Q_BOX + off, 16, 1024), idS,
                               (h > 0 || kk > 0) ? 1u : 0u);
                    }
                    mma_commit(bar(C::B_EMPTY + st));
                    ++piece;
                }
                mma_commit(bar(C::B_SFULL + (i & 1)));
                if (i < 12) FR_STAMP(8 + 4 * i + 2);     // S_i issued
            };
            auto issue_pv = [&](int i) {
                wait(bar(C::B_PFULL + (i & 1)), (i >> 1) & 1);
                tc_fence_after();
                const uint32_t pb = smem_addr(sm + C::P_OFF + (i & 1) * C::P_BYTES);
                for (int h = 0; h < C::HALVES; ++h) {
                    const int st = piece % C::R;
                    wait(bar(C::B_FULL + st), (piece / C::R) & 1);
                    tc_fence_after();
                    const uint32_t vb = smem_addr(sm + C::RING_OFF + st * kStage);
                    const uint32_t d = tbase + C::TM_O + h * C::N2;
#pragma unroll
                    for (int ks = 0; ks < 8; ++ks)               // 16 keys per MMA
                        mma_ss(d, sdesc_sw128(vb + ks * 2048, kBox, 1024), sdesc_sw128(pb + ks * 2048, kBox, 1024),
                               idO, (i > 0 || ks > 0) ? 1u : 0u);
                    mma_commit(bar(C::B_EMPTY + st));
                    ++piece;
                }
                mma_commit(bar(C::B_ODONE));
                if (i < 12) FR_STAMP(8 + 4 * i + 3);     // PV_i issued
            };
            // S_{i+1} before PV_i: no cycle, since S_{i+1}'s stages precede V_i's
            // in the ring order. S_i completing also means PV_{i-2} is complete
            // (one issuing thread, in-order completion), which frees the P
            // buffer the softmax of tile i writes.
            if (n_my > 0) issue_s(0);
            for (int i = 0; i < n_my; ++i) {
                if (i + 1 < n_my) issue_s(i + 1);
                issue_pv(i);
            }
            // drain: no MMA may still be running when TMEM is freed
            mma_commit(bar(C::B_MMADONE));
            if (!mbar_wait(bar(C::B_MMADONE), 0, limit)) record_timeout(a.status, 1u);
        }
    } else {
        // ---- softmax: thread = (key k of the tile, row half rh) ----------------
        const int qd = warp & 3, rh = warp >> 2;
        const uint32_t lane_base = (uint32_t)(qd * 32) << 16;
        const int k = qd * 32 + lane;
        const int r0 = rh * RH;                          // this thread's rows [r0, r0 + RH)
        if (a.rope_in_kernel) {
            // the f16 Q tile from the f32 rows, with qkv_post's arithmetic (the
            // same device routines, so the bits equal fr_qkv_post's rows): one
            // cos/sin per (token, pair), shared by the token's heads; rows >= M
            // are zero
            RopeTable& stb = *reinterpret_cast<RopeTable*>(sm + C::AUX_OFF + C::AUX_TB);
            copy_rope_table(stb, tb, tid, kSmaxThreads);
            asm volatile("griddepcontrol.wait;" ::: "memory");     // pos may come from the grid before
            // the positions now, before the K/V stream starts (the RoPE needs them)
            int* sPos = reinterpret_cast<int*>(sm + C::AUX_OFF + C::AUX_POS);
            if (tid < a.n_tok) sPos[tid] = __ldg(a.pos + tid);
            unsigned char* sQ = sm + C::Q_OFF;
            for (int i = tid; i < (NQ - r_n) * (HD / 8); i += kSmaxThreads) {      // zero rows [r_n, NQ)
                const int r = r_n + i / (HD / 8), ch = i % (HD / 8);
                *reinterpret_cast<uint4*>(sQ + (ch >> 3) * C::Q_BOX + r * 128 + ((ch & 7) << 4)) =
                    make_uint4(0u, 0u, 0u, 0u);
            }
            softmax_bar_sync<kSmaxThreads>();
            if (tid == 0) FR_STAMP(5);
            wait(bar(C::B_QF32), 0);
            if (tid == 0) FR_STAMP(6);           // the f32 Q rows have landed
            rope_rows_to_tile<HD>(reinterpret_cast<const float*>(sm + C::P_OFF), sPos, stb, a.n_head, r_lo, r_n, sQ,
                                  C::Q_BOX, tid, kSmaxThreads);
            if (tid == 0) FR_STAMP(7);               // rows roped
            softmax_bar_sync<kSmaxThreads>();                  // every f32 row read: the P buffers are free again
        }
        // P^T columns [2NQ, N2) stay zero (the MMA's N is at least 64)
        if constexpr (2 * NQ < C::N2) {
            for (int i = tid; i < 2 * kKeys * ((C::N2 - 2 * NQ) / 8); i += kSmaxThreads) {
                const int buf = i / (kKeys * ((C::N2 - 2 * NQ) / 8));
                const int rem = i - buf * (kKeys * ((C::N2 - 2 * NQ) / 8));
                const int kr = rem / ((C::N2 - 2 * NQ) / 8), ch = 2 * NQ / 8 + rem % ((C::N2 - 2 * NQ) / 8);
                *reinterpret_cast<uint4*>(sm + C::P_OFF + buf * C::P_BYTES + kr * 128 + ((ch ^ (kr & 7)) << 4)) =
                    make_uint4(0u, 0u, 0u, 0u);
            }
        }
        fence_proxy_async_cta();                 // the Q tile and the zeros are read by the tensor cores
        if (a.rope_in_kernel) mbar_arrive(bar(C::B_QFULL));

        // token of each of this thread's rows, four bytes per word
        uint32_t tokp[(RH + 3) / 4];
#pragma unroll
        for (int w4 = 0; w4 < (RH + 3) / 4; ++w4) {
            uint32_t pk = 0;
#pragma unroll
            for (int u = 0; u < 4; ++u)
                pk |= (uint32_t)min((r_lo + r0 + w4 * 4 + u) / a.n_head, a.n_tok - 1) << (8 * u);
            tokp[w4] = pk;
        }
        const int rb = rs_row<RH>(lane);
        const bool writer = (lane & (32 / RH - 1)) == 0;
        const float kq = a.kq_log2;
        float l_part[RH], mref[RH];
#pragma unroll
        for (int u = 0; u < RH; ++u) {
            l_part[u] = 0.f;
            mref[u] = -INFINITY;
        }
        for (int i = 0; i < n_my; ++i) {
            wait(bar(C::B_SFULL + (i & 1)), (i >> 1) & 1);
            if (tid == 0 && i < 12) FR_STAMP(8 + 4 * i);         // softmax of tile i starts
            tc_fence_after();
            float x[RH];
            tmem_ld_cols<RH>(tbase + lane_base + C::TM_S + (i & 1) * NQ + r0, x);
            tmem_wait_ld();
            const bool key_ok = k_begin + i * kKeys + k < k_end;
            if (a.has_mask) {
                wait(bar(C::B_MFULL + i % C::MS), (i / C::MS) & 1);
                const unsigned char* mk = sm + C::M_OFF + (i % C::MS) * C::MASK_BYTES + (k >> 6) * C::MASK_BOX +
                                          (k & 63) * 2;
#pragma unroll
                for (int u = 0; u < RH; ++u) {
                    const int t = (tokp[u >> 2] >> (8 * (u & 3))) & 0xff;
                    const float mv = __half2float(*reinterpret_cast<const __half*>(mk + t * 128));
                    x[u] = fmaf(mv, kLog2e, x[u] * kq);
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(bar(C::B_MEMPTY + i % C::MS));
            } else {
#pragma unroll
                for (int u = 0; u < RH; ++u) x[u] *= kq;
            }
            bool over = false;
#pragma unroll
            for (int u = 0; u < RH; ++u) {
                if (!key_ok || r0 + u >= r_n) x[u] = -INFINITY;
                over |= x[u] > mref[u] + kTau;           // -inf + tau = -inf: a first finite score counts
            }
            // the row references change only when some score exceeds its row's
            // reference by more than 2^8: then the row maxima of this tile are
            // reduced (warp shuffles, then the four lane quadrants), and every
            // row whose maximum exceeded its reference takes it
            if (softmax_bar_any<kSmaxThreads>(over)) {
                float v[RH];
#pragma unroll
                for (int u = 0; u < RH; ++u) v[u] = x[u];
                ReduceScatter<16, RH, RH, true>::run(v, lane);
                if (writer) sRed[qd * NQ + r0 + rb] = v[0];
                softmax_bar_sync<kSmaxThreads>();
                if (tid < NQ) {
                    const float tm = fmaxf(fmaxf(sRed[tid], sRed[NQ + tid]), fmaxf(sRed[2 * NQ + tid], sRed[3 * NQ + tid]));
                    const float m_old = sM[tid];
                    float m_new = m_old;
                    if (tm > m_old + kTau) m_new = fmaxf(tm, m_old);
                    const bool grow = m_old != -INFINITY && m_new != m_old;
                    sA[tid] = grow ? ex2(m_old - m_new) : 1.f;
                    sM[tid] = m_new;
                    if (grow) sFlag[0] = 1;
                }
                softmax_bar_sync<kSmaxThreads>();
                const bool grew = sFlag[0] != 0;
#pragma unroll
                for (int u = 0; u < RH; ++u) mref[u] = sM[r0 + u];
                if (grew) {
                    // rescale this thread's partial sums, and the O^T columns of
                    // its rows in its TMEM lane (head dim k of each half) once
                    // PV_{i-1} is complete
#pragma unroll
                    for (int u = 0; u < RH; ++u) l_part[u] *= sA[r0 + u];
                    if (i > 0) {
                        wait(bar(C::B_ODONE), (i - 1) & 1);
                        tc_fence_after();
#pragma unroll 1
                        for (int h = 0; h < C::HALVES; ++h)
#pragma unroll 1
                            for (int lo = 0; lo < 2; ++lo)
#pragma unroll 1
                                for (int c8 = 0; c8 < RH; c8 += 8) {
                                    const uint32_t col = tbase + lane_base + C::TM_O + h * C::N2 + lo * NQ + r0 + c8;
                                    float o[8];
                                    tmem_ld_x8(col, reinterpret_cast<uint32_t*>(o));
                                    tmem_wait_ld();
#pragma unroll
                                    for (int u = 0; u < 8; ++u) o[u] *= sA[r0 + c8 + u];
                                    tmem_st_x8(col, reinterpret_cast<const uint32_t*>(o));
                                }
                        tmem_wait_st();
                    }
                }
                softmax_bar_sync<kSmaxThreads>();                      // everyone has read sFlag and sM
                if (tid == 0) sFlag[0] = 0;
            }
            // P = 2^(x - m) as f16 P_hi and P_lo: row k of the MN-major B operand
            // P^T, columns r (P_hi) and NQ + r (P_lo), 16-byte chunks
            unsigned char* prow = sm + C::P_OFF + (i & 1) * C::P_BYTES + k * 128;
#pragma unroll
            for (int c8 = 0; c8 < RH; c8 += 8) {
                uint32_t hw[4], lw[4];
#pragma unroll
                for (int u2 = 0; u2 < 4; ++u2) {
                    const int u = c8 + 2 * u2;
                    const float m0 = mref[u] == -INFINITY ? 0.f : mref[u];
                    const float m1 = mref[u + 1] == -INFINITY ? 0.f : mref[u + 1];
                    const float p0 = ex2(x[u] - m0), p1 = ex2(x[u + 1] - m1);
                    l_part[u] += p0;
                    l_part[u + 1] += p1;
                    hw[u2] = pack_half2(p0, p1);
                    const float2 hf = __half22float2(*reinterpret_cast<const __half2*>(&hw[u2]));
                    lw[u2] = pack_half2(p0 - hf.x, p1 - hf.y);
                }
                const int ch_hi = (r0 + c8) >> 3, ch_lo = (NQ + r0 + c8) >> 3;     // 16-byte chunks of 8 columns
                unsigned char* bh = prow + (ch_hi >> 3) * kBox;
                unsigned char* bl = prow + (ch_lo >> 3) * kBox;
                *reinterpret_cast<uint4*>(bh + (((ch_hi & 7) ^ (k & 7)) << 4)) = make_uint4(hw[0], hw[1], hw[2], hw[3]);
                *reinterpret_cast<uint4*>(bl + (((ch_lo & 7) ^ (k & 7)) << 4)) = make_uint4(lw[0], lw[1], lw[2], lw[3]);
            }
            fence_proxy_async_cta();            // the tile is read by the tensor cores
            tc_fence_before();
            if (tid == 0 && i < 12) FR_STAMP(8 + 4 * i + 1);     // P_i written
            mbar_arrive(bar(C::B_PFULL + (i & 1)));
        }
        // every MMA is complete: the issuer commits this barrier once, after the
        // last PV (waiting on ODONE by parity could pass while PV_{n-2} is still
        // running, the barrier then being two phases behind)
        if (!mbar_wait(bar(C::B_MMADONE), 0, limit)) record_timeout(a.status, 1u);
        if (tid == 0) FR_STAMP(1);               // every MMA complete
        tc_fence_after();
        // row sums: this thread's partials over the warp's keys, then the four
        // lane quadrants, always in the same order
        ReduceScatter<16, RH, RH, false>::run(l_part, lane);
        if (writer) sRed[qd * NQ + r0 + rb] = l_part[0];
        softmax_bar_sync<kSmaxThreads>();
        if (tid < NQ) sL[tid] = (sRed[tid] + sRed[NQ + tid]) + (sRed[2 * NQ + tid] + sRed[3 * NQ + tid]);
        softmax_bar_sync<kSmaxThreads>();
        if (tid == 0) FR_STAMP(57);              // row sums reduced
        // ---- epilogue: O = O_hi + O_lo; this thread's lane is head dim k of
        // each half, its rows [r0, r0 + RH)
        const int rows = r_n;
        const bool single = a.splits == 1;
        constexpr int EC = RH < 16 ? RH : 16;            // columns per TMEM read
#pragma unroll 1
        for (int h = 0; h < C::HALVES; ++h) {
            const int d = h * 128 + k;
#pragma unroll 1
            for (int c0 = 0; c0 < RH; c0 += EC) {
                const uint32_t col0 = tbase + lane_base + C::TM_O + h * C::N2 + r0 + c0;
                float hi[EC], lo[EC];
                if (n_my > 0) {
                    tmem_ld_cols<EC>(col0, hi);
                    tmem_ld_cols<EC>(col0 + NQ, lo);
                    tmem_wait_ld();
                } else {
#pragma unroll
                    for (int u = 0; u < EC; ++u) hi[u] = lo[u] = 0.f;
                }
#pragma unroll
                for (int u = 0; u < EC; ++u) {
                    const int r = r0 + c0 + u;
                    if (r < rows) {
                        const float o = hi[u] + lo[u];
                        if (single) {
                            const float L = sL[r];
                            a.out[(int64_t)(r_lo + r) * HD + d] = L > 0.f ? o / L : 0.f;
                        } else {
                            a.part_o[((int64_t)split * a.rstride + r_lo + r) * HD + d] = o;
                        }
                    }
                }
            }
        }
        if (!single && tid < rows)
            a.part_ml[(int64_t)split * a.rstride + r_lo + tid] =
                n_my > 0 ? make_float2(sM[tid], sL[tid]) : make_float2(-INFINITY, 0.f);
        if (tid == 0) FR_STAMP(58);              // rows stored
    }

    // ---- the split merge, inside the launch ------------------------------------
    // Every CTA is resident (cooperative launch, one CTA per SM), so a bounded
    // grid barrier is safe: once every split's state is stored, CTA b merges
    // the output in units of (row, 32 columns), spread over every softmax warp
    // of the grid (below). A wait that gives up sets the status word and the
    // CTA carries on.
    if (a.splits > 1) {
        __syncthreads();                         // this CTA's state is stored
        if (tid == 0) {
            FR_STAMP(59);
            if (!split_merge::grid_barrier(a.barrier, gridDim.x, limit)) record_timeout(a.status, 4u);
        }
        __syncthreads();
        if (tid == 0) FR_STAMP(56);              // every split's state stored
        if (warp < kSmaxWarps) {
            // a group of G warps per unit, G the largest power of two with one
            // group per unit over the whole grid (at most every softmax warp of
            // a CTA); warp j of a group folds splits j, j + G, ... in chunks
            // with every load of a chunk in flight (online: the running
            // maximum rescales what is folded so far), and the group combines
            // its warps through shared memory, always in the same order
            constexpr int NCH = HD / 32;
            // one chunk covers a warp's share whenever G = every softmax warp
            constexpr int CHUNK = (tc::kMaxMergeSplits + kSmaxWarps - 1) / kSmaxWarps;
            const int units = a.M * NCH;
            const int S = a.splits;                             // states per row
            const int n_cta = gridDim.x;                        // merging CTAs
            const int per = (n_cta * kSmaxWarps) / units;      // warps of the grid per unit
            int G = 1;
            while (G * 2 <= kSmaxWarps && G * 2 <= per) G *= 2;
            const int groups = kSmaxWarps / G;                  // per CTA
            const int gi = warp / G, j = warp - gi * G;
            float* sAcc = reinterpret_cast<float*>(sm + C::RING_OFF);     // [warps][32] (the ring is idle)
            float* sMw = sAcc + kSmaxWarps * 32;                        // [warps]
            float* sLw = sMw + kSmaxWarps;                              // [warps]
            const int rounds = (units + n_cta * groups - 1) / (n_cta * groups); // the same for every warp
            for (int rd = 0; rd < rounds; ++rd) {
                const int u = (rd * n_cta + (int)blockIdx.x) * groups + gi;
                const bool live = u < units;
                const int r = live ? u / NCH : 0, c0 = live ? (u - (u / NCH) * NCH) * 32 : 0;
                float mx = -INFINITY, acc = 0.f, L = 0.f;
                for (int s0 = j; live && s0 < S; s0 += CHUNK * G) {
                    float2 ml[CHUNK];
                    float ov[CHUNK];
#pragma unroll
                    for (int t = 0; t < CHUNK; ++t) {
                        const int s2 = s0 + t * G;
                        if (s2 < S) {
                            const int64_t row = (int64_t)s2 * a.rstride + r;
                            ml[t] = __ldcg(a.part_ml + row);
                            ov[t] = __ldcg(a.part_o + row * HD + c0 + lane);
                        } else {
                            ml[t] = make_float2(-INFINITY, 0.f);
                            ov[t] = 0.f;
                        }
                    }
                    float cm = mx;
#pragma unroll
                    for (int t = 0; t < CHUNK; ++t) cm = fmaxf(cm, ml[t].x);
                    if (cm != -INFINITY) {
                        const float sc = mx == -INFINITY ? 0.f : ex2(mx - cm);
                        acc *= sc;
                        L *= sc;
#pragma unroll
                        for (int t = 0; t < CHUNK; ++t) {
                            const float w = ml[t].x == -INFINITY ? 0.f : ex2(ml[t].x - cm);
                            L = fmaf(w, ml[t].y, L);
                            acc = fmaf(w, ov[t], acc);
                        }
                        mx = cm;
                    }
                }
                if (G == 1) {
                    if (live) a.out[(int64_t)r * HD + c0 + lane] = L > 0.f ? acc / L : 0.f;
                } else {
                    sAcc[warp * 32 + lane] = acc;
                    if (lane == 0) {
                        sMw[warp] = mx;
                        sLw[warp] = L;
                    }
                    softmax_bar_sync<kSmaxThreads>();
                    if (j == 0 && live) {
                        float gm = -INFINITY;
                        for (int w = 0; w < G; ++w) gm = fmaxf(gm, sMw[warp + w]);
                        float sum = 0.f, Lt = 0.f;
                        for (int w = 0; w < G; ++w) {                  // always the same order
                            const float mw = sMw[warp + w];
                            const float sc = mw == -INFINITY ? 0.f : ex2(mw - gm);
                            sum = fmaf(sc, sAcc[(warp + w) * 32 + lane], sum);
                            Lt = fmaf(sc, sLw[warp + w], Lt);
                        }
                        a.out[(int64_t)r * HD + c0 + lane] = Lt > 0.f ? sum / Lt : 0.f;
                    }
                    softmax_bar_sync<kSmaxThreads>();
                }
            }
        }
    }

    // ---- teardown ----------------------------------------------------------------
    tc_fence_before();
    __syncthreads();
    if (tid == 0) FR_STAMP(2);                   // done
    if (a.splits > 1 && tid == 0) split_merge::grid_barrier_depart(a.barrier, gridDim.x);
    if (warp == kMmaWarp) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tbase, C::TM_COLS);
    }
}

// ---- host side ----------------------------------------------------------------

template <int HD, int NQ>
static cudaError_t ensure_attr(int dev) {
    static unsigned long long done = 0ull;
    if (dev < 64 && (__atomic_load_n(&done, __ATOMIC_ACQUIRE) >> dev & 1ull)) return cudaSuccess;
    cudaError_t e = cudaFuncSetAttribute(attn_sw_kernel<HD, NQ>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         Cfg<HD, NQ>::SMEM);
    if (e == cudaSuccess && dev < 64) __atomic_fetch_or(&done, 1ull << dev, __ATOMIC_RELEASE);
    return e;
}

template <int HD, int NQ>
static fr_status launch(const SwLaunch& L, cudaStream_t stream) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return FR_ERR_CUDA;
    if (ensure_attr<HD, NQ>(dev) != cudaSuccess) return FR_ERR_CUDA;
    SwMaps mp;
    memset(&mp, 0, sizeof(mp));
    const SwArgs& a = L.args;
    if (!tc::encode_f16_2d(&mp.k, L.k, HD, a.n_kv, L.k_rs, 64, kKeys, true)) return FR_ERR_CUDA;
    if (!tc::encode_f16_2d(&mp.v, L.v, HD, a.n_kv, L.v_rs, 64, kKeys, true)) return FR_ERR_CUDA;
    if (!a.rope_in_kernel && !tc::encode_f16_2d(&mp.q16, L.q16, HD, a.M, HD, 64, NQ, true)) return FR_ERR_CUDA;
    if (a.has_mask &&
        !tc::encode_f16_2d(&mp.mask, L.mask, a.n_kv, a.n_tok, L.m_rs, 64,
                           (uint32_t)(a.n_tok < kMaskWin ? a.n_tok : kMaskWin), false))
        return FR_ERR_CUDA;
    cudaLaunchConfig_t cfg;
    memset(&cfg, 0, sizeof(cfg));
    cfg.gridDim = dim3(a.splits * a.slices, 1, 1);
    cfg.blockDim = dim3(Cfg<HD, NQ>::THREADS, 1, 1);
    cfg.dynamicSmemBytes = Cfg<HD, NQ>::SMEM;
    cfg.stream = stream;
    // several splits merge behind a grid barrier: every CTA must be resident
    // (cooperative launch; the grid is at most one CTA per SM)
    cudaLaunchAttribute attr[2];
    int na = 0;
    if (a.splits > 1) {
        attr[na].id = cudaLaunchAttributeCooperative;
        attr[na].val.cooperative = 1;
        ++na;
    }
    if (L.pdl) {
        attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[na].val.programmaticStreamSerializationAllowed = 1;
        ++na;
    }
    cfg.attrs = attr;
    cfg.numAttrs = na;
    cudaError_t e = cudaLaunchKernelEx(&cfg, attn_sw_kernel<HD, NQ>, a, mp, L.tb);
    return e == cudaSuccess ? FR_OK : FR_ERR_CUDA;
}

int rows_n(int M) { return M <= 16 ? 16 : (M <= 32 ? 32 : 64); }

fr_status launch_sw(const SwLaunch& L, int hd, int nq, cudaStream_t stream) {
    if (hd == 128) {
        if (nq == 16) return launch<128, 16>(L, stream);
        if (nq == 32) return launch<128, 32>(L, stream);
        return launch<128, 64>(L, stream);
    }
    if (nq == 16) return launch<256, 16>(L, stream);
    if (nq == 32) return launch<256, 32>(L, stream);
    return launch<256, 64>(L, stream);
}

}  // namespace sw
}  // namespace fr
