// fr_attn_sw.cu -- the decode attention for few query rows with the KV tile
// on the MMA's M side: S^T = K Q^T and O^T = V^T P^T on tcgen05.
//
// FlashRT PR #185, commits "FLASH_ATTN_EXT with q_tokens <= 16 over a single
// padded f16 KV head ..." (QK^T with the K operand shared by every GQA head,
// masked fp32-accurate softmax, PV into [hd, n_head, n_tok]) and "The GQA query
// heads share the one KV head, so the per-head batched QK^T and PV GEMMs
// collapse into single GEMMs over all n_head*n_tok query rows". With M =
// n_tok*n_head <= 64 rows, a 128-row query tile (the MMA's M) would be mostly
// padding; here 128 keys are the MMA's M and the query rows its N (16, 32 or
// 64), so the tensor work follows the real rows.
//
// One CTA = one KV split (one CTA per SM), 192 threads:
//   warps 0-3  softmax, one thread per key of the tile (TMEM lane = key of
//              S^T): kq_scale and the mask, row maxima over the 128 keys (warp
//              shuffles, then the four warps through shared memory), lazy
//              rescaling (only when a row maximum grows by more than 2^8),
//              P = 2^(s - m) as two f16 terms P_hi + P_lo written to shared
//              memory as the B operand [P_hi; P_lo] of the PV MMA, and partial
//              row sums per thread. After the loop the same threads own the
//              TMEM lanes of O^T (lane = head dim) for the epilogue, where
//              O = O_hi + O_lo.
//   warp 4     TMA producer: one ring of 32 KiB stages (128 keys x 128 dims of
//              K or of V, two 64-dim boxes) filled in exactly the order the
//              MMAs consume them, and a ring of mask tiles.
//   warp 5     MMA issuer: S^T_j = K_j Q^T (A = K stage, K-major; B = the Q
//              rows), O^T += V_j^T [P_hi; P_lo]^T (A = V stage read MN-major,
//              N = 2 x rows: the P_lo product accumulates in its own columns).
//              S_{j+1} is issued before PV_j, so the softmax of tile j+1
//              overlaps PV_j.
// Each split writes its unnormalised O rows with its row maxima (log2 units)
// and sums to the workspace, and attn_merge_kernel combines them; a single
// split normalises and writes the output rows itself.
// Every mbarrier wait is bounded; a wait that gives up sets the status word,
// and the CTA still drains its copies and MMAs and frees its TMEM.
#include <math.h>
#include <string.h>

#include <cudaTypedefs.h>

#include "fr_attn.h"
#include "fr_common.cuh"
#include "fr_sm100.cuh"

namespace fr {
namespace sw {

using namespace sm100;

constexpr int kKeys = 128;               // keys per KV tile = the MMA's M
constexpr int kSmaxThreads = 128;        // warps 0-3
constexpr int kProdWarp = 4;
constexpr int kMmaWarp = 5;
constexpr int kThreads = 192;
constexpr float kTau = 8.0f;
constexpr float kLog2e = 1.4426950408889634f;
constexpr int kBox = 16384;              // 128 keys x 64 dims f16 (128-byte rows, 128-byte swizzle)
constexpr int kStage = 2 * kBox;         // 128 keys x 128 dims
constexpr int kSmemLimit = 232448;

template <int HD, int NQ>
struct Cfg {
    static_assert(HD == 128 || HD == 256, "head dims");
    static_assert(NQ == 16 || NQ == 32 || NQ == 64, "query rows");
    static constexpr int HALVES = HD / 128;          // K (and V) stages per tile
    static constexpr int Q_BOX = NQ * 128;           // 64 dims of the NQ rows
    static constexpr int Q_BYTES = (HD / 64) * Q_BOX;
    static constexpr int P_ROWS = 2 * NQ;            // [P_hi; P_lo]
    static constexpr int P_BOX = P_ROWS * 128;       // 64 keys of every P row
    static constexpr int P_BYTES = 2 * P_BOX;        // 128 keys
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
    static_assert(Q_BOX % 1024 == 0 || NQ == 16, "Q boxes");
    static_assert(P_BOX % 1024 == 0 && MASK_BOX % 1024 == 0, "1024-B alignment of swizzled tiles");
    // aux: [4][NQ] per-warp partial maxima / sums, [NQ] row max m, [NQ] rescale
    // factors, [NQ] row sums l, two rescale flags
    static constexpr int AUX_RED = 0;
    static constexpr int AUX_M = 4 * NQ * 4;
    static constexpr int AUX_A = AUX_M + NQ * 4;
    static constexpr int AUX_L = AUX_A + NQ * 4;
    static constexpr int AUX_FLAG = AUX_L + NQ * 4;
    static_assert(AUX_FLAG + 16 <= AUX, "aux");
    static constexpr int B_FULL = 0, B_EMPTY = R, B_MFULL = 2 * R, B_MEMPTY = 2 * R + MS,
                         B_SFULL = 2 * (R + MS), B_PFULL = B_SFULL + 2, B_ODONE = B_SFULL + 4,
                         B_QFULL = B_SFULL + 5, B_MMADONE = B_SFULL + 6, B_PROBE = B_SFULL + 7,
                         N_BARS = B_SFULL + 8;
    static constexpr int TMEM_SLOT = 120 * 8;
    static_assert(N_BARS <= 120, "barrier slots");
    // TMEM columns: S^T double buffer (NQ each), then O^T per 128-dim half
    // (2NQ: O_hi^T, O_lo^T)
    static constexpr int TM_S = 0;
    static constexpr int TM_O = 2 * NQ;
    static constexpr int TM_USED = TM_O + HALVES * 2 * NQ;
    static constexpr uint32_t TM_COLS = TM_USED <= 32 ? 32u : TM_USED <= 64 ? 64u : TM_USED <= 128 ? 128u
                                        : TM_USED <= 256 ? 256u : 512u;
};

// Reduce-scatter across the 32 lanes of a warp (maximum or sum) of CH values
// per lane (CH = 16 or 32): at each step the lanes with bit S set keep the
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

// Barrier over the four softmax warps (named barrier 1).
__device__ __forceinline__ void softmax_bar_sync() {
    asm volatile("bar.sync 1, %0;" :: "n"(kSmaxThreads) : "memory");
}

template <int N>
__device__ __forceinline__ void tmem_ld_cols(uint32_t taddr, float* x) {
    if constexpr (N == 16) {
        tmem_ld_x16(taddr, reinterpret_cast<uint32_t*>(x));
    } else {
#pragma unroll
        for (int c = 0; c < N; c += 32) tmem_ld_x32(taddr + c, reinterpret_cast<uint32_t*>(x) + c);
    }
}

template <int HD, int NQ>
__global__ void __launch_bounds__(kThreads, 1)
attn_sw_kernel(const __grid_constant__ SwArgs a, const __grid_constant__ SwMaps mp) {
    using C = Cfg<HD, NQ>;
    constexpr int CH = NQ < 32 ? NQ : 32;                // rows per reduction chunk
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    unsigned char* sm = reinterpret_cast<unsigned char*>(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    uint64_t* bars = reinterpret_cast<uint64_t*>(sm + C::BAR_OFF);
    uint32_t* sTmemBase = reinterpret_cast<uint32_t*>(sm + C::BAR_OFF + C::TMEM_SLOT);
    float* sRed = reinterpret_cast<float*>(sm + C::AUX_OFF + C::AUX_RED);     // [4][NQ]
    float* sM = reinterpret_cast<float*>(sm + C::AUX_OFF + C::AUX_M);         // [NQ] row max (log2 units)
    float* sA = reinterpret_cast<float*>(sm + C::AUX_OFF + C::AUX_A);         // [NQ] rescale factors
    float* sL = reinterpret_cast<float*>(sm + C::AUX_OFF + C::AUX_L);         // [NQ] row sums
    int* sFlag = reinterpret_cast<int*>(sm + C::AUX_OFF + C::AUX_FLAG);       // [2] some row rescaled

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int split = blockIdx.x;
    const int t0 = split * a.tiles_per_split;
    const int n_my = max(0, min(a.n_tiles, t0 + a.tiles_per_split) - t0);
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
            mbar_init(bar(C::B_MEMPTY + s), 4);              // one arrival per softmax warp
        }
        mbar_init(bar(C::B_SFULL + 0), 1);
        mbar_init(bar(C::B_SFULL + 1), 1);
        mbar_init(bar(C::B_PFULL + 0), kSmaxThreads);
        mbar_init(bar(C::B_PFULL + 1), kSmaxThreads);
        mbar_init(bar(C::B_ODONE), 1);
        mbar_init(bar(C::B_QFULL), 1);
        mbar_init(bar(C::B_MMADONE), 1);
        mbar_init(bar(C::B_PROBE), 1);
        mbar_fence_init();
        prefetch_tmap(&mp.k);
        prefetch_tmap(&mp.v);
        prefetch_tmap(&mp.q16);
    }
    if (tid < NQ) {
        sM[tid] = -INFINITY;
        sA[tid] = 1.f;
        sL[tid] = 0.f;
    }
    if (tid < 2) sFlag[tid] = 0;
    if (warp == kMmaWarp) tmem_alloc(smem_addr(sTmemBase), C::TM_COLS);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tbase = *sTmemBase;
    // a dependent grid (the merge kernel, or the next call's qkv_post) may be
    // scheduled now; it waits for this grid's completion before reading what
    // this grid writes. Only when this grid is one wave.
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
                const int y = (t0 + tile) * kKeys;
                mbar_expect_tx(bar(C::B_FULL + st), (uint32_t)kStage);
                tma_load_2d(dst, m, (2 * h) * 64, y, bar(C::B_FULL + st));
                tma_load_2d(dst + kBox, m, (2 * h + 1) * 64, y, bar(C::B_FULL + st));
            };
            auto load_mask = [&](int i) {
                const int st = i % C::MS;
                const uint32_t dst = smem_addr(sm + C::M_OFF + st * C::MASK_BYTES);
                mbar_expect_tx(bar(C::B_MFULL + st), mask_tx);
                tma_load_2d(dst, &mp.mask, (t0 + i) * kKeys, 0, bar(C::B_MFULL + st));
                tma_load_2d(dst + C::MASK_BOX, &mp.mask, (t0 + i) * kKeys + 64, 0, bar(C::B_MFULL + st));
            };
            // K/V and mask tiles need no Q: the first ones go out before the wait
            // for the grid that writes the Q rows
            int np = 0, nm = 0;
            for (; np < min(C::R, n_pieces); ++np) load_piece(np);
            for (; nm < min(C::MS, n_masks); ++nm) load_mask(nm);
            asm volatile("griddepcontrol.wait;" ::: "memory");
            mbar_expect_tx(bar(C::B_QFULL), (uint32_t)C::Q_BYTES);
            for (int b = 0; b < HD / 64; ++b)
                tma_load_2d(smem_addr(sm + C::Q_OFF + b * C::Q_BOX), &mp.q16, b * 64, 0, bar(C::B_QFULL));
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
            if (!mbar_wait(bar(C::B_QFULL), 0, limit)) record_timeout(a.status, 1u);
        }
        if (a.probe_iters && lane == 1) {
            // test hook: a bounded wait on a barrier nothing ever signals
            if (!mbar_wait_polls(bar(C::B_PROBE), 0, a.probe_iters)) record_timeout(a.status, 2u);
        }
    } else if (warp == kMmaWarp) {
        if (lane == 0) {
            if (!mbar_wait(bar(C::B_QFULL), 0, limit)) record_timeout(a.status, 1u);
            tc_fence_after();
            constexpr uint32_t idS = idesc_f16_f32(kKeys, NQ, 0, 0);
            constexpr uint32_t idO = idesc_f16_f32(128, 2 * NQ, 1, 0);
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
                    const uint32_t d = tbase + C::TM_O + h * 2 * NQ;
#pragma unroll
                    for (int ks = 0; ks < 8; ++ks)               // 16 keys per MMA
                        mma_ss(d, sdesc_sw128(vb + ks * 2048, kBox, 1024),
                               sdesc_sw128(pb + (ks >> 2) * C::P_BOX + (ks & 3) * 32, 16, 1024), idO,
                               (i > 0 || ks > 0) ? 1u : 0u);
                    mma_commit(bar(C::B_EMPTY + st));
                    ++piece;
                }
                mma_commit(bar(C::B_ODONE));
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
        // ---- softmax: thread = key k of the tile (S^T lane) ------------------
        const uint32_t lane_base = (uint32_t)(warp * 32) << 16;
        const int k = warp * 32 + lane;
        // token of each query row, four bytes per word
        uint32_t tokp[NQ / 4];
#pragma unroll
        for (int w4 = 0; w4 < NQ / 4; ++w4) {
            uint32_t pk = 0;
#pragma unroll
            for (int u = 0; u < 4; ++u) pk |= (uint32_t)min((w4 * 4 + u) / a.n_head, a.n_tok - 1) << (8 * u);
            tokp[w4] = pk;
        }
        const int rb = rs_row<CH>(lane);
        const bool writer = (lane & (32 / CH - 1)) == 0;
        const float kq = a.kq_log2;
        float l_part[NQ];
#pragma unroll
        for (int r = 0; r < NQ; ++r) l_part[r] = 0.f;
        for (int i = 0; i < n_my; ++i) {
            wait(bar(C::B_SFULL + (i & 1)), (i >> 1) & 1);
            tc_fence_after();
            float x[NQ];
            tmem_ld_cols<NQ>(tbase + lane_base + C::TM_S + (i & 1) * NQ, x);
            tmem_wait_ld();
            const bool key_ok = (t0 + i) * kKeys + k < a.n_kv;
            if (a.has_mask) {
                wait(bar(C::B_MFULL + i % C::MS), (i / C::MS) & 1);
                const unsigned char* mk = sm + C::M_OFF + (i % C::MS) * C::MASK_BYTES + (k >> 6) * C::MASK_BOX +
                                          (k & 63) * 2;
#pragma unroll
                for (int r = 0; r < NQ; ++r) {
                    const int t = (tokp[r >> 2] >> (8 * (r & 3))) & 0xff;
                    const float mv = __half2float(*reinterpret_cast<const __half*>(mk + t * 128));
                    x[r] = fmaf(mv, kLog2e, x[r] * kq);
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(bar(C::B_MEMPTY + i % C::MS));
            } else {
#pragma unroll
                for (int r = 0; r < NQ; ++r) x[r] *= kq;
            }
#pragma unroll
            for (int r = 0; r < NQ; ++r)
                if (!key_ok || r >= a.M) x[r] = -INFINITY;
            // row maxima of this tile: the warp's 32 keys, then the four warps
#pragma unroll
            for (int c0 = 0; c0 < NQ; c0 += CH) {
                float v[CH];
#pragma unroll
                for (int u = 0; u < CH; ++u) v[u] = x[c0 + u];
                ReduceScatter<16, CH, CH, true>::run(v, lane);
                if (writer) sRed[warp * NQ + c0 + rb] = v[0];
            }
            softmax_bar_sync();
            if (tid < NQ) {
                const float tm = fmaxf(fmaxf(sRed[tid], sRed[NQ + tid]), fmaxf(sRed[2 * NQ + tid], sRed[3 * NQ + tid]));
                const float m_old = sM[tid];
                float m_new = m_old;
                if (tm > m_old + kTau || (m_old == -INFINITY && tm > -INFINITY)) m_new = fmaxf(tm, m_old);
                const bool grow = m_old != -INFINITY && m_new != m_old;
                sA[tid] = grow ? ex2(m_old - m_new) : 1.f;
                sM[tid] = m_new;
                if (grow) sFlag[i & 1] = 1;
            }
            if (tid == 0) sFlag[(i + 1) & 1] = 0;        // read next in tile i + 1
            softmax_bar_sync();
            if (sFlag[i & 1]) {
                // some row's reference grew: rescale this thread's partial sums,
                // and the O^T columns of its TMEM lane (head dim k of each half)
                // once PV_{i-1} is complete
#pragma unroll
                for (int r = 0; r < NQ; r += 4) {
                    const float4 al = *reinterpret_cast<const float4*>(sA + r);
                    l_part[r] *= al.x;
                    l_part[r + 1] *= al.y;
                    l_part[r + 2] *= al.z;
                    l_part[r + 3] *= al.w;
                }
                if (i > 0) {
                    wait(bar(C::B_ODONE), (i - 1) & 1);
                    tc_fence_after();
#pragma unroll 1
                    for (int c = 0; c < C::HALVES * 2 * NQ; c += 32) {
                        uint32_t o[32];
                        tmem_ld_x32(tbase + lane_base + C::TM_O + c, o);
                        tmem_wait_ld();
#pragma unroll
                        for (int u = 0; u < 32; ++u)
                            o[u] = __float_as_uint(__uint_as_float(o[u]) * sA[(c + u) % NQ]);
                        tmem_st_x32(tbase + lane_base + C::TM_O + c, o);
                    }
                    tmem_wait_st();
                }
            }
            // P = 2^(x - m) as f16 P_hi and P_lo, key k of rows r and NQ + r of
            // the K-major (128-byte swizzled) B operand of tile i
            unsigned char* pbuf = sm + C::P_OFF + (i & 1) * C::P_BYTES + (k >> 6) * C::P_BOX;
            const int kc = (k & 63) >> 3, kb2 = (k & 7) * 2;
#pragma unroll
            for (int r = 0; r < NQ; r += 4) {
                const float4 m4 = *reinterpret_cast<const float4*>(sM + r);
                const float mm[4] = {m4.x, m4.y, m4.z, m4.w};
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    const int rr = r + u, rl = NQ + r + u;
                    const float msub = mm[u] == -INFINITY ? 0.f : mm[u];
                    const float p = ex2(x[rr] - msub);
                    l_part[rr] += p;
                    const __half hi = __float2half_rn(p);
                    const __half lo = __float2half_rn(p - __half2float(hi));
                    *reinterpret_cast<__half*>(pbuf + rr * 128 + ((kc ^ (rr & 7)) << 4) + kb2) = hi;
                    *reinterpret_cast<__half*>(pbuf + rl * 128 + ((kc ^ (rl & 7)) << 4) + kb2) = lo;
                }
            }
            fence_proxy_async_cta();            // the tile is read by the tensor cores
            tc_fence_before();
            mbar_arrive(bar(C::B_PFULL + (i & 1)));
        }
        // every MMA is complete: the issuer commits this barrier once, after the
        // last PV (waiting on ODONE by parity could pass while PV_{n-2} is still
        // running, the barrier then being two phases behind)
        if (!mbar_wait(bar(C::B_MMADONE), 0, limit)) record_timeout(a.status, 1u);
        tc_fence_after();
        // row sums: this thread's partials over the warp's keys, then the four
        // warps, always in the same order
#pragma unroll
        for (int c0 = 0; c0 < NQ; c0 += CH) {
            float v[CH];
#pragma unroll
            for (int u = 0; u < CH; ++u) v[u] = l_part[c0 + u];
            ReduceScatter<16, CH, CH, false>::run(v, lane);
            if (writer) sRed[warp * NQ + c0 + rb] = v[0];
        }
        softmax_bar_sync();
        if (tid < NQ) sL[tid] = (sRed[tid] + sRed[NQ + tid]) + (sRed[2 * NQ + tid] + sRed[3 * NQ + tid]);
        softmax_bar_sync();
        // ---- epilogue: O = O_hi + O_lo; this thread's lane is head dim k of each half
        const int rows = a.M;
        const bool single = a.splits == 1;
#pragma unroll 1
        for (int h = 0; h < C::HALVES; ++h) {
            const int d = h * 128 + k;
            const uint32_t col0 = tbase + lane_base + C::TM_O + h * 2 * NQ;
#pragma unroll 1
            for (int c0 = 0; c0 < NQ; c0 += CH) {
                float hi[CH], lo[CH];
                if (n_my > 0) {
                    if constexpr (NQ == 16) {
                        uint32_t o[32];
                        tmem_ld_x32(col0, o);
                        tmem_wait_ld();
#pragma unroll
                        for (int u = 0; u < 16; ++u) {
                            hi[u] = __uint_as_float(o[u]);
                            lo[u] = __uint_as_float(o[16 + u]);
                        }
                    } else {
                        tmem_ld_x32(col0 + c0, reinterpret_cast<uint32_t*>(hi));
                        tmem_ld_x32(col0 + NQ + c0, reinterpret_cast<uint32_t*>(lo));
                        tmem_wait_ld();
                    }
                } else {
#pragma unroll
                    for (int u = 0; u < CH; ++u) hi[u] = lo[u] = 0.f;
                }
#pragma unroll
                for (int u = 0; u < CH; ++u) {
                    const int r = c0 + u;
                    if (r < rows) {
                        const float o = hi[u] + lo[u];
                        if (single) {
                            const float L = sL[r];
                            a.out[(int64_t)r * HD + d] = L > 0.f ? o / L : 0.f;
                        } else {
                            a.part_o[((int64_t)split * a.rstride + r) * HD + d] = o;
                        }
                    }
                }
            }
        }
        if (!single && tid < rows)
            a.part_ml[(int64_t)split * a.rstride + tid] =
                n_my > 0 ? make_float2(sM[tid], sL[tid]) : make_float2(-INFINITY, 0.f);
    }

    // ---- teardown ----------------------------------------------------------------
    tc_fence_before();
    __syncthreads();
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
    if (!tc::encode_f16_2d(&mp.q16, L.q16, HD, a.M, HD, 64, NQ, true)) return FR_ERR_CUDA;
    if (a.has_mask &&
        !tc::encode_f16_2d(&mp.mask, L.mask, a.n_kv, a.n_tok, L.m_rs, 64,
                           (uint32_t)(a.n_tok < kMaskWin ? a.n_tok : kMaskWin), false))
        return FR_ERR_CUDA;
    cudaLaunchConfig_t cfg;
    memset(&cfg, 0, sizeof(cfg));
    cfg.gridDim = dim3(a.splits, 1, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = Cfg<HD, NQ>::SMEM;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = L.pdl ? 1 : 0;
    cudaError_t e = cudaLaunchKernelEx(&cfg, attn_sw_kernel<HD, NQ>, a, mp);
    return e == cudaSuccess ? FR_OK : FR_ERR_CUDA;
}

int rows_n(int M) { return M <= 16 ? 16 : (M <= 32 ? 32 : 64); }

fr_status launch_sw(const SwLaunch& L, int hd, cudaStream_t stream) {
    const int nq = rows_n(L.args.M);
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
