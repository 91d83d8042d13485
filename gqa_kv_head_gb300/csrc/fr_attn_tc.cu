// fr_attn_tc.cu -- the tensor-core (tcgen05 / TMEM / TMA) decode attention:
// collapsed GQA QK^T over 128 t-major query rows per CTA, masked fp32
// softmax, PV, split over n_kv with the split combine fused into the launch.
//
// FlashRT PR #185, commits "FLASH_ATTN_EXT with q_tokens <= 16 over a single
// padded f16 KV head ..." (QK^T with the K operand shared by every GQA head,
// masked fp32-accurate softmax, PV into [hd, n_head, n_tok]) and "The GQA query
// heads share the one KV head, so the per-head batched QK^T and PV GEMMs
// collapse into single GEMMs over all n_head*n_tok query rows".
//
// One CTA = 128 query rows (the MMA M; rows >= M are zero) x one KV split.
// Warp roles (320 threads):
//   warps 0-7  softmax: TMEM lane i = query row i is shared by warps i/32 and
//              i/32 + 4, each taking half of the S tile's columns; the halves
//              exchange their maxima per tile. Applies kq_scale and the mask,
//              keeps the running max m and sum l (lazy rescale of O only when
//              the max grows by > 2^8), and writes P back into TMEM as two f16
//              terms, P = P_hi + P_lo (P_lo = f16(p - P_hi)), so the weights
//              keep ~22 bits and the softmax stays fp32-accurate even where |V|
//              is large.
//   warp 8     TMA producer: one thread fills separate rings of K, V and
//              mask tiles, refilling whichever slot frees first (a K slot is
//              free again once S_j is computed, so K runs ahead of V); it
//              also loads the Q tile, after the first K tile and before the
//              rest of the first ring fill.
//   warp 9     MMA issuer: S_j = Q K_j^T (SS form, S double-buffered in TMEM),
//              O += P_hi,j V_j + P_lo,j V_j (A operand from TMEM, V read
//              MN-major), commits.
// Splits of one row tile form thread-block clusters of C CTAs (cluster dim y):
//   prologue   each CTA loads the whole 128-row f16 Q tile by TMA on its own
//              (the rows sit in L2). In the fused call they come from the
//              qkv_post kernel launched just before (programmatic dependent
//              launch: this kernel's set-up and first K/V loads overlap it).
//   epilogue   each CTA stores its (m, l, O) rows straight from TMEM into the
//              shared memory of the CTA that owns them (rank c owns rows
//              [c*128/C, (c+1)*128/C)); owners merge the C states locally, in
//              rank order. With several clusters per row
//              tile the merged slices go to the workspace and the last CTA to
//              arrive for each (row tile, rank) slice merges them (atomic ticket,
//              reset afterwards). No CTA ever waits for another cluster.
// Merge-kernel mode, for plans with many splits: no clusters, up to one split
// per SM; each CTA writes its unnormalised (m, l, O) rows to the workspace and
// attn_merge_kernel, chained by programmatic dependent launch, combines them
// with the whole GPU instead of one CTA per slice.
// Every mbarrier wait is bounded; a wait that gives up sets the workspace's
// status word and the CTA still runs through every cluster barrier, drains
// its copies and frees its TMEM.
#include <math.h>
#include <string.h>

#include <cudaTypedefs.h>

#include "fr_attn.h"
#include "fr_common.cuh"
#include "fr_sm100.cuh"
#include "fr_trace.cuh"

namespace fr {
namespace tc {

using namespace sm100;

constexpr int kRows = 128;
constexpr int kSmaxWarps = 8;                // two warps per TMEM lane quadrant
constexpr int kSmaxThreads = kSmaxWarps * 32;
constexpr int kProdWarp = 8;
constexpr int kMmaWarp = 9;
constexpr int kThreads = (kSmaxWarps + 2) * 32;
constexpr float kTau = 8.0f;
constexpr float kLog2e = 1.4426950408889634f;
constexpr uint32_t kTmemCols = 512;
constexpr int kOutBoxRows = 32;              // rows per TMA store box of the split states
static_assert(kOutBoxRows == 32, "one box block = the 32 rows of one softmax warp");

// Keys per KV tile: 64, or 128 at hd 128 for long KV ranges (half the S MMA
// instructions per key: the N = 64 QK^T MMAs run at ~40 % of the tensor
// peak). At hd 256 a 128-key K tile does not fit next to Q and a two-deep ring.
template <int HD, int BN_>
struct Cfg {
    static constexpr int BN = BN_;
    static_assert(BN == 64 || (BN == 128 && HD == 128), "tile shapes");
    // At BN = 128 the f16 P_hi / P_lo words go over the S columns the softmax
    // thread has just read (TMEM: O, then two S buffers); else P has its own
    // columns.
    static constexpr bool PALIAS = BN == 128;
    // Separate rings for K, V and mask tiles: a K slot frees when S_j is
    // computed, a V slot when PV_j is, a mask slot when the softmax has read
    // it, so K tiles run ahead of the V tiles they travel with.
    static constexpr int KS = HD == 64 ? 8 : (HD == 128 && BN == 64 ? 3 : 2);   // K slots
    static constexpr int VS = KS;                                     // V slots
    static constexpr int MS = 4;                                      // mask slots
    static constexpr int NB = HD / 64;                     // 128-byte column boxes per row
    static constexpr int Q_BYTES = kRows * HD * 2;
    static constexpr int Q_BOX = kRows * 128;              // one 64-column box of Q
    static constexpr int KV_BOX = BN * 128;                // one 64-column box of a K or V tile
    static constexpr int K_BYTES = BN * HD * 2;
    static constexpr int MASK_BOX = 2048;                  // <= 16 rows x 128 B, 1024-aligned slots
    static constexpr int MASK_BYTES = (BN / 64) * MASK_BOX;
    static constexpr int K_OFF = 0, V_OFF = KS * K_BYTES, M_OFF = V_OFF + VS * K_BYTES;   // in the stage area
    static constexpr int STAGE_AREA = M_OFF + MS * MASK_BYTES;
    static constexpr int BODY = Q_BYTES + STAGE_AREA;
    static constexpr int DATA = BODY;
    static constexpr int AUX = 20480;                      // cos/sin table; then exchange + merge weights
    static constexpr int AUX_MAXX = 0;                     // [2][2][128] f32 half-row maxima
    static constexpr int AUX_LX = 2048;                    // [2][128] f32 half-row sums
    static constexpr int AUX_ML = 3072;                    // [C][R] (m, l) pushed by the cluster's CTAs
    static constexpr int AUX_W = 4096;                     // merge weights (<= 16 KiB)
    // After the KV loop, each CTA stores its O rows straight into the shared
    // memory of the CTA that owns them: [C][R][RS] fp32 at RECV_OFF (past the
    // Q tile). Each softmax warp transposes its rows through a 32 x 36 fp32
    // buffer at TB_OFF so that its DSMEM stores write whole 128-byte segments.
    static constexpr int RS = HD + 4;
    static constexpr int RECV_OFF = Q_BYTES;
    static constexpr int RECV_BYTES = kRows * RS * 4;
    static constexpr int TB_BYTES = 8 * 32 * 36 * 4;
    static constexpr int TB_OFF = HD == 256 ? 0 : RECV_OFF + RECV_BYTES;
    // merge-kernel mode: O rows leave as HD/32 TMA boxes of [128][32] fp32 in the stage area
    static constexpr int OBOX = kRows * 128;
    static_assert((HD / 32) * OBOX <= STAGE_AREA, "O boxes inside the stage area");
    static constexpr int BAR_OFF = DATA + AUX;
    // mbarrier slots (8 bytes each), laid out from the ring depths
    static constexpr int B_KFULL = 0, B_KEMPTY = KS, B_VFULL = 2 * KS, B_VEMPTY = 2 * KS + VS,
                         B_MFULL = 2 * (KS + VS), B_MEMPTY = 2 * (KS + VS) + MS, B_SFULL = 2 * (KS + VS + MS),
                         B_PFULL = B_SFULL + 2, B_ODONE = B_SFULL + 4, B_QFULL = B_SFULL + 5,
                         B_PROBE = B_SFULL + 6, B_MMADONE = B_SFULL + 7, N_BARS = B_SFULL + 8;
    static constexpr int TMEM_SLOT = 120 * 8;              // TMEM base word after 120 barrier slots
    static_assert(N_BARS <= 120, "barrier slots");
    static_assert(RECV_OFF + RECV_BYTES <= BODY, "receive area inside the data region");
    static_assert(HD == 256 ? TB_BYTES <= Q_BYTES : TB_OFF + TB_BYTES <= BODY, "transposition buffer");
    static constexpr int SMEM = BAR_OFF + 1024 + 1024;     // barriers + TMEM word, + alignment slack
    // TMEM columns
    static constexpr int TM_O = 0;
    static constexpr int TM_S = HD;
    static constexpr int TM_P = HD + 2 * BN;               // P_hi, 2 x BN/2 columns (not PALIAS)
    static constexpr int TM_PL = TM_P + BN;                // P_lo, 2 x BN/2 columns (not PALIAS)
    static_assert((PALIAS ? TM_S + 2 * BN : TM_PL + BN) <= (int)kTmemCols, "TMEM budget");
    // TMEM column of softmax half h's f16 P_hi (lo = 0) or P_lo (lo = 1) words
    // for S buffer b: BN/4 columns (two keys per 32-bit column)
    __host__ __device__ static constexpr int p_col(int b, int h, int lo) {
        return PALIAS ? TM_S + b * BN + h * (BN / 2) + lo * (BN / 4)
                      : (lo ? TM_PL : TM_P) + b * (BN / 2) + h * (BN / 4);
    }
    static_assert(K_BYTES % 1024 == 0 && MASK_BYTES % 1024 == 0 && Q_BYTES % 1024 == 0,
                  "1024-B alignment of swizzled tiles");
    static_assert(SMEM <= 232448, "shared memory budget");
};

struct Maps {
    CUtensorMap k, v, mask, q16;
    CUtensorMap po;           // merge-kernel mode: split O rows [row_tiles * splits * 128][HD] fp32
};

__device__ __forceinline__ void record_timeout(unsigned* status, unsigned bit) {
    atomicOr(status, bit);
}

// Barrier over the two softmax warps that share TMEM lane quadrant q (named
// barriers 1..4, 64 threads each).
__device__ __forceinline__ void quad_bar_sync(int q) {
    asm volatile("bar.sync %0, 64;" :: "r"(q + 1) : "memory");
}
// Barrier over all softmax warps (named barrier 5).
__device__ __forceinline__ void softmax_bar_sync() {
    asm volatile("bar.sync 5, %0;" :: "n"(kSmaxThreads) : "memory");
}

template <int HD, int BN_>
__global__ void __launch_bounds__(kThreads, 1)
attn_tc_kernel(const __grid_constant__ TcArgs a, const __grid_constant__ Maps mp) {
    using C = Cfg<HD, BN_>;
    constexpr int BN = C::BN;
    constexpr int HB = BN / 2;                           // S columns per softmax half
    constexpr int OH = HD / 2;                           // O columns per softmax half
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    unsigned char* sm = reinterpret_cast<unsigned char*>(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    unsigned char* sQ = sm;
    unsigned char* sStage = sm + C::Q_BYTES;
    float* sRecvO = reinterpret_cast<float*>(sm + C::RECV_OFF);                     // after the KV loop
    float* sTB = reinterpret_cast<float*>(sm + C::TB_OFF);                          // [8 warps][32][36]
    unsigned char* aux = sm + C::DATA;
    float* sMaxX = reinterpret_cast<float*>(aux + C::AUX_MAXX);       // loop: [2][2][128] half-row maxima
    float* sLX = reinterpret_cast<float*>(aux + C::AUX_LX);           // [2][128] half-row sums
    float2* sML = reinterpret_cast<float2*>(aux + C::AUX_ML);         // [C][R] (m, l) from the cluster
    float* sW = reinterpret_cast<float*>(aux + C::AUX_W);             // merge weights
    uint64_t* bars = reinterpret_cast<uint64_t*>(sm + C::BAR_OFF);
    uint32_t* sTmemBase = reinterpret_cast<uint32_t*>(sm + C::BAR_OFF + C::TMEM_SLOT);
    __shared__ int s_last;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const uint32_t rank = cluster_rank();
    const int CS = a.C;                                  // cluster size
    const int R = kRows / CS;                            // rows owned per rank
    const int rt = blockIdx.x;                           // row tile
    const int split = blockIdx.y;
    const int cl = split / CS;                           // cluster index within the row tile
    const int row0 = rt * kRows;
    const int rows_real = min(kRows, a.M - row0);
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
    auto sK = [&](int s) { return sStage + C::K_OFF + s * C::K_BYTES; };
    auto sV = [&](int s) { return sStage + C::V_OFF + s * C::K_BYTES; };
    auto sMask = [&](int s) { return sStage + C::M_OFF + s * C::MASK_BYTES; };

    // ---- set-up ------------------------------------------------------------
    if (tid == 0) {
        for (int s = 0; s < C::KS; ++s) {
            mbar_init(bar(C::B_KFULL + s), 1);
            mbar_init(bar(C::B_KEMPTY + s), 1);
        }
        for (int s = 0; s < C::VS; ++s) {
            mbar_init(bar(C::B_VFULL + s), 1);
            mbar_init(bar(C::B_VEMPTY + s), 1);
        }
        for (int s = 0; s < C::MS; ++s) {
            mbar_init(bar(C::B_MFULL + s), 1);
            mbar_init(bar(C::B_MEMPTY + s), kSmaxWarps);      // one arrival per softmax warp
        }
        mbar_init(bar(C::B_SFULL + 0), 1);
        mbar_init(bar(C::B_SFULL + 1), 1);
        mbar_init(bar(C::B_PFULL + 0), kSmaxThreads);
        mbar_init(bar(C::B_PFULL + 1), kSmaxThreads);
        mbar_init(bar(C::B_ODONE), 1);
        mbar_init(bar(C::B_QFULL), 1);
        mbar_init(bar(C::B_PROBE), 1);
        mbar_init(bar(C::B_MMADONE), 1);
        mbar_fence_init();
        // the whole Q tile arrives by TMA (each CTA loads it on its own)
        mbar_expect_tx(bar(C::B_QFULL), (uint32_t)C::Q_BYTES);
        prefetch_tmap(&mp.k);
        prefetch_tmap(&mp.v);
    }
    if (warp == kMmaWarp) tmem_alloc(smem_addr(sTmemBase), kTmemCols);
    tc_fence_before();
    if (CS > 1) cluster_sync();         // #1: barriers of every CTA initialised and armed
    else __syncthreads();               //     (one-CTA cluster: a CTA barrier is enough)
    tc_fence_after();
    const uint32_t tbase = *sTmemBase;
    if (tid == 0) {
        FR_STAMP(0);                             // set-up done
        FR_STAMP_SMID();
    }
    // a dependent grid (the merge kernel, or the next call's qkv_post) may be
    // scheduled now; it waits for this grid's completion before reading what it
    // writes. Only when this grid is one wave: otherwise waiting dependent CTAs
    // could hold SMs that later CTAs of this grid need.
    if (a.early_dep) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

    // mask rows: all tokens when n_tok <= kMaskWin, else the kMaskWin tokens
    // from this row tile's first one (they hold every token of the tile)
    const int mask_rows = min(a.n_tok, kMaskWin);
    const int mask_t0 = a.n_tok <= kMaskWin ? 0 : row0 / a.n_head;
    const uint32_t mask_tx = a.has_mask ? (uint32_t)(BN / 64) * 128u * (uint32_t)mask_rows : 0u;
    auto load_k = [&](int i) {
        const int st = i % C::KS;
        mbar_expect_tx(bar(C::B_KFULL + st), (uint32_t)C::K_BYTES);
#pragma unroll
        for (int b = 0; b < C::NB; ++b)
            tma_load_2d(smem_addr(sK(st) + b * C::KV_BOX), &mp.k, b * 64, (t0 + i) * BN, bar(C::B_KFULL + st));
    };
    auto load_v = [&](int i) {
        const int st = i % C::VS;
        mbar_expect_tx(bar(C::B_VFULL + st), (uint32_t)C::K_BYTES);
#pragma unroll
        for (int b = 0; b < C::NB; ++b)
            tma_load_2d(smem_addr(sV(st) + b * C::KV_BOX), &mp.v, b * 64, (t0 + i) * BN, bar(C::B_VFULL + st));
    };
    auto load_m = [&](int i) {
        const int st = i % C::MS;
        mbar_expect_tx(bar(C::B_MFULL + st), mask_tx);
#pragma unroll
        for (int mb = 0; mb < BN / 64; ++mb)
            tma_load_2d(smem_addr(sMask(st) + mb * C::MASK_BOX), &mp.mask, (t0 + i) * BN + mb * 64, mask_t0,
                        bar(C::B_MFULL + st));
    };
    // ---- prologue: one producer thread requests the first K tile (and its
    // mask tile), then the 128 Q rows as f16 (SW128 K-major, every CTA of a
    // cluster loads the whole tile itself: the rows are in L2, qkv_post has
    // just written them), then the rest of the slots every ring starts with.
    // When the rows come from the qkv_post grid launched just before this one
    // (programmatic dependent launch), the wait for that grid sits between
    // the first K tile and the Q rows: the K tile overlaps it, and the Q rows
    // are not queued behind the whole first ring fill (requesting that ring
    // before the wait put the rows in place ~2 us after it ended, and the
    // whole call 0.1-0.5 us slower; requesting no tile before it, or both
    // first K tiles, was slower too).
    if (warp == kProdWarp && lane == 0) {
        if (n_my > 0) {
            load_k(0);
            if (a.has_mask) load_m(0);
        }
        asm volatile("griddepcontrol.wait;" ::: "memory");
        FR_STAMP(4);                                 // the grids ahead are complete
        for (int b = 0; b < C::NB; ++b)
            tma_load_2d(smem_addr(sQ + b * C::Q_BOX), &mp.q16, b * 64, row0, bar(C::B_QFULL));
        for (int i = 0; i < max(C::KS, max(C::VS, C::MS)) && i < n_my; ++i) {
            if (i > 0 && i < C::KS) load_k(i);
            if (a.has_mask && i > 0 && i < C::MS) load_m(i);
            if (i < C::VS) load_v(i);
        }
    }

    if (a.probe_iters && tid == 0) {
        // test hook: a bounded wait on a barrier nothing ever signals
        if (!mbar_wait_polls(bar(C::B_PROBE), 0, a.probe_iters)) record_timeout(a.status, 2u);
    }

    // ---- main phase ----------------------------------------------------------
    const int qd = warp & 3, half = (warp >> 2) & 1;     // softmax: lane quadrant, column half
    const int r = qd * 32 + lane;                        // softmax: row of the tile
    const uint32_t lane_base = (uint32_t)(qd * 32) << 16;
    const bool quad_active = row0 + qd * 32 < a.M;
    float m_ref = -INFINITY, l_part = 0.f;
    if (warp == kProdWarp) {
        if (lane == 0) {
            // Refill whichever slot frees first (non-blocking probes, K first: it
            // gates the next S). No progress for the time limit = a timeout.
            int nk = min(C::KS, n_my), nv = min(C::VS, n_my), nm = a.has_mask ? min(C::MS, n_my) : n_my;
            uint64_t t_last = global_ns();
            while (nk < n_my || nv < n_my || nm < n_my) {
                bool moved = false;
                if (nk < n_my && mbar_ready(bar(C::B_KEMPTY + nk % C::KS), ((nk / C::KS) - 1) & 1)) {
                    load_k(nk++);
                    moved = true;
                }
                if (nm < n_my && mbar_ready(bar(C::B_MEMPTY + nm % C::MS), ((nm / C::MS) - 1) & 1)) {
                    load_m(nm++);
                    moved = true;
                }
                if (nv < n_my && mbar_ready(bar(C::B_VEMPTY + nv % C::VS), ((nv / C::VS) - 1) & 1)) {
                    load_v(nv++);
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
            // drain: every issued load has landed before the slot memory is reused
            // (full time limit even after a failure: no copy may outlive the CTA)
            for (int i = max(0, nk - C::KS); i < nk; ++i)
                if (!mbar_wait(bar(C::B_KFULL + i % C::KS), (i / C::KS) & 1, limit)) record_timeout(a.status, 1u);
            for (int i = max(0, nv - C::VS); i < nv; ++i)
                if (!mbar_wait(bar(C::B_VFULL + i % C::VS), (i / C::VS) & 1, limit)) record_timeout(a.status, 1u);
            if (a.has_mask)
                for (int i = max(0, nm - C::MS); i < nm; ++i)
                    if (!mbar_wait(bar(C::B_MFULL + i % C::MS), (i / C::MS) & 1, limit))
                        record_timeout(a.status, 1u);
        }
    } else if (warp == kMmaWarp) {
        if (lane == 0) {
            // the Q tile must have landed (full limit: the copy writes this
            // CTA's shared memory)
            if (!mbar_wait(bar(C::B_QFULL), 0, limit)) record_timeout(a.status, 1u);
            FR_STAMP(3);                             // the Q tile is in place
            tc_fence_after();
            constexpr uint32_t idS = idesc_f16_f32(kRows, BN, 0, 0);
            constexpr uint32_t idO = idesc_f16_f32(kRows, HD, 0, 1);
            const uint32_t q_base = smem_addr(sQ);
            auto issue_s = [&](int i) {
                const int st = i % C::KS;
                wait(bar(C::B_KFULL + st), (i / C::KS) & 1);
                if (i < 8) FR_STAMP(36 + i);             // K_i has landed
                tc_fence_after();
                const uint32_t k_base = smem_addr(sK(st));
                const uint32_t d = tbase + C::TM_S + (i & 1) * BN;
#pragma unroll
                for (int kk = 0; kk < HD / 16; ++kk) {
                    const int b = kk >> 2, off = (kk & 3) * 32;
                    mma_ss(d, sdesc_sw128(q_base + b * C::Q_BOX + off, 16, 1024),
                           sdesc_sw128(k_base + b * C::KV_BOX + off, 16, 1024), idS, kk > 0);
                }
                mma_commit(bar(C::B_SFULL + (i & 1)));
                mma_commit(bar(C::B_KEMPTY + st));
                if (i < 7) FR_STAMP(8 + 4 * i + 2);      // S_i issued
            };
            // S_{i+1} is issued ahead of PV_i, waiting for its K tile if need be, so
            // the softmax of tile i+1 can start as soon as that of tile i ends. No
            // cycle: the K slot it needs was freed by S_{i+1-KS}, already issued,
            // and K and V have separate rings. (Issuing it only when K_{i+1} had
            // already landed was 0.1-0.6 us per call slower.)
            int s_next = 0;
            if (n_my > 0) issue_s(s_next++);
            for (int i = 0; i < n_my; ++i) {
                if (s_next == i + 1 && s_next < n_my) issue_s(s_next++);
                wait(bar(C::B_PFULL + (i & 1)), (i >> 1) & 1);
                wait(bar(C::B_VFULL + i % C::VS), (i / C::VS) & 1);
                if (i < 8) FR_STAMP(44 + i);             // P_i written and V_i landed
                tc_fence_after();
                const uint32_t v_base = smem_addr(sV(i % C::VS));
#pragma unroll
                for (int ks = 0; ks < BN / 16; ++ks) {
                    // keys [16 ks, 16 ks + 16): softmax half h, k-step kk within it
                    const int h = ks / (BN / 32), kk = ks % (BN / 32);
                    const uint32_t p_tm = tbase + C::p_col(i & 1, h, 0) + kk * 8;
                    const uint32_t pl_tm = tbase + C::p_col(i & 1, h, 1) + kk * 8;
                    const uint64_t vd = sdesc_sw128(v_base + ks * 2048, C::KV_BOX, 1024);
                    mma_ts(tbase + C::TM_O, p_tm, vd, idO, (i > 0 || ks > 0) ? 1u : 0u);
                    mma_ts(tbase + C::TM_O, pl_tm, vd, idO, 1u);
                }
                mma_commit(bar(C::B_ODONE));
                mma_commit(bar(C::B_VEMPTY + i % C::VS));
                if (i < 7) FR_STAMP(8 + 4 * i + 3);      // PV_i issued
            }
            // drain: no MMA may still be running when TMEM is freed
            mma_commit(bar(C::B_MMADONE));
            if (!mbar_wait(bar(C::B_MMADONE), 0, limit)) record_timeout(a.status, 1u);
        }
    } else {
        // softmax: warps w and w+4 share TMEM lanes [32(w%4), +32) (row r); warp
        // w < 4 takes S columns [0, BN/2), warp w+4 takes [BN/2, BN). The two
        // halves of a row exchange their maxima through shared memory per tile.
        const int grow = row0 + r;
        const int t = (grow < a.M ? grow / a.n_head : a.n_tok - 1) - mask_t0;   // row of the mask window
        const int c_base = half * HB;
        for (int i = 0; i < n_my; ++i) {
            wait(bar(C::B_SFULL + (i & 1)), (i >> 1) & 1);
            if (tid == 0 && i < 7) FR_STAMP(8 + 4 * i);          // softmax of tile i starts
            tc_fence_after();
            float x[HB];
            float pm = -INFINITY;
            const int j0 = (t0 + i) * BN + c_base;
            if (quad_active) {
#pragma unroll
                for (int c = 0; c < HB; c += 32)
                    tmem_ld_x32(tbase + lane_base + C::TM_S + (i & 1) * BN + c_base + c,
                                reinterpret_cast<uint32_t*>(x) + c);
                tmem_wait_ld();
                const float kq = a.kq_log2;
                if (a.has_mask) {
                    wait(bar(C::B_MFULL + i % C::MS), (i / C::MS) & 1);
                    const unsigned char* mk = sMask(i % C::MS);
#pragma unroll
                    for (int c8 = 0; c8 < HB / 8; ++c8) {
                        const int col = c_base + c8 * 8;
                        const int mb = col >> 6, ch = (col & 63) >> 3;
                        const uint4 raw = *reinterpret_cast<const uint4*>(mk + mb * C::MASK_BOX + t * 128 +
                                                                         ((ch ^ (t & 7)) << 4));
                        const __half2* h2 = reinterpret_cast<const __half2*>(&raw);
#pragma unroll
                        for (int u = 0; u < 4; ++u) {
                            const float2 f = __half22float2(h2[u]);
                            x[c8 * 8 + 2 * u] = fmaf(f.x, kLog2e, x[c8 * 8 + 2 * u] * kq);
                            x[c8 * 8 + 2 * u + 1] = fmaf(f.y, kLog2e, x[c8 * 8 + 2 * u + 1] * kq);
                        }
                    }
                } else {
#pragma unroll
                    for (int c = 0; c < HB; ++c) x[c] *= kq;
                }
                if (j0 + HB > a.n_kv) {               // ragged last tile only
#pragma unroll
                    for (int c = 0; c < HB; ++c)
                        if (j0 + c >= a.n_kv) x[c] = -INFINITY;
                }
                float pm4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
                for (int c = 0; c < HB; ++c) pm4[c & 3] = fmaxf(pm4[c & 3], x[c]);
                pm = fmaxf(fmaxf(pm4[0], pm4[1]), fmaxf(pm4[2], pm4[3]));
            }
            if (a.has_mask) {                     // this warp is done with mask slot i % MS
                __syncwarp();
                if (lane == 0) mbar_arrive(bar(C::B_MEMPTY + i % C::MS));
            }
            sMaxX[((i & 1) * 2 + half) * kRows + r] = pm;
            quad_bar_sync(qd);
            const float mx = fmaxf(pm, sMaxX[((i & 1) * 2 + (half ^ 1)) * kRows + r]);
            float m_new = m_ref;
            if (mx > m_ref + kTau || (m_ref == -INFINITY && mx > -INFINITY)) m_new = fmaxf(mx, m_ref);
            const bool grow_ref = m_ref != -INFINITY && m_new != m_ref;
            const float alpha = grow_ref ? ex2(m_ref - m_new) : 1.f;
            if (quad_active) {
                if (__any_sync(0xffffffffu, grow_ref) && i > 0) {
                    // O holds PV up to tile i-1: wait for it, then rescale this half of the row
                    wait(bar(C::B_ODONE), (i - 1) & 1);
                    tc_fence_after();
#pragma unroll 1
                    for (int c = 0; c < OH; c += 32) {
                        uint32_t o[32];
                        tmem_ld_x32(tbase + lane_base + C::TM_O + half * OH + c, o);
                        tmem_wait_ld();
#pragma unroll
                        for (int u = 0; u < 32; ++u) o[u] = __float_as_uint(__uint_as_float(o[u]) * alpha);
                        tmem_st_x32(tbase + lane_base + C::TM_O + half * OH + c, o);
                    }
                    tmem_wait_st();
                }
                const float m_sub = m_new == -INFINITY ? 0.f : m_new;
                float sum4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                for (int cc = 0; cc < HB; cc += 32) {       // 32 columns at a time
                    uint32_t pk[16], pl[16];
#pragma unroll
                    for (int c = 0; c < 32; c += 2) {
                        const float p0 = ex2(x[cc + c] - m_sub), p1 = ex2(x[cc + c + 1] - m_sub);
                        sum4[(c >> 1) & 3] += p0 + p1;
                        const uint32_t hbits = pack_half2(p0, p1);
                        const float2 hf = __half22float2(*reinterpret_cast<const __half2*>(&hbits));
                        pk[c / 2] = hbits;
                        pl[c / 2] = pack_half2(p0 - hf.x, p1 - hf.y);
                    }
                    tmem_st_x16(tbase + lane_base + C::p_col(i & 1, half, 0) + cc / 2, pk);
                    tmem_st_x16(tbase + lane_base + C::p_col(i & 1, half, 1) + cc / 2, pl);
                }
                const float sum = (sum4[0] + sum4[1]) + (sum4[2] + sum4[3]);
                l_part = fmaf(l_part, alpha, sum);
                tmem_wait_st();
            }
            m_ref = m_new;
            if (tid == 0 && i < 7) FR_STAMP(8 + 4 * i + 1);      // P_i written
            tc_fence_before();
            mbar_arrive(bar(C::B_PFULL + (i & 1)));
        }
        if (n_my > 0) {
            if (!mbar_wait(bar(C::B_ODONE), (n_my - 1) & 1, limit)) record_timeout(a.status, 1u);
            if (tid == 0) FR_STAMP(1);           // every MMA complete
            tc_fence_after();
        }
        // the row sum is the sum of both halves' partial sums
        sLX[half * kRows + r] = l_part;
        quad_bar_sync(qd);
        l_part += sLX[(half ^ 1) * kRows + r];
    }
    __syncthreads();                    // every async load drained, every MMA done
    if (tid == 0) FR_STAMP(57);
    tc_fence_before();
    if (CS > 1) cluster_sync();         // #3: every CTA is done with its data region

    if (a.merge_kernel) {
        // ---- merge-kernel mode: this split's (m, l, O) rows go to the workspace;
        // attn_merge_kernel merges them. O leaves TMEM into the stage area (free
        // now) as HD/32 boxes of [128 rows][32 fp32] in the 128-byte swizzle.
        // Each softmax warp fills the [32 rows][32 fp32] block of one box per
        // TMEM chunk and stores it by TMA at once, so the stores of the first
        // chunks overlap the TMEM reads of the later ones. Warps whose 32 rows
        // hold no real row store nothing.
        if (warp < kSmaxWarps && quad_active) {
            unsigned char* sOut = sStage;
            const int y = (rt * a.splits + split) * kRows + qd * 32;
            tc_fence_after();
#pragma unroll 1
            for (int c = 0; c < OH; c += 32) {
                uint32_t o[32];
                if (n_my > 0) {
                    tmem_ld_x32(tbase + lane_base + C::TM_O + half * OH + c, o);
                    tmem_wait_ld();
                } else {
#pragma unroll
                    for (int u = 0; u < 32; ++u) o[u] = 0u;
                }
                const int bx = (half * OH + c) >> 5;
                unsigned char* rowp = sOut + bx * C::OBOX + r * 128;
#pragma unroll
                for (int j = 0; j < 8; ++j)
                    *reinterpret_cast<uint4*>(rowp + ((j ^ (r & 7)) << 4)) =
                        make_uint4(o[4 * j], o[4 * j + 1], o[4 * j + 2], o[4 * j + 3]);
                fence_proxy_async_cta();        // the block is read by the TMA engine
                __syncwarp();
                if (lane == 0) tma_store_2d(&mp.po, bx * 32, y, smem_addr(sOut + bx * C::OBOX + qd * 32 * 128));
            }
            if (lane == 0) bulk_commit();
            if (half == 0 && r < rows_real)
                a.part_ml[(int64_t)(rt * a.splits + split) * kRows + r] =
                    n_my > 0 ? make_float2(m_ref, l_part) : make_float2(-INFINITY, 0.f);
            if (lane == 0) bulk_wait_all();     // performed before the grid completes
            if (tid == 0) FR_STAMP(58);          // this split's state is stored
        }
    } else {
    // ---- push (m, l, O) rows to the CTA that owns them in this cluster ------
    // rank c owns rows [c*R, (c+1)*R) of the tile: sML[src][row], sRecvO[src][row][RS]
    if (warp < kSmaxWarps && quad_active) {
        tc_fence_after();
        float* tb_w = sTB + warp * (32 * 36);
        const int srow = lane >> 3, scol = (lane & 7) * 4;   // 4 rows x 32 columns per step
#pragma unroll 1
        for (int c = 0; c < OH; c += 32) {
            uint32_t o[32];
            if (n_my > 0) {
                tmem_ld_x32(tbase + lane_base + C::TM_O + half * OH + c, o);
                tmem_wait_ld();
            } else {
#pragma unroll
                for (int u = 0; u < 32; ++u) o[u] = 0u;
            }
#pragma unroll
            for (int u = 0; u < 32; u += 4)
                *reinterpret_cast<uint4*>(tb_w + lane * 36 + u) = make_uint4(o[u], o[u + 1], o[u + 2], o[u + 3]);
            __syncwarp();
#pragma unroll
            for (int st = 0; st < 8; ++st) {
                const int rr = qd * 32 + st * 4 + srow;          // tile row this lane stores
                if (rr < rows_real) {
                    const int ow = rr / R, olr = rr - ow * R;
                    const uint4 v = *reinterpret_cast<const uint4*>(tb_w + (st * 4 + srow) * 36 + scol);
                    st_cluster_v4(map_rank(smem_addr(sRecvO + ((int)rank * R + olr) * C::RS + half * OH + c + scol),
                                           (uint32_t)ow), v);
                }
            }
            __syncwarp();
        }
        if (half == 0 && r < rows_real) {
            const int owner = r / R, lr = r - owner * R;
            const float2 ml = n_my > 0 ? make_float2(m_ref, l_part) : make_float2(-INFINITY, 0.f);
            const uint32_t dml = map_rank(smem_addr(sML + (int)rank * R + lr), (uint32_t)owner);
            asm volatile("st.shared::cluster.v2.f32 [%0], {%1, %2};" :: "r"(dml), "f"(ml.x), "f"(ml.y) : "memory");
        }
    }
    tc_fence_before();
    cluster_sync();                     // #4: every push has landed; no remote access after this

    // ---- merge the cluster's states for rows [rank*R, rank*R + R) ----------
    const int mr0 = (int)rank * R;
    const int mrows = max(0, min(R, rows_real - mr0));
    float* wts = sW;                         // [R][CS]
    float* rowM = sW + R * CS;               // [R]
    float* rowL = rowM + R;                  // [R]
    if (tid < mrows) {
        float mmax = -INFINITY;
        for (int p = 0; p < CS; ++p) mmax = fmaxf(mmax, sML[p * R + tid].x);
        const float ref = mmax == -INFINITY ? 0.f : mmax;
        float L = 0.f;
        for (int p = 0; p < CS; ++p) {
            const float2 ml = sML[p * R + tid];
            const float w = ml.x == -INFINITY ? 0.f : ex2(ml.x - ref);
            wts[tid * CS + p] = w;
            L = fmaf(w, ml.y, L);
        }
        rowM[tid] = mmax;
        rowL[tid] = L;
    }
    __syncthreads();
    const bool single = a.n_clusters == 1;
    {
        constexpr int Q4 = HD / 4;
        for (int i = tid; i < mrows * Q4; i += kThreads) {
            const int lr = i / Q4, q4 = i - lr * Q4;
            float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
            for (int p = 0; p < CS; ++p) {            // rank order: deterministic
                const float w = wts[lr * CS + p];
                const float4 v = *reinterpret_cast<const float4*>(sRecvO + (p * R + lr) * C::RS + q4 * 4);
                acc.x = fmaf(w, v.x, acc.x);
                acc.y = fmaf(w, v.y, acc.y);
                acc.z = fmaf(w, v.z, acc.z);
                acc.w = fmaf(w, v.w, acc.w);
            }
            if (single) {
                const float L = rowL[lr];
                float4 o;
                o.x = L > 0.f ? acc.x / L : 0.f;
                o.y = L > 0.f ? acc.y / L : 0.f;
                o.z = L > 0.f ? acc.z / L : 0.f;
                o.w = L > 0.f ? acc.w / L : 0.f;
                *reinterpret_cast<float4*>(a.out + (int64_t)(row0 + mr0 + lr) * HD + q4 * 4) = o;
            } else {
                const int64_t slot = ((int64_t)rt * a.n_clusters + cl) * kRows + mr0 + lr;
                *reinterpret_cast<float4*>(a.part_o + slot * HD + q4 * 4) = acc;
                if (q4 == 0) a.part_ml[slot] = make_float2(rowM[lr], rowL[lr]);
            }
        }
    }

    // ---- merge across clusters: the last CTA of each (row tile, rank) slice ---
    if (!single) {
        __threadfence();
        __syncthreads();
        if (tid == 0) {
            const unsigned prev = atomicAdd(a.tickets + rt * CS + rank, 1u);
            s_last = prev == (unsigned)(a.n_clusters - 1);
        }
        __syncthreads();
        if (s_last) {
            __threadfence();
            const int NC = a.n_clusters;
            float* w2 = sW;                          // [R][NC]
            float* L2 = sW + R * NC;                 // [R]
            float2* ml2 = reinterpret_cast<float2*>(sRecvO);      // [R][NC] (m, l), local scratch
            for (int i = tid; i < mrows * NC; i += kThreads) {    // every (row, cluster) at once
                const int lr = i / NC, c2 = i - lr * NC;
                ml2[i] = __ldcg(a.part_ml + ((int64_t)rt * NC + c2) * kRows + mr0 + lr);
            }
            __syncthreads();
            if (tid < mrows) {
                float mmax = -INFINITY;
                for (int c2 = 0; c2 < NC; ++c2) mmax = fmaxf(mmax, ml2[tid * NC + c2].x);
                const float ref = mmax == -INFINITY ? 0.f : mmax;
                float L = 0.f;
                for (int c2 = 0; c2 < NC; ++c2) {
                    const float2 ml = ml2[tid * NC + c2];
                    const float w = ml.x == -INFINITY ? 0.f : ex2(ml.x - ref);
                    w2[tid * NC + c2] = w;
                    L = fmaf(w, ml.y, L);
                }
                L2[tid] = L;
            }
            __syncthreads();
            constexpr int Q4 = HD / 4;
            for (int i = tid; i < mrows * Q4; i += kThreads) {
                const int lr = i / Q4, q4 = i - lr * Q4;
                const int rr = mr0 + lr;
                const float* src = a.part_o + (((int64_t)rt * NC) * kRows + rr) * HD + q4 * 4;
                const int64_t cstride = (int64_t)kRows * HD;
                float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
                for (int c0 = 0; c0 < NC; c0 += 8) {
                    float4 v[8];
#pragma unroll
                    for (int u = 0; u < 8; ++u)          // eight independent loads in flight
                        v[u] = c0 + u < NC ? __ldcg(reinterpret_cast<const float4*>(src + (c0 + u) * cstride))
                                           : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
                    for (int u = 0; u < 8; ++u) {
                        const float w = c0 + u < NC ? w2[lr * NC + c0 + u] : 0.f;
                        acc.x = fmaf(w, v[u].x, acc.x);
                        acc.y = fmaf(w, v[u].y, acc.y);
                        acc.z = fmaf(w, v[u].z, acc.z);
                        acc.w = fmaf(w, v[u].w, acc.w);
                    }
                }
                const float L = L2[lr];
                float4 o;
                o.x = L > 0.f ? acc.x / L : 0.f;
                o.y = L > 0.f ? acc.y / L : 0.f;
                o.z = L > 0.f ? acc.z / L : 0.f;
                o.w = L > 0.f ? acc.w / L : 0.f;
                *reinterpret_cast<float4*>(a.out + (int64_t)(row0 + rr) * HD + q4 * 4) = o;
            }
            if (tid == 0) a.tickets[rt * CS + rank] = 0u;
        }
    }

    }   // in-kernel merge

    // ---- teardown --------------------------------------------------------------
    tc_fence_before();
    __syncthreads();
    if (tid == 0) FR_STAMP(2);                   // done
    if (warp == kMmaWarp) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tbase, kTmemCols);
    }
}

// Merge of the split states written in merge-kernel mode: split s of row tile
// rt holds rows [rt*rstride, (rt+1)*rstride) at part_o[((rt*splits + s)*rstride
// + rr)*HD] (rstride = 128 for the 128-row tiles, M for the keys-on-M kernel).
// A unit is one (row,
// 128-column chunk); it gets nw warps (one per split when that fits the GPU in
// one wave, else one per 5 or 6 splits, see launch_merge) and a CTA of up to
// kMergeWarps warps holds several units. Warp w of a unit takes splits
// w, w + nw, ... (at most a handful each, so the loads of the whole CTA are in
// flight together). Each warp weighs its splits by 2^(m_s - m_w) against its
// own maximum m_w; the unit's warp sums are then combined in warp order
// against the row maximum. The order of every sum is fixed: the result does
// not depend on timing.
constexpr int kMergeWarps = 32;
// Splits per warp when a unit cannot have one warp per split: nw = ceil(splits /
// this) warps per unit. At hd <= 128 a row is one unit, so there are half as
// many units and 5 splits per warp (more warps each) pays: hd 128 / 16 tokens
// / 65536 keys 18.70 -> 17.75 us per call, long decode 25.06 -> 23.82 us,
// while at hd 256 it cost 0.2-0.4 us (same-process A/B).
__host__ __device__ constexpr int merge_splits_per_warp(int hd) { return hd >= 256 ? 6 : 5; }

// The FR_TRACE build holds the untraced kernel's register count (two CTAs of
// up to 1024 threads per SM), so that its stamps do not change the occupancy.
#ifdef FR_TRACE
#define FR_MERGE_BOUNDS __launch_bounds__(kMergeWarps * 32, 2)
#else
#define FR_MERGE_BOUNDS __launch_bounds__(kMergeWarps * 32)
#endif
template <int HD>
__global__ void FR_MERGE_BOUNDS
attn_merge_kernel(const float* __restrict__ part_o, const float2* __restrict__ part_ml, float* __restrict__ out,
                  int M, int splits, int nw, int early, int rstride, unsigned* trace_ws) {
    constexpr int CWM = HD < 128 ? HD : 128;
    constexpr int NCH = HD / CWM;
    constexpr int LANES = CWM / 4;
    constexpr int PER_WARP = merge_splits_per_warp(HD);
    static_assert(PER_WARP <= 32, "one (m, l) pair per lane");
    static_assert((kMaxMergeSplits + PER_WARP - 1) / PER_WARP <= kMergeWarps,
                  "every split count fits in one CTA");
    __shared__ float s_acc[kMergeWarps][CWM];
    __shared__ float s_m[kMergeWarps], s_l[kMergeWarps];
    const int tid = threadIdx.x, lane = tid & 31;
    const int uw = (tid >> 5) / nw, warp = (tid >> 5) - uw * nw;      // unit in the CTA, warp in the unit
    const int upc = (int)(blockDim.x >> 5) / nw;                        // units per CTA
    const int unit = blockIdx.x * upc + uw;
    const bool live = uw < upc && unit < M * NCH;
    const int row = live ? unit / NCH : 0, chunk = live ? unit - (unit / NCH) * NCH : 0;
    const int rt = row / rstride, rr = row - rt * rstride;
    if (tid == 0) {
        FR_STAMP_AT(trace_ws, 0);                           // resident
        FR_STAMP_SMID_AT(trace_ws);
    }
    asm volatile("griddepcontrol.wait;" ::: "memory");     // the attention grid is complete
    if (tid == 0) FR_STAMP_AT(trace_ws, 1);
    // A dependent launch (the next call's qkv_post) may start now only when this
    // grid fits in one wave; otherwise its waiting CTAs would hold the SMs the
    // later merge CTAs need.
    if (early) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    const int n_w = live && splits > warp ? (splits - warp + nw - 1) / nw : 0;   // this warp's splits
    const float2* ml = part_ml + (int64_t)rt * splits * rstride + rr;
    const float2 my_ml =
        lane < n_w ? __ldcg(ml + (int64_t)(warp + nw * lane) * rstride) : make_float2(-INFINITY, 0.f);
    float4 v[PER_WARP];
    const float* base = part_o + ((int64_t)rt * splits * rstride + rr) * HD + chunk * CWM + (lane % LANES) * 4;
    const int64_t sstride = (int64_t)rstride * HD;
#pragma unroll
    for (int u = 0; u < PER_WARP; ++u)
        v[u] = (u < n_w && lane < LANES)
                   ? __ldcg(reinterpret_cast<const float4*>(base + (warp + nw * u) * sstride))
                   : make_float4(0.f, 0.f, 0.f, 0.f);
    float mw = my_ml.x;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) mw = fmaxf(mw, __shfl_xor_sync(0xffffffffu, mw, o));
    const float ref = mw == -INFINITY ? 0.f : mw;
    const float my_w = my_ml.x == -INFINITY ? 0.f : ex2(my_ml.x - ref);
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    float lw = 0.f;
#pragma unroll
    for (int u = 0; u < PER_WARP; ++u) {
        const float w = __shfl_sync(0xffffffffu, my_w, u);
        const float l = __shfl_sync(0xffffffffu, my_ml.y, u);
        lw = fmaf(w, l, lw);
        acc.x = fmaf(w, v[u].x, acc.x);
        acc.y = fmaf(w, v[u].y, acc.y);
        acc.z = fmaf(w, v[u].z, acc.z);
        acc.w = fmaf(w, v[u].w, acc.w);
    }
    const int sw = tid >> 5;                                            // warp slot in the CTA
    if (lane < LANES) *reinterpret_cast<float4*>(&s_acc[sw][lane * 4]) = acc;
    if (lane == 0) {
        s_m[sw] = mw;
        s_l[sw] = lw;
    }
    __syncthreads();
    if (live) {
        const int w0 = uw * nw;                                         // the unit's first warp slot
        float mx = -INFINITY;
        for (int w = 0; w < nw; ++w) mx = fmaxf(mx, s_m[w0 + w]);
        const float mref = mx == -INFINITY ? 0.f : mx;
        for (int c = warp * 32 + lane; c < CWM; c += nw * 32) {   // fewer threads than columns when nw < 4
            float sum = 0.f, L = 0.f;
#pragma unroll 4
            for (int w = 0; w < nw; ++w) {
                const float sc = s_m[w0 + w] == -INFINITY ? 0.f : ex2(s_m[w0 + w] - mref);
                sum = fmaf(sc, s_acc[w0 + w][c], sum);
                L = fmaf(sc, s_l[w0 + w], L);
            }
            out[(int64_t)row * HD + chunk * CWM + c] = L > 0.f ? sum / L : 0.f;
        }
    }
#ifdef FR_TRACE
    __syncthreads();
    if (tid == 0) FR_STAMP_AT(trace_ws, 2);                 // done
#endif
}

// The same merge for a few splits (<= kSmallMergeSplits): one warp per unit,
// each lane merging its 4 columns over all splits in registers, units strided
// over a one-wave grid. Same weights, same order of every sum.
constexpr int kSmallMergeSplits = 8;

template <int HD>
__global__ void __launch_bounds__(256)
attn_merge_small_kernel(const float* __restrict__ part_o, const float2* __restrict__ part_ml,
                        float* __restrict__ out, int M, int splits, int rstride) {
    constexpr int CWM = HD < 128 ? HD : 128;
    constexpr int NCH = HD / CWM;
    constexpr int LANES = CWM / 4;
    asm volatile("griddepcontrol.wait;" ::: "memory");     // the attention grid is complete
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    const int lane = threadIdx.x & 31;
    const int64_t sstride = (int64_t)rstride * HD;
    for (int64_t unit = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5; unit < (int64_t)M * NCH;
         unit += ((int64_t)gridDim.x * blockDim.x) >> 5) {
        const int row = (int)(unit / NCH), chunk = (int)(unit - (int64_t)row * NCH);
        const int rt = row / rstride, rr = row - rt * rstride;
        const float2* ml = part_ml + (int64_t)rt * splits * rstride + rr;
        const float* base = part_o + ((int64_t)rt * splits * rstride + rr) * HD + chunk * CWM + (lane % LANES) * 4;
        float2 st[kSmallMergeSplits];
        float4 v[kSmallMergeSplits];
#pragma unroll
        for (int s2 = 0; s2 < kSmallMergeSplits; ++s2) {
            st[s2] = s2 < splits ? __ldcg(ml + (int64_t)s2 * rstride) : make_float2(-INFINITY, 0.f);
            v[s2] = (s2 < splits && lane < LANES) ? __ldcg(reinterpret_cast<const float4*>(base + s2 * sstride))
                                                 : make_float4(0.f, 0.f, 0.f, 0.f);
        }
        float mx = -INFINITY;
#pragma unroll
        for (int s2 = 0; s2 < kSmallMergeSplits; ++s2) mx = fmaxf(mx, st[s2].x);
        const float ref = mx == -INFINITY ? 0.f : mx;
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
        float L = 0.f;
#pragma unroll
        for (int s2 = 0; s2 < kSmallMergeSplits; ++s2) {
            const float w = st[s2].x == -INFINITY ? 0.f : ex2(st[s2].x - ref);
            L = fmaf(w, st[s2].y, L);
            acc.x = fmaf(w, v[s2].x, acc.x);
            acc.y = fmaf(w, v[s2].y, acc.y);
            acc.z = fmaf(w, v[s2].z, acc.z);
            acc.w = fmaf(w, v[s2].w, acc.w);
        }
        if (lane < LANES) {
            float4 o;
            o.x = L > 0.f ? acc.x / L : 0.f;
            o.y = L > 0.f ? acc.y / L : 0.f;
            o.z = L > 0.f ? acc.z / L : 0.f;
            o.w = L > 0.f ? acc.w / L : 0.f;
            *reinterpret_cast<float4*>(out + (int64_t)row * HD + chunk * CWM + lane * 4) = o;
        }
    }
}

fr_status launch_merge(const float* part_o, const float2* part_ml, float* out, int M, int splits, int hd,
                       int rstride, unsigned* ws, cudaStream_t stream) {
    if (splits < 1 || splits > kMaxMergeSplits) return FR_ERR_UNSUPPORTED;
    cudaLaunchConfig_t cfg;
    memset(&cfg, 0, sizeof(cfg));
    if (splits <= kSmallMergeSplits) {
        int dev = 0, sms = 152;
        if (cudaGetDevice(&dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            return FR_ERR_CUDA;
        const int64_t units = (int64_t)M * (hd < 128 ? 1 : hd / 128);
        const int64_t want = (units + 7) / 8;                       // 8 warps (units) per CTA
        cfg.gridDim = dim3((unsigned)(want < (int64_t)sms * 8 ? want : (int64_t)sms * 8), 1, 1);
        cfg.blockDim = dim3(256, 1, 1);
        cfg.stream = stream;
        cudaLaunchAttribute at[1];
        at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        at[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = at;
        cfg.numAttrs = 1;
        cudaError_t e;
        switch (hd) {
            case 64: e = cudaLaunchKernelEx(&cfg, attn_merge_small_kernel<64>, part_o, part_ml, out, M, splits, rstride); break;
            case 128: e = cudaLaunchKernelEx(&cfg, attn_merge_small_kernel<128>, part_o, part_ml, out, M, splits, rstride); break;
            default: e = cudaLaunchKernelEx(&cfg, attn_merge_small_kernel<256>, part_o, part_ml, out, M, splits, rstride); break;
        }
        return e == cudaSuccess ? FR_OK : FR_ERR_CUDA;
    }
    const int nch = hd < 128 ? 1 : hd / 128;
    const int units = M * nch;
    int dev = 0, sms = 152;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return FR_ERR_CUDA;
    // Warps per unit and units per CTA. When one warp per split fits the GPU in
    // one wave, take that (the fewest dependent loads per warp). Otherwise up to
    // 5 (hd <= 128) or 6 splits per warp (fewer instructions per split), with
    // few enough units per CTA that the grid still covers the SMs.
    int nw, upc;
    if ((int64_t)units * splits <= (int64_t)sms * kMergeWarps && splits <= kMergeWarps) {
        nw = splits;
        upc = kMergeWarps / nw;
    } else {
        const int spw = merge_splits_per_warp(hd);
        nw = (splits + spw - 1) / spw;
        upc = kMergeWarps / nw;
        if (upc > units / sms) upc = units / sms > 0 ? units / sms : 1;
    }
    cfg.gridDim = dim3((units + upc - 1) / upc, 1, 1);
    cfg.blockDim = dim3(upc * nw * 32, 1, 1);
    const int early = (int64_t)cfg.gridDim.x * cfg.blockDim.x <= (int64_t)sms * 2048 ? 1 : 0;   // one wave
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaError_t e;
    switch (hd) {
        case 64: e = cudaLaunchKernelEx(&cfg, attn_merge_kernel<64>, part_o, part_ml, out, M, splits, nw, early, rstride, ws); break;
        case 128: e = cudaLaunchKernelEx(&cfg, attn_merge_kernel<128>, part_o, part_ml, out, M, splits, nw, early, rstride, ws); break;
        default: e = cudaLaunchKernelEx(&cfg, attn_merge_kernel<256>, part_o, part_ml, out, M, splits, nw, early, rstride, ws); break;
    }
    return e == cudaSuccess ? FR_OK : FR_ERR_CUDA;
}

// ---- host side ----------------------------------------------------------------

static PFN_cuTensorMapEncodeTiled_v12000 get_encoder() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    if (!fn) {
        cudaDriverEntryPointQueryResult q;
        void* p = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess && q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    }
    return fn;
}

// 2-D f16 tensor [rows][inner] with a row stride in elements; 128-byte swizzle.
static bool encode_2d(CUtensorMap* m, const void* base, uint64_t inner, uint64_t rows, uint64_t row_stride,
                      uint32_t box_inner, uint32_t box_rows) {
    auto enc = get_encoder();
    if (!enc) return false;
    cuuint64_t dims[2] = {inner, rows};
    cuuint64_t strides[1] = {row_stride * 2};
    cuuint32_t box[2] = {box_inner, box_rows};
    cuuint32_t es[2] = {1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<void*>(base), dims, strides, box, es,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool encode_f16_2d(CUtensorMap* m, const void* base, uint64_t inner, uint64_t rows, uint64_t row_stride,
                   uint32_t box_inner, uint32_t box_rows, bool swizzle128) {
    auto enc = get_encoder();
    if (!enc) return false;
    cuuint64_t dims[2] = {inner, rows};
    cuuint64_t strides[1] = {row_stride * 2};
    cuuint32_t box[2] = {box_inner, box_rows};
    cuuint32_t es[2] = {1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<void*>(base), dims, strides, box, es,
               CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 2-D fp32 tensor [rows][inner], contiguous rows; boxes of 32 columns (128 B) x
// box_rows in the 128-byte swizzle (the layout the merge-kernel epilogue writes).
static bool encode_2d_f32(CUtensorMap* m, void* base, uint64_t inner, uint64_t rows, uint32_t box_rows) {
    auto enc = get_encoder();
    if (!enc) return false;
    cuuint64_t dims[2] = {inner, rows};
    cuuint64_t strides[1] = {inner * 4};
    cuuint32_t box[2] = {32, box_rows};
    cuuint32_t es[2] = {1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, base, dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
               CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int HD, int BN>
static cudaError_t ensure_attr(int dev) {
    static unsigned long long done = 0ull;
    if (dev < 64 && (__atomic_load_n(&done, __ATOMIC_ACQUIRE) >> dev & 1ull)) return cudaSuccess;
    cudaError_t e = cudaFuncSetAttribute(attn_tc_kernel<HD, BN>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         Cfg<HD, BN>::SMEM);
    if (e == cudaSuccess && dev < 64) __atomic_fetch_or(&done, 1ull << dev, __ATOMIC_RELEASE);
    return e;
}

// 128-key tiles at hd 128 when there is at least one for each SM of a row
// tile's share (measured: 65536 keys 1.0-1.5 us faster per call, 32768 keys on
// 4 row tiles 3.3 us faster; even at 16384 keys; 1.7-2.4 us slower at 4096
// keys, where they would halve the CTAs).
int tile_keys(int hd, int n_kv, int row_tiles, int num_sms) {
    if (hd != 128) return 64;
    const int share = row_tiles > 0 ? num_sms / row_tiles : num_sms;
    return n_kv / 128 >= share ? 128 : 64;
}

template <int HD, int BN_>
static fr_status launch(const TcLaunch& L, cudaStream_t stream) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return FR_ERR_CUDA;
    if (ensure_attr<HD, BN_>(dev) != cudaSuccess) return FR_ERR_CUDA;
    Maps mp;
    memset(&mp, 0, sizeof(mp));
    const TcArgs& a = L.args;
    constexpr int BN = Cfg<HD, BN_>::BN;
    if (!encode_2d(&mp.k, L.k, HD, a.n_kv, L.k_rs, 64, BN)) return FR_ERR_CUDA;
    if (!encode_2d(&mp.v, L.v, HD, a.n_kv, L.v_rs, 64, BN)) return FR_ERR_CUDA;
    if (a.has_mask &&
        !encode_2d(&mp.mask, L.mask, a.n_kv, a.n_tok, L.m_rs, 64, (uint32_t)(a.n_tok < kMaskWin ? a.n_tok : kMaskWin)))
        return FR_ERR_CUDA;
    if (!a.q16 || !encode_2d(&mp.q16, a.q16, HD, a.M, HD, 64, kRows)) return FR_ERR_CUDA;
    if (a.merge_kernel &&
        !encode_2d_f32(&mp.po, a.part_o, HD, (uint64_t)L.row_tiles * a.splits * kRows, kOutBoxRows))
        return FR_ERR_CUDA;

    cudaLaunchConfig_t cfg;
    memset(&cfg, 0, sizeof(cfg));
    cfg.gridDim = dim3(L.row_tiles, L.splits, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = Cfg<HD, BN_>::SMEM;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 1;
    attr[0].val.clusterDim.y = a.C;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = L.pdl ? 2 : 1;
    cudaError_t e = cudaLaunchKernelEx(&cfg, attn_tc_kernel<HD, BN_>, a, mp);
    return e == cudaSuccess ? FR_OK : FR_ERR_CUDA;
}

fr_status launch_tc(const TcLaunch& L, int hd, cudaStream_t stream) {
    switch (hd) {
        case 64: return launch<64, 64>(L, stream);
        case 128: return L.bn == 128 ? launch<128, 128>(L, stream) : launch<128, 64>(L, stream);
        default: return launch<256, 64>(L, stream);
    }
}

}  // namespace tc
}  // namespace fr
