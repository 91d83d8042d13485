// fr_decode_attn.cu -- collapsed GQA decode attention over one shared f16 KV
// head, split over n_kv with the fix-up (split combine) fused into the kernel.
//
// FlashRT PR #185, commit "FLASH_ATTN_EXT with q_tokens <= 16 over a single
// padded f16 KV head runs as a batched QK^T GEMM (GQA heads share the stride-0
// K operand), a masked fp32-accurate softmax, and a batched PV GEMM whose fp32
// result lands directly in the node's [hd, n_head, n_tok] layout"; commit "The
// GQA query heads share the one KV head, so the per-head batched QK^T and PV
// GEMMs collapse into single GEMMs over all n_head*n_tok query rows. Ordering
// the rows t-major makes the PV output land contiguously". The same commit
// names the stream-k flash kernel and its fixup pass as the alternative; here
// the split-KV partial states are merged inside the same launch by the last
// CTA to arrive for each row block, so there is no second pass.
//
// Work decomposition (one launch):
//   grid = (row blocks of 16 t-major query rows) x (KV splits)
//   CTA  = 4 warps; every 64-key tile is staged in shared memory with cp.async
//          (multi-stage ring); warp w takes keys [16w, 16w+16) of each tile
//          against all 16 rows: S = Q K^T and O += P V on mma.sync m16n8k16
//          (f16 in, fp32 accumulate), online softmax in the log2 domain.
//   end  = the 4 warps' states merge in shared memory; with one split the CTA
//          writes the normalised rows, otherwise it writes its (m, l, O) to the
//          workspace and the last-arriving CTA of the row block merges all
//          splits (atomic ticket, reset to zero afterwards; nothing waits).
#include <math.h>
#include <string.h>

#include "fr_attn.h"
#include "fr_common.cuh"

namespace fr {

constexpr int kBN = 64;          // keys per KV tile
constexpr int kRB = 16;          // t-major query rows per CTA
constexpr int kWarps = 4;
constexpr int kThreads = kWarps * 32;
constexpr int kMaxSplits = 32;
constexpr size_t kWsHeader = 1024;     // [0,4): status word; [256, 256+4*32): tickets
constexpr size_t kWsTickets = 256;
constexpr size_t kWsSwBarrier = 512;   // [512, 520): the keys-on-M kernel's grid barrier (arrivals, departures)
constexpr float kLog2e = 1.4426950408889634f;

template <int HD>
struct V1Cfg {
    static constexpr int STAGES = HD == 256 ? 2 : (HD == 128 ? 3 : 4);
    static constexpr int LDS = HD + 8;          // f16 row stride in shared memory
    static constexpr int LDM = kBN + 8;         // mask row stride (f16)
    static constexpr int RS = HD + 4;           // fp32 row stride of the merge area
    static constexpr int Q_BYTES = kRB * LDS * 2;
    static constexpr int KV_BYTES = kBN * LDS * 2;
    static constexpr int MASK_BYTES = kMaxTok * LDM * 2;
    static constexpr int STAGE_BYTES = 2 * KV_BYTES + MASK_BYTES;
    static constexpr int RED_BYTES = kWarps * kRB * RS * 4 + 2 * kWarps * kRB * 4;
    static constexpr int FIX_BYTES = kMaxSplits * kRB * 12 + 2 * kRB * 4;
    static constexpr int BODY = STAGES * STAGE_BYTES;
    static constexpr int AFTER = RED_BYTES > FIX_BYTES ? RED_BYTES : FIX_BYTES;
    static constexpr int TABLE_BYTES = kMaxPairs * 8;
    static constexpr int SMEM = Q_BYTES + TABLE_BYTES + (BODY > AFTER ? BODY : AFTER);
};

struct AttnArgs {
    const __half* q16;
    const float* q;
    int64_t q_tok_stride;
    const int32_t* pos;
    const __half* k;
    int64_t k_rs;
    const __half* v;
    int64_t v_rs;
    const __half* mask;
    int64_t m_rs;
    float* out;
    float* part_o;         // [n_splits][M][HD]
    float2* part_ml;       // [n_splits][M]  (row max in log2 units, row sum)
    unsigned* tickets;     // [n_row_blocks]
    int n_tok, n_head, M, n_kv, n_tiles, n_splits, tiles_per_split;
    float kq_log2;         // kq_scale * log2(e)
};

template <int HD>
__global__ void __launch_bounds__(kThreads, 1)
attn_v1_kernel(const __grid_constant__ AttnArgs a, const __grid_constant__ RopeTable tb) {
    using C = V1Cfg<HD>;
    extern __shared__ __align__(128) unsigned char smem[];
    __half* sQ = reinterpret_cast<__half*>(smem);
    uint64_t* sTurns = reinterpret_cast<uint64_t*>(smem + C::Q_BYTES);
    unsigned char* body = smem + C::Q_BYTES + C::TABLE_BYTES;
    __shared__ int s_last;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int rb = blockIdx.x, split = blockIdx.y;
    const int row0 = rb * kRB;
    const int tile0 = split * a.tiles_per_split;
    const int ntl = min(a.n_tiles, tile0 + a.tiles_per_split) - tile0;   // >= 1
    const int nrows = min(kRB, a.M - row0);

    auto sK = [&](int s) { return reinterpret_cast<__half*>(body + s * C::STAGE_BYTES); };
    auto sV = [&](int s) { return reinterpret_cast<__half*>(body + s * C::STAGE_BYTES + C::KV_BYTES); };
    auto sMk = [&](int s) { return reinterpret_cast<__half*>(body + s * C::STAGE_BYTES + 2 * C::KV_BYTES); };

    auto load_tile = [&](int s, int tile) {
        constexpr int CH = HD / 8;                  // 16-byte chunks per row
        const int j0 = tile * kBN;
        __half* dk = sK(s);
        __half* dv = sV(s);
        for (int idx = tid; idx < kBN * CH; idx += kThreads) {
            const int jj = idx / CH, cc = idx - jj * CH;
            const int j = j0 + jj;
            const bool ok = j < a.n_kv;
            const __half* gk = a.k + (ok ? (int64_t)j * a.k_rs + cc * 8 : 0);
            const __half* gv = a.v + (ok ? (int64_t)j * a.v_rs + cc * 8 : 0);
            cp_async16(smem_u32(dk + jj * C::LDS + cc * 8), gk, ok ? 16 : 0);
            cp_async16(smem_u32(dv + jj * C::LDS + cc * 8), gv, ok ? 16 : 0);
        }
        if (a.mask) {
            __half* dm = sMk(s);
            constexpr int MC = kBN / 8;
            for (int idx = tid; idx < a.n_tok * MC; idx += kThreads) {
                const int t = idx / MC, cc = idx - t * MC;
                const int j = j0 + cc * 8;
                const int nb = max(0, min(16, (a.n_kv - j) * 2));
                const __half* gm = a.mask + (nb ? (int64_t)t * a.m_rs + j : 0);
                cp_async16(smem_u32(dm + t * C::LDM + cc * 8), gm, nb);
            }
        }
    };

    // ---- prologue: Q rows (given, or rope'd here) and the first tiles -----
    if (a.q16) {
        constexpr int CH = HD / 8;
        for (int idx = tid; idx < kRB * CH; idx += kThreads) {
            const int rr = idx / CH, cc = idx - rr * CH;
            const bool ok = rr < nrows;
            const __half* g = a.q16 + (ok ? (int64_t)(row0 + rr) * HD + cc * 8 : 0);
            cp_async16(smem_u32(sQ + rr * C::LDS + cc * 8), g, ok ? 16 : 0);
        }
    }
    for (int s = 0; s < C::STAGES - 1; ++s) {
        if (s < ntl) load_tile(s, tile0 + s);
        cp_async_commit();
    }
    if (!a.q16) {
        for (int i = tid; i < tb.half; i += kThreads) sTurns[i] = tb.turns[i];
        __syncthreads();
        RopeTable const& T = tb;
        constexpr int SL = HD / 2;
        for (int idx = tid; idx < kRB * SL; idx += kThreads) {
            const int rr = idx / SL, c = idx - rr * SL;
            __half* qrow_s = sQ + rr * C::LDS;
            if (rr >= nrows) {
                qrow_s[2 * c] = __float2half_rn(0.f);
                qrow_s[2 * c + 1] = __float2half_rn(0.f);
                continue;
            }
            const int r = row0 + rr;
            const int t = r / a.n_head, h = r - t * a.n_head;
            const float* qrow = a.q + (int64_t)t * a.q_tok_stride + (int64_t)h * HD;
            const int p = __ldg(a.pos + t);
            int d0, d1;
            float y0, y1;
            if (c < T.half && T.mode == FR_ROPE_EXACT) {
                d0 = c;
                d1 = c + T.half;
                float cs, sn;
                rope_cs(p, sTurns[c], T.mscale, cs, sn);
                y0 = rope_lo(qrow[d0], qrow[d1], cs, sn, T.q_scale);
                y1 = rope_hi(qrow[d0], qrow[d1], cs, sn, T.q_scale);
            } else {
                rope_slot(qrow, c, p, T, d0, d1, y0, y1);
            }
            qrow_s[d0] = __float2half_rn(y0);
            qrow_s[d1] = __float2half_rn(y1);
        }
    }

    const int g = lane >> 2, qd = lane & 3;
    const int t_lo = min((row0 + g) / a.n_head, a.n_tok - 1);
    const int t_hi = min((row0 + g + 8) / a.n_head, a.n_tok - 1);
    const int kw = warp * 16;

    float o[HD / 8][4];
#pragma unroll
    for (int i = 0; i < HD / 8; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
    float m_lo = -INFINITY, m_hi = -INFINITY, l_lo = 0.f, l_hi = 0.f;

    // ---- main loop over this split's KV tiles ---------------------------
    for (int it = 0; it < ntl; ++it) {
        cp_async_wait<C::STAGES - 2>();
        __syncthreads();
        {
            const int nt = it + C::STAGES - 1;
            if (nt < ntl) load_tile(nt % C::STAGES, tile0 + nt);
            cp_async_commit();
        }
        const int s = it % C::STAGES;
        const int j0 = (tile0 + it) * kBN;
        const __half* K = sK(s);
        const __half* V = sV(s);
        const __half* Mk = sMk(s);

        float sc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll
        for (int kk = 0; kk < HD / 16; ++kk) {
            uint32_t af[4], b0, b1, b2, b3;
            ldsm_x4(smem_u32(sQ + (lane & 15) * C::LDS + kk * 16 + (lane >> 4) * 8),
                    af[0], af[1], af[2], af[3]);
            ldsm_x4(smem_u32(K + (kw + (lane & 7) + (lane >> 4) * 8) * C::LDS + kk * 16 +
                             ((lane >> 3) & 1) * 8),
                    b0, b1, b2, b3);
            mma_16816(sc[0], af, b0, b1);
            mma_16816(sc[1], af, b2, b3);
        }

        float mx_lo = -INFINITY, mx_hi = -INFINITY;
#pragma unroll
        for (int n = 0; n < 2; ++n) {
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int key = kw + n * 8 + 2 * qd + (e & 1);
                const int t = e < 2 ? t_lo : t_hi;
                float x = sc[n][e] * a.kq_log2;
                if (a.mask) x = fmaf(__half2float(Mk[t * C::LDM + key]), kLog2e, x);
                if (j0 + key >= a.n_kv) x = -INFINITY;
                sc[n][e] = x;
                if (e < 2) mx_lo = fmaxf(mx_lo, x); else mx_hi = fmaxf(mx_hi, x);
            }
        }
        mx_lo = fmaxf(mx_lo, __shfl_xor_sync(0xffffffffu, mx_lo, 1));
        mx_lo = fmaxf(mx_lo, __shfl_xor_sync(0xffffffffu, mx_lo, 2));
        mx_hi = fmaxf(mx_hi, __shfl_xor_sync(0xffffffffu, mx_hi, 1));
        mx_hi = fmaxf(mx_hi, __shfl_xor_sync(0xffffffffu, mx_hi, 2));
        const float mn_lo = fmaxf(m_lo, mx_lo), mn_hi = fmaxf(m_hi, mx_hi);
        const float ref_lo = mn_lo == -INFINITY ? 0.f : mn_lo;
        const float ref_hi = mn_hi == -INFINITY ? 0.f : mn_hi;
        const float al_lo = exp2f(m_lo - ref_lo), al_hi = exp2f(m_hi - ref_hi);
        m_lo = mn_lo;
        m_hi = mn_hi;
        float sum_lo = 0.f, sum_hi = 0.f;
#pragma unroll
        for (int n = 0; n < 2; ++n) {
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const float p = exp2f(sc[n][e] - (e < 2 ? ref_lo : ref_hi));
                sc[n][e] = p;
                if (e < 2) sum_lo += p; else sum_hi += p;
            }
        }
        l_lo = fmaf(l_lo, al_lo, sum_lo);
        l_hi = fmaf(l_hi, al_hi, sum_hi);
#pragma unroll
        for (int i = 0; i < HD / 8; ++i) {
            o[i][0] *= al_lo;
            o[i][1] *= al_lo;
            o[i][2] *= al_hi;
            o[i][3] *= al_hi;
        }
        uint32_t pa[4];
        pa[0] = pack_half2(sc[0][0], sc[0][1]);
        pa[1] = pack_half2(sc[0][2], sc[0][3]);
        pa[2] = pack_half2(sc[1][0], sc[1][1]);
        pa[3] = pack_half2(sc[1][2], sc[1][3]);
#pragma unroll
        for (int dd = 0; dd < HD / 16; ++dd) {
            uint32_t b0, b1, b2, b3;
            ldsm_x4_t(smem_u32(V + (kw + (lane & 7) + ((lane >> 3) & 1) * 8) * C::LDS + dd * 16 +
                               (lane >> 4) * 8),
                      b0, b1, b2, b3);
            mma_16816(o[2 * dd], pa, b0, b1);
            mma_16816(o[2 * dd + 1], pa, b2, b3);
        }
    }

    // ---- merge the four warps' states -----------------------------------
    cp_async_wait<0>();
    __syncthreads();
    l_lo += __shfl_xor_sync(0xffffffffu, l_lo, 1);
    l_lo += __shfl_xor_sync(0xffffffffu, l_lo, 2);
    l_hi += __shfl_xor_sync(0xffffffffu, l_hi, 1);
    l_hi += __shfl_xor_sync(0xffffffffu, l_hi, 2);
    float* redO = reinterpret_cast<float*>(body);                 // [warp][row][RS]
    float* redM = redO + kWarps * kRB * C::RS;                    // [warp][row]
    float* redL = redM + kWarps * kRB;                            // [warp][row]
    {
        float* wO = redO + warp * kRB * C::RS;
#pragma unroll
        for (int i = 0; i < HD / 8; ++i) {
            const int d = i * 8 + 2 * qd;
            wO[g * C::RS + d] = o[i][0];
            wO[g * C::RS + d + 1] = o[i][1];
            wO[(g + 8) * C::RS + d] = o[i][2];
            wO[(g + 8) * C::RS + d + 1] = o[i][3];
        }
        if (qd == 0) {
            redM[warp * kRB + g] = m_lo;
            redM[warp * kRB + g + 8] = m_hi;
            redL[warp * kRB + g] = l_lo;
            redL[warp * kRB + g + 8] = l_hi;
        }
    }
    __syncthreads();
    for (int idx = tid; idx < nrows * HD; idx += kThreads) {
        const int rr = idx / HD, d = idx - rr * HD;
        float mrow = -INFINITY;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) mrow = fmaxf(mrow, redM[w * kRB + rr]);
        const float ref = mrow == -INFINITY ? 0.f : mrow;
        float O = 0.f, L = 0.f;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) {
            const float sw = exp2f(redM[w * kRB + rr] - ref);
            O = fmaf(sw, redO[(w * kRB + rr) * C::RS + d], O);
            L = fmaf(sw, redL[w * kRB + rr], L);
        }
        const int r = row0 + rr;
        if (a.n_splits == 1) {
            a.out[(int64_t)r * HD + d] = L > 0.f ? O / L : 0.f;
        } else {
            a.part_o[((int64_t)split * a.M + r) * HD + d] = O;
            if (d == 0) a.part_ml[(int64_t)split * a.M + r] = make_float2(mrow, L);
        }
    }
    if (a.n_splits == 1) return;

    // ---- fused fix-up: the last CTA of this row block merges all splits ---
    __threadfence();
    __syncthreads();
    if (tid == 0) {
        const unsigned prev = atomicAdd(a.tickets + rb, 1u);
        s_last = prev == (unsigned)(a.n_splits - 1);
    }
    __syncthreads();
    if (!s_last) return;
    __threadfence();
    float2* sml = reinterpret_cast<float2*>(body);                // [split][row]
    float* sw = reinterpret_cast<float*>(sml + kMaxSplits * kRB); // [split][row] weights
    float* sL = sw + kMaxSplits * kRB;                            // [row]
    for (int idx = tid; idx < a.n_splits * kRB; idx += kThreads) {
        const int s = idx / kRB, rr = idx - s * kRB;
        sml[idx] = rr < nrows ? __ldcg(a.part_ml + (int64_t)s * a.M + row0 + rr)
                              : make_float2(-INFINITY, 0.f);
    }
    __syncthreads();
    if (tid < kRB) {
        float mrow = -INFINITY;
        for (int s = 0; s < a.n_splits; ++s) mrow = fmaxf(mrow, sml[s * kRB + tid].x);
        const float ref = mrow == -INFINITY ? 0.f : mrow;
        float L = 0.f;
        for (int s = 0; s < a.n_splits; ++s) {
            const float w = exp2f(sml[s * kRB + tid].x - ref);
            sw[s * kRB + tid] = w;
            L = fmaf(w, sml[s * kRB + tid].y, L);
        }
        sL[tid] = L;
    }
    __syncthreads();
    for (int idx = tid; idx < nrows * HD; idx += kThreads) {
        const int rr = idx / HD, d = idx - rr * HD;
        const int r = row0 + rr;
        float O = 0.f;
        for (int s = 0; s < a.n_splits; ++s)
            O = fmaf(sw[s * kRB + rr], __ldcg(a.part_o + ((int64_t)s * a.M + r) * HD + d), O);
        const float L = sL[rr];
        a.out[(int64_t)r * HD + d] = L > 0.f ? O / L : 0.f;
    }
    if (tid == 0) a.tickets[rb] = 0u;
}

struct Plan {
    int n_rb, n_tiles, n_splits, tiles_per_split;
};

static Plan make_plan(int M, int n_kv, int num_sms, int force_splits) {
    Plan p;
    p.n_rb = (M + kRB - 1) / kRB;
    p.n_tiles = (n_kv + kBN - 1) / kBN;
    int s = force_splits > 0 ? force_splits : (2 * num_sms + p.n_rb - 1) / p.n_rb;
    s = max(1, min(s, min(p.n_tiles, kMaxSplits)));
    p.tiles_per_split = (p.n_tiles + s - 1) / s;
    p.n_splits = (p.n_tiles + p.tiles_per_split - 1) / p.tiles_per_split;
    return p;
}

static size_t v1_workspace_bytes(int M, int hd, int n_kv) {
    const int n_tiles = (n_kv + kBN - 1) / kBN;
    const size_t splits = (size_t)min(n_tiles, kMaxSplits);
    return kWsHeader + splits * M * hd * sizeof(float) + splits * M * sizeof(float2);
}

// Tensor-core kernel workspace: [header][f16 Q rows handed from qkv_post]
// [cluster partial O][cluster partial (m, l)].
static size_t tc_q16_bytes(int M, int hd) { return ((size_t)M * hd * 2 + 1023) & ~(size_t)1023; }

// Up to kMaxClusters clusters per row tile for at most kMaxRowTilesMulti row
// tiles; more row tiles fill the GPU alone and get one cluster each.
constexpr int kMaxRowTilesMulti = 4;

static size_t tc_workspace_bytes(int M, int hd) {
    const size_t row_tiles = (size_t)(M + 127) / 128;
    const size_t slots = row_tiles * (row_tiles <= (size_t)kMaxRowTilesMulti ? tc::kMaxClusters : 1) * 128;
    return kWsHeader + tc_q16_bytes(M, hd) + slots * hd * sizeof(float) + slots * sizeof(float2);
}

// merge-kernel mode: [header][f16 Q rows][split O [row_tiles][splits][128][hd]][split (m, l)]
static size_t tc_merge_fixed_bytes(int M, int hd) { return kWsHeader + tc_q16_bytes(M, hd); }
static size_t tc_merge_split_bytes(int M, int hd) {      // per split of every row tile
    return (size_t)((M + 127) / 128) * 128 * (hd * sizeof(float) + sizeof(float2));
}
static int tc_merge_max_splits(int M) { return tc::kMaxMergeSplits / ((M + 127) / 128); }
static size_t tc_merge_workspace_bytes(int M, int hd) {
    return tc_merge_fixed_bytes(M, hd) + (size_t)tc_merge_max_splits(M) * tc_merge_split_bytes(M, hd);
}

// The kernel with the KV tile on the MMA's M side: M <= 64 decode rows, hd 128
// or 256, library-chosen clusters and merge. One KV split of 128-key tiles per
// SM; the split count is cut to what the workspace holds (a single split
// needs no partial states).
static bool sw_shape_ok(int n_tok, int n_head, int hd) {
    return (hd == 128 || hd == 256) && n_tok <= kMaskWin && (int64_t)n_tok * n_head <= sw::kMaxRows;
}
// The library's choice of the keys-on-M kernel and its slice size (measured
// on GB300, graph replay of fused calls, against the 128-row kernel):
//  (a) 16-row slices when the KV range is short: n_kv >= 1024 and
//      ceil(M/16) * n_kv <= 32768 at hd 256, <= 16384 at hd 128 (the slices'
//      repeated reads of each K/V tile, served by L2, stay cheaper than the
//      128-row kernel's split states): at hd 256 4-20 % faster up to the
//      limit (128 rows / 4096 keys 12.42 vs 12.95 us, 64 / 8192 12.57 vs
//      13.63, 32 / 16384 12.86 vs 13.69), slower past it (128 / 8192 16.01 vs
//      14.58); at hd 128 the limit is 16384 (128 / 4096: 10.62 vs 10.23);
//      below 1024 keys the 128-row kernel's short call wins;
//  (b) one slice of all rows for M <= 32 and n_kv >= max(1024, 256 M):
//      10-25 % faster on long KV;
// else the 128-row kernel (32-row slices for 33-64 rows at hd 128 were 3-7 %
// faster once, and tie or lose since the merge kernel takes 5 splits per
// warp there: 64 rows / 65536 keys 17.76 vs 17.28 us). Returns the rows per
// slice, or 0 for layout 1.
static constexpr int kSwShortKeys = 1024;
static int64_t sw_short_work(int hd) { return hd == 256 ? 32768 : 16384; }
static int auto_sw_rows(int n_tok, int n_head, int hd, int n_kv) {
    if (!sw_shape_ok(n_tok, n_head, hd)) return 0;
    const int M = n_tok * n_head;
    if (n_kv >= kSwShortKeys && (int64_t)((M + 15) / 16) * n_kv <= sw_short_work(hd)) return 16;
    if (M <= 32 && n_kv >= kSwShortKeys && n_kv >= 256 * M) return sw::rows_n(M);
    return 0;
}
// Kernel of a call: 1 = 128-row query tiles (fr_attn_tc.cu, or the mma.sync
// engine), 2 = keys on M (fr_attn_sw.cu). A forced layout 2 is validated by
// the caller.
static int pick_layout(int n_tok, int n_head, int hd, int n_kv, const fr_attn_opts& o) {
    if (o.engine != 0) return 1;
    if (o.layout == 2) return 2;
    if (o.layout == 1 || o.force_cluster != 0 || o.merge_mode == 1) return 1;
    return auto_sw_rows(n_tok, n_head, hd, n_kv) > 0 ? 2 : 1;
}

// Smallest workspace the plan a call with these options takes accepts: the
// keys-on-M kernel needs only the header and the f16 Q slot (it cuts its split
// count to what the workspace holds); the 128-row kernel its in-launch merge
// plan; the mma.sync engine's needs count for the shapes it takes.
static size_t workspace_bytes_for(int n_tok, int n_head, int hd, int n_kv, const fr_attn_opts& o) {
    const int M = n_tok * n_head;
    if (pick_layout(n_tok, n_head, hd, n_kv, o) != 1) return kWsHeader + tc_q16_bytes(M, hd);
    const size_t b = tc_workspace_bytes(M, hd);
    if (!decode_shape(n_tok, n_head)) return b;
    const size_t a = v1_workspace_bytes(M, hd, n_kv);
    return a > b ? a : b;
}

// Splits and cluster size of the tensor-core kernel. One 128-row tile per
// ceil(M/128); splits of a row tile form clusters of C CTAs; at most as many
// CTAs as are co-resident for that cluster size (1 CTA per SM).
struct TcPlan {
    int row_tiles, n_tiles, C, n_clusters, splits, tiles_per_split;
    int bn;                // keys per KV tile
    int merge_kernel;      // 1: separate merge kernel (C == 1, splits over the whole GPU)
};

static TcPlan make_tc_plan(int M, int hd, int n_kv, int num_sms, int force_splits, int force_cluster) {
    TcPlan p;
    p.row_tiles = (M + 127) / 128;
    const int bn = tc::tile_keys(hd, n_kv, p.row_tiles, num_sms);
    p.bn = bn;
    p.n_tiles = (n_kv + bn - 1) / bn;
    // clusters of 8 for one row tile; with several row tiles (whose CTAs share
    // each K/V tile through L2) clusters of 4, which fit more CTAs per GPU
    int C = force_cluster > 0 ? force_cluster : (p.row_tiles > 1 ? 4 : 8);
    while (C > 1 && C > p.n_tiles) C >>= 1;
    int n_cl;
    if (force_splits > 0) {
        n_cl = (force_splits + C - 1) / C;
    } else {
        // co-resident CTAs at one CTA per SM for this cluster size
        const int budget = C >= 8 ? (num_sms * 120) / 152 : (C == 4 ? (num_sms * 144) / 152 : num_sms);
        n_cl = budget / (p.row_tiles * C);
        // at least two KV tiles per CTA: below that the merge costs more than
        // the extra streaming
        n_cl = min(n_cl, (p.n_tiles + 2 * C - 1) / (2 * C));
    }
    n_cl = max(1, min(n_cl, min(tc::kMaxClusters, (p.n_tiles + C - 1) / C)));
    if (p.row_tiles > kMaxRowTilesMulti) n_cl = 1;   // many row tiles fill the GPU without more splits
    int S = C * n_cl;
    p.tiles_per_split = (p.n_tiles + S - 1) / S;
    // drop clusters that would get no tile at all
    const int used = (p.n_tiles + p.tiles_per_split - 1) / p.tiles_per_split;
    n_cl = max(1, (used + C - 1) / C);
    p.C = C;
    p.n_clusters = n_cl;
    p.splits = C * n_cl;
    p.merge_kernel = 0;
    return p;
}

// Beyond two splits the in-launch merge (DSMEM pushes at a few tens of GB/s
// per SM, then the last CTA per slice reading every cluster's slice) costs
// more than a second launch; then every SM takes one split without clusters
// and a separate merge kernel reduces the states with the whole GPU. The
// split count is cut to what the workspace holds; in the automatic choice a
// workspace too small for the full count keeps the in-launch plan.
static TcPlan choose_tc_plan(int M, int hd, int n_kv, int num_sms, const fr_attn_opts& o, size_t ws_bytes,
                             bool* ok) {
    TcPlan p = make_tc_plan(M, hd, n_kv, num_sms, o.force_splits, o.force_cluster);
    *ok = true;
    bool use;
    if (o.merge_mode == 2) use = true;
    else if (o.merge_mode == 1 || o.force_cluster != 0) use = false;
    else use = p.splits > 2;
    if (!use) return p;
    const int cap = tc_merge_max_splits(M);
    if (cap < 1) {                                    // more row tiles than split slots
        if (o.merge_mode == 2) *ok = false;
        return p;
    }
    int S = o.force_splits > 0 ? o.force_splits : max(1, num_sms / p.row_tiles);
    S = max(1, min(S, min(cap, p.n_tiles)));
    const size_t fixed = tc_merge_fixed_bytes(M, hd);
    const int fit = ws_bytes > fixed ? (int)min((size_t)cap, (ws_bytes - fixed) / tc_merge_split_bytes(M, hd)) : 0;
    if (fit < S) {
        if (o.merge_mode != 2) return p;
        if (o.force_splits > 0 || fit < 1) {
            *ok = false;
            return p;
        }
        S = fit;
    }
    p.tiles_per_split = (p.n_tiles + S - 1) / S;
    p.splits = (p.n_tiles + p.tiles_per_split - 1) / p.tiles_per_split;
    p.C = 1;
    p.n_clusters = p.splits;
    p.merge_kernel = 1;
    return p;
}

static size_t sw_split_bytes(int M, int hd) { return (size_t)M * (hd * sizeof(float) + sizeof(float2)); }

// Splits cover equal key ranges in multiples of 16 keys, at least 128 (so every
// SM gets a share even when the 128-key tiles do not divide evenly); a split's
// last tile may be short, its keys past the range masked.
struct SwPlan {
    int splits, keys_per_split;
    int nq, slices;        // rows per slice (the MMA's N) and slices per split
};

// Rows per slice: the caller's choice (16, 32 or 64), else the library's
// (auto_sw_rows), else (layout 2 forced where the library would not pick it)
// all rows in one slice up to 64 and 32-row slices beyond.
static int sw_slice_rows(int n_tok, int n_head, int hd, int n_kv, const fr_attn_opts& o) {
    if (o.slice_rows > 0) return o.slice_rows;
    const int a = auto_sw_rows(n_tok, n_head, hd, n_kv);
    if (a > 0) return a;
    const int M = n_tok * n_head;
    return M <= sw::kMaxSliceRows ? sw::rows_n(M) : 32;
}

static SwPlan make_sw_plan(int n_tok, int n_head, int hd, int n_kv, int num_sms, const fr_attn_opts& o,
                           size_t ws_bytes) {
    SwPlan p;
    const int M = n_tok * n_head;
    p.nq = sw_slice_rows(n_tok, n_head, hd, n_kv, o);
    p.slices = (M + p.nq - 1) / p.nq;
    num_sms = max(1, num_sms / p.slices);                 // one CTA per SM: KV splits per slice
    const int force_splits = o.force_splits;
    const int units = (n_kv + 15) / 16;
    int S = force_splits > 0 ? force_splits : num_sms;
    S = max(1, min(S, min(units, min(num_sms, tc::kMaxMergeSplits))));
    if (S > 1) {
        const size_t fixed = kWsHeader + tc_q16_bytes(M, hd);
        const size_t fit = ws_bytes > fixed ? (ws_bytes - fixed) / sw_split_bytes(M, hd) : 0;
        if ((size_t)S > fit) S = fit > 1 ? (int)fit : 1;
    }
    // at least one full 128-key tile per split: below that a split still loads
    // a whole tile and adds a state to merge
    p.keys_per_split = max((units + S - 1) / S * 16, min(128, units * 16));
    p.splits = (n_kv + p.keys_per_split - 1) / p.keys_per_split;
    return p;
}

template <int HD>
static cudaError_t ensure_smem_attr(int dev) {
    static unsigned long long done = 0ull;     // one bit per device (idempotent)
    if (dev < 64 && (__atomic_load_n(&done, __ATOMIC_ACQUIRE) >> dev & 1ull)) return cudaSuccess;
    cudaError_t e = cudaFuncSetAttribute(attn_v1_kernel<HD>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         V1Cfg<HD>::SMEM);
    if (e == cudaSuccess && dev < 64) __atomic_fetch_or(&done, 1ull << dev, __ATOMIC_RELEASE);
    return e;
}

template <int HD>
static fr_status launch_v1(const AttnArgs& a, const RopeTable& tb, const Plan& p, cudaStream_t st) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return FR_ERR_CUDA;
    if (ensure_smem_attr<HD>(dev) != cudaSuccess) return FR_ERR_CUDA;
    dim3 grid(p.n_rb, p.n_splits);
    attn_v1_kernel<HD><<<grid, kThreads, V1Cfg<HD>::SMEM, st>>>(a, tb);
    return cudaGetLastError() == cudaSuccess ? FR_OK : FR_ERR_CUDA;
}

static fr_status decode_attn_impl(const uint16_t* q16, const float* q, int64_t q_tok_stride,
                                  const int32_t* pos, const fr_rope_params* rp, float q_scale,
                                  const uint16_t* k, int64_t k_rs, const uint16_t* v, int64_t v_rs,
                                  const uint16_t* mask, int64_t m_rs, int n_tok, int n_head, int hd,
                                  int n_kv, float kq_scale, float* out, void* ws, size_t ws_bytes,
                                  const fr_attn_opts* opts, cudaStream_t stream) {
    fr_attn_opts o;
    memset(&o, 0, sizeof(o));
    if (opts) o = *opts;
    if (o.engine < 0 || o.engine > 1 || o.force_splits < 0 || o.wait_probe_iters < 0) return FR_ERR_INVALID_ARG;
    if (o.merge_mode < 0 || o.merge_mode > 2 || o.layout < 0 || o.layout > 2) return FR_ERR_INVALID_ARG;
    if (o.slice_rows != 0 && o.slice_rows != 16 && o.slice_rows != 32 && o.slice_rows != 64) return FR_ERR_INVALID_ARG;
    if (o.layout == 2 && (o.engine != 0 || !sw_shape_ok(n_tok, n_head, hd))) return FR_ERR_UNSUPPORTED;
    if (o.force_cluster != 0 && o.force_cluster != 1 && o.force_cluster != 2 && o.force_cluster != 4 &&
        o.force_cluster != 8)
        return FR_ERR_INVALID_ARG;
    if (!k || !v || !out || !ws) return FR_ERR_INVALID_ARG;
    if (n_tok < 1 || n_head < 1 || n_kv < 1) return FR_ERR_INVALID_ARG;
    if (hd != 64 && hd != 128 && hd != 256) return FR_ERR_UNSUPPORTED;
    if (!tc_shape_ok(n_tok, n_head)) return FR_ERR_UNSUPPORTED;
    if (o.engine == 1 && !decode_shape(n_tok, n_head)) return FR_ERR_UNSUPPORTED;
    if (n_kv > (1 << 26)) return FR_ERR_UNSUPPORTED;
    if (!isfinite(kq_scale)) return FR_ERR_INVALID_ARG;
    if (k_rs < hd || (k_rs & 7) || v_rs < hd || (v_rs & 7)) return FR_ERR_INVALID_ARG;
    if (!aligned16(k) || !aligned16(v) || !aligned16(out) || !aligned16(ws)) return FR_ERR_INVALID_ARG;
    if (mask && (m_rs < n_kv || (m_rs & 7) || !aligned16(mask))) return FR_ERR_INVALID_ARG;
    RopeTable tb;
    memset(&tb, 0, sizeof(tb));
    if (q16) {
        if (!aligned16(q16)) return FR_ERR_INVALID_ARG;
    } else {
        if (!q || !pos || !rp) return FR_ERR_INVALID_ARG;
        if (!aligned16(q) || q_tok_stride < (int64_t)n_head * hd || (q_tok_stride & 3))
            return FR_ERR_INVALID_ARG;
        if (!build_rope_table(rp, resolve_q_scale(q_scale, hd), hd, &tb)) return FR_ERR_INVALID_ARG;
    }
    const int M = n_tok * n_head;
    if (ws_bytes < workspace_bytes_for(n_tok, n_head, hd, n_kv, o)) return FR_ERR_WORKSPACE;

    int dev = 0, sms = 152;
    if (cudaGetDevice(&dev) != cudaSuccess) return FR_ERR_CUDA;
    // every buffer must be memory of the current GPU (not host memory, not a peer's)
    if (!device_ptr_ok(k, dev) || !device_ptr_ok(v, dev) || !device_ptr_ok(out, dev) || !device_ptr_ok(ws, dev) ||
        (mask && !device_ptr_ok(mask, dev)) || (q16 && !device_ptr_ok(q16, dev)) ||
        (!q16 && (!device_ptr_ok(q, dev) || !device_ptr_ok(pos, dev))))
        return FR_ERR_INVALID_ARG;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return FR_ERR_CUDA;
    unsigned char* w = static_cast<unsigned char*>(ws);

    if (pick_layout(n_tok, n_head, hd, n_kv, o) == 2) {
        const SwPlan p = make_sw_plan(n_tok, n_head, hd, n_kv, sms, o, ws_bytes);
        sw::SwLaunch L;
        memset(&L, 0, sizeof(L));
        sw::SwArgs& a = L.args;
        unsigned char* qslot = w + kWsHeader;
        unsigned char* parts = qslot + tc_q16_bytes(M, hd);
        if (q16) {
            L.q16 = q16;
        } else {
            // qkv_post inside the attention kernel: one launch per call
            a.rope_in_kernel = 1;
            a.q = q;
            a.q_tok_stride = q_tok_stride;
            a.pos = pos;
            L.tb = tb;
            L.pdl = true;
        }
        a.out = out;
        a.status = reinterpret_cast<unsigned*>(w);
        a.part_o = reinterpret_cast<float*>(parts);
        a.part_ml = reinterpret_cast<float2*>(parts + (size_t)p.splits * M * hd * sizeof(float));
        a.has_mask = mask != nullptr;
        a.n_tok = n_tok;
        a.n_head = n_head;
        a.M = M;
        a.n_kv = n_kv;
        a.keys_per_split = p.keys_per_split;
        a.splits = p.splits;
        a.rstride = M;
        a.barrier = reinterpret_cast<unsigned*>(w + kWsSwBarrier);
        a.early_dep = 1;                     // at most one CTA per SM: one wave
        a.kq_log2 = kq_scale * kLog2e;
        a.wait_limit_ns = tc::kWaitLimitNs;
        a.probe_iters = (uint32_t)o.wait_probe_iters;
        L.k = k;
        L.v = v;
        L.mask = mask;
        L.k_rs = k_rs;
        L.v_rs = v_rs;
        L.m_rs = m_rs;
        a.slices = p.slices;
        return sw::launch_sw(L, hd, p.nq, stream);     // the split merge happens inside the launch
    }

    if (o.engine == 0) {
        bool plan_ok = true;
        const TcPlan p = choose_tc_plan(M, hd, n_kv, sms, o, ws_bytes, &plan_ok);
        if (!plan_ok) return FR_ERR_WORKSPACE;
        const size_t slots = (size_t)p.row_tiles * (p.merge_kernel ? p.splits : p.n_clusters) * 128;
        tc::TcLaunch L;
        memset(&L, 0, sizeof(L));
        tc::TcArgs& a = L.args;
        unsigned char* qslot = w + kWsHeader;
        unsigned char* parts = qslot + tc_q16_bytes(M, hd);
        if (q16) {
            a.q16 = reinterpret_cast<const __half*>(q16);
        } else {
            // qkv_post hands its f16 rows to the attention through the workspace
            const fr_status st = launch_qkv_post(q, q_tok_stride, pos, n_tok, n_head, hd, tb,
                                                 reinterpret_cast<uint16_t*>(qslot), nullptr, stream);
            if (st != FR_OK) return st;
            a.q16 = reinterpret_cast<const __half*>(qslot);
            L.pdl = true;
        }
        a.out = out;
        a.status = reinterpret_cast<unsigned*>(w);
        a.tickets = reinterpret_cast<unsigned*>(w + kWsTickets);
        a.part_o = reinterpret_cast<float*>(parts);
        a.part_ml = reinterpret_cast<float2*>(parts + slots * hd * sizeof(float));
        a.has_mask = mask != nullptr;
        a.n_tok = n_tok;
        a.n_head = n_head;
        a.M = M;
        a.n_kv = n_kv;
        a.n_tiles = p.n_tiles;
        a.tiles_per_split = p.tiles_per_split;
        a.n_clusters = p.n_clusters;
        a.C = p.C;
        a.merge_kernel = p.merge_kernel;
        {   // one wave: at one CTA per SM, the co-resident CTAs for this cluster size
            const int cap = p.C >= 8 ? (sms * 120) / 152 : (p.C == 4 ? (sms * 144) / 152 : sms);
            a.early_dep = p.row_tiles * p.splits <= cap ? 1 : 0;
        }
        a.splits = p.splits;
        a.kq_log2 = kq_scale * kLog2e;
        a.wait_limit_ns = tc::kWaitLimitNs;
        a.probe_iters = (uint32_t)o.wait_probe_iters;
        L.k = k;
        L.v = v;
        L.mask = mask;
        L.k_rs = k_rs;
        L.v_rs = v_rs;
        L.m_rs = m_rs;
        L.row_tiles = p.row_tiles;
        L.splits = p.splits;
        L.bn = p.bn;
        const fr_status st = tc::launch_tc(L, hd, stream);
        if (st != FR_OK || !p.merge_kernel) return st;
        return tc::launch_merge(a.part_o, a.part_ml, out, M, p.splits, hd, 128, a.status, stream);
    }

    const Plan p = make_plan(M, n_kv, sms, o.force_splits);
    const size_t splits_cap = (size_t)min(p.n_tiles, kMaxSplits);
    AttnArgs a;
    a.q16 = reinterpret_cast<const __half*>(q16);
    a.q = q;
    a.q_tok_stride = q_tok_stride;
    a.pos = pos;
    a.k = reinterpret_cast<const __half*>(k);
    a.k_rs = k_rs;
    a.v = reinterpret_cast<const __half*>(v);
    a.v_rs = v_rs;
    a.mask = reinterpret_cast<const __half*>(mask);
    a.m_rs = m_rs;
    a.out = out;
    a.tickets = reinterpret_cast<unsigned*>(w + kWsTickets);
    a.part_o = reinterpret_cast<float*>(w + kWsHeader);
    a.part_ml = reinterpret_cast<float2*>(w + kWsHeader + splits_cap * M * hd * sizeof(float));
    a.n_tok = n_tok;
    a.n_head = n_head;
    a.M = M;
    a.n_kv = n_kv;
    a.n_tiles = p.n_tiles;
    a.n_splits = p.n_splits;
    a.tiles_per_split = p.tiles_per_split;
    a.kq_log2 = kq_scale * kLog2e;
    switch (hd) {
        case 64: return launch_v1<64>(a, tb, p, stream);
        case 128: return launch_v1<128>(a, tb, p, stream);
        default: return launch_v1<256>(a, tb, p, stream);
    }
}

}  // namespace fr

using namespace fr;

extern "C" size_t fr_decode_attn_workspace_size(int n_tok, int n_head, int hd, int n_kv) {
    if (!tc_shape_ok(n_tok, n_head)) return 0;
    if ((hd != 64 && hd != 128 && hd != 256) || n_kv < 1 || n_kv > (1 << 26)) return 0;
    const int M = n_tok * n_head;
    // room for every plan, forced ones and the merge-kernel one included
    fr_attn_opts o;
    memset(&o, 0, sizeof(o));
    o.layout = 1;                        // the 128-row kernel's in-launch plan (and engine 1's)
    const size_t base = workspace_bytes_for(n_tok, n_head, hd, n_kv, o);
    const size_t merge = tc_merge_max_splits(M) >= 1 ? tc_merge_workspace_bytes(M, hd) : 0;
    const size_t sw_full = sw_shape_ok(n_tok, n_head, hd)
                               ? kWsHeader + tc_q16_bytes(M, hd) + (size_t)tc::kMaxMergeSplits * sw_split_bytes(M, hd)
                               : 0;
    size_t r = merge > base ? merge : base;
    return sw_full > r ? sw_full : r;
}

extern "C" fr_status fr_decode_attn_plan(int n_tok, int n_head, int hd, int n_kv, int fused_qkv_post,
                                         size_t workspace_bytes, const fr_attn_opts* opts, fr_attn_plan* plan) {
    if (!plan) return FR_ERR_INVALID_ARG;
    if (fr_decode_attn_workspace_size(n_tok, n_head, hd, n_kv) == 0) return FR_ERR_UNSUPPORTED;
    fr_attn_opts o;
    memset(&o, 0, sizeof(o));
    if (opts) o = *opts;
    if (o.engine < 0 || o.engine > 1 || o.force_splits < 0 || o.merge_mode < 0 || o.merge_mode > 2 ||
        o.layout < 0 || o.layout > 2 ||
        (o.slice_rows != 0 && o.slice_rows != 16 && o.slice_rows != 32 && o.slice_rows != 64))
        return FR_ERR_INVALID_ARG;
    if (o.layout == 2 && (o.engine != 0 || !sw_shape_ok(n_tok, n_head, hd))) return FR_ERR_UNSUPPORTED;
    if (o.force_cluster != 0 && o.force_cluster != 1 && o.force_cluster != 2 && o.force_cluster != 4 &&
        o.force_cluster != 8)
        return FR_ERR_INVALID_ARG;
    const int M = n_tok * n_head;
    if (o.engine == 1 && !decode_shape(n_tok, n_head)) return FR_ERR_UNSUPPORTED;
    if (workspace_bytes < workspace_bytes_for(n_tok, n_head, hd, n_kv, o)) return FR_ERR_WORKSPACE;
    int dev = 0, sms = 152;
    if (cudaGetDevice(&dev) != cudaSuccess) return FR_ERR_CUDA;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return FR_ERR_CUDA;
    memset(plan, 0, sizeof(*plan));
    plan->engine = o.engine;
    plan->row_slices = 1;
    plan->layout = pick_layout(n_tok, n_head, hd, n_kv, o);
    if (plan->layout == 2) {
        const SwPlan p = make_sw_plan(n_tok, n_head, hd, n_kv, sms, o, workspace_bytes);
        plan->row_tiles = 1;
        plan->splits = p.splits;
        plan->cluster = 1;
        plan->merge_kernel = 0;              // merged inside the launch
        plan->keys_on_m = 1;
        plan->row_slices = p.slices;
    } else if (o.engine == 0) {
        bool ok = true;
        const TcPlan p = choose_tc_plan(M, hd, n_kv, sms, o, workspace_bytes, &ok);
        if (!ok) return FR_ERR_WORKSPACE;
        plan->row_tiles = p.row_tiles;
        plan->splits = p.splits;
        plan->cluster = p.C;
        plan->merge_kernel = p.merge_kernel;
    } else {
        const Plan p = make_plan(M, n_kv, sms, o.force_splits);
        plan->row_tiles = p.n_rb;
        plan->splits = p.n_splits;
        plan->cluster = 1;
        plan->merge_kernel = 0;
    }
    // the keys-on-M kernel (layout 2) ropes the Q rows itself: no separate
    // qkv_post launch
    plan->launches = (fused_qkv_post && o.engine == 0 && plan->layout == 1 ? 1 : 0) + 1 + plan->merge_kernel;
    return FR_OK;
}

namespace fr {
size_t decode_attn_min_workspace_bytes(int n_tok, int n_head, int hd, int n_kv) {
    if (fr_decode_attn_workspace_size(n_tok, n_head, hd, n_kv) == 0) return 0;
    fr_attn_opts o;
    memset(&o, 0, sizeof(o));
    return workspace_bytes_for(n_tok, n_head, hd, n_kv, o);
}
}  // namespace fr

extern "C" fr_status fr_workspace_init(void* ws, size_t ws_bytes, cudaStream_t stream) {
    if (!ws || ws_bytes < kWsHeader) return FR_ERR_INVALID_ARG;
    return cudaMemsetAsync(ws, 0, ws_bytes, stream) == cudaSuccess ? FR_OK : FR_ERR_CUDA;
}

extern "C" fr_status fr_workspace_check(void* ws, cudaStream_t stream) {
    if (!ws) return FR_ERR_INVALID_ARG;
    unsigned word = 0;
    if (cudaMemcpyAsync(&word, ws, sizeof(word), cudaMemcpyDeviceToHost, stream) != cudaSuccess)
        return FR_ERR_CUDA;
    if (cudaStreamSynchronize(stream) != cudaSuccess) return FR_ERR_CUDA;
    if (word == 0) return FR_OK;
    if (cudaMemsetAsync(ws, 0, sizeof(word), stream) != cudaSuccess) return FR_ERR_CUDA;
    return FR_ERR_DEVICE_TIMEOUT;
}

extern "C" fr_status fr_decode_attn(const uint16_t* q16, const float* q, int64_t q_tok_stride,
                                    const int32_t* pos, const fr_rope_params* rp, float q_scale,
                                    const uint16_t* k, int64_t k_row_stride, const uint16_t* v,
                                    int64_t v_row_stride, const uint16_t* mask,
                                    int64_t mask_row_stride, int n_tok, int n_head, int hd, int n_kv,
                                    float kq_scale, float* out, void* workspace,
                                    size_t workspace_bytes, cudaStream_t stream) {
    return decode_attn_impl(q16, q, q_tok_stride, pos, rp, q_scale, k, k_row_stride, v, v_row_stride,
                            mask, mask_row_stride, n_tok, n_head, hd, n_kv, kq_scale, out, workspace,
                            workspace_bytes, nullptr, stream);
}

extern "C" fr_status fr_decode_attn_ex(const uint16_t* q16, const float* q, int64_t q_tok_stride,
                                       const int32_t* pos, const fr_rope_params* rp, float q_scale,
                                       const uint16_t* k, int64_t k_row_stride, const uint16_t* v,
                                       int64_t v_row_stride, const uint16_t* mask, int64_t mask_row_stride,
                                       int n_tok, int n_head, int hd, int n_kv, float kq_scale, float* out,
                                       void* workspace, size_t workspace_bytes, const fr_attn_opts* opts,
                                       cudaStream_t stream) {
    return decode_attn_impl(q16, q, q_tok_stride, pos, rp, q_scale, k, k_row_stride, v, v_row_stride,
                            mask, mask_row_stride, n_tok, n_head, hd, n_kv, kq_scale, out, workspace,
                            workspace_bytes, opts, stream);
}
