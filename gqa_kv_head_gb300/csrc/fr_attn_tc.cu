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
// Warp roles (192 threads):
//   warps 0-3  softmax: thread i owns TMEM lane i = query row i. Reads its S
//              row, applies kq_scale and the mask, keeps the running max m and
//              sum l (lazy rescale of O only when the max grows by > 2^8), and
//              writes P back into TMEM as two f16 terms, P = P_hi + P_lo
//              (P_lo = f16(p - P_hi)), so the weights keep ~22 bits and the
//              softmax stays fp32-accurate even where |V| is large.
//   warp 4     TMA producer: K, V and mask tiles into a ring of stages.
//   warp 5     MMA issuer: S_j = Q K_j^T (SS form, S double-buffered in TMEM),
//              O += P_hi,j V_j + P_lo,j V_j (A operand from TMEM, V read
//              MN-major), commits.
// Splits of one row tile form thread-block clusters of C CTAs (cluster dim y):
//   prologue   each CTA ropes 1/C of the Q rows (fused qkv_post) and stores
//              the f16 rows into every peer's shared memory (DSMEM); with given
//              f16 Q rows each CTA multicasts its 1/C slice by TMA instead.
//   epilogue   the C partial states (m, l, O) are merged over DSMEM; CTA rank c
//              owns rows [c*128/C, (c+1)*128/C). With several clusters per row
//              tile the merged slices go to the workspace and the last CTA to
//              arrive for each (row tile, rank) slice merges them (atomic ticket,
//              reset afterwards). No CTA ever waits for another cluster.
// Every mbarrier wait is bounded; a wait that gives up sets the workspace's
// status word and the CTA still runs through every cluster barrier, drains
// its copies and frees its TMEM.
#include <math.h>
#include <string.h>

#include <cudaTypedefs.h>

#include "fr_attn.h"
#include "fr_common.cuh"
#include "fr_sm100.cuh"

namespace fr {
namespace tc {

using namespace sm100;

constexpr int kRows = 128;
constexpr int kThreads = 192;
constexpr int kProdWarp = 4;
constexpr int kMmaWarp = 5;
constexpr float kTau = 8.0f;
constexpr float kLog2e = 1.4426950408889634f;
constexpr uint32_t kTmemCols = 512;

template <int HD>
struct Cfg {
    static constexpr int BN = 64;                          // keys per tile
    static constexpr int STAGES = HD == 256 ? 2 : (HD == 128 ? 5 : 8);
    static constexpr int NB = HD / 64;                     // 128-byte column boxes per row
    static constexpr int Q_BYTES = kRows * HD * 2;
    static constexpr int Q_BOX = kRows * 128;              // one 64-column box of Q
    static constexpr int KV_BOX = BN * 128;                // one 64-column box of a K or V tile
    static constexpr int K_BYTES = BN * HD * 2;
    static constexpr int MASK_BOX = 2048;                  // <= 16 rows x 128 B, 1024-aligned slots
    static constexpr int MASK_BYTES = (BN / 64) * MASK_BOX;
    static constexpr int STAGE_BYTES = 2 * K_BYTES + MASK_BYTES;
    static constexpr int BODY = Q_BYTES + STAGES * STAGE_BYTES;
    static constexpr int RED_STRIDE = HD + 4;              // fp32 staging row stride
    static constexpr int RED_BYTES = kRows * RED_STRIDE * 4 + kRows * 8;
    static constexpr int DATA = BODY > RED_BYTES ? BODY : RED_BYTES;
    static constexpr int AUX = 16384;                      // cos/sin table, then merge weights
    static constexpr int BAR_OFF = DATA + AUX;
    // mbarrier slots (8 bytes each), laid out from STAGES
    static constexpr int B_FULL = 0, B_EMPTY = STAGES, B_SFULL = 2 * STAGES, B_PFULL = 2 * STAGES + 2,
                         B_ODONE = 2 * STAGES + 4, B_QFULL = 2 * STAGES + 5, B_PROBE = 2 * STAGES + 6,
                         B_MMADONE = 2 * STAGES + 7, N_BARS = 2 * STAGES + 8;
    static constexpr int TMEM_SLOT = 32 * 8;               // TMEM base word after 32 barrier slots
    static_assert(N_BARS <= 32, "barrier slots");
    static constexpr int SMEM = BAR_OFF + 512 + 1024;      // barriers + TMEM word, + alignment slack
    // TMEM columns
    static constexpr int TM_O = 0;
    static constexpr int TM_S = HD;
    static constexpr int TM_P = HD + 2 * BN;               // P_hi, 2 x BN/2 columns
    static constexpr int TM_PL = TM_P + BN;                // P_lo, 2 x BN/2 columns
    static_assert(TM_PL + BN <= (int)kTmemCols, "TMEM budget");
    static_assert(STAGE_BYTES % 1024 == 0 && Q_BYTES % 1024 == 0, "1024-B alignment of swizzled tiles");
    static_assert(SMEM <= 232448, "shared memory budget");
};

struct Maps {
    CUtensorMap k, v, mask, q16;
};

__device__ __forceinline__ void record_timeout(unsigned* status, unsigned bit) {
    atomicOr(status, bit);
}

template <int HD>
__global__ void __launch_bounds__(kThreads, 1)
attn_tc_kernel(const __grid_constant__ TcArgs a, const __grid_constant__ RopeTable tb,
               const __grid_constant__ Maps mp) {
    using C = Cfg<HD>;
    constexpr int BN = C::BN;
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    unsigned char* sm = reinterpret_cast<unsigned char*>(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    unsigned char* sQ = sm;
    unsigned char* sStage = sm + C::Q_BYTES;
    float* sRedO = reinterpret_cast<float*>(sm);                                   // after the KV loop
    float2* sRedML = reinterpret_cast<float2*>(sm + kRows * C::RED_STRIDE * 4);
    float2* sCS = reinterpret_cast<float2*>(sm + C::DATA);                        // [16][128] (cos, sin)
    float* sW = reinterpret_cast<float*>(sm + C::DATA);                           // merge weights (later)
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
    auto sK = [&](int s) { return sStage + s * C::STAGE_BYTES; };
    auto sV = [&](int s) { return sStage + s * C::STAGE_BYTES + C::K_BYTES; };
    auto sMask = [&](int s) { return sStage + s * C::STAGE_BYTES + 2 * C::K_BYTES; };

    // ---- set-up ------------------------------------------------------------
    if (tid == 0) {
        for (int s = 0; s < C::STAGES; ++s) {
            mbar_init(bar(C::B_FULL + s), 1);
            mbar_init(bar(C::B_EMPTY + s), 1);
        }
        mbar_init(bar(C::B_SFULL + 0), 1);
        mbar_init(bar(C::B_SFULL + 1), 1);
        mbar_init(bar(C::B_PFULL + 0), 128);
        mbar_init(bar(C::B_PFULL + 1), 128);
        mbar_init(bar(C::B_ODONE), 1);
        mbar_init(bar(C::B_QFULL), 1);
        mbar_init(bar(C::B_PROBE), 1);
        mbar_init(bar(C::B_MMADONE), 1);
        mbar_fence_init();
        if (a.q16) mbar_expect_tx(bar(C::B_QFULL), C::Q_BYTES);
        prefetch_tmap(&mp.k);
        prefetch_tmap(&mp.v);
    }
    if (warp == kMmaWarp) tmem_alloc(smem_addr(sTmemBase), kTmemCols);
    tc_fence_before();
    cluster_sync();                     // barriers of every CTA initialised
    tc_fence_after();
    const uint32_t tbase = *sTmemBase;

    // ---- prologue: the 128 Q rows as f16, SW128 K-major in every CTA --------
    const int my_r0 = (int)rank * R;
    if (a.q16) {
        if (tid == 0) {
            for (int b = 0; b < C::NB; ++b) {
                const uint32_t dst = smem_addr(sQ + b * C::Q_BOX + my_r0 * 128);
                if (CS == 1)
                    tma_load_2d(dst, &mp.q16, b * 64, row0 + my_r0, bar(C::B_QFULL));
                else
                    tma_load_2d_mc(dst, &mp.q16, b * 64, row0 + my_r0, bar(C::B_QFULL),
                                   (uint16_t)((1u << CS) - 1u));
            }
        }
    } else {
        // cos/sin of every (token, pair) the owned rows need; heads share them
        const int r_beg = my_r0, r_end = min(my_r0 + R, rows_real);
        if (r_beg < r_end) {
            const int tk0 = (row0 + r_beg) / a.n_head, tk1 = (row0 + r_end - 1) / a.n_head;
            const int ntk = tk1 - tk0 + 1;
            for (int i = tid; i < ntk * tb.half; i += kThreads) {
                const int tt = i / tb.half, pr = i - tt * tb.half;
                float c, s;
                rope_cs(__ldg(a.pos + tk0 + tt), tb.turns[pr], tb.mscale, c, s);
                sCS[tt * kMaxPairs + pr] = make_float2(c, s);
            }
            __syncthreads();
            constexpr int CH = HD / 8;
            for (int i = tid; i < (r_end - r_beg) * CH; i += kThreads) {
                const int rr = r_beg + i / CH, ch = i % CH;
                const int r = row0 + rr;
                const int t = r / a.n_head, h = r - t * a.n_head;
                const float* x = a.q + (int64_t)t * a.q_tok_stride + (int64_t)h * HD;
                const float2* cs = sCS + (t - tk0) * kMaxPairs;
                uint32_t pk[4];
#pragma unroll
                for (int e = 0; e < 8; e += 2) {
                    float y[2];
#pragma unroll
                    for (int u = 0; u < 2; ++u) {
                        const int d = ch * 8 + e + u;
                        if (d < tb.half) {
                            const float2 v = cs[d];
                            y[u] = rope_lo(x[d], x[d + tb.half], v.x, v.y, tb.q_scale);
                        } else if (d < tb.n_dims) {
                            const int p = d - tb.half;
                            const float2 v = cs[p];
                            y[u] = rope_hi(x[p], x[d], v.x, v.y, tb.q_scale);
                        } else {
                            y[u] = __fmul_rn(x[d], tb.q_scale);
                        }
                    }
                    pk[e / 2] = pack_half2(y[0], y[1]);
                }
                const int b = ch >> 3, c8 = ch & 7;
                const uint32_t dst = smem_addr(sQ + b * C::Q_BOX + (rr >> 3) * 1024 + (rr & 7) * 128 +
                                               ((c8 ^ (rr & 7)) << 4));
                const uint4 val = make_uint4(pk[0], pk[1], pk[2], pk[3]);
                for (int p = 0; p < CS; ++p) st_cluster_v4(map_rank(dst, (uint32_t)p), val);
            }
        }
        // rows >= M of this tile are zero in every CTA
        constexpr int CH = HD / 8;
        for (int i = tid; i < (kRows - rows_real) * CH; i += kThreads) {
            const int rr = rows_real + i / CH, ch = i % CH;
            const int b = ch >> 3, c8 = ch & 7;
            *reinterpret_cast<uint4*>(sQ + b * C::Q_BOX + (rr >> 3) * 1024 + (rr & 7) * 128 + ((c8 ^ (rr & 7)) << 4)) =
                make_uint4(0, 0, 0, 0);
        }
        fence_proxy_async_cta();
        fence_proxy_async_cluster();
    }
    cluster_sync();                     // Q rows (fused path) visible cluster-wide
    tc_fence_after();

    if (a.probe_iters && tid == 0) {
        // test hook: a bounded wait on a barrier nothing ever signals
        if (!mbar_wait_polls(bar(C::B_PROBE), 0, a.probe_iters)) record_timeout(a.status, 2u);
    }

    // ---- main phase ----------------------------------------------------------
    float m_ref = -INFINITY, l_sum = 0.f;
    if (warp == kProdWarp) {
        if (lane == 0) {
            const uint32_t mask_tx = a.has_mask ? (uint32_t)(BN / 64) * 128u * (uint32_t)a.n_tok : 0u;
            for (int i = 0; i < n_my; ++i) {
                const int st = i % C::STAGES;
                if (i >= C::STAGES) wait(bar(C::B_EMPTY + st), ((i / C::STAGES) - 1) & 1);
                mbar_expect_tx(bar(C::B_FULL + st), 2u * C::K_BYTES + mask_tx);
                const int j0 = (t0 + i) * BN;
#pragma unroll
                for (int b = 0; b < C::NB; ++b) {
                    tma_load_2d(smem_addr(sK(st) + b * C::KV_BOX), &mp.k, b * 64, j0, bar(C::B_FULL + st));
                    tma_load_2d(smem_addr(sV(st) + b * C::KV_BOX), &mp.v, b * 64, j0, bar(C::B_FULL + st));
                }
                if (a.has_mask) {
#pragma unroll
                    for (int mb = 0; mb < BN / 64; ++mb)
                        tma_load_2d(smem_addr(sMask(st) + mb * C::MASK_BOX), &mp.mask, j0 + mb * 64, 0,
                                    bar(C::B_FULL + st));
                }
            }
            // drain: every issued load has landed before the stage memory is reused
            // (full time limit even after a failure: no copy may outlive the CTA)
            for (int i = max(0, n_my - C::STAGES); i < n_my; ++i)
                if (!mbar_wait(bar(C::B_FULL + i % C::STAGES), (i / C::STAGES) & 1, limit))
                    record_timeout(a.status, 1u);
        }
    } else if (warp == kMmaWarp) {
        if (lane == 0) {
            // given f16 Q: every CTA's multicast slices must have landed (full limit:
            // peers write this CTA's shared memory)
            if (a.q16 && !mbar_wait(bar(C::B_QFULL), 0, limit)) record_timeout(a.status, 1u);
            tc_fence_after();
            constexpr uint32_t idS = idesc_f16_f32(kRows, BN, 0, 0);
            constexpr uint32_t idO = idesc_f16_f32(kRows, HD, 0, 1);
            const uint32_t q_base = smem_addr(sQ);
            auto issue_s = [&](int i) {
                const int st = i % C::STAGES;
                wait(bar(C::B_FULL + st), (i / C::STAGES) & 1);
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
            };
            // S_{i+1} goes ahead of PV_i only when its K tile has already landed, so
            // PV_i (which frees a stage for the producer) never waits on a load.
            int s_next = 0;
            if (n_my > 0) issue_s(s_next++);
            for (int i = 0; i < n_my; ++i) {
                if (s_next == i + 1 && s_next < n_my &&
                    mbar_test(bar(C::B_FULL + s_next % C::STAGES), (s_next / C::STAGES) & 1))
                    issue_s(s_next++);
                wait(bar(C::B_PFULL + (i & 1)), (i >> 1) & 1);
                tc_fence_after();
                const uint32_t v_base = smem_addr(sV(i % C::STAGES));
                const uint32_t p_tm = tbase + C::TM_P + (i & 1) * (BN / 2);
                const uint32_t pl_tm = tbase + C::TM_PL + (i & 1) * (BN / 2);
#pragma unroll
                for (int ks = 0; ks < BN / 16; ++ks) {
                    const uint64_t vd = sdesc_sw128(v_base + ks * 2048, C::KV_BOX, 1024);
                    mma_ts(tbase + C::TM_O, p_tm + ks * 8, vd, idO, (i > 0 || ks > 0) ? 1u : 0u);
                    mma_ts(tbase + C::TM_O, pl_tm + ks * 8, vd, idO, 1u);
                }
                mma_commit(bar(C::B_ODONE));
                mma_commit(bar(C::B_EMPTY + i % C::STAGES));
                if (s_next == i + 1 && s_next < n_my) issue_s(s_next++);
            }
            // drain: no MMA may still be running when TMEM is freed
            mma_commit(bar(C::B_MMADONE));
            if (!mbar_wait(bar(C::B_MMADONE), 0, limit)) record_timeout(a.status, 1u);
        }
    } else {
        // softmax warps: thread `tid` owns row `tid` of the tile
        const int r = tid;
        const int grow = row0 + r;
        const int t = grow < a.M ? grow / a.n_head : a.n_tok - 1;
        const bool warp_active = row0 + warp * 32 < a.M;
        const uint32_t lane_base = (uint32_t)(warp * 32) << 16;
        for (int i = 0; i < n_my; ++i) {
            wait(bar(C::B_SFULL + (i & 1)), (i >> 1) & 1);
            tc_fence_after();
            if (warp_active) {
                float x[BN];
#pragma unroll
                for (int c = 0; c < BN; c += 32)
                    tmem_ld_x32(tbase + lane_base + C::TM_S + (i & 1) * BN + c, reinterpret_cast<uint32_t*>(x + c));
                tmem_wait_ld();
                const int j0 = (t0 + i) * BN;
                const unsigned char* mk = sMask(i % C::STAGES);
                const float kq = a.kq_log2;
                if (a.has_mask) {
#pragma unroll
                    for (int c8 = 0; c8 < BN / 8; ++c8) {
                        const int mb = c8 >> 3, ch = c8 & 7;
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
                    for (int c = 0; c < BN; ++c) x[c] *= kq;
                }
                if (j0 + BN > a.n_kv) {               // ragged last tile only
#pragma unroll
                    for (int c = 0; c < BN; ++c)
                        if (j0 + c >= a.n_kv) x[c] = -INFINITY;
                }
                float mx = -INFINITY;
#pragma unroll
                for (int c = 0; c < BN; ++c) mx = fmaxf(mx, x[c]);
                float m_new = m_ref;
                if (mx > m_ref + kTau || (m_ref == -INFINITY && mx > -INFINITY)) m_new = fmaxf(mx, m_ref);
                const bool grow_ref = m_ref != -INFINITY && m_new != m_ref;
                const float alpha = grow_ref ? ex2(m_ref - m_new) : 1.f;
                if (__any_sync(0xffffffffu, grow_ref) && i > 0) {
                    // O holds PV up to tile i-1: wait for it, then rescale this warp's rows
                    wait(bar(C::B_ODONE), (i - 1) & 1);
                    tc_fence_after();
#pragma unroll 1
                    for (int c = 0; c < HD; c += 32) {
                        uint32_t o[32];
                        tmem_ld_x32(tbase + lane_base + C::TM_O + c, o);
                        tmem_wait_ld();
#pragma unroll
                        for (int u = 0; u < 32; ++u) o[u] = __float_as_uint(__uint_as_float(o[u]) * alpha);
                        tmem_st_x32(tbase + lane_base + C::TM_O + c, o);
                    }
                    tmem_wait_st();
                }
                m_ref = m_new;
                const float m_sub = m_ref == -INFINITY ? 0.f : m_ref;
                float sum = 0.f;
                uint32_t pk[BN / 2], pl[BN / 2];
#pragma unroll
                for (int c = 0; c < BN; c += 2) {
                    const float p0 = ex2(x[c] - m_sub), p1 = ex2(x[c + 1] - m_sub);
                    sum += p0 + p1;
                    const uint32_t h = pack_half2(p0, p1);
                    const float2 hf = __half22float2(*reinterpret_cast<const __half2*>(&h));
                    pk[c / 2] = h;
                    pl[c / 2] = pack_half2(p0 - hf.x, p1 - hf.y);
                }
                l_sum = fmaf(l_sum, alpha, sum);
#pragma unroll
                for (int c = 0; c < BN / 2; c += 32) {
                    tmem_st_x32(tbase + lane_base + C::TM_P + (i & 1) * (BN / 2) + c, pk + c);
                    tmem_st_x32(tbase + lane_base + C::TM_PL + (i & 1) * (BN / 2) + c, pl + c);
                }
                tmem_wait_st();
            }
            tc_fence_before();
            mbar_arrive(bar(C::B_PFULL + (i & 1)));
        }
        if (n_my > 0) {
            if (!mbar_wait(bar(C::B_ODONE), (n_my - 1) & 1, limit)) record_timeout(a.status, 1u);
            tc_fence_after();
        }
    }
    __syncthreads();                    // every async load drained, every MMA done

    // ---- stage this CTA's (m, l, O) for the cluster merge ------------------
    if (warp < 4) {
        const int r = tid;
        const uint32_t lane_base = (uint32_t)(warp * 32) << 16;
        float* dst = sRedO + r * C::RED_STRIDE;
        const bool have = n_my > 0 && row0 + warp * 32 < a.M;
#pragma unroll 1
        for (int c = 0; c < HD; c += 32) {
            uint32_t o[32];
            if (have) {
                tmem_ld_x32(tbase + lane_base + C::TM_O + c, o);
                tmem_wait_ld();
            } else {
#pragma unroll
                for (int u = 0; u < 32; ++u) o[u] = 0u;
            }
#pragma unroll
            for (int u = 0; u < 32; u += 4)
                *reinterpret_cast<uint4*>(dst + c + u) = make_uint4(o[u], o[u + 1], o[u + 2], o[u + 3]);
        }
        sRedML[r] = have ? make_float2(m_ref, l_sum) : make_float2(-INFINITY, 0.f);
    }
    tc_fence_before();
    cluster_sync();                     // every CTA's staging complete

    // ---- cluster merge of rows [rank*R, rank*R + R) -------------------------
    const int mr0 = (int)rank * R;
    const int mrows = max(0, min(R, rows_real - mr0));
    float* wts = sW;                         // [R][CS]
    float* rowM = sW + R * CS;               // [R]
    float* rowL = rowM + R;                  // [R]
    if (tid < mrows) {
        const int rr = mr0 + tid;
        float mv[8], lv[8];
        float mmax = -INFINITY;
        for (int p = 0; p < CS; ++p) {
            const float2 ml = ld_cluster_v2f(map_rank(smem_addr(sRedML + rr), (uint32_t)p));
            mv[p] = ml.x;
            lv[p] = ml.y;
            mmax = fmaxf(mmax, ml.x);
        }
        const float ref = mmax == -INFINITY ? 0.f : mmax;
        float L = 0.f;
        for (int p = 0; p < CS; ++p) {
            const float w = mv[p] == -INFINITY ? 0.f : ex2(mv[p] - ref);
            wts[tid * CS + p] = w;
            L = fmaf(w, lv[p], L);
        }
        rowM[tid] = mmax;
        rowL[tid] = L;
    }
    __syncthreads();
    const bool single = a.n_clusters == 1;
    constexpr int Q4 = HD / 4;
    for (int i = tid; i < mrows * Q4; i += kThreads) {
        const int lr = i / Q4, q4 = i - lr * Q4;
        const int rr = mr0 + lr;
        const uint32_t src = smem_addr(sRedO + rr * C::RED_STRIDE + q4 * 4);
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int p = 0; p < CS; ++p) {
            const float w = wts[lr * CS + p];
            const float4 v = ld_cluster_v4f(map_rank(src, (uint32_t)p));
            acc.x = fmaf(w, v.x, acc.x);
            acc.y = fmaf(w, v.y, acc.y);
            acc.z = fmaf(w, v.z, acc.z);
            acc.w = fmaf(w, v.w, acc.w);
        }
        const int grow = row0 + rr;
        if (single) {
            const float L = rowL[lr];
            float4 o;
            o.x = L > 0.f ? acc.x / L : 0.f;
            o.y = L > 0.f ? acc.y / L : 0.f;
            o.z = L > 0.f ? acc.z / L : 0.f;
            o.w = L > 0.f ? acc.w / L : 0.f;
            *reinterpret_cast<float4*>(a.out + (int64_t)grow * HD + q4 * 4) = o;
        } else {
            const int64_t slot = ((int64_t)rt * a.n_clusters + cl) * kRows + rr;
            *reinterpret_cast<float4*>(a.part_o + slot * HD + q4 * 4) = acc;
            if (q4 == 0) a.part_ml[slot] = make_float2(rowM[lr], rowL[lr]);
        }
    }
    cluster_sync();                     // peers finished reading this CTA's staging

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
            if (tid < mrows) {
                const int rr = mr0 + tid;
                float mmax = -INFINITY;
                for (int c2 = 0; c2 < NC; ++c2)
                    mmax = fmaxf(mmax, __ldcg(a.part_ml + ((int64_t)rt * NC + c2) * kRows + rr).x);
                const float ref = mmax == -INFINITY ? 0.f : mmax;
                float L = 0.f;
                for (int c2 = 0; c2 < NC; ++c2) {
                    const float2 ml = __ldcg(a.part_ml + ((int64_t)rt * NC + c2) * kRows + rr);
                    const float w = ml.x == -INFINITY ? 0.f : ex2(ml.x - ref);
                    w2[tid * NC + c2] = w;
                    L = fmaf(w, ml.y, L);
                }
                L2[tid] = L;
            }
            __syncthreads();
            for (int i = tid; i < mrows * Q4; i += kThreads) {
                const int lr = i / Q4, q4 = i - lr * Q4;
                const int rr = mr0 + lr;
                float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
                for (int c2 = 0; c2 < NC; ++c2) {
                    const float w = w2[lr * NC + c2];
                    const float4 v = __ldcg(reinterpret_cast<const float4*>(
                        a.part_o + (((int64_t)rt * NC + c2) * kRows + rr) * HD + q4 * 4));
                    acc.x = fmaf(w, v.x, acc.x);
                    acc.y = fmaf(w, v.y, acc.y);
                    acc.z = fmaf(w, v.z, acc.z);
                    acc.w = fmaf(w, v.w, acc.w);
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

    // ---- teardown --------------------------------------------------------------
    tc_fence_before();
    __syncthreads();
    if (warp == kMmaWarp) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tbase, kTmemCols);
    }
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

template <int HD>
static cudaError_t ensure_attr(int dev) {
    static unsigned long long done = 0ull;
    if (dev < 64 && (__atomic_load_n(&done, __ATOMIC_ACQUIRE) >> dev & 1ull)) return cudaSuccess;
    cudaError_t e = cudaFuncSetAttribute(attn_tc_kernel<HD>, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg<HD>::SMEM);
    if (e == cudaSuccess && dev < 64) __atomic_fetch_or(&done, 1ull << dev, __ATOMIC_RELEASE);
    return e;
}

int tile_keys(int hd) { return hd == 256 ? Cfg<256>::BN : (hd == 128 ? Cfg<128>::BN : Cfg<64>::BN); }

template <int HD>
static fr_status launch(const TcLaunch& L, cudaStream_t stream) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return FR_ERR_CUDA;
    if (ensure_attr<HD>(dev) != cudaSuccess) return FR_ERR_CUDA;
    Maps mp;
    memset(&mp, 0, sizeof(mp));
    const TcArgs& a = L.args;
    constexpr int BN = Cfg<HD>::BN;
    if (!encode_2d(&mp.k, L.k, HD, a.n_kv, L.k_rs, 64, BN)) return FR_ERR_CUDA;
    if (!encode_2d(&mp.v, L.v, HD, a.n_kv, L.v_rs, 64, BN)) return FR_ERR_CUDA;
    if (a.has_mask && !encode_2d(&mp.mask, L.mask, a.n_kv, a.n_tok, L.m_rs, 64, a.n_tok)) return FR_ERR_CUDA;
    if (a.q16 && !encode_2d(&mp.q16, a.q16, HD, a.M, HD, 64, kRows / a.C)) return FR_ERR_CUDA;

    cudaLaunchConfig_t cfg;
    memset(&cfg, 0, sizeof(cfg));
    cfg.gridDim = dim3(L.row_tiles, L.splits, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = Cfg<HD>::SMEM;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 1;
    attr[0].val.clusterDim.y = a.C;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaError_t e = cudaLaunchKernelEx(&cfg, attn_tc_kernel<HD>, a, L.tb, mp);
    return e == cudaSuccess ? FR_OK : FR_ERR_CUDA;
}

fr_status launch_tc(const TcLaunch& L, int hd, cudaStream_t stream) {
    switch (hd) {
        case 64: return launch<64>(L, stream);
        case 128: return launch<128>(L, stream);
        default: return launch<256>(L, stream);
    }
}

}  // namespace tc
}  // namespace fr
