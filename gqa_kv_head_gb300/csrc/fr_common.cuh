// fr_common.cuh -- pieces shared by the qkv_post kernel and the decode
// attention kernels: the RoPE table passed by value to every launch, the one
// device routine that rotates a Q element pair (so the fused and the two-call
// paths emit bit-identical f16 rows), argument checks and small PTX wrappers.
#pragma once

#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include "fr_kernels.h"

namespace fr {

constexpr int kMaxPairs = 128;     // hd 256 -> 128 rotated pairs at most
constexpr int kMaxTok = 16;        // q_tokens <= 16 (decode; the mma.sync engine's bound)
constexpr int kMaxRows = 512;      // M = n_tok * n_head (decode)
// The tcgen05 engine also takes longer query windows (prefill): each 128-row
// tile reads a window of kMaskWin consecutive tokens' mask rows, which holds
// every token of the tile when n_tok <= kMaskWin or n_head >= 8.
constexpr int kMaxTokTc = 8192;
constexpr int kMaxRowsTc = 65536;
constexpr int kMaskWin = 16;
inline bool tc_shape_ok(int n_tok, int n_head) {
    return n_tok >= 1 && n_head >= 1 && n_tok <= kMaxTokTc && (int64_t)n_tok * n_head <= kMaxRowsTc &&
           (n_tok <= kMaskWin || n_head >= 8);
}
inline bool decode_shape(int n_tok, int n_head) {
    return n_tok >= 1 && n_head >= 1 && n_tok <= kMaxTok && (int64_t)n_tok * n_head <= kMaxRows;
}

// Per-launch RoPE constants (kernel parameter, by value).
// Mode FR_ROPE_EXACT:
//   turns[i] = frac(w_i / 2pi) * 2^64, w_i = effective angle per position of
//   pair i (base^(-2i/n_dims) / ff_i times the YaRN interpolation factor). The
//   angle of pair i at integer position p is then 2pi * ((p * turns[i]) mod
//   2^64) / 2^64: the product wraps exactly modulo one turn, so large
//   positions lose no precision to the range reduction.
// Mode FR_ROPE_GGML_F32 (ggml's fp32 evaluation, one IEEE fp32 operation per
// step): theta_0 = fl(p), theta_i = fl(theta_{i-1} * theta_scale); theta_ext =
// fl(theta_i / ff_i); theta_int = fl(freq_scale * theta_ext); with YaRN,
// theta = fl(fl(theta_int * fl(1 - mix_i)) + fl(theta_ext * mix_i)).
struct RopeTable {
    uint64_t turns[kMaxPairs];   // exact mode
    float mix[kMaxPairs];        // fp32 mode: fl(ramp_i * ext_factor)
    float ff[kMaxPairs];         // fp32 mode: freq factor of pair i (1 when absent)
    float mscale;       // attn_factor (* (1 + 0.1 ln(1/freq_scale)) with YaRN)
    float q_scale;      // applied after the rotation
    float theta_scale;  // fp32 mode: fl(base ^ fl(-2/n_dims))
    float freq_scale;   // fp32 mode
    int half;           // n_dims / 2
    int n_dims;
    int mode;           // FR_ROPE_EXACT or FR_ROPE_GGML_F32
    int yarn;           // ext_factor != 0
};

// Host: validate the parameters and fill the table. Returns false if invalid.
bool build_rope_table(const fr_rope_params* rp, float q_scale, int hd, RopeTable* t);

// Host: enqueue the qkv_post kernel (arguments already validated). The kernel
// lets a programmatically dependent launch start early.
fr_status launch_qkv_post(const float* q, int64_t q_tok_stride, const int32_t* pos, int n_tok, int n_head,
                          int hd, const RopeTable& tb, uint16_t* q16_out, float* q32_out, cudaStream_t stream);
// Threads per qkv_post CTA and query heads per work item (one cos/sin each).
constexpr int kQkvThreads = 256;
constexpr int kQkvHeads = 4;

// Scaled cosine and sine of pair i at integer position pos (exact mode).
__device__ __forceinline__ void rope_cs(int pos, uint64_t turns, float mscale, float& c, float& s) {
    const uint64_t a = (uint64_t)(int64_t)pos * turns;      // mod 2^64 = mod one turn
    const float half_turns = (float)(int64_t)a * 0x1p-63f;   // angle / pi in [-1, 1)
    sincospif(half_turns, &s, &c);
    c = __fmul_rn(c, mscale);
    s = __fmul_rn(s, mscale);
}

// Angle of pair i at position pos in ggml's fp32 evaluation (see RopeTable).
__device__ __forceinline__ float rope_theta_f32(int pos, int i, const RopeTable& tb) {
    float th = __int2float_rn(pos);
    const float ts = tb.theta_scale;
    for (int j = 0; j < i; ++j) th = __fmul_rn(th, ts);
    const float te = __fdiv_rn(th, tb.ff[i]);
    const float ti = __fmul_rn(tb.freq_scale, te);
    if (!tb.yarn) return ti;
    const float m = tb.mix[i];
    return __fadd_rn(__fmul_rn(ti, __fsub_rn(1.0f, m)), __fmul_rn(te, m));
}

// Scaled cosine and sine of pair i at position pos, either mode.
__device__ __forceinline__ void rope_cs_tab(int pos, int i, const RopeTable& tb, float& c, float& s) {
    if (tb.mode == FR_ROPE_GGML_F32) {
        sincosf(rope_theta_f32(pos, i, tb), &s, &c);
        c = __fmul_rn(c, tb.mscale);
        s = __fmul_rn(s, tb.mscale);
    } else {
        rope_cs(pos, tb.turns[i], tb.mscale, c, s);
    }
}

// The two rotated outputs of a pair, from the scaled cos/sin. Plain IEEE fp32
// ops with explicit rounding intrinsics, so every kernel that calls these
// produces the same bits.
__device__ __forceinline__ float rope_lo(float x0, float x1, float c, float s, float q_scale) {
    return __fmul_rn(__fmaf_rn(x0, c, -__fmul_rn(x1, s)), q_scale);
}
__device__ __forceinline__ float rope_hi(float x0, float x1, float c, float s, float q_scale) {
    return __fmul_rn(__fmaf_rn(x0, s, __fmul_rn(x1, c)), q_scale);
}


// One "slot" of a Q row: slot c < half rotates dims (c, c + half); slot
// c >= half passes dims n_dims + 2(c - half) and +1 through (scaled).
// hd/2 slots cover the row exactly.
// The two dims of slot c.
__device__ __forceinline__ void rope_slot_dims(int c, const RopeTable& tb, int& d0, int& d1) {
    if (c < tb.half) {
        d0 = c;
        d1 = c + tb.half;
    } else {
        d0 = tb.n_dims + 2 * (c - tb.half);
        d1 = d0 + 1;
    }
}
// Slot c applied to its two inputs x0 = row[d0], x1 = row[d1].
__device__ __forceinline__ void rope_slot_apply(int c, float x0, float x1, int pos, const RopeTable& tb,
                                                float& y0, float& y1) {
    if (c < tb.half) {
        float cs, sn;
        rope_cs_tab(pos, c, tb, cs, sn);
        y0 = rope_lo(x0, x1, cs, sn, tb.q_scale);
        y1 = rope_hi(x0, x1, cs, sn, tb.q_scale);
    } else {
        y0 = __fmul_rn(x0, tb.q_scale);
        y1 = __fmul_rn(x1, tb.q_scale);
    }
}
__device__ __forceinline__ void rope_slot(const float* __restrict__ qrow, int c, int pos,
                                          const RopeTable& tb, int& d0, int& d1,
                                          float& y0, float& y1) {
    rope_slot_dims(c, tb, d0, d1);
    rope_slot_apply(c, qrow[d0], qrow[d1], pos, tb, y0, y1);
}

// The f16 Q tile of an attention kernel that ropes its own rows: query rows
// [r_lo, r_lo + r_n) (row r = t*n_head + h, t-major, the order qkv_post emits)
// from the f32 rows staged in shared memory at q32[(r - r_lo)*HD], written as
// tile rows r - r_lo, K-major in the 128-byte swizzle (64 dims per box of
// q_box bytes, 128 bytes per row). One work item is (token, slot, group of
// kQkvHeads heads) with one cos/sin, and every value goes through rope_cs_tab /
// rope_lo / rope_hi like qkv_post's: the bits equal its f16 rows. Called by
// threads [0, nthreads) with their index tid.
template <int HD>
__device__ __forceinline__ void rope_rows_to_tile(const float* q32, const int* pos, const RopeTable& tb, int n_head,
                                                  int r_lo, int r_n, unsigned char* tile, int q_box, int tid,
                                                  int nthreads) {
    const int groups = (n_head + kQkvHeads - 1) / kQkvHeads;
    const int t_lo = r_lo / n_head, n_t = (r_lo + r_n - 1) / n_head - t_lo + 1;
    for (int it = tid; it < n_t * groups * (HD / 2); it += nthreads) {
        const int c = it % (HD / 2), tg = it / (HD / 2);
        const int t = t_lo + tg / groups, h0 = (tg % groups) * kQkvHeads;
        const int ha = max(h0, r_lo - t * n_head);                      // heads of the group inside the rows
        const int hb = min(min(h0 + kQkvHeads, n_head), r_lo + r_n - t * n_head);
        if (ha >= hb) continue;
        int d0, d1;
        rope_slot_dims(c, tb, d0, d1);
        const bool rot = c < tb.half;
        float cs = 0.f, sn = 0.f;
        if (rot) rope_cs_tab(pos[t], c, tb, cs, sn);
        for (int h = ha; h < hb; ++h) {
            const int r = t * n_head + h - r_lo;                        // tile row
            const float x0 = q32[r * HD + d0], x1 = q32[r * HD + d1];
            const float y0 = rot ? rope_lo(x0, x1, cs, sn, tb.q_scale) : __fmul_rn(x0, tb.q_scale);
            const float y1 = rot ? rope_hi(x0, x1, cs, sn, tb.q_scale) : __fmul_rn(x1, tb.q_scale);
            unsigned char* row = tile + r * 128;
            *reinterpret_cast<__half*>(row + (d0 >> 6) * q_box + ((((d0 & 63) >> 3) ^ (r & 7)) << 4) + (d0 & 7) * 2) =
                __float2half_rn(y0);
            *reinterpret_cast<__half*>(row + (d1 >> 6) * q_box + ((((d1 & 63) >> 3) ^ (r & 7)) << 4) + (d1 & 7) * 2) =
                __float2half_rn(y1);
        }
    }
}

// Copy of the RoPE table into shared memory by threads [0, nthreads).
__device__ __forceinline__ void copy_rope_table(RopeTable& dst, const RopeTable& src, int tid, int nthreads) {
    for (int c = tid; c < kMaxPairs; c += nthreads) {
        dst.turns[c] = src.turns[c];
        dst.mix[c] = src.mix[c];
        dst.ff[c] = src.ff[c];
    }
    if (tid == 0) {
        dst.mscale = src.mscale;
        dst.q_scale = src.q_scale;
        dst.theta_scale = src.theta_scale;
        dst.freq_scale = src.freq_scale;
        dst.half = src.half;
        dst.n_dims = src.n_dims;
        dst.mode = src.mode;
        dst.yarn = src.yarn;
    }
}

inline bool aligned16(const void* p) { return (((uintptr_t)p) & 15u) == 0; }

// Host: p is device memory of GPU `dev` (or managed memory). A host pointer,
// an unregistered address or memory of another GPU fails, before any launch.
inline bool device_ptr_ok(const void* p, int dev) {
    cudaPointerAttributes at;
    if (cudaPointerGetAttributes(&at, p) != cudaSuccess) {
        (void)cudaGetLastError();          // reset the last-error state this call set
        return false;
    }
    if (at.type == cudaMemoryTypeManaged) return true;
    return at.type == cudaMemoryTypeDevice && at.device == dev;
}

// Host: the Q scale a call applies; FR_Q_SCALE_DEFAULT (0) selects 1/sqrt(hd)
// (a zero scale has no use: it would make every score equal).
inline float resolve_q_scale(float q_scale, int hd) {
    return q_scale == 0.0f ? (float)(1.0 / sqrt((double)hd)) : q_scale;
}

// ---- PTX wrappers ---------------------------------------------------------

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return (uint32_t)__cvta_generic_to_shared(p);
}

// 16-byte async copy global -> shared; src_bytes 0 zero-fills the destination.
__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, int src_bytes) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n"
                 :: "r"(dst), "l"(src), "r"(src_bytes) : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
    asm volatile("cp.async.commit_group;\n" ::: "memory");
}
template <int N>
__device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;\n" :: "n"(N) : "memory");
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1,
                                        uint32_t& r2, uint32_t& r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];\n"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3) : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1,
                                          uint32_t& r2, uint32_t& r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];\n"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3) : "r"(addr));
}

// D (16x8 f32) += A (16x16 f16, row) * B (16x8 f16, col)
__device__ __forceinline__ void mma_16816(float* d, const uint32_t* a, uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 "
        "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};\n"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t pack_half2(float lo, float hi) {
    __half2 h = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&h);
}

}  // namespace fr
