// fr_qkv_post.cu -- the Q leg of qkv_post: NEOX RoPE with the YaRN terms,
// scale by q_scale, one round to f16, rows written t-major (r = t*n_head + h).
//
// FlashRT PR #185, commits "Fuses the prefix layers' q/k/v projections, RoPE,
// scale, KV padding ..." and "qkv_post optionally stores the rope'd+scaled Q
// rows as f16 alongside the f32 tensor; its [M, Nq] layout is exactly the
// t-major gather order the decomposed decode attention consumes".
// FlashRT-llama.cpp development guide, "Invariants and pitfalls": RoPE mirrors
// ggml's rope_neox with the YaRN corrections; non-NEOX modes are not offered.
#include <math.h>
#include <string.h>

#include "fr_common.cuh"

namespace fr {

// YaRN correction range (YaRN paper, Peng et al. 2023, as ggml applies it):
// d(beta) = n_dims * ln(n_ctx_orig / (2 pi beta)) / (2 ln base);
// c0 = max(0, floor(d(beta_fast))), c1 = min(n_dims - 1, ceil(d(beta_slow))).
static void yarn_corr_dims(int n_dims, int n_ctx_orig, double base, double beta_fast,
                           double beta_slow, double* c0, double* c1) {
    const double two_pi = 6.283185307179586476925286766559;
    auto d = [&](double beta) {
        return n_dims * log((double)n_ctx_orig / (two_pi * beta)) / (2.0 * log(base));
    };
    *c0 = fmax(0.0, floor(d(beta_fast)));
    *c1 = fmin((double)(n_dims - 1), ceil(d(beta_slow)));
}

bool build_rope_table(const fr_rope_params* rp, float q_scale, int hd, RopeTable* t) {
    if (!rp || !t) return false;
    memset(t, 0, sizeof(*t));
    const int n = rp->n_dims;
    if (n < 2 || (n & 1) || n > hd || n / 2 > kMaxPairs) return false;
    if (!(rp->freq_base > 0.0f) || !(rp->freq_scale > 0.0f)) return false;
    if (!isfinite(rp->freq_base) || !isfinite(rp->freq_scale)) return false;
    if (!isfinite(rp->ext_factor) || !isfinite(rp->attn_factor) || !isfinite(q_scale)) return false;
    if (rp->mode != FR_ROPE_EXACT && rp->mode != FR_ROPE_GGML_F32) return false;
    const int half = n / 2;
    if (rp->freq_factors)
        for (int i = 0; i < half; ++i)
            if (!(rp->freq_factors[i] > 0.0f) || !isfinite(rp->freq_factors[i])) return false;
    const bool yarn = rp->ext_factor != 0.0f;
    double c0 = 0.0, c1 = 0.0;
    if (yarn) {
        if (rp->n_ctx_orig <= 0 || !(rp->beta_fast > 0.0f) || !(rp->beta_slow > 0.0f)) return false;
        yarn_corr_dims(n, rp->n_ctx_orig, rp->freq_base, rp->beta_fast, rp->beta_slow, &c0, &c1);
    }
    t->half = half;
    t->n_dims = n;
    t->mode = rp->mode;
    t->yarn = yarn ? 1 : 0;
    t->q_scale = q_scale;
    for (int i = 0; i < half; ++i) t->ff[i] = rp->freq_factors ? rp->freq_factors[i] : 1.0f;
    if (rp->mode == FR_ROPE_GGML_F32) {
        // one IEEE fp32 operation per step (the host objects are built with
        // floating-point contraction off, so no step is fused); powf and logf
        // are the correctly rounded values, taken in double and rounded once
        const float e = -2.0f / (float)n;
        t->theta_scale = (float)pow((double)rp->freq_base, (double)e);
        t->freq_scale = rp->freq_scale;
        const float lo = (float)c0, hi = (float)c1;
        for (int i = 0; i < half; ++i) {
            if (!yarn) {
                t->mix[i] = 0.0f;
                continue;
            }
            const float y = ((float)i - lo) / fmaxf(0.001f, hi - lo);
            const float ramp = 1.0f - fminf(1.0f, fmaxf(0.0f, y));
            t->mix[i] = ramp * rp->ext_factor;
        }
        float ms = rp->attn_factor;
        if (yarn) {
            const float lg = (float)log((double)(1.0f / rp->freq_scale));
            const float f = 1.0f + 0.1f * lg;
            ms = ms * f;
        }
        t->mscale = ms;
        return true;
    }
    const double two_pi = 6.283185307179586476925286766559;
    const double step = pow((double)rp->freq_base, -2.0 / n);   // ratio between pairs
    const double fs = rp->freq_scale;
    double w_base = 1.0;
    for (int i = 0; i < half; ++i) {
        const double w_ext = w_base / (double)t->ff[i];
        double w = fs * w_ext;                                   // interpolation
        if (yarn) {
            const double y = ((double)i - c0) / fmax(0.001, c1 - c0);
            const double ramp = 1.0 - fmin(1.0, fmax(0.0, y));
            const double mix = ramp * (double)rp->ext_factor;
            w = w * (1.0 - mix) + w_ext * mix;
        }
        double f = w / two_pi;
        f -= floor(f);                                           // turns per step, mod 1
        const double scaled = ldexp(f, 64);
        t->turns[i] = scaled >= 18446744073709551616.0 ? 0ull : (uint64_t)scaled;
        w_base *= step;
    }
    double mscale = rp->attn_factor;
    if (yarn) mscale *= 1.0 + 0.1 * log(1.0 / fs);
    t->mscale = (float)mscale;
    return true;
}

// Every query head of a token rotates its pairs by the same angles, so a work
// item is (token t, slot c, group of kQkvHeads heads): one cos/sin for the
// group, then the group's pairs loaded together and rotated. Items are
// strided over the grid.
template <int HD>
__global__ void __launch_bounds__(kQkvThreads)
qkv_post_kernel(const float* __restrict__ q, int64_t q_tok_stride, const int32_t* __restrict__ pos,
                int n_tok, int n_head, __half* __restrict__ q16, float* __restrict__ q32,
                const __grid_constant__ RopeTable tb) {
    // Launched with programmatic stream serialization: wait until the grids
    // before this one on the stream are complete and their writes visible. A
    // dependent attention launch may then start its set-up and K/V loads; it
    // waits for this grid's completion before it reads the rows.
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    // Each item reads its pair's constants straight from the parameter block:
    // no shared-memory copy and no block barrier, so the table, position and Q
    // loads of an item all go out at once (the kernel is latency-bound).
    const RopeTable& stb = tb;
    constexpr int SLOTS = HD / 2;
    const int groups = (n_head + kQkvHeads - 1) / kQkvHeads;
    const int64_t items = (int64_t)n_tok * groups * SLOTS;
    const float q_scale = stb.q_scale;
    for (int64_t it = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; it < items;
         it += (int64_t)gridDim.x * blockDim.x) {
        const int c = (int)(it % SLOTS);                    // consecutive threads: consecutive slots
        const int64_t tg = it / SLOTS;
        const int t = (int)(tg / groups), h0 = (int)(tg - (int64_t)t * groups) * kQkvHeads;
        int d0, d1;
        rope_slot_dims(c, stb, d0, d1);
        const float* qh = q + (int64_t)t * q_tok_stride + (int64_t)h0 * HD;
        float x0[kQkvHeads], x1[kQkvHeads];
#pragma unroll
        for (int u = 0; u < kQkvHeads; ++u) {
            x0[u] = h0 + u < n_head ? __ldg(qh + u * HD + d0) : 0.f;
            x1[u] = h0 + u < n_head ? __ldg(qh + u * HD + d1) : 0.f;
        }
        const bool rot = c < stb.half;
        float cs = 0.f, sn = 0.f;
        if (rot) rope_cs_tab(__ldg(pos + t), c, stb, cs, sn);
        const int64_t r0 = (int64_t)t * n_head + h0;       // t-major row of head h0
#pragma unroll
        for (int u = 0; u < kQkvHeads; ++u) {
            if (h0 + u >= n_head) break;
            // the same operations as rope_slot_apply, so the bits match
            const float y0 = rot ? rope_lo(x0[u], x1[u], cs, sn, q_scale) : __fmul_rn(x0[u], q_scale);
            const float y1 = rot ? rope_hi(x0[u], x1[u], cs, sn, q_scale) : __fmul_rn(x1[u], q_scale);
            __half* orow = q16 + (r0 + u) * HD;
            orow[d0] = __float2half_rn(y0);
            orow[d1] = __float2half_rn(y1);
            if (q32) {
                float* frow = q32 + (r0 + u) * HD;
                frow[d0] = y0;
                frow[d1] = y1;
            }
        }
    }
}

// at most 8 CTAs of 256 threads on each of 152 SMs: one wave, so a dependent
// launch is released as soon as every CTA has started
constexpr int kQkvMaxCtas = 1216;

fr_status launch_qkv_post(const float* q, int64_t q_tok_stride, const int32_t* pos, int n_tok, int n_head,
                          int hd, const RopeTable& tb, uint16_t* q16_out, float* q32_out, cudaStream_t stream) {
    const int64_t items = (int64_t)n_tok * ((n_head + kQkvHeads - 1) / kQkvHeads) * (hd / 2);
    const int threads = items < kQkvThreads ? (int)((items + 31) / 32 * 32) : kQkvThreads;
    int64_t ctas = (items + threads - 1) / threads;
    if (ctas > kQkvMaxCtas) ctas = kQkvMaxCtas;
    __half* o16 = reinterpret_cast<__half*>(q16_out);
    // programmatic dependent launch: this grid may be scheduled while the
    // previous one on the stream finishes (the kernel waits before any access)
    cudaLaunchConfig_t cfg;
    memset(&cfg, 0, sizeof(cfg));
    cfg.gridDim = dim3((unsigned)ctas);
    cfg.blockDim = dim3(threads);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaError_t e;
    switch (hd) {
        case 64: e = cudaLaunchKernelEx(&cfg, qkv_post_kernel<64>, q, q_tok_stride, pos, n_tok, n_head, o16, q32_out, tb); break;
        case 128: e = cudaLaunchKernelEx(&cfg, qkv_post_kernel<128>, q, q_tok_stride, pos, n_tok, n_head, o16, q32_out, tb); break;
        default: e = cudaLaunchKernelEx(&cfg, qkv_post_kernel<256>, q, q_tok_stride, pos, n_tok, n_head, o16, q32_out, tb); break;
    }
    return e == cudaSuccess ? FR_OK : FR_ERR_CUDA;
}

// K/V leg: one grid-stride pass over three kinds of work item — rotated K
// pairs (the same device routine as the Q rows, scale 1), groups of 8 V
// elements (one 16-byte f16 store) and 16-byte zero stores of the pad rows.
template <int HD>
__global__ void __launch_bounds__(256)
kv_append_kernel(const float* __restrict__ k_new, int64_t k_stride, const float* __restrict__ v_new,
                 int64_t v_stride, const int32_t* __restrict__ pos, int n_tok, __half* __restrict__ k_cache,
                 int64_t k_rs, __half* __restrict__ v_cache, int64_t v_rs, int64_t row0, int64_t pad_begin,
                 int64_t pad_rows, float* __restrict__ k32, float* __restrict__ v32,
                 const __grid_constant__ RopeTable tb) {
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    const RopeTable& stb = tb;                                 // see qkv_post_kernel
    constexpr int G = HD / 8;                                  // 8-element groups per row
    const int64_t nK = (int64_t)n_tok * (HD / 2), nV = (int64_t)n_tok * G, nP = pad_rows * G;
    for (int64_t w = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; w < nK + nV + nP;
         w += (int64_t)gridDim.x * blockDim.x) {
        if (w < nK) {
            const int t = (int)(w / (HD / 2)), c = (int)(w - (int64_t)t * (HD / 2));
            int d0, d1;
            float y0, y1;
            rope_slot(k_new + (int64_t)t * k_stride, c, __ldg(pos + t), stb, d0, d1, y0, y1);
            __half* krow = k_cache + (row0 + t) * k_rs;
            krow[d0] = __float2half_rn(y0);
            krow[d1] = __float2half_rn(y1);
            if (k32) {
                k32[(int64_t)t * HD + d0] = y0;
                k32[(int64_t)t * HD + d1] = y1;
            }
        } else if (w < nK + nV) {
            const int64_t u = w - nK;
            const int t = (int)(u / G), g = (int)(u - (int64_t)t * G);
            const float4* src = reinterpret_cast<const float4*>(v_new + (int64_t)t * v_stride + g * 8);
            const float4 a = src[0], b = src[1];
            uint4 h;
            h.x = pack_half2(a.x, a.y);
            h.y = pack_half2(a.z, a.w);
            h.z = pack_half2(b.x, b.y);
            h.w = pack_half2(b.z, b.w);
            *reinterpret_cast<uint4*>(v_cache + (row0 + t) * v_rs + g * 8) = h;
            if (v32) {
                float4* dst = reinterpret_cast<float4*>(v32 + (int64_t)t * HD + g * 8);
                dst[0] = a;
                dst[1] = b;
            }
        } else {
            const int64_t u = w - nK - nV;
            const int64_t row = pad_begin + u / G;
            const int g = (int)(u % G);
            const uint4 z = make_uint4(0u, 0u, 0u, 0u);
            *reinterpret_cast<uint4*>(k_cache + row * k_rs + g * 8) = z;
            *reinterpret_cast<uint4*>(v_cache + row * v_rs + g * 8) = z;
        }
    }
}

}  // namespace fr

using namespace fr;

extern "C" fr_status fr_kv_append(const float* k_new, int64_t k_stride, const float* v_new, int64_t v_stride,
                                  const int32_t* pos, int n_tok, int hd, const fr_rope_params* rp,
                                  uint16_t* k_cache, int64_t k_row_stride, uint16_t* v_cache,
                                  int64_t v_row_stride, int64_t n_ctx, int64_t row0, int64_t pad_begin,
                                  int64_t pad_end, float* k32_out, float* v32_out, cudaStream_t stream) {
    if (!k_new || !v_new || !pos || !rp || !k_cache || !v_cache) return FR_ERR_INVALID_ARG;
    if (n_tok < 1 || hd < 1) return FR_ERR_INVALID_ARG;
    if (hd != 64 && hd != 128 && hd != 256) return FR_ERR_UNSUPPORTED;
    if (n_tok > kMaxTokTc) return FR_ERR_UNSUPPORTED;
    if (k_stride < hd || (k_stride & 3) || v_stride < hd || (v_stride & 3)) return FR_ERR_INVALID_ARG;
    if (k_row_stride < hd || (k_row_stride & 7) || v_row_stride < hd || (v_row_stride & 7))
        return FR_ERR_INVALID_ARG;
    if (!aligned16(k_new) || !aligned16(v_new) || !aligned16(k_cache) || !aligned16(v_cache) ||
        (k32_out && !aligned16(k32_out)) || (v32_out && !aligned16(v32_out)))
        return FR_ERR_INVALID_ARG;
    if (row0 < 0 || row0 + n_tok > n_ctx) return FR_ERR_INVALID_ARG;            // tail inside the cache
    if (pad_begin < 0 || pad_end < pad_begin || pad_end > n_ctx) return FR_ERR_INVALID_ARG;
    if (pad_end > pad_begin && pad_begin < row0 + n_tok && row0 < pad_end) return FR_ERR_INVALID_ARG;
    RopeTable tb;
    if (!build_rope_table(rp, 1.0f, hd, &tb)) return FR_ERR_INVALID_ARG;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return FR_ERR_CUDA;
    if (!device_ptr_ok(k_new, dev) || !device_ptr_ok(v_new, dev) || !device_ptr_ok(pos, dev) ||
        !device_ptr_ok(k_cache, dev) || !device_ptr_ok(v_cache, dev) || (k32_out && !device_ptr_ok(k32_out, dev)) ||
        (v32_out && !device_ptr_ok(v32_out, dev)))
        return FR_ERR_INVALID_ARG;
    const int64_t total = (int64_t)n_tok * (hd / 2) + ((int64_t)n_tok + (pad_end - pad_begin)) * (hd / 8);
    const int blocks = (int)(total < 256 * 1184 ? (total + 255) / 256 : 1184);
    cudaLaunchConfig_t cfg;
    memset(&cfg, 0, sizeof(cfg));
    cfg.gridDim = dim3(blocks);
    cfg.blockDim = dim3(256);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    __half* kc = reinterpret_cast<__half*>(k_cache);
    __half* vc = reinterpret_cast<__half*>(v_cache);
    const int64_t pr = pad_end - pad_begin;
    cudaError_t e;
    switch (hd) {
        case 64: e = cudaLaunchKernelEx(&cfg, kv_append_kernel<64>, k_new, k_stride, v_new, v_stride, pos, n_tok, kc,
                                        k_row_stride, vc, v_row_stride, row0, pad_begin, pr, k32_out, v32_out, tb); break;
        case 128: e = cudaLaunchKernelEx(&cfg, kv_append_kernel<128>, k_new, k_stride, v_new, v_stride, pos, n_tok, kc,
                                         k_row_stride, vc, v_row_stride, row0, pad_begin, pr, k32_out, v32_out, tb); break;
        default: e = cudaLaunchKernelEx(&cfg, kv_append_kernel<256>, k_new, k_stride, v_new, v_stride, pos, n_tok, kc,
                                        k_row_stride, vc, v_row_stride, row0, pad_begin, pr, k32_out, v32_out, tb); break;
    }
    return e == cudaSuccess ? FR_OK : FR_ERR_CUDA;
}

extern "C" const char* fr_status_string(fr_status s) {
    switch (s) {
        case FR_OK: return "FR_OK";
        case FR_ERR_INVALID_ARG: return "FR_ERR_INVALID_ARG: null pointer, bad size, alignment or stride";
        case FR_ERR_UNSUPPORTED: return "FR_ERR_UNSUPPORTED: shape outside the supported set";
        case FR_ERR_WORKSPACE: return "FR_ERR_WORKSPACE: workspace missing or too small";
        case FR_ERR_CUDA: return "FR_ERR_CUDA: a CUDA call or kernel launch failed";
        case FR_ERR_DEVICE_TIMEOUT: return "FR_ERR_DEVICE_TIMEOUT: a bounded device wait gave up";
    }
    return "unknown fr_status";
}

extern "C" int fr_abi_version(void) { return (4 << 16) | 0; }

extern "C" fr_status fr_qkv_post(const float* q, int64_t q_tok_stride, const int32_t* pos,
                                 int n_tok, int n_head, int hd, const fr_rope_params* rp,
                                 float q_scale, uint16_t* q16_out, float* q32_out,
                                 cudaStream_t stream) {
    if (!q || !pos || !rp || !q16_out) return FR_ERR_INVALID_ARG;
    if (n_tok < 1 || n_head < 1 || hd < 1) return FR_ERR_INVALID_ARG;
    if (hd != 64 && hd != 128 && hd != 256) return FR_ERR_UNSUPPORTED;
    if (n_tok > kMaxTokTc || (int64_t)n_tok * n_head > kMaxRowsTc) return FR_ERR_UNSUPPORTED;
    if (q_tok_stride < (int64_t)n_head * hd || (q_tok_stride & 3)) return FR_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(q16_out) || (q32_out && !aligned16(q32_out)))
        return FR_ERR_INVALID_ARG;
    RopeTable tb;
    if (!build_rope_table(rp, resolve_q_scale(q_scale, hd), hd, &tb)) return FR_ERR_INVALID_ARG;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return FR_ERR_CUDA;
    if (!device_ptr_ok(q, dev) || !device_ptr_ok(pos, dev) || !device_ptr_ok(q16_out, dev) ||
        (q32_out && !device_ptr_ok(q32_out, dev)))
        return FR_ERR_INVALID_ARG;
    return launch_qkv_post(q, q_tok_stride, pos, n_tok, n_head, hd, tb, q16_out, q32_out, stream);
}
