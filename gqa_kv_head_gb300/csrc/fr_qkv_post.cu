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
    const int n = rp->n_dims;
    if (n < 2 || (n & 1) || n > hd || n / 2 > kMaxPairs) return false;
    if (!(rp->freq_base > 0.0f) || !(rp->freq_scale > 0.0f)) return false;
    if (!isfinite(rp->ext_factor) || !isfinite(rp->attn_factor) || !isfinite(q_scale)) return false;
    const bool yarn = rp->ext_factor != 0.0f;
    double c0 = 0.0, c1 = 0.0;
    if (yarn) {
        if (rp->n_ctx_orig <= 0 || !(rp->beta_fast > 0.0f) || !(rp->beta_slow > 0.0f)) return false;
        yarn_corr_dims(n, rp->n_ctx_orig, rp->freq_base, rp->beta_fast, rp->beta_slow, &c0, &c1);
    }
    const double two_pi = 6.283185307179586476925286766559;
    const double step = pow((double)rp->freq_base, -2.0 / n);   // ratio between pairs
    const double fs = rp->freq_scale;
    double w_ext = 1.0;
    t->half = n / 2;
    t->n_dims = n;
    for (int i = 0; i < t->half; ++i) {
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
        w_ext *= step;
    }
    for (int i = t->half; i < kMaxPairs; ++i) t->turns[i] = 0;
    double mscale = rp->attn_factor;
    if (yarn) mscale *= 1.0 + 0.1 * log(1.0 / fs);
    t->mscale = (float)mscale;
    t->q_scale = q_scale;
    return true;
}

// One thread per slot (hd/2 slots per row); blockDim.x = hd/2 rows-slots,
// blockDim.y rows per block.
template <int HD>
__global__ void __launch_bounds__(256)
qkv_post_kernel(const float* __restrict__ q, int64_t q_tok_stride, const int32_t* __restrict__ pos,
                int n_head, int M, __half* __restrict__ q16, float* __restrict__ q32,
                const __grid_constant__ RopeTable tb) {
    // Launched with programmatic stream serialization: wait until the grids
    // before this one on the stream are complete and their writes visible. A
    // dependent attention launch may then start its set-up and K/V loads; it
    // waits for this grid's completion before it reads the rows.
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    const int r = blockIdx.x * blockDim.y + threadIdx.y;
    if (r >= M) return;
    const int c = threadIdx.x;                 // slot 0 .. HD/2-1
    const int t = r / n_head, h = r - t * n_head;
    const float* qrow = q + (int64_t)t * q_tok_stride + (int64_t)h * HD;
    int d0, d1;
    float y0, y1;
    rope_slot(qrow, c, __ldg(pos + t), tb, d0, d1, y0, y1);
    __half* orow = q16 + (int64_t)r * HD;
    orow[d0] = __float2half_rn(y0);
    orow[d1] = __float2half_rn(y1);
    if (q32) {
        float* frow = q32 + (int64_t)r * HD;
        frow[d0] = y0;
        frow[d1] = y1;
    }
}

fr_status launch_qkv_post(const float* q, int64_t q_tok_stride, const int32_t* pos, int n_tok, int n_head,
                          int hd, const RopeTable& tb, uint16_t* q16_out, float* q32_out, cudaStream_t stream) {
    const int M = n_tok * n_head;
    const int slots = hd / 2;
    const int rows_per_block = 256 / slots;
    dim3 block(slots, rows_per_block);
    dim3 grid((M + rows_per_block - 1) / rows_per_block);
    __half* o16 = reinterpret_cast<__half*>(q16_out);
    // programmatic dependent launch: this grid may be scheduled while the
    // previous one on the stream finishes (the kernel waits before any access)
    cudaLaunchConfig_t cfg;
    memset(&cfg, 0, sizeof(cfg));
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaError_t e;
    switch (hd) {
        case 64: e = cudaLaunchKernelEx(&cfg, qkv_post_kernel<64>, q, q_tok_stride, pos, n_head, M, o16, q32_out, tb); break;
        case 128: e = cudaLaunchKernelEx(&cfg, qkv_post_kernel<128>, q, q_tok_stride, pos, n_head, M, o16, q32_out, tb); break;
        default: e = cudaLaunchKernelEx(&cfg, qkv_post_kernel<256>, q, q_tok_stride, pos, n_head, M, o16, q32_out, tb); break;
    }
    return e == cudaSuccess ? FR_OK : FR_ERR_CUDA;
}

}  // namespace fr

using namespace fr;

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

extern "C" int fr_abi_version(void) { return (1 << 16) | 0; }

extern "C" fr_status fr_qkv_post(const float* q, int64_t q_tok_stride, const int32_t* pos,
                                 int n_tok, int n_head, int hd, const fr_rope_params* rp,
                                 float q_scale, uint16_t* q16_out, float* q32_out,
                                 cudaStream_t stream) {
    if (!q || !pos || !rp || !q16_out) return FR_ERR_INVALID_ARG;
    if (n_tok < 1 || n_head < 1 || hd < 1) return FR_ERR_INVALID_ARG;
    if (hd != 64 && hd != 128 && hd != 256) return FR_ERR_UNSUPPORTED;
    if (n_tok > kMaxTok || (int64_t)n_tok * n_head > kMaxRows) return FR_ERR_UNSUPPORTED;
    if (q_tok_stride < (int64_t)n_head * hd || (q_tok_stride & 3)) return FR_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(q16_out) || (q32_out && !aligned16(q32_out)))
        return FR_ERR_INVALID_ARG;
    RopeTable tb;
    if (!build_rope_table(rp, q_scale, hd, &tb)) return FR_ERR_INVALID_ARG;
    return launch_qkv_post(q, q_tok_stride, pos, n_tok, n_head, hd, tb, q16_out, q32_out, stream);
}
