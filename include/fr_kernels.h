/*
 * fr_kernels.h -- C ABI of the GB300 (sm_103a) decode-attention hot path:
 * qkv_post (NEOX RoPE with YaRN terms, 1/sqrt(hd) scale, f16 t-major Q rows)
 * and the collapsed GQA decode attention over one shared f16 KV head.
 *
 * Plain C: raw pointers, sizes and a cudaStream_t; no framework types.
 *
 * Sources (the FlashRT pages):
 *  - FlashRT PR #185 "ggml host adapter", commit "qkv_post optionally stores
 *    the rope'd+scaled Q rows as f16": the [M, Nq] layout is the t-major order
 *    the decode attention consumes; the f16 values round from the same fp32
 *    registers.
 *  - FlashRT PR #185, commit "FLASH_ATTN_EXT with q_tokens <= 16 over a single
 *    padded f16 KV head": QK^T with a stride-0 K operand shared by the GQA
 *    heads, a masked fp32-accurate softmax, PV whose fp32 result lands in the
 *    node's [hd, n_head, n_tok] layout.
 *  - FlashRT PR #185, commit "The GQA query heads share the one KV head": one
 *    GEMM over all n_head*n_tok t-major rows; the PV output lands contiguously.
 *  - FlashRT-llama.cpp development guide, "Architecture": launch interface with
 *    raw pointers + cudaStream_t, consumable from plain C++; "Caches": no
 *    allocation while a CUDA graph is being captured; "Invariants and
 *    pitfalls": RoPE mirrors ggml's rope_neox with the YaRN corrections;
 *    "SM120 target": runtime dimensions dispatched onto compile-time
 *    specialisations at the launch boundary.
 *
 * Conventions for every entry point
 *  - Device pointers unless stated otherwise: memory of the GPU that is
 *    current when the call is made (cudaMalloc'd or managed). Host memory and
 *    another GPU's memory are rejected with FR_ERR_INVALID_ARG before any
 *    launch; the library is for calls on one GPU. f16 tensors are IEEE
 *    binary16 stored as uint16_t. Every pointer and every row stride (in
 *    bytes) must be 16-byte aligned.
 *  - Row index r = t*n_head + h ("t-major"): Q16 rows and output rows.
 *  - Ownership: the caller owns every buffer. The library keeps no pointer
 *    after a call returns, never allocates or frees device memory and holds no
 *    mutable global state, so calls may be captured in a CUDA graph and made
 *    from several host threads (each concurrent call needs its own workspace).
 *    The one exception is fr_decode_attn_noalloc (end of this file): its
 *    calls share a scratch array inside the library and must not overlap.
 *  - Errors: arguments are validated on the host before any launch; an invalid
 *    call returns a status != FR_OK and launches nothing. A failed launch
 *    returns FR_ERR_CUDA. Nothing prints or aborts.
 *  - Work is enqueued on `stream` and is asynchronous, like a kernel launch.
 */
#ifndef FR_KERNELS_H
#define FR_KERNELS_H

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum fr_status {
    FR_OK = 0,
    FR_ERR_INVALID_ARG = 1,    /* null pointer, bad size, bad alignment or stride */
    FR_ERR_UNSUPPORTED = 2,    /* valid but outside the supported shapes (hd, n_tok, M) */
    FR_ERR_WORKSPACE = 3,      /* workspace missing or smaller than required */
    FR_ERR_CUDA = 4,           /* a CUDA runtime call or a launch failed */
    FR_ERR_DEVICE_TIMEOUT = 5  /* a bounded device-side wait gave up (see fr_workspace_check) */
} fr_status;

/* RoPE parameters, NEOX mode, with the YaRN terms as ggml's rope_ext takes
 * them (FlashRT-llama.cpp development guide, "Invariants and pitfalls": RoPE
 * mirrors ggml's rope_neox, YaRN corrections included).
 * Pair i < n_dims/2 rotates (x[i], x[i + n_dims/2]); dims >= n_dims pass
 * through. theta_ext = pos * freq_base^(-2i/n_dims) / ff_i, theta_int =
 * freq_scale * theta_ext; with ext_factor != 0 they are mixed by the YaRN ramp
 * between the correction dims of beta_fast/beta_slow (n_ctx_orig) and the
 * magnitude is attn_factor * (1 + 0.1 ln(1/freq_scale)); otherwise theta =
 * theta_int and the magnitude is attn_factor.
 *
 * mode selects how the angles are evaluated:
 *   FR_ROPE_EXACT     pos * w_i reduced exactly modulo one turn (64-bit fixed
 *                     point; w_i from double on the host), sincospi in fp32.
 *   FR_ROPE_GGML_F32  ggml's fp32 evaluation, one IEEE fp32 operation per step
 *                     in ggml's order: theta_scale = fl(freq_base ^ fl(-2/n_dims))
 *                     (correctly rounded), theta_0 = fl(pos), theta_i =
 *                     fl(theta_{i-1} * theta_scale), theta_ext = fl(theta_i / ff_i),
 *                     theta_int = fl(freq_scale * theta_ext), YaRN mix
 *                     fl(fl(theta_int * fl(1 - m_i)) + fl(theta_ext * m_i)) with
 *                     m_i = fl(ramp_i * ext_factor); then fp32 sincos and the
 *                     fp32 magnitude fl(attn_factor * fl(1 + fl(0.1 * ln(1/freq_scale)))).
 *                     The angles are bit-exact with that recurrence; at large
 *                     positions they carry its fp32 error (~1e-7 relative per step).
 * freq_factors: nullable host pointer to n_dims/2 floats (finite, > 0), the
 * per-pair divisors ff_i of rope_ext (1 when NULL); read during the call only. */
#define FR_ROPE_EXACT 0
#define FR_ROPE_GGML_F32 1
typedef struct fr_rope_params {
    int   n_dims;        /* rotated dims: even, 2 <= n_dims <= hd */
    float freq_base;     /* > 0 */
    float freq_scale;    /* > 0 */
    float ext_factor;    /* YaRN mix strength; 0 = pure interpolation */
    float attn_factor;
    float beta_fast;
    float beta_slow;
    int   n_ctx_orig;    /* > 0 when ext_factor != 0 */
    int   mode;          /* FR_ROPE_EXACT or FR_ROPE_GGML_F32 */
    const float* freq_factors;   /* nullable, n_dims/2 host floats */
} fr_rope_params;

/* Pass as q_scale to apply 1/sqrt(hd), the attention's usual scale (a zero
 * scale has no use: it would make every score equal). */
#define FR_Q_SCALE_DEFAULT 0.0f

/* Human-readable name of a status code (static storage). */
const char* fr_status_string(fr_status s);

/* ABI version: (major << 16) | minor. */
int fr_abi_version(void);

/*
 * fr_qkv_post -- the Q leg of qkv_post (FlashRT PR #185, commits "Fuses the
 * prefix layers' q/k/v projections, RoPE, scale ..." and "qkv_post optionally
 * stores the rope'd+scaled Q rows as f16").
 *
 *   q        f32, element (t, h, d) at q[t*q_tok_stride + h*hd + d]
 *            (the QKV GEMM's [M = n_tok, Nq] rows; q_tok_stride >= n_head*hd,
 *            a multiple of 4 elements)
 *   pos      int32 [n_tok] token positions (shared by all heads of a token)
 *   rp       RoPE parameters (host pointer, read during the call only)
 *   q_scale  multiplier applied after the rotation; FR_Q_SCALE_DEFAULT (0)
 *            selects 1/sqrt(hd), rounded once to fp32
 *   q16_out  f16 [n_tok*n_head][hd], row r = t*n_head + h, contiguous
 *   q32_out  nullable; f32, same layout, the values q16_out is rounded from
 *
 * Arithmetic: angles as rp->mode says (fr_rope_params), rotation and scale
 * in fp32, one round-to-nearest to f16.
 * Supported: 1 <= n_tok <= 8192, 1 <= n_head, M = n_tok*n_head <= 65536,
 * hd in {64, 128, 256}.
 */
fr_status fr_qkv_post(const float* q, int64_t q_tok_stride, const int32_t* pos,
                      int n_tok, int n_head, int hd,
                      const fr_rope_params* rp, float q_scale,
                      uint16_t* q16_out, float* q32_out, cudaStream_t stream);

/*
 * fr_kv_append -- the K/V leg of qkv_post with the write of the new rows into
 * the persistent KV cache (FlashRT PR #185, commit "Fuses the prefix layers'
 * q/k/v projections, RoPE, scale, KV padding to the FA KQ stride, and the
 * permuted f16 materializations ..."; its full variant re-emits the rope'd K
 * and plain V as f32 rows and zeroes the pad rows).
 *
 * For each new token t < n_tok:
 *   k_cache[row0 + t] = f16_RN(mscale * NEOX-RoPE(k_new[t], pos[t]))   no 1/sqrt(hd)
 *   v_cache[row0 + t] = f16_RN(v_new[t])
 * with the same angles, YaRN terms and fp32 arithmetic as fr_qkv_post's Q rows,
 * and rows [pad_begin, pad_end) of both caches set to zero. No other row is
 * touched.
 *
 *   k_new, v_new  f32, row t at k_new + t*k_stride (elements, >= hd, multiple
 *                 of 4), hd contiguous values — e.g. the K and V columns of a
 *                 fused QKV GEMM output.
 *   k_cache, v_cache  f16 [n_ctx][hd], row strides >= hd, multiples of 8.
 *   row0          first cache row written; [row0, row0 + n_tok) and
 *                 [pad_begin, pad_end) must lie in [0, n_ctx) and not overlap.
 *   k32_out, v32_out  optional f32 [n_tok][hd] copies (rope'd K, plain V).
 * All pointers 16-byte aligned. Launched with programmatic stream
 * serialization; the kernel waits for the grids before it on the stream
 * before reading. A following fr_decode_attn on the same stream sees the new
 * rows: its qkv_post kernel waits for this grid before it releases the
 * attention launch.
 * Supported: 1 <= n_tok <= 8192, hd in {64, 128, 256}.
 */
fr_status fr_kv_append(const float* k_new, int64_t k_stride, const float* v_new, int64_t v_stride,
                       const int32_t* pos, int n_tok, int hd, const fr_rope_params* rp,
                       uint16_t* k_cache, int64_t k_row_stride, uint16_t* v_cache, int64_t v_row_stride,
                       int64_t n_ctx, int64_t row0, int64_t pad_begin, int64_t pad_end,
                       float* k32_out, float* v32_out, cudaStream_t stream);

/*
 * Workspace bytes for this shape that admit every plan of fr_decode_attn,
 * the separate merge kernel's included (0 for unsupported shapes). The
 * workspace holds the split-KV partial states, self-resetting arrival tickets
 * and a device status word. Zero it once after allocating it
 * (fr_workspace_init); every call leaves the tickets at zero again.
 */
size_t fr_decode_attn_workspace_size(int n_tok, int n_head, int hd, int n_kv);

/* Zero a freshly allocated workspace on `stream` (cudaMemsetAsync). */
fr_status fr_workspace_init(void* workspace, size_t workspace_bytes, cudaStream_t stream);

/*
 * Reads the workspace's device status word (synchronises `stream`), clears it
 * and returns FR_ERR_DEVICE_TIMEOUT if a bounded device-side wait of an
 * earlier call on this workspace gave up, else FR_OK.
 */
fr_status fr_workspace_check(void* workspace, cudaStream_t stream);

/*
 * fr_decode_attn -- decode attention for q_tokens <= 16 over one padded f16
 * KV head shared by all n_head query heads (FlashRT PR #185, commits
 * "FLASH_ATTN_EXT with q_tokens <= 16 ..." and "The GQA query heads share the
 * one KV head ...").
 *
 * For every row r = t*n_head + h (M = n_tok*n_head rows):
 *   s_j    = kq_scale * <Q16[r], K[j]> + mask[t][j]      j < n_kv
 *   out[r] = sum_j softmax(s)_j V[j]                     fp32
 * with fp32 accumulation and softmax. Columns whose mask is -inf get weight 0;
 * a row whose every column is masked yields 0.
 *
 *   q16      f16 [M][hd], rope'd and scaled (fr_qkv_post's output), or NULL
 *            to fuse qkv_post: then q, q_tok_stride, pos, rp and q_scale are
 *            used exactly as in fr_qkv_post and the f16 rows are bit-identical
 *            to what fr_qkv_post would have written.
 *   k, v     f16 [n_kv][hd] with row strides k_row_stride / v_row_stride
 *            (elements, >= hd, multiple of 8); one KV head, already rope'd.
 *   mask     nullable; f16 additive [n_tok][n_kv], row stride mask_row_stride
 *            (elements, >= n_kv, multiple of 8), shared by all heads
 *            (ggml FA semantics with max_bias = 0 and softcap = 0).
 *   out      f32 [n_tok][n_head][hd] contiguous == ggml [hd, n_head, n_tok].
 *   workspace, workspace_bytes: >= fr_decode_attn_workspace_size(...), zeroed
 *            once; one workspace per concurrently running call.
 *
 * Supported: hd in {64, 128, 256}, n_kv >= 1, and
 *   decode windows: 1 <= n_tok <= 16, M <= 512 (both engines);
 *   longer query windows (prefill, e.g. a prefix with KV length = query
 *   count and a pad-only mask): n_tok <= 8192, M <= 65536, with n_tok <= 16
 *   or n_head >= 8 (every 128-row tile then spans at most 16 consecutive
 *   tokens, whose mask rows it reads as one window); tcgen05 engine only.
 */
fr_status fr_decode_attn(const uint16_t* q16,
                         const float* q, int64_t q_tok_stride, const int32_t* pos,
                         const fr_rope_params* rp, float q_scale,
                         const uint16_t* k, int64_t k_row_stride,
                         const uint16_t* v, int64_t v_row_stride,
                         const uint16_t* mask, int64_t mask_row_stride,
                         int n_tok, int n_head, int hd, int n_kv, float kq_scale,
                         float* out, void* workspace, size_t workspace_bytes,
                         cudaStream_t stream);

/*
 * Test and tuning hook (not needed by ordinary callers): fr_decode_attn with
 * explicit choices. Results agree with fr_decode_attn within fp32
 * rounding-order differences. opts may be NULL (all defaults).
 */
typedef struct fr_attn_opts {
    int engine;            /* 0 = default (tcgen05 tensor-core kernel); 1 = mma.sync kernel */
    int force_splits;      /* 0 = library's choice; else KV splits per 128-row tile */
    int force_cluster;     /* 0 = library's choice; else 1, 2, 4 or 8 CTAs per cluster */
    int wait_probe_iters;  /* > 0: every CTA also polls, this many times, a barrier that is
                              never signalled; fr_workspace_check then reports
                              FR_ERR_DEVICE_TIMEOUT (exercises the timeout path) */
    int merge_mode;        /* 0 = library's choice; 1 = merge the split states inside the
                              attention launch (clusters + arrival tickets); 2 = a separate
                              merge kernel (split count cut to what the workspace holds;
                              FR_ERR_WORKSPACE if forced splits do not fit) */
    int layout;            /* 0 = library's choice; 1 = 128-row query tiles (the query rows
                              are the MMA's M); 2 = 128-key tiles as the MMA's M and the
                              query rows as its N (M <= 128 rows, hd 128 or 256, n_tok <= 16:
                              FR_ERR_UNSUPPORTED otherwise). The library's choice (measured
                              faster there) is 2 with 16-row slices when n_kv >= 1024 and
                              ceil(M/16) * n_kv <= 32768 (hd 256) or 16384 (hd 128); 2 with
                              one slice of all rows when M <= 32 and n_kv >= max(1024, 256 M);
                              else 1 — unless
                              force_cluster or merge_mode 1 is given (then 1). */
    int slice_rows;        /* layout 2 only: 0 = library's choice; else 16, 32 or 64 query
                              rows per CTA (the MMA's N): the M rows are cut into
                              ceil(M / slice_rows) slices, each KV split is then read by that
                              many CTAs (one per slice; the later reads served by L2), and
                              the KV splits are the SMs / slices. With layout 2 forced where
                              the library would not pick it, the default is one slice up to
                              64 rows and 32-row slices beyond. */
} fr_attn_opts;

fr_status fr_decode_attn_ex(const uint16_t* q16,
                            const float* q, int64_t q_tok_stride, const int32_t* pos,
                            const fr_rope_params* rp, float q_scale,
                            const uint16_t* k, int64_t k_row_stride,
                            const uint16_t* v, int64_t v_row_stride,
                            const uint16_t* mask, int64_t mask_row_stride,
                            int n_tok, int n_head, int hd, int n_kv, float kq_scale,
                            float* out, void* workspace, size_t workspace_bytes,
                            const fr_attn_opts* opts, cudaStream_t stream);

/*
 * Launch shape fr_decode_attn / fr_decode_attn_ex would use for this shape on
 * the current device, with a workspace of workspace_bytes and these options
 * (opts may be NULL); nothing is launched. fused_qkv_post != 0 describes the
 * call with q16 == NULL. FlashRT PR #185 has no counterpart: the pages' host
 * adapter sizes its launches internally.
 */
typedef struct fr_attn_plan {
    int engine;            /* 0 tcgen05 kernel, 1 mma.sync kernel */
    int row_tiles;         /* query-row tiles (128 rows tcgen05, 64 mma.sync) */
    int splits;            /* KV splits per row tile */
    int cluster;           /* CTAs per thread-block cluster (1 = none) */
    int merge_kernel;      /* 1: split states merged by a separate kernel */
    int launches;          /* kernels one call launches (qkv_post, attention, merge) */
    int keys_on_m;         /* 1: 128-key tiles are the MMA's M, the query rows its N */
    int layout;            /* kernel: 1 = 128-row query tiles, 2 = keys on M (see
                              fr_attn_opts.layout) */
    int row_slices;        /* layout 2: CTAs per KV split (slices of the query rows); else 1 */
} fr_attn_plan;

fr_status fr_decode_attn_plan(int n_tok, int n_head, int hd, int n_kv, int fused_qkv_post,
                              size_t workspace_bytes, const fr_attn_opts* opts, fr_attn_plan* plan);

/*
 * fr_decode_attn_noalloc -- fr_decode_attn without a workspace argument, for
 * callers that cannot allocate device memory (their memory is planned up front
 * by an allocator they do not control, or they must not allocate once running).
 * The FlashRT pages have no counterpart to this entry point.
 *
 * Same arguments and result as fr_decode_attn, minus the workspace. The split
 * state lives in a 9 MiB scratch array inside the library, present on every GPU
 * that loads the library until the process exits. Within it the library picks
 * only plans that fit; shapes whose smallest accepted workspace exceeds 9 MiB
 * return FR_ERR_WORKSPACE. With M = n_tok*n_head those are: hd 64 with
 * M >= 24065; hd 128 with M >= 12161; hd 256 with 257 <= M <= 512 or
 * M >= 6047 (the f16 Q slot plus one partial state per row of the 128-row
 * kernel's in-launch plan). No device memory is allocated.
 * The first call on each device looks up the array's device address
 * (cudaGetSymbolAddress); make that first call before any stream capture. Each
 * call clears the array's arrival tickets on `stream` before launching; its
 * status word is kept, so a bounded device-side wait that gave up in any call
 * is reported by the next fr_decode_attn_noalloc_check. Every call shares the
 * one array: calls that overlap on the GPU (other streams, other host threads)
 * race and must be serialised by the caller.
 */
fr_status fr_decode_attn_noalloc(const uint16_t* q16,
                                 const float* q, int64_t q_tok_stride, const int32_t* pos,
                                 const fr_rope_params* rp, float q_scale,
                                 const uint16_t* k, int64_t k_row_stride,
                                 const uint16_t* v, int64_t v_row_stride,
                                 const uint16_t* mask, int64_t mask_row_stride,
                                 int n_tok, int n_head, int hd, int n_kv, float kq_scale,
                                 float* out, cudaStream_t stream);

/*
 * fr_decode_attn_noalloc_check -- fr_workspace_check for the scratch array of
 * fr_decode_attn_noalloc on the current device: synchronises `stream`, returns
 * FR_ERR_DEVICE_TIMEOUT (and clears the word) if a bounded device-side wait of
 * an earlier fr_decode_attn_noalloc call gave up, else FR_OK. Allocates
 * nothing. The pages have no counterpart to this entry point.
 */
fr_status fr_decode_attn_noalloc_check(cudaStream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* FR_KERNELS_H */
