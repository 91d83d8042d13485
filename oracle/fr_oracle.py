"""fp64 CPU oracle: qkv_post (NEOX RoPE + YaRN, scale, f16 t-major Q rows)
followed by the collapsed GQA decode attention over one KV head.

TEST INFRASTRUCTURE ONLY: imported by tests/, __graft_entry__.smoke() and the
benchmark's CPU baseline, never by the product path. Shares no code with the
CUDA kernels. Everything is computed in float64 with numpy; matrix products
use numpy's matmul as a library primitive, with no blocking or fusion beyond
what each definition states.

Sources (the FlashRT pages):
  * FlashRT PR #185 "ggml host adapter", commit "qkv_post ... f16 Q rows":
    qkv_post stores rope'd+scaled Q rows as f16 in the [M, Nq] = t-major order
    the decode attention consumes.
  * FlashRT PR #185, commit "FLASH_ATTN_EXT with q_tokens <= 16": batched QK^T
    with a stride-0 K operand shared by the GQA heads, masked fp32-accurate
    softmax, PV whose fp32 result lands in [hd, n_head, n_tok].
  * FlashRT PR #185, commit "The GQA query heads share the one KV head": the
    per-head GEMMs collapse into one GEMM over n_head*n_tok t-major rows,
    numerically identical to the batched form.
  * FlashRT-llama.cpp development guide, "Invariants and pitfalls": RoPE
    mirrors ggml's rope_neox with the YaRN corrections; non-NEOX modes are
    rejected.

The pages name the YaRN corrections but do not print them. They are taken from
ggml's published rope_ext semantics, which follow the YaRN paper (Peng et al.,
2023, "YaRN: Efficient Context Window Extension of Large Language Models"):
correction dimensions from beta_fast/beta_slow, a ramp that is linear in the
pair index between them, and the attention-magnitude factor 1 + 0.1 ln(s).

Parity pins: every function here is checked by tests/test_oracle_*.py against
closed forms, hand-derived fixtures (tests/golden/), invariants and an
independent library routine (torch scaled_dot_product_attention in float64).
"""
import math
import numpy as np


def f16_round(x):
    """Round-to-nearest-even to IEEE binary16 (numpy's exact double->half)."""
    return np.asarray(x, dtype=np.float64).astype(np.float16)


# ---------------------------------------------------------------------------
# RoPE (NEOX) with YaRN
# ---------------------------------------------------------------------------

def yarn_corr_dims(n_dims, n_ctx_orig, freq_base, beta_fast, beta_slow):
    """Correction range [c0, c1] of pair indices (YaRN, as ggml applies it).

    The pair index d whose wavelength 2*pi*base^(2d/n_dims) fits n_ctx_orig/beta
    times into the original context is
        d(beta) = n_dims * ln(n_ctx_orig / (2*pi*beta)) / (2 ln base).
    c0 = max(0, floor(d(beta_fast))), c1 = min(n_dims - 1, ceil(d(beta_slow))).
    """
    def d(beta):
        return n_dims * math.log(n_ctx_orig / (2.0 * math.pi * beta)) / (2.0 * math.log(freq_base))
    c0 = max(0.0, float(math.floor(d(beta_fast))))
    c1 = min(float(n_dims - 1), float(math.ceil(d(beta_slow))))
    return c0, c1


def _freq_factors(rp):
    """rope_ext's optional per-pair divisors of the angle (1 when absent). They
    are an fp32 input (ggml's rope_ext takes an F32 tensor), so they are
    rounded to fp32 first, like the Q rows."""
    half = rp.n_dims // 2
    ff = getattr(rp, "freq_factors", None)
    if ff is None:
        return np.ones(half)
    ff = np.asarray(ff, dtype=np.float32).astype(np.float64)
    assert ff.shape == (half,)
    return ff


def rope_theta(pos, rp):
    """Angles theta[t, i] for pairs i < n_dims/2 and the magnitude factor mscale.

    theta_ext = pos * base^(-2i/n_dims) / ff_i; theta_int = freq_scale * theta_ext.
    With ext_factor != 0 the two are mixed by ramp(i) * ext_factor, where
    ramp(i) = 1 - clamp((i - c0) / max(0.001, c1 - c0), 0, 1), and mscale is
    attn_factor * (1 + 0.1 ln(1/freq_scale)); otherwise theta = theta_int and
    mscale = attn_factor.
    """
    half = rp.n_dims // 2
    i = np.arange(half, dtype=np.float64)
    pos = np.asarray(pos, dtype=np.float64).reshape(-1, 1)
    theta_ext = pos * np.power(float(rp.freq_base), -2.0 * i / rp.n_dims) / _freq_factors(rp)
    theta_int = float(rp.freq_scale) * theta_ext
    mscale = float(rp.attn_factor)
    if rp.ext_factor != 0.0:
        c0, c1 = yarn_corr_dims(rp.n_dims, rp.n_ctx_orig, rp.freq_base,
                                rp.beta_fast, rp.beta_slow)
        y = (i - c0) / max(0.001, c1 - c0)
        ramp = 1.0 - np.minimum(1.0, np.maximum(0.0, y))
        mix = ramp * float(rp.ext_factor)
        theta = theta_int * (1.0 - mix) + theta_ext * mix
        mscale *= 1.0 + 0.1 * math.log(1.0 / float(rp.freq_scale))
    else:
        theta = theta_int
    return theta, mscale


def rope_theta_scale_f32(rp):
    """ggml's fp32 ratio between consecutive pairs' angles: base raised to the
    fp32 exponent fl(-2/n_dims), rounded once to fp32 (the correctly rounded
    powf; computed here in double, then rounded)."""
    e = np.float32(-2.0) / np.float32(rp.n_dims)
    return np.float32(math.pow(float(np.float32(rp.freq_base)), float(e)))


def rope_theta_f32(pos, rp):
    """Angles of ggml's fp32 RoPE evaluation (mode 1) and its fp32 mscale.

    Every step is one IEEE fp32 operation, rounded to nearest, in the order
    ggml's rope cache takes them (no fused multiply-add):
      theta_0 = fl(pos); theta_i = fl(theta_{i-1} * theta_scale)
      theta_ext = fl(theta_i / ff_i); theta_int = fl(freq_scale * theta_ext)
      ext_factor != 0:  y = fl(fl(i - c0) / max(0.001, fl(c1 - c0)))
                        ramp_mix = fl(fl(1 - clamp(y, 0, 1)) * ext_factor)
                        theta = fl(fl(theta_int * fl(1 - ramp_mix)) + fl(theta_ext * ramp_mix))
                        mscale = fl(attn_factor * fl(1 + fl(0.1 * fl(ln(fl(1 / freq_scale))))))
      else:             theta = theta_int, mscale = attn_factor
    The correction dims c0, c1 are the integers yarn_corr_dims gives. The
    logarithm is rounded once to fp32 from double. Returns (theta float32
    [n_tok, n_dims/2], mscale float32)."""
    f32 = np.float32
    half = rp.n_dims // 2
    ts = rope_theta_scale_f32(rp)
    pos = np.asarray(pos).reshape(-1)
    theta = np.empty((pos.shape[0], half), dtype=f32)
    cur = pos.astype(f32)
    for i in range(half):
        if i > 0:
            cur = (cur * ts).astype(f32)
        theta[:, i] = cur
    ff = _freq_factors(rp).astype(f32)
    th_ext = (theta / ff[None, :]).astype(f32)
    th_int = (f32(rp.freq_scale) * th_ext).astype(f32)
    mscale = f32(rp.attn_factor)
    if rp.ext_factor != 0.0:
        c0, c1 = yarn_corr_dims(rp.n_dims, rp.n_ctx_orig, rp.freq_base, rp.beta_fast, rp.beta_slow)
        c0, c1 = f32(c0), f32(c1)
        i = np.arange(half).astype(f32)
        y = ((i - c0).astype(f32) / np.maximum(f32(0.001), f32(c1 - c0))).astype(f32)
        ramp = (f32(1.0) - np.minimum(f32(1.0), np.maximum(f32(0.0), y))).astype(f32)
        mix = (ramp * f32(rp.ext_factor)).astype(f32)
        a = (th_int * (f32(1.0) - mix).astype(f32)[None, :]).astype(f32)
        b = (th_ext * mix[None, :]).astype(f32)
        th = (a + b).astype(f32)
        lg = f32(math.log(float(f32(1.0) / f32(rp.freq_scale))))
        mscale = f32(mscale * f32(f32(1.0) + f32(f32(0.1) * lg)))
    else:
        th = th_int
    return th, mscale


def rope_neox(x, pos, rp):
    """NEOX rotation of x [n_tok, n_head, hd] at positions pos [n_tok].

    Pair i rotates (x[i], x[i + n_dims/2]) by theta[t, i] (rope_theta, or
    rope_theta_f32 when rp.mode == 1), scaled by mscale:
        y[i]          = x[i] * c - x[i + n/2] * s
        y[i + n/2]    = x[i] * s + x[i + n/2] * c,   c = mscale cos, s = mscale sin
    Dimensions >= n_dims pass through unchanged. Every head of token t uses the
    same angles (the GQA heads share the token position).
    """
    x = np.asarray(x, dtype=np.float64)
    n = rp.n_dims
    half = n // 2
    if getattr(rp, "mode", 0) == 1:
        th32, ms32 = rope_theta_f32(pos, rp)             # ggml's fp32 angles, cos/sin in fp64
        theta, mscale = th32.astype(np.float64), float(ms32)
    else:
        theta, mscale = rope_theta(pos, rp)
    c = (mscale * np.cos(theta))[:, None, :]          # [n_tok, 1, half]
    s = (mscale * np.sin(theta))[:, None, :]
    y = x.copy()
    x0 = x[..., :half]
    x1 = x[..., half:n]
    y[..., :half] = x0 * c - x1 * s
    y[..., half:n] = x0 * s + x1 * c
    return y


def qkv_post(q, pos, rp, q_scale):
    """The Q leg of qkv_post.

    q [n_tok, n_head, hd] (f32, the QKV GEMM's [M=n_tok, Nq] rows) ->
      y   [n_tok*n_head, hd] float64: rope'd then scaled, row r = t*n_head + h
      q16 [n_tok*n_head, hd] float16: y rounded once to f16 (the emitted rows)
    """
    n_tok, n_head, hd = q.shape
    y = rope_neox(q, pos, rp) * float(q_scale)
    rows = y.reshape(n_tok * n_head, hd)          # t-major: r = t*n_head + h
    return rows, f16_round(rows)


def kv_append(k_cache, v_cache, k_new, v_new, pos, rp, row0, pad=None):
    """The K/V leg of qkv_post with the write of the new rows into the
    persistent KV cache (FlashRT PR #185, commit "Fuses the prefix layers'
    q/k/v projections, RoPE, scale, KV padding to the FA KQ stride, and the
    permuted f16 materializations ..."; the full variant "re-emits the rope'd K
    and plain V as f32 rows" and "pad rows are zeroed").

    The new K rows are rotated exactly as the Q rows of the same tokens (same
    angles and mscale, no 1/sqrt(hd) scale); K and V are rounded once to f16
    and written at cache rows row0 + t. pad = (begin, end) rows of both caches
    are set to zero (the attention reads a padded length). Nothing else changes.

    k_cache, v_cache: f16 [n_ctx, hd]; k_new, v_new: [n_tok, hd]; pos: [n_tok].
    Returns (k_cache', v_cache', k_rope fp64 [n_tok, hd], v fp64 [n_tok, hd]).
    """
    k_new = np.asarray(k_new, dtype=np.float64)
    v_new = np.asarray(v_new, dtype=np.float64)
    n_tok = k_new.shape[0]
    k_rope = rope_neox(k_new[:, None, :], pos, rp)[:, 0, :]
    kc = np.array(k_cache, dtype=np.float16, copy=True)
    vc = np.array(v_cache, dtype=np.float16, copy=True)
    kc[row0:row0 + n_tok] = f16_round(k_rope)
    vc[row0:row0 + n_tok] = f16_round(v_new)
    if pad is not None:
        kc[pad[0]:pad[1]] = 0
        vc[pad[0]:pad[1]] = 0
    return kc, vc, k_rope, v_new


# ---------------------------------------------------------------------------
# Attention over one shared KV head
# ---------------------------------------------------------------------------

def _scores(qrows, k, mask, row_tok, kq_scale):
    s = float(kq_scale) * (np.asarray(qrows, np.float64) @ np.asarray(k, np.float64).T)
    if mask is not None:
        s = s + np.asarray(mask, np.float64)[row_tok, :]
    return s


def _softmax_pv(s, v):
    """Masked softmax of score rows s, then P V. -inf columns get weight 0;
    a row with every column masked yields 0."""
    m = np.max(s, axis=1, keepdims=True)
    m_safe = np.where(np.isfinite(m), m, 0.0)
    p = np.exp(s - m_safe)
    l = np.sum(p, axis=1, keepdims=True)
    o = p @ np.asarray(v, np.float64)
    l_safe = np.where(l > 0.0, l, 1.0)
    return np.where(l > 0.0, o / l_safe, 0.0)


def attention_collapsed(qrows, k, v, mask, n_tok, n_head, kq_scale=1.0):
    """One QK^T over all M = n_tok*n_head t-major rows (K shared, stride 0 across
    heads), masked softmax, one PV. Row r uses mask row t = r // n_head.
    Returns [M, hd] float64 == [n_tok][n_head][hd] == ggml [hd, n_head, n_tok]."""
    M = n_tok * n_head
    row_tok = np.arange(M) // n_head
    return _softmax_pv(_scores(qrows, k, mask, row_tok, kq_scale), v)


def attention_batched(qrows, k, v, mask, n_tok, n_head, kq_scale=1.0):
    """The per-head batched form: for each head h, a GEMM over its n_tok rows
    against the shared K, softmax, a GEMM against the shared V, stored
    strided into [n_tok][n_head][hd]."""
    hd = k.shape[1]
    q3 = np.asarray(qrows, np.float64).reshape(n_tok, n_head, hd)
    out = np.zeros((n_tok, n_head, hd))
    for h in range(n_head):
        s = _scores(q3[:, h, :], k, mask, np.arange(n_tok), kq_scale)
        out[:, h, :] = _softmax_pv(s, v)
    return out.reshape(n_tok * n_head, hd)


def attention_rows(qrows, k, v, mask, rows, n_head, kq_scale=1.0):
    """Selected output rows only (for sampled checks at full size)."""
    rows = np.asarray(rows)
    row_tok = rows // n_head
    return _softmax_pv(_scores(np.asarray(qrows)[rows], k, mask, row_tok, kq_scale), v)


def split_partials(qrows, k, v, mask, n_tok, n_head, kq_scale, n_splits):
    """Per-split (m, l, O): the softmax state of each contiguous KV chunk."""
    M = n_tok * n_head
    n_kv = k.shape[0]
    row_tok = np.arange(M) // n_head
    bounds = np.linspace(0, n_kv, n_splits + 1).astype(int)
    parts = []
    for a, b in zip(bounds[:-1], bounds[1:]):
        s = _scores(qrows, k[a:b], None if mask is None else np.asarray(mask)[:, a:b],
                    row_tok, kq_scale)
        if b == a:
            parts.append((np.full((M, 1), -np.inf), np.zeros((M, 1)), np.zeros((M, k.shape[1]))))
            continue
        m = np.max(s, axis=1, keepdims=True)
        m_safe = np.where(np.isfinite(m), m, 0.0)
        p = np.exp(s - m_safe)
        parts.append((m, np.sum(p, axis=1, keepdims=True), p @ np.asarray(v[a:b], np.float64)))
    return parts


def merge_partials(parts):
    """Combine split states: m = max_s m_s, O = sum e^(m_s-m) O_s / sum e^(m_s-m) l_s."""
    ms = np.concatenate([p[0] for p in parts], axis=1)
    m = np.max(ms, axis=1, keepdims=True)
    m_safe = np.where(np.isfinite(m), m, 0.0)
    num = 0.0
    den = 0.0
    for (ms_, ls_, os_) in parts:
        ms_safe = np.where(np.isfinite(ms_), ms_, 0.0)
        w = np.where(np.isfinite(ms_), np.exp(ms_safe - m_safe), 0.0)
        num = num + w * os_
        den = den + w * ls_
    den_safe = np.where(den > 0.0, den, 1.0)
    return np.where(den > 0.0, num / den_safe, 0.0)


def attention_split_merge(qrows, k, v, mask, n_tok, n_head, kq_scale=1.0, n_splits=4):
    return merge_partials(split_partials(qrows, k, v, mask, n_tok, n_head, kq_scale, n_splits))


# ---------------------------------------------------------------------------
# The whole path
# ---------------------------------------------------------------------------

def decode_attn(q, pos, k, v, mask, rp, q_scale, kq_scale=1.0, rows=None):
    """qkv_post then attention. The attention consumes the f16 Q rows that
    qkv_post emits; everything after that rounding is float64.
    Returns float64 [M, hd] (t-major rows r = t*n_head + h), or only `rows`."""
    n_tok, n_head, _ = q.shape
    _, q16 = qkv_post(q, pos, rp, q_scale)
    qrows = np.asarray(q16, np.float64)
    if rows is not None:
        return attention_rows(qrows, k, v, mask, rows, n_head, kq_scale)
    return attention_collapsed(qrows, k, v, mask, n_tok, n_head, kq_scale)
