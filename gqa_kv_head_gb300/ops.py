"""Python binding of the C ABI: argument marshalling only.

Every function takes torch CUDA tensors, passes their device pointers, strides
and the current CUDA stream to the library, and raises FrError on a non-OK
status. All arithmetic happens in the library's kernels.
"""
import ctypes

import torch

from . import _abi
from ._abi import FrAttnOpts, FrError, FrRopeParams


def rope_params(n_dims, freq_base=10000.0, freq_scale=1.0, ext_factor=0.0, attn_factor=1.0,
                beta_fast=32.0, beta_slow=1.0, n_ctx_orig=4096, mode=0, freq_factors=None):
    """fr_rope_params. mode: 0 = FR_ROPE_EXACT, 1 = FR_ROPE_GGML_F32;
    freq_factors: None or n_dims/2 floats (kept alive by the returned struct)."""
    ff = None
    if freq_factors is not None:
        ff = (ctypes.c_float * len(freq_factors))(*[float(x) for x in freq_factors])
    rp = FrRopeParams(int(n_dims), float(freq_base), float(freq_scale), float(ext_factor),
                      float(attn_factor), float(beta_fast), float(beta_slow), int(n_ctx_orig), int(mode),
                      ctypes.cast(ff, ctypes.POINTER(ctypes.c_float)) if ff is not None else None)
    rp._ff_keepalive = ff
    return rp


def _as_rope(rp):
    if rp is None or isinstance(rp, FrRopeParams):
        return rp
    return rope_params(rp.n_dims, rp.freq_base, rp.freq_scale, rp.ext_factor, rp.attn_factor,
                       rp.beta_fast, rp.beta_slow, rp.n_ctx_orig, getattr(rp, "mode", 0),
                       getattr(rp, "freq_factors", None))


def _stream(stream):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _q_scale(q_scale):
    """None -> FR_Q_SCALE_DEFAULT (0): the library applies 1/sqrt(hd)."""
    return 0.0 if q_scale is None else float(q_scale)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _check_dev(*ts):
    for t in ts:
        if t is not None and not t.is_cuda:
            raise ValueError("tensors must be CUDA tensors")


def _q_tok_stride(q, n_head, hd):
    """q is [n_tok, n_head, hd] (or [n_tok, >= n_head*hd]) f32 with unit inner strides."""
    if q.dtype != torch.float32:
        raise TypeError("q must be float32")
    if q.dim() == 3:
        if q.stride(2) != 1 or q.stride(1) != hd:
            raise ValueError("q [n_tok, n_head, hd] needs contiguous heads")
        return q.stride(0)
    if q.dim() == 2 and q.stride(1) == 1:
        return q.stride(0)
    raise ValueError("q must be [n_tok, n_head, hd] or [n_tok, Nq]")


def qkv_post(q, pos, n_head, hd, rope, q_scale=None, q16_out=None, q32_out=None, stream=None):
    """fr_qkv_post. Returns (q16 [n_tok*n_head, hd] f16, q32 or None)."""
    lib = _abi.load()
    _check_dev(q, pos, q16_out, q32_out)
    n_tok = q.shape[0]
    if q16_out is None:
        q16_out = torch.empty((n_tok * n_head, hd), dtype=torch.float16, device=q.device)
    rp = _as_rope(rope)
    st = lib.fr_qkv_post(_ptr(q), _q_tok_stride(q, n_head, hd), _ptr(pos), n_tok, n_head, hd,
                         ctypes.byref(rp), _q_scale(q_scale), _ptr(q16_out), _ptr(q32_out),
                         _stream(stream))
    _abi.check(st, "fr_qkv_post")
    return q16_out, q32_out


def kv_append(k_new, v_new, pos, rope, k_cache, v_cache, row0, pad=None, k32_out=None, v32_out=None,
              stream=None):
    """fr_kv_append: rope the new K rows, round K and V to f16 and write them at
    cache rows row0 .. row0 + n_tok - 1; zero the pad rows (pad = (begin, end)).
    k_new, v_new: f32 [n_tok, hd] (row stride may exceed hd, e.g. columns of a
    fused QKV buffer); k_cache, v_cache: f16 [n_ctx, hd] (row stride >= hd)."""
    lib = _abi.load()
    _check_dev(k_new, v_new, pos, k_cache, v_cache, k32_out, v32_out)
    for name, t in (("k_new", k_new), ("v_new", v_new), ("k32_out", k32_out), ("v32_out", v32_out)):
        if t is not None and t.dtype != torch.float32:
            raise TypeError(f"{name} must be float32")
    for name, t in (("k_cache", k_cache), ("v_cache", v_cache)):
        if t.dtype != torch.float16:
            raise TypeError(f"{name} must be float16")
    if pos.dtype != torch.int32:
        raise TypeError("pos must be int32")
    n_tok, hd = k_new.shape[0], k_new.shape[1]
    if tuple(v_new.shape) != (n_tok, hd) or k_cache.shape[1] != hd or tuple(v_cache.shape) != tuple(k_cache.shape):
        raise ValueError("shape mismatch")
    pb, pe = pad if pad is not None else (0, 0)
    rp = _as_rope(rope)
    st = lib.fr_kv_append(_ptr(k_new), _row_stride(k_new, "k_new"), _ptr(v_new), _row_stride(v_new, "v_new"),
                          _ptr(pos), n_tok, hd, ctypes.byref(rp), _ptr(k_cache), _row_stride(k_cache, "k_cache"),
                          _ptr(v_cache), _row_stride(v_cache, "v_cache"), k_cache.shape[0], int(row0), int(pb),
                          int(pe), _ptr(k32_out), _ptr(v32_out), _stream(stream))
    _abi.check(st, "fr_kv_append")


def workspace_size(n_tok, n_head, hd, n_kv):
    return int(_abi.load().fr_decode_attn_workspace_size(n_tok, n_head, hd, n_kv))


def make_workspace(n_tok, n_head, hd, n_kv, device="cuda", stream=None):
    """Allocate (torch) and zero (library) a workspace for this shape."""
    n = workspace_size(n_tok, n_head, hd, n_kv)
    if n == 0:
        raise FrError(2, "fr_decode_attn_workspace_size")
    ws = torch.empty(n, dtype=torch.uint8, device=device)
    _abi.check(_abi.load().fr_workspace_init(_ptr(ws), n, _stream(stream)), "fr_workspace_init")
    return ws


def workspace_check(ws, stream=None):
    _abi.check(_abi.load().fr_workspace_check(_ptr(ws), _stream(stream)), "fr_workspace_check")


def _row_stride(t, name):
    if t.dim() != 2 or t.stride(1) != 1:
        raise ValueError(f"{name} must be 2-D with unit inner stride")
    return t.stride(0)


def decode_attn(k, v, n_tok, n_head, *, q16=None, q=None, pos=None, rope=None, q_scale=None,
                mask=None, kq_scale=1.0, out=None, workspace=None, splits=None, cluster=None,
                engine=None, wait_probe_iters=0, merge_mode=None, layout=None, slice_rows=None, stream=None):
    """fr_decode_attn (fused qkv_post when q16 is None). Returns out
    [n_tok, n_head, hd] f32. splits / cluster / engine / wait_probe_iters /
    merge_mode / layout / slice_rows go through the fr_decode_attn_ex test
    hook."""
    lib = _abi.load()
    _check_dev(k, v, q16, q, pos, mask, out, workspace)
    n_kv, hd = k.shape[0], k.shape[1]
    for name, t in (("k", k), ("v", v), ("mask", mask), ("q16", q16)):
        if t is not None and t.dtype != torch.float16:
            raise TypeError(f"{name} must be float16")
    if out is None:
        out = torch.empty((n_tok, n_head, hd), dtype=torch.float32, device=k.device)
    if workspace is None:
        workspace = make_workspace(n_tok, n_head, hd, n_kv, device=k.device, stream=stream)
    q_stride = 0
    rp = None
    if q16 is None:
        if q is None or pos is None or rope is None:
            raise ValueError("pass q16, or q + pos + rope for the fused path")
        q_stride = _q_tok_stride(q, n_head, hd)
        rp = _as_rope(rope)
    args = [_ptr(q16), _ptr(q), q_stride, _ptr(pos), ctypes.byref(rp) if rp is not None else None,
            _q_scale(q_scale), _ptr(k), _row_stride(k, "k"), _ptr(v), _row_stride(v, "v"),
            _ptr(mask), 0 if mask is None else _row_stride(mask, "mask"), n_tok, n_head, hd, n_kv,
            float(kq_scale), _ptr(out), _ptr(workspace), workspace.numel()]
    if (splits is None and cluster is None and engine is None and not wait_probe_iters and not merge_mode
            and not layout and not slice_rows):
        st = lib.fr_decode_attn(*args, _stream(stream))
        _abi.check(st, "fr_decode_attn")
    else:
        opts = FrAttnOpts(int(engine or 0), int(splits or 0), int(cluster or 0), int(wait_probe_iters),
                          int(merge_mode or 0), int(layout or 0), int(slice_rows or 0))
        st = lib.fr_decode_attn_ex(*args, ctypes.byref(opts), _stream(stream))
        _abi.check(st, "fr_decode_attn_ex")
    return out


def decode_attn_plan(n_tok, n_head, hd, n_kv, *, fused_qkv_post=True, workspace_bytes=None,
                     splits=None, cluster=None, engine=None, merge_mode=None, layout=None, slice_rows=None):
    """fr_decode_attn_plan: the launch shape a call with these arguments would
    use on the current device (nothing is launched). Returns a dict with
    engine, row_tiles, splits, cluster, merge_kernel, launches, keys_on_m,
    layout, row_slices."""
    lib = _abi.load()
    if workspace_bytes is None:
        workspace_bytes = workspace_size(n_tok, n_head, hd, n_kv)
    opts = FrAttnOpts(int(engine or 0), int(splits or 0), int(cluster or 0), 0, int(merge_mode or 0),
                      int(layout or 0), int(slice_rows or 0))
    plan = _abi.FrAttnPlan()
    st = lib.fr_decode_attn_plan(n_tok, n_head, hd, n_kv, 1 if fused_qkv_post else 0, int(workspace_bytes),
                                 ctypes.byref(opts), ctypes.byref(plan))
    _abi.check(st, "fr_decode_attn_plan")
    return {name: getattr(plan, name) for name, _ in plan._fields_}


def decode_attn_noalloc(k, v, n_tok, n_head, *, q16=None, q=None, pos=None, rope=None, q_scale=None,
                        mask=None, kq_scale=1.0, out=None, stream=None):
    """fr_decode_attn_noalloc: the same attention without a workspace, for
    callers that cannot allocate device memory (the library's fixed scratch is
    used instead; see include/fr_kernels.h for its limit and sharing rules).
    Returns out [n_tok, n_head, hd] f32 (allocated here only if not given)."""
    lib = _abi.load()
    _check_dev(k, v, q16, q, pos, mask, out)
    n_kv, hd = k.shape[0], k.shape[1]
    if out is None:
        out = torch.empty((n_tok, n_head, hd), dtype=torch.float32, device=k.device)
    q_stride = 0
    rp = None
    if q16 is None:
        if q is None or pos is None or rope is None:
            raise ValueError("pass q16, or q + pos + rope for the fused path")
        q_stride = _q_tok_stride(q, n_head, hd)
        rp = _as_rope(rope)
    st = lib.fr_decode_attn_noalloc(
        _ptr(q16), _ptr(q), q_stride, _ptr(pos), ctypes.byref(rp) if rp is not None else None,
        _q_scale(q_scale), _ptr(k), _row_stride(k, "k"), _ptr(v), _row_stride(v, "v"), _ptr(mask),
        0 if mask is None else _row_stride(mask, "mask"), n_tok, n_head, hd, n_kv, float(kq_scale),
        _ptr(out), _stream(stream))
    _abi.check(st, "fr_decode_attn_noalloc")
    return out


def decode_attn_noalloc_check(stream=None):
    """fr_decode_attn_noalloc_check: raise FrError (FR_ERR_DEVICE_TIMEOUT) if a
    bounded device-side wait of an earlier decode_attn_noalloc call gave up."""
    _abi.check(_abi.load().fr_decode_attn_noalloc_check(_stream(stream)), "fr_decode_attn_noalloc_check")
