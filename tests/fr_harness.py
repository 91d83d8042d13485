"""Shared helpers for the GPU tests: move a gen.Workload to the device (with
optional padded strides), run the library through its C ABI, and compare
against the oracle with the parity tolerance."""
import functools

import numpy as np
import torch

import gqa_kv_head_gb300 as fr

# spec tolerance for the f16-in / fp32-out attention
MAX_ABS = 2e-3
REL_L2 = 1e-3


def rel_err(got, ref):
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    d = got - ref
    max_abs = float(np.max(np.abs(d))) if d.size else 0.0
    den = float(np.linalg.norm(ref))
    rel = float(np.linalg.norm(d)) / den if den > 0 else float(np.linalg.norm(d))
    return max_abs, rel


def assert_close(got, ref, what=""):
    max_abs, rel = rel_err(got, ref)
    assert np.all(np.isfinite(got)), f"{what}: non-finite output"
    assert max_abs <= MAX_ABS and rel <= REL_L2, f"{what}: max_abs={max_abs:.3e} rel_l2={rel:.3e}"
    return max_abs, rel


@functools.lru_cache(maxsize=16)
def _kv_cached(hd, n_kv, n_kv_real, sigma, outlier_p, outlier_mult, seed):
    # K/V depend only on these fields (not on n_tok / n_head)
    from gen import Workload, RopeParams
    w = Workload("kv", n_head=1, n_tok=1, hd=hd, n_kv=n_kv, rope=RopeParams(n_dims=hd),
                 positions=(0,), n_kv_real=n_kv_real, kv_sigma=sigma, outlier_p=outlier_p,
                 outlier_mult=outlier_mult, seed=seed)
    return w.k(), w.v()


def host_kv(w):
    return _kv_cached(w.hd, w.n_kv, w.n_kv_real, w.kv_sigma, w.outlier_p, w.outlier_mult, w.seed)


def _strided_2d(a, row_stride, dev, fill=0.0):
    rows, cols = a.shape
    buf = torch.full((rows, row_stride), fill, dtype=torch.from_numpy(a[:0]).dtype, device=dev)
    view = buf[:, :cols]
    view.copy_(torch.from_numpy(np.ascontiguousarray(a)))
    return view


def to_device(w, k_pad=0, mask_pad=0, q_extra_heads=0, dev="cuda"):
    """Device tensors for workload w. k_pad/mask_pad add elements to the row
    strides; q_extra_heads widens the Q token stride (as in a fused QKV
    GEMM output whose K and V columns follow the Q heads)."""
    k, v = host_kv(w)
    q = w.q()
    qt = torch.zeros((w.n_tok, (w.n_head + q_extra_heads) * w.hd), dtype=torch.float32, device=dev)
    qt[:, :w.n_head * w.hd] = torch.from_numpy(q.reshape(w.n_tok, -1))
    qv = qt[:, :w.n_head * w.hd] if q_extra_heads else qt
    d = {
        "q": qv,
        "pos": torch.from_numpy(w.pos()).to(dev),
        "k": _strided_2d(k, w.hd + k_pad, dev),
        "v": _strided_2d(v, w.hd + k_pad, dev),
        "mask": None,
    }
    m = w.mask()
    if m is not None:
        stride = ((w.n_kv + 7) // 8) * 8 + mask_pad
        d["mask"] = _strided_2d(m, stride, dev)
    return d


def run_fused(w, d, **kw):
    return fr.decode_attn(d["k"], d["v"], w.n_tok, w.n_head, q=d["q"], pos=d["pos"], rope=w.rope,
                          q_scale=w.q_scale, mask=d["mask"], kq_scale=w.kq_scale, **kw)


def run_two_call(w, d, **kw):
    q16, _ = fr.qkv_post(d["q"], d["pos"], w.n_head, w.hd, w.rope, w.q_scale)
    out = fr.decode_attn(d["k"], d["v"], w.n_tok, w.n_head, q16=q16, mask=d["mask"],
                         kq_scale=w.kq_scale, **kw)
    return out, q16


def oracle_out(w, rows=None):
    import oracle
    k, v = host_kv(w)
    return oracle.decode_attn(w.q(), w.pos(), k, v, w.mask(), w.rope, w.q_scale, w.kq_scale,
                              rows=rows)
