"""GPU parity of the ggml float-compat RoPE mode (FR_ROPE_GGML_F32) and of
freq_factors (both modes) against the oracle, through the C ABI.

FlashRT-llama.cpp development guide, "Invariants and pitfalls": RoPE mirrors
ggml's rope_neox (YaRN corrections included) and must stay bit-exact with it.
The angles follow ggml's fp32 recurrence step for step; the kernel then takes
fp32 sincos, the oracle fp64 cos/sin of the same fp32 angles, so the f32 rows
agree within fp32 sincos and rotation rounding: |q32 - y| <= 16 * 2^-24 *
(|x0| + |x1|) * mscale * q_scale per element (an angle off by the fp32
recurrence error at these positions, ~1e-3 rad, is ~100x that)."""
import numpy as np
import pytest
import torch

import oracle
from gen import RopeParams, make_workload, named_config
import gqa_kv_head_gb300 as fr
from fr_harness import assert_close, host_kv, oracle_out, run_fused, run_two_call, to_device

pytestmark = pytest.mark.gpu

LLAMA_FF = tuple(1.0 if i < 20 else (8.0 if i > 44 else 1.0 + 7.0 * (i - 20) / 24.0) for i in range(64))


def _ulp_diff(a16, b16):
    a = np.asarray(a16, np.float16).view(np.int16).astype(np.int32)
    b = np.asarray(b16, np.float16).view(np.int16).astype(np.int32)
    a = np.where(a < 0, -32768 - a, a)
    b = np.where(b < 0, -32768 - b, b)
    return np.abs(a - b)


def _bound(w):
    """Per-element bound of the f32 rows (see the module docstring)."""
    q = w.q().astype(np.float64)
    n, half = w.rope.n_dims, w.rope.n_dims // 2
    if w.rope.mode == 1:
        _, ms = oracle.rope_theta_f32(w.pos(), w.rope)
    else:
        _, ms = oracle.rope_theta(w.pos(), w.rope)
    pair = np.abs(q[..., :half]) + np.abs(q[..., half:n])
    b = np.zeros_like(q)
    b[..., :half] = pair
    b[..., half:n] = pair
    b[..., n:] = np.abs(q[..., n:])
    return (16 * 2.0 ** -24 * b * float(ms) * abs(w.q_scale) + 2.0 ** -40).reshape(w.M, w.hd)


CASES = [
    ("long_decode", dict(mode=1)),
    ("long_decode", dict(mode=1, freq_factors=LLAMA_FF)),
    ("long_decode", dict(mode=0, freq_factors=LLAMA_FF)),
    ("pi05", dict(mode=1)),
    ("c3", dict(mode=1)),
    ("sweep:128:4:65536", dict(mode=1)),
    ("tiny", dict(mode=1)),
]


def _workload(name, kw):
    w = make_workload(name)
    ff = kw.get("freq_factors")
    if ff is not None and len(ff) != w.rope.n_dims // 2:
        ff = tuple(ff[i % len(ff)] for i in range(w.rope.n_dims // 2))
    rp = RopeParams(**{**w.rope.__dict__, "mode": kw.get("mode", 0), "freq_factors": ff})
    return w.with_(rope=rp)


@pytest.mark.parametrize("name,kw", CASES)
def test_qkv_post_rows(name, kw):
    w = _workload(name, kw)
    q = torch.from_numpy(w.q()).cuda()
    pos = torch.from_numpy(w.pos()).cuda()
    q32 = torch.empty((w.M, w.hd), dtype=torch.float32, device="cuda")
    q16, _ = fr.qkv_post(q, pos, w.n_head, w.hd, w.rope, w.q_scale, q32_out=q32)
    torch.cuda.synchronize()
    rows, want16 = oracle.qkv_post(w.q(), w.pos(), w.rope, w.q_scale)
    got32 = q32.cpu().numpy().astype(np.float64)
    if w.rope.mode == 1:
        assert np.all(np.abs(got32 - rows) <= _bound(w)), np.max(np.abs(got32 - rows) / _bound(w))
    else:
        assert np.max(np.abs(got32 - rows)) <= 2e-6 * max(1.0, np.abs(rows).max())
    ulps = _ulp_diff(q16.cpu().numpy(), want16)
    assert ulps.max() <= 1 and (ulps == 0).mean() >= 0.99


def test_float_mode_differs_from_exact_mode_at_large_positions():
    """At positions ~32k the fp32 recurrence's angles differ from the exact
    ones by ~1e-3 rad: the two modes must give visibly different rows (the
    mode flag reaches the kernel)."""
    w0 = _workload("long_decode", dict(mode=0))
    w1 = _workload("long_decode", dict(mode=1))
    outs = []
    for w in (w0, w1):
        q32 = torch.empty((w.M, w.hd), dtype=torch.float32, device="cuda")
        fr.qkv_post(torch.from_numpy(w.q()).cuda(), torch.from_numpy(w.pos()).cuda(), w.n_head, w.hd, w.rope,
                    w.q_scale, q32_out=q32)
        outs.append(q32.cpu().numpy())
    assert np.max(np.abs(outs[0] - outs[1])) > 1e-5


@pytest.mark.parametrize("name,kw", [CASES[0], CASES[1], CASES[3]])
def test_attention_and_fused_equals_two_call(name, kw):
    w = _workload(name, kw)
    d = to_device(w)
    a = run_fused(w, d)
    b, _ = run_two_call(w, d)
    torch.cuda.synchronize()
    assert torch.equal(a, b)
    assert_close(a.reshape(w.M, w.hd).cpu().numpy().astype(np.float64), oracle_out(w), f"{name} {kw}")


def test_kv_append_float_mode():
    w = _workload("long_decode", dict(mode=1, freq_factors=LLAMA_FF))
    hd = w.hd
    rng = np.random.default_rng(5)
    k_new = rng.standard_normal((w.n_tok, hd)).astype(np.float32)
    v_new = rng.standard_normal((w.n_tok, hd)).astype(np.float32)
    k0 = rng.standard_normal((w.n_kv, hd)).astype(np.float16)
    kc = torch.from_numpy(k0.copy()).cuda()
    vc = torch.from_numpy(k0.copy()).cuda()
    row0 = w.n_kv - w.n_tok
    fr.kv_append(torch.from_numpy(k_new).cuda(), torch.from_numpy(v_new).cuda(), torch.from_numpy(w.pos()).cuda(),
                 w.rope, kc, vc, row0)
    torch.cuda.synchronize()
    kw_, vw_, _, _ = oracle.kv_append(k0, k0, k_new, v_new, w.pos(), w.rope, row0)
    got = kc.cpu().numpy()
    ulps = _ulp_diff(got[row0:], kw_[row0:])
    assert ulps.max() <= 1 and (ulps == 0).mean() >= 0.99
    assert np.array_equal(got[:row0].view(np.uint16), k0[:row0].view(np.uint16))
