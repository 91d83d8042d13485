"""fr_kv_append on the GPU against the oracle's kv_append: K rows within one
f16 ulp of the oracle's rounding (>= 99 % exact, bitwise at position 0), V
rows and pad rows bitwise, every other cache row untouched, the f32 copies,
inputs taken from the K/V columns of a fused QKV buffer, and the append
followed by the fused decode attention against the oracle on the updated
cache."""
import numpy as np
import pytest
import torch

import gqa_kv_head_gb300 as fr
import oracle
from fr_harness import assert_close, host_kv
from gen import RopeParams, named_config

pytestmark = pytest.mark.gpu


def _f16_ulps(a, b):
    """Distance in f16 ulps (sign-magnitude bits mapped to an ordered integer)."""
    def ordered(x):
        u = x.view(np.uint16).astype(np.int32)
        return np.where(u & 0x8000, 0x8000 - u, u)
    return np.abs(ordered(a) - ordered(b))


def _case(w, seed=21):
    """New K/V rows for w's query tokens (cache rows = their positions) inside
    a fused QKV buffer [n_tok][(n_head + 2) hd], and a random f16 cache."""
    rng = np.random.default_rng(seed)
    n_ctx, hd = w.n_kv, w.hd
    qkv = rng.standard_normal((w.n_tok, (w.n_head + 2) * hd)).astype(np.float32)
    k0 = rng.standard_normal((n_ctx, hd)).astype(np.float16)
    v0 = rng.standard_normal((n_ctx, hd)).astype(np.float16)
    return qkv, k0, v0


def _run(w, qkv, k0, v0, row0, pad, pos, want_f32=True):
    hd = w.hd
    d_qkv = torch.from_numpy(qkv).cuda()
    k_new = d_qkv[:, w.n_head * hd:(w.n_head + 1) * hd]
    v_new = d_qkv[:, (w.n_head + 1) * hd:(w.n_head + 2) * hd]
    kc = torch.from_numpy(k0.copy()).cuda()
    vc = torch.from_numpy(v0.copy()).cuda()
    k32 = torch.empty((w.n_tok, hd), dtype=torch.float32, device="cuda") if want_f32 else None
    v32 = torch.empty((w.n_tok, hd), dtype=torch.float32, device="cuda") if want_f32 else None
    fr.kv_append(k_new, v_new, torch.from_numpy(np.asarray(pos, np.int32)).cuda(), w.rope, kc, vc, row0,
                 pad=pad, k32_out=k32, v32_out=v32)
    torch.cuda.synchronize()
    return (kc.cpu().numpy(), vc.cpu().numpy(), None if k32 is None else k32.cpu().numpy(),
            None if v32 is None else v32.cpu().numpy())


@pytest.mark.parametrize("name", ["tiny", "pi05", "c3", "long_decode"])
def test_kv_append_matches_oracle(name):
    w = named_config(name)
    qkv, k0, v0 = _case(w)
    pos = w.pos()
    row0 = w.n_kv_real - w.n_tok                  # the last real rows of the cache
    pad = (w.n_kv_real, w.n_kv) if w.n_kv_real < w.n_kv else None
    kc, vc, k32, v32 = _run(w, qkv, k0, v0, row0, pad, pos)
    hd = w.hd
    k_new = qkv[:, w.n_head * hd:(w.n_head + 1) * hd]
    v_new = qkv[:, (w.n_head + 1) * hd:]
    ok, ov, okr, _ = oracle.kv_append(k0, v0, k_new, v_new, pos, w.rope, row0, pad)
    tail = slice(row0, row0 + w.n_tok)
    ulps = _f16_ulps(kc[tail], ok[tail])
    assert ulps.max() <= 1 and (ulps == 0).mean() >= 0.99, (ulps.max(), (ulps == 0).mean())
    assert np.array_equal(vc[tail].view(np.uint16), ov[tail].view(np.uint16))
    others = np.ones(w.n_kv, bool)
    others[tail] = False
    assert np.array_equal(kc[others].view(np.uint16), ok[others].view(np.uint16))    # untouched or zeroed pad
    assert np.array_equal(vc[others].view(np.uint16), ov[others].view(np.uint16))
    assert np.abs(k32 - okr).max() <= 4e-6 * max(1.0, np.abs(okr).max())
    assert np.array_equal(v32, v_new)


def test_kv_append_identity_at_pos0_bitwise():
    w = named_config("pi05")
    qkv, k0, v0 = _case(w, seed=3)
    pos = np.zeros(w.n_tok, np.int32)
    kc, vc, _, _ = _run(w, qkv, k0, v0, 5, None, pos, want_f32=False)
    hd = w.hd
    want = qkv[:, w.n_head * hd:(w.n_head + 1) * hd].astype(np.float16)
    assert np.array_equal(kc[5:5 + w.n_tok].view(np.uint16), want.view(np.uint16))


@pytest.mark.parametrize("name", ["pi05", "long_decode"])
def test_append_then_fused_attention_matches_oracle(name):
    """The new K/V rows written by fr_kv_append are what the following fused
    fr_decode_attn on the same stream attends to (long decode: hd 128 over
    32768 keys, the 128-key tile path)."""
    w = named_config(name)
    rng = np.random.default_rng(8)
    hd = w.hd
    kc0, vc0 = host_kv(w)
    k_new = rng.standard_normal((w.n_tok, hd)).astype(np.float32)
    v_new = rng.standard_normal((w.n_tok, hd)).astype(np.float32) * 0.5
    pos = w.pos()
    row0 = int(pos[0])
    pad = (w.n_kv_real, w.n_kv) if w.n_kv_real < w.n_kv else None
    okc, ovc, _, _ = oracle.kv_append(kc0, vc0, k_new, v_new, pos, w.rope, row0, pad)
    want = oracle.decode_attn(w.q(), pos, okc, ovc, w.mask(), w.rope, w.q_scale, w.kq_scale)
    kc = torch.from_numpy(kc0.copy()).cuda()
    vc = torch.from_numpy(vc0.copy()).cuda()
    d_pos = torch.from_numpy(pos).cuda()
    st = torch.cuda.Stream()
    with torch.cuda.stream(st):
        fr.kv_append(torch.from_numpy(k_new).cuda(), torch.from_numpy(v_new).cuda(), d_pos, w.rope, kc, vc,
                     row0, pad=pad, stream=st)
        out = fr.decode_attn(kc, vc, w.n_tok, w.n_head, q=torch.from_numpy(w.q().reshape(w.n_tok, -1)).cuda(),
                             pos=d_pos, rope=w.rope, q_scale=w.q_scale,
                             mask=torch.from_numpy(w.mask()).cuda(), kq_scale=w.kq_scale, stream=st)
    st.synchronize()
    assert_close(out.cpu().numpy().reshape(w.n_tok * w.n_head, hd), want, f"{name}: append + attention")
