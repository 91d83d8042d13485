"""GPU parity of fr_qkv_post against the oracle (FlashRT PR #185, qkv_post
commits): t-major layout bit-exact, values within one f16 ulp of the fp64
oracle's rounding, and the optional f32 copy rounding to the same f16 bits."""
import numpy as np
import pytest
import torch

import oracle
from gen import RopeParams, make_workload, named_config
import gqa_kv_head_gb300 as fr

pytestmark = pytest.mark.gpu


def _ulp_diff(a16, b16):
    a = np.asarray(a16, np.float16).view(np.int16).astype(np.int32)
    b = np.asarray(b16, np.float16).view(np.int16).astype(np.int32)
    # map sign-magnitude to a monotone integer line
    a = np.where(a < 0, -32768 - a, a)
    b = np.where(b < 0, -32768 - b, b)
    return np.abs(a - b)


@pytest.mark.parametrize("hd,n_tok,n_head", [(64, 3, 4), (128, 16, 32), (256, 10, 8), (256, 1, 1)])
def test_layout_bit_exact_at_pos0(hd, n_tok, n_head):
    """pos 0 is the identity and q_scale a power of two, so every f16 must be
    exactly f16(q[t, h, d] * scale) at row t*n_head + h; inputs encode (t, h, d)."""
    t_, h_, d_ = np.meshgrid(np.arange(n_tok), np.arange(n_head), np.arange(hd), indexing="ij")
    q = (t_ * 1000 + h_ * 64 + d_ * 0.25 + 0.5).astype(np.float32)
    scale = 2.0 ** -4
    qd = torch.from_numpy(q).cuda()
    pos = torch.zeros(n_tok, dtype=torch.int32, device="cuda")
    q32 = torch.empty((n_tok * n_head, hd), dtype=torch.float32, device="cuda")
    q16, _ = fr.qkv_post(qd, pos, n_head, hd, RopeParams(n_dims=hd), scale, q32_out=q32)
    torch.cuda.synchronize()
    want = (q.reshape(n_tok * n_head, hd).astype(np.float64) * scale).astype(np.float16)
    assert np.array_equal(q16.cpu().numpy().view(np.uint16), want.view(np.uint16))
    assert np.array_equal(q32.cpu().numpy(), q.reshape(n_tok * n_head, hd) * np.float32(scale))


@pytest.mark.parametrize("name", ["tiny", "pi05", "c3", "long_decode", "sweep:128:16:65536",
                                  "sweep:256:1:256"])
def test_matches_oracle_within_one_ulp(name):
    w = make_workload(name)
    q = torch.from_numpy(w.q()).cuda()
    pos = torch.from_numpy(w.pos()).cuda()
    q32 = torch.empty((w.M, w.hd), dtype=torch.float32, device="cuda")
    q16, _ = fr.qkv_post(q, pos, w.n_head, w.hd, w.rope, w.q_scale, q32_out=q32)
    torch.cuda.synchronize()
    rows, want16 = oracle.qkv_post(w.q(), w.pos(), w.rope, w.q_scale)
    got16 = q16.cpu().numpy()
    ulps = _ulp_diff(got16, want16)
    assert ulps.max() <= 1, f"max ulp diff {ulps.max()}"
    assert (ulps == 0).mean() >= 0.99
    # the f32 values the f16 rows round from agree with the fp64 rotation
    assert np.max(np.abs(q32.cpu().numpy() - rows)) <= 2e-6 * max(1.0, np.abs(rows).max())
    # "convert once" claim: casting the f32 copy to f16 gives the same bits
    assert np.array_equal(q32.cpu().numpy().astype(np.float16).view(np.uint16), got16.view(np.uint16))


def test_token_stride_and_pass_through_dims():
    """Q rows taken from a fused-QKV-like buffer ([n_tok, (n_head+2)*hd]) with
    n_dims < hd: the pass-through dims are only scaled."""
    w = named_config("c3").with_(rope=RopeParams(n_dims=64, freq_base=10000.0))
    big = torch.zeros((w.n_tok, (w.n_head + 2) * w.hd), dtype=torch.float32, device="cuda")
    big[:, :w.n_head * w.hd] = torch.from_numpy(w.q().reshape(w.n_tok, -1))
    q16, _ = fr.qkv_post(big[:, :w.n_head * w.hd], torch.from_numpy(w.pos()).cuda(), w.n_head,
                         w.hd, w.rope, w.q_scale)
    torch.cuda.synchronize()
    _, want16 = oracle.qkv_post(w.q(), w.pos(), w.rope, w.q_scale)
    assert _ulp_diff(q16.cpu().numpy(), want16).max() <= 1
    tail = (w.q().reshape(w.M, w.hd)[:, 64:].astype(np.float64) * w.q_scale).astype(np.float16)
    assert np.array_equal(q16.cpu().numpy()[:, 64:].view(np.uint16), tail.view(np.uint16))
