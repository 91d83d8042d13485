"""Pins for the oracle's K/V leg of qkv_post with the KV-cache tail write
(no GPU): the identity at position 0, the NEOX pairing of K on unit vectors
against libm cos/sin, the relative-position property between rope'd Q and K
rows (so K turns with Q, same sign and pairing), the YaRN magnitude on K, and
exactly which cache rows change."""
import math

import numpy as np
import pytest

import oracle
from gen import RopeParams, named_config


def _rand(shape, seed=3):
    return np.random.default_rng(seed).standard_normal(shape)


def _cache(n_ctx, hd, seed=5):
    return _rand((n_ctx, hd), seed).astype(np.float16)


def test_identity_at_pos0_and_plain_v():
    rp = RopeParams(n_dims=64, freq_base=10000.0)
    k, v = _rand((3, 64)), _rand((3, 64), 4)
    kc, vc, kr, _ = oracle.kv_append(_cache(40, 64), _cache(40, 64, 6), k, v, np.zeros(3, np.int32), rp, row0=10)
    assert np.array_equal(kr, k)
    assert np.array_equal(kc[10:13].view(np.uint16), k.astype(np.float16).view(np.uint16))
    assert np.array_equal(vc[10:13].view(np.uint16), v.astype(np.float16).view(np.uint16))


def test_k_pairing_on_unit_vectors():
    """pos 1, base 1e4, n_dims 8: theta_i = 1, 0.1, 0.01, 0.001 and NEOX pairs
    (i, i + 4); K carries no 1/sqrt(hd) scale."""
    rp = RopeParams(n_dims=8, freq_base=10000.0)
    th = [1.0, 0.1, 0.01, 0.001]
    for i in range(4):
        e = np.zeros((1, 8)); e[0, i] = 1.0
        _, _, kr, _ = oracle.kv_append(_cache(4, 8), _cache(4, 8), e, e, [1], rp, row0=0)
        want = np.zeros(8); want[i] = math.cos(th[i]); want[i + 4] = math.sin(th[i])
        assert np.allclose(kr[0], want, rtol=0, atol=1e-15)


@pytest.mark.parametrize("cfg", ["tiny", "long_decode"])
def test_relative_position_property_between_q_and_k(cfg):
    """<R(p) q, R(p') k> depends only on p - p' (angles linear in the
    position, YaRN included): shifting both positions leaves every score."""
    w = named_config(cfg)
    rp = w.rope
    q = _rand((1, 1, w.hd), 7)
    k = _rand((1, w.hd), 8)
    def score(pq, pk):
        qr = oracle.rope_neox(q, [pq], rp)[0, 0]
        _, _, kr, _ = oracle.kv_append(_cache(2, w.hd), _cache(2, w.hd), k, k, [pk], rp, row0=0)
        return float(qr @ kr[0])
    for pq, pk, d in ((5, 2, 100), (300, 17, 1000), (40, 40, 2500)):
        a, b = score(pq, pk), score(pq + d, pk + d)
        assert abs(a - b) <= 1e-9 * max(1.0, abs(a)), (pq, pk, d, a, b)
    # and it is not symmetric in the positions (a sign mistake would make it so)
    assert abs(score(30, 3) - score(3, 30)) > 1e-3


def test_yarn_magnitude_on_k():
    """With YaRN (long-decode parameters) every rotated K pair has norm
    mscale * |pair|, mscale = 1 + 0.1 ln(1 / freq_scale)."""
    w = named_config("long_decode")
    rp = w.rope
    k = _rand((4, w.hd), 9)
    pos = np.array([100, 4095, 20000, 32767])
    _, _, kr, _ = oracle.kv_append(_cache(8, w.hd), _cache(8, w.hd), k, k, pos, rp, row0=0)
    half = rp.n_dims // 2
    mscale = 1.0 + 0.1 * math.log(1.0 / rp.freq_scale)
    n0 = np.hypot(k[:, :half], k[:, half:rp.n_dims])
    n1 = np.hypot(kr[:, :half], kr[:, half:rp.n_dims])
    assert np.allclose(n1, mscale * n0, rtol=1e-12, atol=0)


def test_only_tail_and_pad_rows_change():
    rp = RopeParams(n_dims=128, freq_base=10000.0)
    k, v = _rand((5, 128)), _rand((5, 128), 11)
    k0, v0 = _cache(64, 128, 12), _cache(64, 128, 13)
    kc, vc, kr, vr = oracle.kv_append(k0, v0, k, v, np.arange(20, 25), rp, row0=20, pad=(40, 64))
    keep = np.r_[0:20, 25:40]
    assert np.array_equal(kc[keep].view(np.uint16), k0[keep].view(np.uint16))
    assert np.array_equal(vc[keep].view(np.uint16), v0[keep].view(np.uint16))
    assert not np.any(kc[40:64].astype(np.float64)) and not np.any(vc[40:64].astype(np.float64))
    assert np.array_equal(kc[20:25].view(np.uint16), oracle.f16_round(kr).view(np.uint16))
    assert np.array_equal(vr, v)
    # the inputs are not modified
    assert np.array_equal(k0.view(np.uint16), _cache(64, 128, 12).view(np.uint16))
