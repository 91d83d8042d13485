"""Pins for the oracle's RoPE / YaRN / qkv_post (no GPU).

Each test ties the oracle to something other than itself: closed forms
(cos/sin of known angles via Python's libm, complex rotation), invariants
(pair norms, relative-position property), YaRN's own definitions (wavelength
at the correction dims) and hand-derived fixtures in tests/golden/.
"""
import json
import math
import os

import numpy as np
import pytest

import oracle
from gen import RopeParams, named_config

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rand(shape, seed=1):
    return np.random.default_rng(seed).standard_normal(shape)


def test_identity_at_pos0():
    rp = RopeParams(n_dims=64, freq_base=10000.0)
    x = _rand((3, 4, 64))
    y = oracle.rope_neox(x, np.zeros(3, np.int32), rp)
    assert np.array_equal(y, x)


def test_neox_pairing_unit_vectors():
    """pos 1, base 1e4, n_dims 8: theta_i = 10000^(-i/4) = 1, 0.1, 0.01, 0.001.
    NEOX pairs dimension i with i + n_dims/2 (not 2i with 2i+1)."""
    rp = RopeParams(n_dims=8, freq_base=10000.0)
    thetas = [1.0, 0.1, 0.01, 0.001]
    for i in range(4):
        e = np.zeros((1, 1, 8)); e[0, 0, i] = 1.0
        y = oracle.rope_neox(e, [1], rp)[0, 0]
        want = np.zeros(8); want[i] = math.cos(thetas[i]); want[i + 4] = math.sin(thetas[i])
        assert np.allclose(y, want, rtol=0, atol=1e-15), (i, y, want)
        e = np.zeros((1, 1, 8)); e[0, 0, i + 4] = 1.0
        y = oracle.rope_neox(e, [1], rp)[0, 0]
        want = np.zeros(8); want[i] = -math.sin(thetas[i]); want[i + 4] = math.cos(thetas[i])
        assert np.allclose(y, want, rtol=0, atol=1e-15), (i, y, want)


@pytest.mark.parametrize("n_dims,hd,base,pos", [(64, 64, 1e4, 128), (128, 128, 1e6, 32767),
                                                (32, 64, 1e4, 5), (256, 256, 1e4, 4111)])
def test_complex_rotation_form(n_dims, hd, base, pos):
    """Plain RoPE (RoFormer, Su et al.) as complex multiplication:
    (x_i + j x_{i+n/2}) * exp(j * pos * base^(-2i/n)); dims >= n_dims untouched."""
    rp = RopeParams(n_dims=n_dims, freq_base=base)
    x = _rand((1, 3, hd), seed=pos)
    y = oracle.rope_neox(x, [pos], rp)
    half = n_dims // 2
    z = x[..., :half] + 1j * x[..., half:n_dims]
    ang = np.array([pos * base ** (-2.0 * i / n_dims) for i in range(half)])
    zr = z * np.exp(1j * ang)
    tol = 1e-14 * max(1.0, pos) * 4      # an angle of pos radians carries ~pos*eps
    assert np.allclose(y[..., :half], zr.real, rtol=0, atol=tol)
    assert np.allclose(y[..., half:n_dims], zr.imag, rtol=0, atol=tol)
    assert np.array_equal(y[..., n_dims:], x[..., n_dims:])


def test_pair_norm_scaled_by_mscale():
    w = named_config("long_decode")
    x = _rand((2, 5, 128))
    y = oracle.rope_neox(x, [32000, 32767], w.rope)
    _, mscale = oracle.rope_theta([0], w.rope)
    nx = np.hypot(x[..., :64], x[..., 64:])
    ny = np.hypot(y[..., :64], y[..., 64:])
    assert np.allclose(ny, mscale * nx, rtol=1e-13, atol=0)


@pytest.mark.parametrize("cfg", ["pi05", "long_decode"])
def test_relative_position_property(cfg):
    """<R(p) q, R(p') k> depends only on p - p' (angles are linear in pos)."""
    rp = named_config(cfg).rope
    n = rp.n_dims
    q = _rand((1, 1, n), 3); k = _rand((1, 1, n), 4)
    def dot(p1, p2):
        return float(np.sum(oracle.rope_neox(q, [p1], rp) * oracle.rope_neox(k, [p2], rp)))
    base = dot(100, 37)
    for shift in (1, 999, 30000):
        assert abs(dot(100 + shift, 37 + shift) - base) < 1e-9 * (1 + abs(base))


def test_yarn_golden():
    g = json.load(open(os.path.join(GOLDEN, "yarn_long_decode.json")))
    p = g["params"]
    c0, c1 = oracle.yarn_corr_dims(p["n_dims"], p["n_ctx_orig"], p["freq_base"],
                                   p["beta_fast"], p["beta_slow"])
    assert (c0, c1) == (g["c0"], g["c1"])
    rp = RopeParams(**p)
    theta, mscale = oracle.rope_theta([1000], rp)
    assert mscale == pytest.approx(g["mscale"], rel=1e-15)
    for i, f in g["theta_factor"].items():
        i = int(i)
        theta_ext = 1000 * p["freq_base"] ** (-2.0 * i / p["n_dims"])
        assert theta[0, i] == pytest.approx(f * theta_ext, rel=1e-13), i


def test_yarn_corr_dims_match_wavelength_definition():
    """YaRN: the correction index is where the wavelength 2*pi*base^(2d/n) equals
    n_ctx_orig / beta. Solve that by bisection and compare with floor/ceil."""
    n, L, base = 128, 4096, 1.0e6
    def solve(beta):
        lo, hi = 0.0, float(n)
        for _ in range(200):
            mid = 0.5 * (lo + hi)
            if 2 * math.pi * base ** (2 * mid / n) < L / beta:
                lo = mid
            else:
                hi = mid
        return lo
    c0, c1 = oracle.yarn_corr_dims(n, L, base, 32.0, 1.0)
    assert c0 == math.floor(solve(32.0))
    assert c1 == math.ceil(solve(1.0))


def test_yarn_reduces_to_plain_and_linear():
    x = _rand((1, 2, 128), 7)
    plain = RopeParams(n_dims=128, freq_base=1e6)
    # freq_scale = 1: interpolation and extrapolation coincide, ln 1 = 0.
    yarn1 = RopeParams(n_dims=128, freq_base=1e6, freq_scale=1.0, ext_factor=1.0)
    assert np.allclose(oracle.rope_neox(x, [5000], yarn1), oracle.rope_neox(x, [5000], plain),
                       rtol=0, atol=1e-11)
    _, ms = oracle.rope_theta([0], yarn1)
    assert ms == 1.0
    # ext_factor = 0: pure linear position interpolation == plain RoPE at pos*s.
    lin = RopeParams(n_dims=128, freq_base=1e6, freq_scale=0.125, ext_factor=0.0)
    assert np.allclose(oracle.rope_neox(x, [5000], lin), oracle.rope_neox(x, [625.0], plain),
                       rtol=0, atol=1e-12)


def test_yarn_ramp_regions():
    rp = named_config("long_decode").rope
    c0, c1 = oracle.yarn_corr_dims(rp.n_dims, rp.n_ctx_orig, rp.freq_base, rp.beta_fast, rp.beta_slow)
    theta, _ = oracle.rope_theta([12345], rp)
    i = np.arange(rp.n_dims // 2)
    ext = 12345 * rp.freq_base ** (-2.0 * i / rp.n_dims)
    hi = i <= c0
    lo = i >= c1
    assert np.allclose(theta[0, hi], ext[hi], rtol=1e-14)
    assert np.allclose(theta[0, lo], rp.freq_scale * ext[lo], rtol=1e-14)
    mid = ~(hi | lo)
    r = theta[0, mid] / ext[mid]
    assert np.all(np.diff(r) < 0) and np.all(r < 1) and np.all(r > rp.freq_scale)


def test_qkv_post_t_major_layout_bit_exact():
    """pos 0 (identity), q_scale = 1/8 (exact power of two): every emitted f16
    equals f16(q[t, h, d] / 8) at row r = t*n_head + h. Inputs encode (t, h, d)."""
    n_tok, n_head, hd = 3, 4, 64
    q = np.zeros((n_tok, n_head, hd), np.float32)
    for t in range(n_tok):
        for h in range(n_head):
            for d in range(hd):
                q[t, h, d] = t * 1000 + h * 100 + d + 0.5
    rp = RopeParams(n_dims=64, freq_base=1e4)
    rows, q16 = oracle.qkv_post(q, np.zeros(n_tok, np.int32), rp, 0.125)
    assert q16.dtype == np.float16 and q16.shape == (n_tok * n_head, hd)
    for t in range(n_tok):
        for h in range(n_head):
            r = t * n_head + h
            for d in range(hd):
                assert q16[r, d] == np.float16(q[t, h, d] / 8.0)
                assert rows[r, d] == float(q[t, h, d]) / 8.0
