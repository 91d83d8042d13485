"""Pins for the oracle's ggml float-compat RoPE angles (mode 1) and the
freq_factors input (no GPU).

FlashRT-llama.cpp development guide, "Invariants and pitfalls": RoPE mirrors
ggml's rope_neox (YaRN corrections included) and must stay bit-exact with it.
ggml evaluates the angles in fp32: theta_scale = powf(base, -2/n_dims), then
per position a running product theta_i = theta_{i-1} * theta_scale, divided by
the optional per-pair freq_factors, then the YaRN mix, all in fp32.

The pins tie the oracle to things other than itself: an exact rational
evaluation of the same steps with its own IEEE binary32 rounding (no numpy
float32 arithmetic), a 50-digit evaluation of the power, error bounds against
the exact-angle oracle, and scaling identities."""
import math
from fractions import Fraction

import numpy as np
import pytest

import oracle
from gen import RopeParams


def f32(q):
    """Round a rational to the nearest IEEE binary32 value (ties to even),
    returned as a Fraction; normal range only (what these angles need)."""
    q = Fraction(q)
    if q == 0:
        return Fraction(0)
    sign = -1 if q < 0 else 1
    a = abs(q)
    e = math.floor(math.log2(a.numerator) - math.log2(a.denominator))
    while Fraction(2) ** e > a:
        e -= 1
    while Fraction(2) ** (e + 1) <= a:
        e += 1
    assert -126 <= e <= 127
    scaled = a / Fraction(2) ** (e - 23)            # in [2^23, 2^24)
    m = scaled.numerator // scaled.denominator
    rem = scaled - m
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and m % 2 == 1):
        m += 1
    return sign * Fraction(m) * Fraction(2) ** (e - 23)


def exact_angles(pos, rp, ts):
    """The mode-1 angle steps in exact rationals with binary32 rounding after
    each operation (ts: the fp32 theta_scale as a Fraction)."""
    half = rp.n_dims // 2
    ff = [Fraction(1)] * half if rp.freq_factors is None else [f32(Fraction(x)) for x in rp.freq_factors]
    fs = f32(Fraction(rp.freq_scale))
    out = []
    th = f32(Fraction(pos))
    if rp.ext_factor != 0.0:
        c0, c1 = oracle.yarn_corr_dims(rp.n_dims, rp.n_ctx_orig, rp.freq_base, rp.beta_fast, rp.beta_slow)
        c0, c1 = Fraction(c0), Fraction(c1)
        ef = f32(Fraction(rp.ext_factor))
    for i in range(half):
        if i > 0:
            th = f32(th * ts)
        t_ext = f32(th / ff[i])
        t_int = f32(fs * t_ext)
        if rp.ext_factor != 0.0:
            y = f32((Fraction(i) - c0) / max(f32(Fraction(1, 1000)), f32(c1 - c0)))
            ramp = f32(1 - min(Fraction(1), max(Fraction(0), y)))
            mix = f32(ramp * ef)
            out.append(f32(f32(t_int * f32(1 - mix)) + f32(t_ext * mix)))
        else:
            out.append(t_int)
    return out


@pytest.mark.parametrize("base,n_dims", [(10000.0, 128), (1.0e6, 128), (10000.0, 256), (10000.0, 64),
                                         (500000.0, 96)])
def test_theta_scale_is_the_correctly_rounded_power(base, n_dims):
    """theta_scale = base ^ fl(-2/n_dims), rounded once: 50-digit mpmath value
    rounded by the exact binary32 rounding above."""
    mpmath = pytest.importorskip("mpmath")
    mpmath.mp.dps = 50
    e = Fraction(float(np.float32(-2.0) / np.float32(n_dims)))
    want = f32(Fraction(mpmath.nstr(mpmath.power(mpmath.mpf(base), mpmath.mpf(e.numerator) / e.denominator), 45)))
    got = oracle.rope_theta_scale_f32(RopeParams(n_dims=n_dims, freq_base=base, mode=1))
    assert Fraction(float(got)) == want


@pytest.mark.parametrize("rp", [
    RopeParams(n_dims=128, freq_base=10000.0, mode=1),
    RopeParams(n_dims=128, freq_base=1.0e6, freq_scale=1.0 / 8.0, ext_factor=1.0, n_ctx_orig=4096, mode=1),
    RopeParams(n_dims=64, freq_base=10000.0, freq_scale=0.25, ext_factor=0.5, n_ctx_orig=2048, mode=1,
               freq_factors=tuple(1.0 + 0.37 * (i % 5) for i in range(32))),
])
@pytest.mark.parametrize("pos", [0, 1, 4111, 32767, 65535])
def test_angles_bitwise_against_exact_rational_steps(rp, pos):
    th, _ = oracle.rope_theta_f32([pos], rp)
    ts = Fraction(float(oracle.rope_theta_scale_f32(rp)))
    want = exact_angles(pos, rp, ts)
    got = [Fraction(float(x)) for x in th[0]]
    assert got == want


@pytest.mark.parametrize("pos", [1, 958, 4096, 32767, 65535])
@pytest.mark.parametrize("base,n_dims", [(10000.0, 256), (1.0e6, 128)])
def test_angles_within_fp32_bound_of_exact(pos, base, n_dims):
    """Each pair's fp32 angle is within the error the recurrence can build up:
    i products and the rounding of theta_scale, each <= 2^-24 relative."""
    rp = RopeParams(n_dims=n_dims, freq_base=base, mode=1)
    th, ms = oracle.rope_theta_f32([pos], rp)
    ex, ms64 = oracle.rope_theta([pos], RopeParams(n_dims=n_dims, freq_base=base))
    i = np.arange(n_dims // 2)
    bound = ex[0] * (2.0 * (i + 1) + 1.0) * 2.0 ** -24
    assert np.all(np.abs(th[0].astype(np.float64) - ex[0]) <= bound)
    assert ms == np.float32(1.0) and ms64 == 1.0


def test_freq_factors_of_one_change_nothing():
    for mode in (0, 1):
        a = RopeParams(n_dims=128, freq_base=1e6, freq_scale=0.125, ext_factor=1.0, mode=mode)
        b = RopeParams(n_dims=128, freq_base=1e6, freq_scale=0.125, ext_factor=1.0, mode=mode,
                       freq_factors=(1.0,) * 64)
        x = np.random.default_rng(0).standard_normal((3, 2, 128))
        pos = [7, 4000, 32767]
        assert np.array_equal(oracle.rope_neox(x, pos, a), oracle.rope_neox(x, pos, b))


@pytest.mark.parametrize("mode", [0, 1])
def test_freq_factor_two_halves_the_position(mode):
    """theta_ext = theta_base / ff: ff = 2 at position p is the angle of
    position p/2 (exact in both modes: halving commutes with rounding)."""
    ff = RopeParams(n_dims=64, freq_base=10000.0, mode=mode, freq_factors=(2.0,) * 32)
    plain = RopeParams(n_dims=64, freq_base=10000.0, mode=mode)
    p = np.array([2, 1000, 65534])
    if mode == 1:
        a, _ = oracle.rope_theta_f32(p, ff)
        b, _ = oracle.rope_theta_f32(p // 2, plain)
        assert np.array_equal(a, b)
    else:
        a, _ = oracle.rope_theta(p, ff)
        b, _ = oracle.rope_theta(p // 2, plain)
        assert np.allclose(a, b, rtol=1e-15, atol=0)


def test_freq_factors_divide_each_pair():
    """Exact mode: pair i's angle is pos * base^(-2i/n) / ff_i (closed form)."""
    ffs = tuple(1.0 + i for i in range(16))
    rp = RopeParams(n_dims=32, freq_base=10000.0, freq_factors=ffs)
    th, _ = oracle.rope_theta([321], rp)
    for i in range(16):
        assert math.isclose(th[0, i], 321 * 10000.0 ** (-2.0 * i / 32) / ffs[i], rel_tol=1e-14)


def test_float_mode_rotation_close_to_exact_mode():
    """Mode 1 and mode 0 rotate by angles that differ by the fp32 angle error
    only: |y1 - y0| <= |x_pair| * mscale * |dtheta| per pair."""
    base = dict(n_dims=128, freq_base=1e6, freq_scale=1.0 / 8.0, ext_factor=1.0, n_ctx_orig=4096)
    r0, r1 = RopeParams(**base), RopeParams(mode=1, **base)
    pos = [32752, 32767]
    x = np.random.default_rng(3).standard_normal((2, 4, 128))
    y0, y1 = oracle.rope_neox(x, pos, r0), oracle.rope_neox(x, pos, r1)
    th0, ms = oracle.rope_theta(pos, r0)
    th1, _ = oracle.rope_theta_f32(pos, r1)
    dth = np.abs(th1.astype(np.float64) - th0)[:, None, :]
    norm = np.hypot(x[..., :64], x[..., 64:])
    tol = norm * ms * (dth + 1e-6) * 1.0001
    assert np.all(np.abs(y1[..., :64] - y0[..., :64]) <= tol)
    assert np.all(np.abs(y1[..., 64:] - y0[..., 64:]) <= tol)


def test_fp32_corr_dims_agree_with_double():
    """The correction dims computed with fp32 logarithms (ggml) are the same
    integers as in double for every YaRN setting used here."""
    for n_dims, n_ctx, base in ((128, 4096, 1e6), (64, 2048, 10000.0), (128, 8192, 500000.0)):
        c = oracle.yarn_corr_dims(n_dims, n_ctx, base, 32.0, 1.0)
        f = np.float32
        def d32(beta):
            return f(n_dims) * f(np.log(f(n_ctx) / (f(beta) * f(2.0) * f(math.pi)))) / (f(2.0) * f(np.log(f(base))))
        assert (max(0.0, math.floor(d32(32.0))), min(n_dims - 1.0, math.ceil(d32(1.0)))) == c


def test_position_zero_is_identity_in_float_mode():
    rp = RopeParams(n_dims=64, freq_base=10000.0, mode=1)
    x = np.random.default_rng(1).standard_normal((2, 3, 64))
    assert np.array_equal(oracle.rope_neox(x, [0, 0], rp), x)
