"""Pins for the oracle's attention (no GPU): a library routine (torch
scaled_dot_product_attention in float64), closed forms, invariants and
hand-derived brute-force fixtures."""
import json
import os

import numpy as np
import pytest
import torch

import oracle
from gen import named_config, sweep_config

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _case(n_tok=3, n_head=4, hd=32, n_kv=50, seed=0, masked=True):
    g = np.random.default_rng(seed)
    q = g.standard_normal((n_tok * n_head, hd)) / np.sqrt(hd)
    k = g.standard_normal((n_kv, hd))
    v = g.standard_normal((n_kv, hd))
    mask = None
    if masked:
        mask = np.where(g.random((n_tok, n_kv)) < 0.3, -np.inf, 0.0)
        mask[:, 0] = 0.0                      # no fully masked row
    return q, k, v, mask


def _sdpa(q, k, v, mask, n_tok, n_head, kq_scale):
    hd = k.shape[1]
    qt = torch.tensor(q).reshape(n_tok, n_head, hd).permute(1, 0, 2)[None]   # [1, H, T, hd]
    kt = torch.tensor(k)[None, None].expand(1, n_head, -1, -1)
    vt = torch.tensor(v)[None, None].expand(1, n_head, -1, -1)
    am = None if mask is None else torch.tensor(mask)[None, None].expand(1, n_head, -1, -1)
    o = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, attn_mask=am, scale=kq_scale)
    return o[0].permute(1, 0, 2).reshape(n_tok * n_head, hd).numpy()


@pytest.mark.parametrize("kq_scale", [1.0, 0.37])
@pytest.mark.parametrize("masked", [False, True])
def test_matches_torch_sdpa_float64(kq_scale, masked):
    n_tok, n_head = 3, 4
    q, k, v, mask = _case(n_tok, n_head, masked=masked)
    got = oracle.attention_collapsed(q, k, v, mask, n_tok, n_head, kq_scale)
    ref = _sdpa(q, k, v, mask, n_tok, n_head, kq_scale)
    assert np.allclose(got, ref, rtol=0, atol=1e-12)


def test_batched_equals_collapsed():
    """Same values up to summation order (numpy may pick gemv for one row)."""
    for cfg in ("tiny", "pi05"):
        w = named_config(cfg)
        _, q16 = oracle.qkv_post(w.q(), w.pos(), w.rope, w.q_scale)
        a = oracle.attention_collapsed(q16, w.k(), w.v(), w.mask(), w.n_tok, w.n_head)
        b = oracle.attention_batched(q16, w.k(), w.v(), w.mask(), w.n_tok, w.n_head)
        assert np.allclose(a, b, rtol=0, atol=1e-15)


def test_rows_sum_to_one():
    q, k, v, mask = _case()
    v[:, 5] = 1.0
    o = oracle.attention_collapsed(q, k, v, mask, 3, 4)
    assert np.allclose(o[:, 5], 1.0, rtol=0, atol=1e-14)


def test_single_key_returns_v0_exactly():
    q, k, v, _ = _case(n_kv=1, masked=False)
    o = oracle.attention_collapsed(q, k, v, None, 3, 4)
    assert np.array_equal(o, np.broadcast_to(v[0], o.shape))


def test_zero_q_is_mean_of_unmasked_v():
    q, k, v, mask = _case()
    o = oracle.attention_collapsed(np.zeros_like(q), k, v, mask, 3, 4)
    for r in range(12):
        keep = np.isfinite(mask[r // 4])
        assert np.allclose(o[r], v[keep].mean(axis=0), rtol=0, atol=1e-14)


def test_masked_columns_get_zero_weight():
    q, k, v, mask = _case()
    o = oracle.attention_collapsed(q, k, v, mask, 3, 4)
    # columns masked for EVERY token: garbage there must not matter
    dead = np.all(~np.isfinite(mask), axis=0)
    assert dead.any()
    k2, v2 = k.copy(), v.copy()
    k2[dead] = 1e3; v2[dead] = -7e3
    o2 = oracle.attention_collapsed(q, k2, v2, mask, 3, 4)
    assert np.array_equal(o, o2)


def test_pad_rows_of_pi05_are_inert():
    w = named_config("pi05")
    _, q16 = oracle.qkv_post(w.q(), w.pos(), w.rope, w.q_scale)
    o = oracle.attention_collapsed(q16, w.k(), w.v(), w.mask(), w.n_tok, w.n_head)
    k, v = w.k().copy(), w.v().copy()
    k[968:] = 3.0; v[968:] = -5.0
    o2 = oracle.attention_collapsed(q16, k, v, w.mask(), w.n_tok, w.n_head)
    assert np.array_equal(o, o2)
    # and truncating to the real rows gives the same result (up to summation order)
    o3 = oracle.attention_collapsed(q16, k[:968], v[:968], w.mask()[:, :968], w.n_tok, w.n_head)
    assert np.allclose(o, o3, rtol=0, atol=1e-15)


@pytest.mark.parametrize("n_splits", [1, 2, 5, 17, 50])
def test_split_merge_equals_direct(n_splits):
    q, k, v, mask = _case(n_kv=50)
    mask[:, 10:25] = -np.inf     # whole chunks fully masked for some splits
    direct = oracle.attention_collapsed(q, k, v, mask, 3, 4)
    merged = oracle.attention_split_merge(q, k, v, mask, 3, 4, 1.0, n_splits)
    assert np.allclose(direct, merged, rtol=0, atol=1e-14)


def test_fully_masked_row_is_zero():
    q, k, v, mask = _case()
    mask[1, :] = -np.inf
    o = oracle.attention_collapsed(q, k, v, mask, 3, 4)
    assert np.array_equal(o[4:8], np.zeros((4, k.shape[1])))
    assert np.all(np.isfinite(o))


def test_mask_row_is_token_not_head():
    """Row r = t*n_head + h reads mask row t: a mask that differs per token."""
    n_tok, n_head = 2, 3
    q, k, v, _ = _case(n_tok, n_head, masked=False)
    mask = np.zeros((n_tok, k.shape[0]))
    mask[0, 25:] = -np.inf
    mask[1, :25] = -np.inf
    got = oracle.attention_collapsed(q, k, v, mask, n_tok, n_head)
    ref = _sdpa(q, k, v, mask, n_tok, n_head, 1.0)
    assert np.allclose(got, ref, rtol=0, atol=1e-12)


def test_bruteforce_golden():
    g = json.load(open(os.path.join(GOLDEN, "attn_bruteforce.json")))
    for c in g["cases"]:
        q = np.array(c["q"], np.float64)
        k = np.array(c["k"], np.float64)
        v = np.array(c["v"], np.float64)
        mask = None if c["mask"] is None else np.array(
            [[-np.inf if x == "-inf" else float(x) for x in row] for row in c["mask"]])
        n_tok = c.get("n_tok", 1)
        n_head = c.get("n_head", q.shape[0] // n_tok)
        o = oracle.attention_collapsed(q, k, v, mask, n_tok, n_head, c["kq_scale"])
        assert np.allclose(o, np.array(c["out"]), rtol=0, atol=1e-14), c["name"]


def test_decode_attn_rows_match_full():
    w = sweep_config(128, 4, 1024)
    full = oracle.decode_attn(w.q(), w.pos(), w.k(), w.v(), w.mask(), w.rope, w.q_scale)
    rows = np.array([0, 7, 31])
    sub = oracle.decode_attn(w.q(), w.pos(), w.k(), w.v(), w.mask(), w.rope, w.q_scale, rows=rows)
    assert np.allclose(full[rows], sub, rtol=0, atol=1e-15)
