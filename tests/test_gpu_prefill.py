"""Longer query windows (prefill) through the same C ABI: every 128-row tile
reads its 16-token mask window; parity with the oracle on the pi0.5 prefix
window (968 tokens x 8 heads, KV length = query count, pad-only mask) and on
ragged shapes, both split-merge strategies, fused == two-call bitwise, and the
shapes the mask window cannot hold rejected."""
import numpy as np
import pytest
import torch

import gqa_kv_head_gb300 as fr
from fr_harness import assert_close, oracle_out, run_fused, run_two_call, to_device
from gen import RopeParams, Workload, named_config

pytestmark = pytest.mark.gpu


def _rows(o):
    return o.cpu().numpy().reshape(-1, o.shape[-1])


def test_pi05_prefix_window_matches_oracle():
    w = named_config("pi05_prefill")
    d = to_device(w)
    o = _rows(run_fused(w, d))
    assert_close(o, oracle_out(w), "pi0.5 prefix prefill")


@pytest.mark.parametrize("n_head,n_tok,hd,n_kv,n_real,mask", [
    (12, 100, 128, 112, 100, "none"),      # 1200 rows, tiles span 10-11 tokens, pad columns
    (8, 40, 64, 40, 40, "causal"),         # causal inside the window
    (9, 77, 256, 80, 77, "causal"),        # 693 rows, unaligned tiles
    (16, 64, 128, 1000, 1000, "random5"),  # 1024 rows, per-token random mask
])
def test_ragged_prefill_windows(n_head, n_tok, hd, n_kv, n_real, mask):
    w = Workload(f"prefill_{n_head}_{n_tok}", n_head=n_head, n_tok=n_tok, hd=hd, n_kv=n_kv, n_kv_real=n_real,
                 rope=RopeParams(n_dims=hd, freq_base=10000.0),
                 positions=tuple(range(n_real - n_tok, n_real)), mask_kind=mask, seed=4)
    d = to_device(w)
    o = _rows(run_fused(w, d))
    assert_close(o, oracle_out(w), f"prefill {n_head}x{n_tok}")


@pytest.mark.parametrize("merge_mode", [1, 2])
def test_prefill_split_strategies_agree(merge_mode):
    w = Workload("prefill_merge", n_head=8, n_tok=200, hd=128, n_kv=2048, n_kv_real=2000,
                 rope=RopeParams(n_dims=128, freq_base=10000.0), positions=tuple(range(1800, 2000)),
                 mask_kind="causal", seed=6)
    d = to_device(w)
    o = _rows(run_fused(w, d, merge_mode=merge_mode))
    assert_close(o, oracle_out(w), f"prefill merge mode {merge_mode}")


def test_prefill_fused_equals_two_call():
    w = Workload("prefill_2call", n_head=8, n_tok=300, hd=256, n_kv=512, n_kv_real=500,
                 rope=RopeParams(n_dims=256, freq_base=10000.0), positions=tuple(range(200, 500)),
                 mask_kind="none", seed=7)
    d = to_device(w)
    a = run_fused(w, d)
    b, _ = run_two_call(w, d)
    torch.cuda.synchronize()
    assert torch.equal(a, b)


def _sampled_rows(w, n_random, seed):
    rng = np.random.default_rng(seed)
    toks = np.unique(np.concatenate([[0, w.n_tok - 1], rng.integers(0, w.n_tok, size=6)]))
    return np.unique(np.concatenate([toks * w.n_head, toks * w.n_head + w.n_head - 1,
                                     rng.integers(0, w.M, size=n_random)]))


def test_largest_window_sampled_rows():
    """The largest window the API takes: 8192 tokens x 8 heads = 65536 query
    rows (512 row tiles) against 8192 keys, causal; the oracle checks a sample
    of rows (first and last head of sampled tokens, plus random rows)."""
    w = Workload("prefill_max", n_head=8, n_tok=8192, hd=128, n_kv=8192, n_kv_real=8192,
                 rope=RopeParams(n_dims=128, freq_base=10000.0), positions=tuple(range(8192)),
                 mask_kind="causal", seed=13)
    d = to_device(w)
    o = _rows(run_fused(w, d))
    rows = _sampled_rows(w, 24, 13)
    assert_close(o[rows], oracle_out(w, rows=rows), "65536-row window")


def test_many_heads_one_kv_head_sampled_rows():
    """4096 query heads sharing the KV head, 16 tokens: 65536 rows, ragged
    KV length and a random mask."""
    w = Workload("heads_max", n_head=4096, n_tok=16, hd=64, n_kv=300, n_kv_real=300,
                 rope=RopeParams(n_dims=64, freq_base=10000.0), positions=tuple(range(284, 300)),
                 mask_kind="random5", seed=14)
    d = to_device(w)
    o = _rows(run_fused(w, d))
    rows = _sampled_rows(w, 24, 14)
    assert_close(o[rows], oracle_out(w, rows=rows), "4096 heads x 16 tokens")


def test_more_row_tiles_than_sms_short_kv():
    """256 row tiles (more than SMs) over only 50 keys at hd 128: 128-key tiles
    whose second softmax half lies wholly past the last key."""
    w = Workload("tiles_short_kv", n_head=2048, n_tok=16, hd=128, n_kv=50, n_kv_real=50,
                 rope=RopeParams(n_dims=128, freq_base=10000.0), positions=tuple(range(34, 50)),
                 mask_kind="random5", seed=16)
    d = to_device(w)
    o = _rows(run_fused(w, d))
    rows = _sampled_rows(w, 24, 16)
    assert_close(o[rows], oracle_out(w, rows=rows), "256 row tiles, 50 keys")


def test_window_too_wide_is_rejected():
    # 4 heads: a 128-row tile spans 32 tokens, more than the 16-token mask window
    w = Workload("prefill_narrow", n_head=4, n_tok=40, hd=64, n_kv=64, n_kv_real=64,
                 rope=RopeParams(n_dims=64, freq_base=10000.0), positions=tuple(range(24, 64)),
                 mask_kind="causal", seed=8)
    d = to_device(w)
    with pytest.raises(fr.FrError, match="UNSUPPORTED"):
        run_fused(w, d, workspace=torch.zeros(1 << 20, dtype=torch.uint8, device="cuda"))
