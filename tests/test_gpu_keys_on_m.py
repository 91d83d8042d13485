"""The kernel with 128-key tiles on the MMA's M side and the query rows on
its N (layout 2: M = n_tok*n_head <= 128, hd 128 or 256), against the fp64
oracle through the C ABI: every row count up to 64 (N = 16, 32, 64 with
padded rows), rows cut into slices of 16, 32 or 64 (up to 128 rows, CTAs of
one split sharing its K/V tiles), ragged KV lengths, masks, padded strides,
forced split counts, a workspace that holds fewer split states, and the same
result as the 128-row query-tile kernel (layout 1).

FlashRT PR #185, commits "FLASH_ATTN_EXT with q_tokens <= 16 ..." and "The
GQA query heads share the one KV head ...": one QK^T and one PV over all
t-major rows; here computed transposed (S^T = K Q^T, O^T = V^T P^T)."""
import numpy as np
import pytest
import torch

from gen import RopeParams, Workload, make_workload, named_config
import gqa_kv_head_gb300 as fr
from fr_harness import assert_close, oracle_out, run_fused, run_two_call, to_device

pytestmark = pytest.mark.gpu


def _rows(out):
    return out.reshape(-1, out.shape[-1]).cpu().numpy().astype(np.float64)


def _plan(w, **kw):
    return fr.decode_attn_plan(w.n_tok, w.n_head, w.hd, w.n_kv, layout=2, **kw)


KOM = dict(layout=2)


def _auto_rows(w):
    """Rows per slice of the library's own keys-on-M choice (0: the 128-row
    kernel), as include/fr_kernels.h documents it: 16-row slices for a short
    KV range (n_kv >= 1024 and ceil(M/16)*n_kv <= 32768 at hd 256, 16384 at
    hd 128), one slice of all rows for M <= 32 and n_kv >= max(1024, 256 M)."""
    M = w.n_tok * w.n_head
    if w.hd not in (128, 256) or w.n_tok > 16 or M > 128:
        return 0
    if w.n_kv >= 1024 and -(-M // 16) * w.n_kv <= (32768 if w.hd == 256 else 16384):
        return 16
    if M <= 32 and w.n_kv >= max(1024, 256 * M):
        return 16 if M <= 16 else 32
    return 0


@pytest.mark.parametrize("hd", [128, 256])
@pytest.mark.parametrize("n_tok,n_head", [(1, 1), (1, 8), (2, 8), (3, 5), (4, 8), (7, 5), (8, 8), (16, 4), (1, 64),
                                          (11, 3)])
def test_row_counts(hd, n_tok, n_head):
    w = Workload("keys-on-m", n_head=n_head, n_tok=n_tok, hd=hd, n_kv=3000,
                 rope=RopeParams(n_dims=hd, freq_base=10000.0), positions=tuple(range(2999 - n_tok + 1, 3000)),
                 mask_kind="causal", seed=n_tok * 7 + n_head)
    assert _plan(w)["keys_on_m"] == 1
    auto = fr.decode_attn_plan(w.n_tok, w.n_head, w.hd, w.n_kv)
    rows = _auto_rows(w)
    assert auto["keys_on_m"] == (1 if rows else 0)
    assert auto["row_slices"] == (-(-w.M // rows) if rows else 1)
    d = to_device(w)
    out = _rows(run_fused(w, d, **KOM))
    ref = oracle_out(w)
    assert_close(out, ref, f"{n_tok}x{n_head} hd {hd}")
    assert_close(_rows(run_fused(w, d, layout=1)), ref, f"{n_tok}x{n_head} hd {hd} query tiles")


@pytest.mark.parametrize("n_kv", [1, 5, 127, 128, 129, 1000, 20037])
@pytest.mark.parametrize("hd", [128, 256])
def test_ragged_kv_masks_and_strides(n_kv, hd):
    w = Workload(f"ragged-kom{n_kv}", n_head=5, n_tok=7, hd=hd, n_kv=n_kv,
                 rope=RopeParams(n_dims=hd, freq_base=10000.0),
                 positions=tuple(range(n_kv - 1, n_kv + 6)), mask_kind="random5", seed=n_kv % 97)
    d = to_device(w, k_pad=16, mask_pad=8, q_extra_heads=2)
    assert_close(_rows(run_fused(w, d, **KOM)), oracle_out(w), w.name)


@pytest.mark.parametrize("name", ["sweep:256:1:65536", "sweep:128:8:16384", "sweep:256:4:4096"])
@pytest.mark.parametrize("splits", [1, 2, 7, 1000])
def test_forced_splits(name, splits):
    w = make_workload(name)
    d = to_device(w)
    p = _plan(w, splits=splits)
    assert p["keys_on_m"] == 1 and p["splits"] <= max(1, splits)
    assert_close(_rows(run_fused(w, d, splits=splits, **KOM)), oracle_out(w), f"{name} splits={splits}")


def test_workspace_holding_fewer_split_states():
    """A workspace of the smallest accepted size: the split count is cut to
    the states it holds (down to one split, which needs none)."""
    w = make_workload("sweep:256:8:65536")
    d = to_device(w)
    lib = fr.load()
    full = fr.workspace_size(w.n_tok, w.n_head, w.hd, w.n_kv)
    ref = oracle_out(w)
    for nbytes in (full, 2 << 20, 300 << 10):
        ws = torch.zeros(max(nbytes, 1 << 20), dtype=torch.uint8, device="cuda")[:nbytes]
        p = _plan(w, workspace_bytes=nbytes)
        out = _rows(run_fused(w, d, workspace=ws, **KOM))
        assert_close(out, ref, f"workspace {nbytes}: plan {p}")
    assert _plan(w, workspace_bytes=full)["splits"] > _plan(w, workspace_bytes=2 << 20)["splits"]


@pytest.mark.parametrize("name", ["sweep:128:1:65536", "sweep:256:8:4096", "sweep:256:2:1024"])
def test_fused_equals_two_call_bitwise(name):
    w = make_workload(name)
    d = to_device(w)
    a = run_fused(w, d, **KOM)
    b, _ = run_two_call(w, d, **KOM)
    torch.cuda.synchronize()
    assert torch.equal(a, b)


def test_repeatable_and_graph_captured():
    w = make_workload("sweep:256:2:16384")
    d = to_device(w)
    ws = fr.make_workspace(w.n_tok, w.n_head, w.hd, w.n_kv)
    out = torch.empty((w.n_tok, w.n_head, w.hd), dtype=torch.float32, device="cuda")
    ref = run_fused(w, d, workspace=ws, **KOM).clone()
    assert torch.equal(run_fused(w, d, workspace=ws, **KOM), ref)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        run_fused(w, d, workspace=ws, out=out, stream=s, **KOM)
    out.zero_()
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(out, ref)
    fr.workspace_check(ws)


def test_device_timeout_is_reported_and_recoverable():
    w = make_workload("sweep:128:4:4096")
    d = to_device(w)
    ws = fr.make_workspace(w.n_tok, w.n_head, w.hd, w.n_kv)
    run_fused(w, d, workspace=ws, wait_probe_iters=1000, **KOM)
    with pytest.raises(fr.FrError) as e:
        fr.workspace_check(ws)
    assert e.value.status == 5
    out = _rows(run_fused(w, d, workspace=ws, **KOM))
    fr.workspace_check(ws)
    assert_close(out, oracle_out(w), "after timeout")


def test_fully_masked_token_is_zero():
    w = make_workload("sweep:256:4:4096")
    d = to_device(w)
    d["mask"][2, :] = float("-inf")
    out = run_fused(w, d, **KOM)
    torch.cuda.synchronize()
    assert torch.all(torch.isfinite(out)) and torch.equal(out[2], torch.zeros_like(out[2]))


def test_layout_option_validation():
    w = Workload("wide", n_head=9, n_tok=16, hd=256, n_kv=512, rope=RopeParams(n_dims=256),
                 positions=tuple(range(496, 512)), mask_kind="causal")      # 144 rows: no keys-on-M plan
    d = to_device(w)
    with pytest.raises(fr.FrError) as e:
        run_fused(w, d, layout=2)
    assert e.value.status == 2
    with pytest.raises(fr.FrError) as e:                                     # not 16, 32 or 64 rows per slice
        run_fused(named_config("c3"), to_device(named_config("c3")), layout=2, slice_rows=48)
    assert e.value.status == 1
    t = named_config("tiny")                    # hd 64
    with pytest.raises(fr.FrError):
        run_fused(t, to_device(t), layout=2)


@pytest.mark.parametrize("hd", [128, 256])
@pytest.mark.parametrize("slice_rows", [16, 32, 64])
@pytest.mark.parametrize("n_tok,n_head", [(16, 8), (8, 8), (4, 8), (3, 5), (9, 11), (2, 64), (13, 7), (1, 20)])
def test_row_slices(hd, slice_rows, n_tok, n_head):
    """The query rows cut into slices of slice_rows (the MMA's N): one CTA per
    (KV split, slice), each roping or loading only its own rows (slices may
    cut through a token's heads), the merge over every slice's rows."""
    w = Workload("slices", n_head=n_head, n_tok=n_tok, hd=hd, n_kv=5000,
                 rope=RopeParams(n_dims=hd, freq_base=10000.0), positions=tuple(range(4999 - n_tok + 1, 5000)),
                 mask_kind="random5", seed=n_tok * 13 + n_head + slice_rows)
    p = _plan(w, slice_rows=slice_rows)
    assert p["keys_on_m"] == 1 and p["row_slices"] == (w.M + slice_rows - 1) // slice_rows
    d = to_device(w, k_pad=8, q_extra_heads=1)
    ref = oracle_out(w)
    fused = run_fused(w, d, slice_rows=slice_rows, **KOM)
    assert_close(_rows(fused), ref, f"{n_tok}x{n_head} hd {hd} / {slice_rows}")
    two_call, _ = run_two_call(w, d, slice_rows=slice_rows, **KOM)
    torch.cuda.synchronize()
    assert torch.equal(fused, two_call)          # the kernel's own RoPE gives qkv_post's bits


@pytest.mark.parametrize("name", ["sweep:256:16:65536", "sweep:128:16:4096", "sweep:256:8:1024"])
@pytest.mark.parametrize("splits", [1, 3, 1000])
def test_row_slices_forced_splits(name, splits):
    w = make_workload(name)
    d = to_device(w)
    p = _plan(w, splits=splits, slice_rows=32)
    assert p["row_slices"] == (w.M + 31) // 32 and p["splits"] <= max(1, splits)
    assert_close(_rows(run_fused(w, d, splits=splits, slice_rows=32, **KOM)), oracle_out(w), f"{name} splits={splits}")


@pytest.mark.parametrize("n_kv", [1, 129, 20037])
def test_row_slices_ragged_kv(n_kv):
    w = Workload(f"slices-ragged{n_kv}", n_head=8, n_tok=16, hd=256, n_kv=n_kv,
                 rope=RopeParams(n_dims=256, freq_base=10000.0), positions=tuple(range(n_kv - 1, n_kv + 15)),
                 mask_kind="causal", seed=n_kv % 31)
    d = to_device(w, k_pad=16, mask_pad=8)
    assert_close(_rows(run_fused(w, d, slice_rows=32, **KOM)), oracle_out(w), w.name)


def test_barrier_words_across_grid_sizes():
    """The grid barrier's words in one workspace return to zero after every
    call, so calls with different grids (40 sliced CTAs, 152 CTAs, one split
    without a barrier, a timed-out probe) can follow each other on it in any
    order, captured in a graph too."""
    shapes = [make_workload("pi05"), make_workload("sweep:256:1:65536"), make_workload("sweep:128:4:4096"),
              make_workload("sweep:256:16:2048")]
    devs = [to_device(w) for w in shapes]
    refs = [oracle_out(w) for w in shapes]
    nbytes = max(fr.workspace_size(w.n_tok, w.n_head, w.hd, w.n_kv) for w in shapes)
    ws = torch.zeros(nbytes, dtype=torch.uint8, device="cuda")
    order = [0, 1, 2, 3, 1, 0, 3, 2, 0]
    for i in order:
        w, d = shapes[i], devs[i]
        assert_close(_rows(run_fused(w, d, workspace=ws, **KOM)), refs[i], f"{w.name} in sequence")
        assert_close(_rows(run_fused(w, d, workspace=ws, splits=1, **KOM)), refs[i], f"{w.name} one split")
    fr.workspace_check(ws)
    # graph of mixed calls on the same workspace
    outs = [torch.empty((w.n_tok, w.n_head, w.hd), dtype=torch.float32, device="cuda") for w in shapes]
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        for i in order:
            run_fused(shapes[i], devs[i], workspace=ws, out=outs[i], stream=s, **KOM)
    for o in outs:
        o.zero_()
    g.replay()
    g.replay()
    torch.cuda.synchronize()
    for i, w in enumerate(shapes):
        assert_close(_rows(outs[i]), refs[i], f"{w.name} replayed")
    fr.workspace_check(ws)
