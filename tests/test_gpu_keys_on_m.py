"""The kernel with 128-key tiles on the MMA's M side and the query rows on
its N (layout 2: M = n_tok*n_head <= 64, hd 128 or 256), against the fp64
oracle through the C ABI: every row count up to 64 (N = 16, 32, 64 with
padded rows), ragged KV lengths, masks, padded strides, forced split counts,
a workspace that holds fewer split states, and the same result as the
128-row query-tile kernel (layout 1).

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


KOM = dict(layout=2)      # the library picks this layout itself for M <= 32 rows and n_kv >= max(1024, 256 M)


@pytest.mark.parametrize("hd", [128, 256])
@pytest.mark.parametrize("n_tok,n_head", [(1, 1), (1, 8), (2, 8), (3, 5), (4, 8), (7, 5), (8, 8), (16, 4), (1, 64),
                                          (11, 3)])
def test_row_counts(hd, n_tok, n_head):
    w = Workload("keys-on-m", n_head=n_head, n_tok=n_tok, hd=hd, n_kv=3000,
                 rope=RopeParams(n_dims=hd, freq_base=10000.0), positions=tuple(range(2999 - n_tok + 1, 3000)),
                 mask_kind="causal", seed=n_tok * 7 + n_head)
    assert _plan(w)["keys_on_m"] == 1
    auto = fr.decode_attn_plan(w.n_tok, w.n_head, w.hd, w.n_kv)["keys_on_m"]
    assert auto == (1 if w.M <= 32 and w.n_kv >= max(1024, 256 * w.M) else 0)
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
    w = named_config("c3")                      # 128 rows: no keys-on-M plan
    d = to_device(w)
    with pytest.raises(fr.FrError) as e:
        run_fused(w, d, layout=2)
    assert e.value.status == 2
    t = named_config("tiny")                    # hd 64
    with pytest.raises(fr.FrError):
        run_fused(t, to_device(t), layout=2)
