"""GPU parity of fr_decode_attn against the fp64 oracle, through the C ABI.

Bar: max-abs <= 2e-3 and relative L2 <= 1e-3 for the fp32 output; bitwise
equality where the pages claim it (fused qkv_post == the two-call form,
masked/pad columns inert, head permutation) or where the arithmetic is exact
(one key returns V[0])."""
import numpy as np
import pytest
import torch

import oracle
from gen import RopeParams, Workload, named_config
import gqa_kv_head_gb300 as fr
from fr_harness import assert_close, host_kv, oracle_out, run_fused, run_two_call, to_device

pytestmark = pytest.mark.gpu


def _out_rows(out):
    return out.reshape(-1, out.shape[-1]).cpu().numpy().astype(np.float64)


@pytest.mark.parametrize("name", ["tiny", "pi05", "c3", "long_decode"])
def test_named_configs_full(name):
    w = named_config(name)
    d = to_device(w)
    out = run_fused(w, d)
    torch.cuda.synchronize()
    assert_close(_out_rows(out), oracle_out(w), name)


@pytest.mark.parametrize("name", ["tiny", "pi05", "c3", "long_decode"])
def test_fused_equals_two_call_bitwise(name):
    """FlashRT PR #185: the f16 Q from qkv_post is bit-identical to what the
    attention's own gather would produce."""
    w = named_config(name)
    d = to_device(w)
    a = run_fused(w, d)
    b, _ = run_two_call(w, d)
    torch.cuda.synchronize()
    assert torch.equal(a, b)


@pytest.mark.parametrize("n_kv", [1, 7, 63, 65, 1000, 4097])
@pytest.mark.parametrize("hd", [64, 128, 256])
def test_ragged_kv_and_strides(n_kv, hd):
    """Ragged KV lengths (partial last tile, partial mask chunk), padded K/V and
    mask row strides, and Q rows read from a fused-QKV-shaped buffer."""
    w = Workload(f"ragged{n_kv}", n_head=5, n_tok=7, hd=hd, n_kv=n_kv,
                 rope=RopeParams(n_dims=hd, freq_base=10000.0),
                 positions=tuple(range(n_kv - 1, n_kv + 6)), mask_kind="random5", seed=3)
    d = to_device(w, k_pad=16, mask_pad=8, q_extra_heads=2)
    out = _out_rows(run_fused(w, d))
    assert_close(out, oracle_out(w), w.name)


def test_128_key_tiles_ragged_tail():
    """hd 128 over a long KV range takes 128-key tiles (P written over S in
    TMEM); 20037 keys leave a last tile of 69 keys, across the boundary of the
    two softmax halves. Padded strides, random mask, extra Q heads."""
    w = Workload("tile128", n_head=8, n_tok=16, hd=128, n_kv=20037,
                 rope=RopeParams(n_dims=128, freq_base=10000.0),
                 positions=tuple(range(20021, 20037)), mask_kind="random5", seed=15)
    d = to_device(w, k_pad=16, mask_pad=8, q_extra_heads=2)
    out = _out_rows(run_fused(w, d))
    assert_close(out, oracle_out(w), "128-key tiles, ragged tail")
    ref = oracle_out(w)
    for splits, cluster in ((1, 1), (5, 1), (8, 8)):
        o = _out_rows(run_fused(w, d, splits=splits, cluster=cluster))
        assert_close(o, ref, f"128-key tiles, splits={splits} cluster={cluster}")


@pytest.mark.parametrize("hd", [64, 128, 256])
@pytest.mark.parametrize("n_head,n_tok", [(1, 1), (32, 16), (3, 11), (512, 1)])
def test_edge_shapes(hd, n_head, n_tok):
    w = Workload("edge", n_head=n_head, n_tok=n_tok, hd=hd, n_kv=777,
                 rope=RopeParams(n_dims=hd, freq_base=10000.0),
                 positions=tuple(range(760, 760 + n_tok)), mask_kind="causal", seed=5)
    out = _out_rows(run_fused(w, to_device(w)))
    assert_close(out, oracle_out(w), f"edge {n_head}x{n_tok} hd{hd}")


@pytest.mark.parametrize("name", ["pi05", "c3", "long_decode"])
def test_split_and_cluster_invariance(name):
    """Any split count / cluster size (including one split, one CTA per cluster,
    several clusters per row tile) gives the oracle's result."""
    w = named_config(name)
    d = to_device(w)
    ref = oracle_out(w)
    outs = []
    for splits, cluster in ((1, 1), (2, 2), (3, 1), (8, 8), (16, 4), (48, 8), (1000, 2)):
        o = _out_rows(run_fused(w, d, splits=splits, cluster=cluster))
        assert_close(o, ref, f"{name} splits={splits} cluster={cluster}")
        outs.append(o)
    for o in outs[1:]:
        # fp32 summation order only: relative to the output scale (outlier rows reach ~50)
        assert np.max(np.abs(o - outs[0])) <= 2e-5 * max(1.0, np.abs(outs[0]).max())


@pytest.mark.parametrize("name", ["tiny", "pi05", "c3"])
def test_mma_sync_engine_matches(name):
    """The mma.sync kernel (engine 1) stays a valid path through the same ABI."""
    w = named_config(name)
    d = to_device(w)
    assert_close(_out_rows(run_fused(w, d, engine=1)), oracle_out(w), f"{name} engine 1")
    for s in (1, 2, 1000):
        assert_close(_out_rows(run_fused(w, d, engine=1, splits=s)), oracle_out(w), f"{name} v1 s{s}")


def test_q16_input_path_with_clusters():
    """Given f16 Q rows, every cluster size gives the fused result bitwise (each
    CTA of a cluster loads the whole Q tile itself)."""
    w = named_config("c3")
    d = to_device(w)
    q16, _ = fr.qkv_post(d["q"], d["pos"], w.n_head, w.hd, w.rope, w.q_scale)
    for cluster in (1, 2, 4, 8):
        o = fr.decode_attn(d["k"], d["v"], w.n_tok, w.n_head, q16=q16, mask=d["mask"], cluster=cluster)
        assert torch.equal(o, run_fused(w, d, cluster=cluster))


def test_device_timeout_is_reported_and_recoverable():
    """A bounded wait on a barrier that nothing signals gives up, the status
    word reports it, the context stays usable and the next call is clean."""
    w = named_config("pi05")
    d = to_device(w)
    ws = fr.make_workspace(w.n_tok, w.n_head, w.hd, w.n_kv)
    run_fused(w, d, workspace=ws, wait_probe_iters=1000)
    with pytest.raises(fr.FrError) as e:
        fr.workspace_check(ws)
    assert e.value.status == 5
    fr.workspace_check(ws)                       # cleared
    out = _out_rows(run_fused(w, d, workspace=ws))
    fr.workspace_check(ws)
    assert_close(out, oracle_out(w), "after timeout")


def test_single_key_is_v0_bitwise():
    w = Workload("one", n_head=4, n_tok=3, hd=128, n_kv=1, rope=RopeParams(n_dims=128),
                 positions=(0, 5, 9), seed=2)
    d = to_device(w)
    out = run_fused(w, d)
    torch.cuda.synchronize()
    v0 = d["v"][0].float()
    assert torch.equal(out.reshape(-1, 128), v0.expand(w.M, 128))


def test_zero_q_is_mean_of_visible_v():
    w = named_config("pi05")
    d = to_device(w)
    q16 = torch.zeros((w.M, w.hd), dtype=torch.float16, device="cuda")
    out = _out_rows(fr.decode_attn(d["k"], d["v"], w.n_tok, w.n_head, q16=q16, mask=d["mask"]))
    k, v = host_kv(w)
    ref = oracle.attention_collapsed(np.zeros((w.M, w.hd)), k, v, w.mask(), w.n_tok, w.n_head)
    assert_close(out, ref, "zero q")


def test_masked_and_pad_columns_inert_bitwise():
    """Pad rows zero and masked by -inf (FlashRT PR #185, qkv_post pads KV to
    the KQ stride): replacing their contents with finite garbage changes nothing."""
    w = named_config("pi05")
    d = to_device(w)
    a = run_fused(w, d)
    d["k"][968:] = 37.0
    d["v"][968:] = -1234.0
    b = run_fused(w, d)
    torch.cuda.synchronize()
    assert torch.equal(a, b)


def test_head_permutation_permutes_rows_bitwise():
    """The collapsed GEMM treats every t-major row alike (FlashRT PR #185,
    'numerically identical to the batched form')."""
    w = named_config("c3")
    d = to_device(w)
    a = run_fused(w, d)
    perm = torch.randperm(w.n_head, generator=torch.Generator().manual_seed(0))
    q3 = d["q"].reshape(w.n_tok, w.n_head, w.hd)
    d2 = dict(d, q=q3[:, perm.cuda(), :].contiguous().reshape(w.n_tok, -1))
    b = run_fused(w, d2)
    torch.cuda.synchronize()
    assert torch.equal(a[:, perm.cuda(), :], b)


def test_fully_masked_token_is_zero():
    w = named_config("c3")
    d = to_device(w)
    d["mask"][3, :] = float("-inf")
    out = run_fused(w, d)
    torch.cuda.synchronize()
    assert torch.all(torch.isfinite(out))
    assert torch.equal(out[3], torch.zeros_like(out[3]))
    others = [t for t in range(w.n_tok) if t != 3]
    m = w.mask().copy()
    m[3, :] = -np.inf
    k, v = host_kv(w)
    ref = oracle.decode_attn(w.q(), w.pos(), k, v, m, w.rope, w.q_scale).reshape(w.n_tok, w.n_head, -1)
    assert_close(out.cpu().numpy()[others], ref[others], "other tokens")


def test_repeated_calls_reuse_workspace():
    """Arrival tickets reset themselves: back-to-back calls on one workspace
    give identical results."""
    w = named_config("c3")
    d = to_device(w)
    ws = fr.make_workspace(w.n_tok, w.n_head, w.hd, w.n_kv)
    outs = [run_fused(w, d, workspace=ws).clone() for _ in range(3)]
    torch.cuda.synchronize()
    assert torch.equal(outs[0], outs[1]) and torch.equal(outs[1], outs[2])
    fr.workspace_check(ws)


def test_graph_capture_replay():
    """No allocation inside the call: it can be captured and replayed."""
    w = named_config("pi05")
    d = to_device(w)
    ws = fr.make_workspace(w.n_tok, w.n_head, w.hd, w.n_kv)
    out = torch.empty((w.n_tok, w.n_head, w.hd), dtype=torch.float32, device="cuda")
    ref = run_fused(w, d, workspace=ws).clone()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        run_fused(w, d, workspace=ws, out=out, stream=s)
    out.zero_()
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(out, ref)


def test_unsupported_returns_status():
    w = named_config("tiny")
    d = to_device(w)
    with pytest.raises(fr.FrError):
        fr.decode_attn(d["k"], d["v"], 17, 1, q16=torch.zeros((17, 64), dtype=torch.float16,
                                                                device="cuda"))


@pytest.mark.parametrize("name", ["tiny", "pi05", "c3", "long_decode"])
@pytest.mark.parametrize("splits", [None, 1, 3])
def test_merge_kernel_mode(name, splits):
    """Split states merged by the separate merge kernel (every SM one split)."""
    w = named_config(name)
    d = to_device(w)
    o = _out_rows(run_fused(w, d, merge_mode=2, splits=splits))
    assert_close(o, oracle_out(w), f"{name} merge kernel splits={splits}")


def test_merge_kernel_mode_ragged_and_repeatable():
    w = Workload("ragged-merge", n_head=5, n_tok=7, hd=64, n_kv=4097,
                 rope=RopeParams(n_dims=64, freq_base=10000.0),
                 positions=tuple(range(4096, 4103)), mask_kind="random5", seed=9)
    d = to_device(w, k_pad=16, mask_pad=8, q_extra_heads=2)
    ws = fr.make_workspace(w.n_tok, w.n_head, w.hd, w.n_kv)
    a = run_fused(w, d, merge_mode=2, workspace=ws).clone()
    b = run_fused(w, d, merge_mode=2, workspace=ws)
    torch.cuda.synchronize()
    assert torch.equal(a, b)
    assert_close(_out_rows(a), oracle_out(w), "ragged merge kernel")


def test_plan_reports_the_launch_shape():
    """fr_decode_attn_plan: one or two splits keep the in-launch merge, more
    splits go to the merge kernel; launches count qkv_post, attention, merge."""
    tiny = named_config("tiny")
    p = fr.decode_attn_plan(tiny.n_tok, tiny.n_head, tiny.hd, tiny.n_kv)
    assert p["engine"] == 0 and p["merge_kernel"] == 0 and p["launches"] == 2 and p["splits"] <= 2
    w = named_config("pi05")
    # the library's own choice here: the keys-on-M kernel, five 16-row slices, one launch
    pa = fr.decode_attn_plan(w.n_tok, w.n_head, w.hd, w.n_kv)
    assert pa["keys_on_m"] == 1 and pa["row_slices"] == 5 and pa["launches"] == 1 and pa["merge_kernel"] == 0
    p = fr.decode_attn_plan(w.n_tok, w.n_head, w.hd, w.n_kv, layout=1)
    assert p["merge_kernel"] == 1 and p["cluster"] == 1 and p["launches"] == 3 and p["row_slices"] == 1
    assert p["splits"] == 16                        # one 64-key tile per split
    assert fr.decode_attn_plan(w.n_tok, w.n_head, w.hd, w.n_kv, fused_qkv_post=False, layout=1)["launches"] == 2
    p1 = fr.decode_attn_plan(w.n_tok, w.n_head, w.hd, w.n_kv, merge_mode=1)
    assert p1["merge_kernel"] == 0 and p1["cluster"] > 1 and p1["launches"] == 2
    # a workspace of the in-launch size only keeps the in-launch plan, or cuts
    # the split count when the merge kernel is forced
    lw = named_config("long_decode")
    small = 9 << 20
    assert fr.decode_attn_plan(lw.n_tok, lw.n_head, lw.hd, lw.n_kv, workspace_bytes=small)["merge_kernel"] == 0
    pf = fr.decode_attn_plan(lw.n_tok, lw.n_head, lw.hd, lw.n_kv, workspace_bytes=small, merge_mode=2)
    assert pf["merge_kernel"] == 1 and pf["splits"] * pf["row_tiles"] * 128 * (lw.hd * 4 + 8) <= small
    assert fr.decode_attn_plan(w.n_tok, w.n_head, w.hd, w.n_kv, engine=1)["launches"] == 1


def test_forced_merge_kernel_with_cut_split_count():
    """merge_mode 2 with a workspace that holds fewer splits than the default:
    the split count is cut to fit and the result still matches the oracle."""
    w = named_config("long_decode")
    d = to_device(w)
    nbytes = 9 << 20
    ws = torch.zeros(nbytes, dtype=torch.uint8, device="cuda")
    p = fr.decode_attn_plan(w.n_tok, w.n_head, w.hd, w.n_kv, workspace_bytes=nbytes, merge_mode=2)
    assert p["merge_kernel"] == 1
    o = _out_rows(run_fused(w, d, merge_mode=2, workspace=ws))
    assert_close(o, oracle_out(w), "long decode, merge kernel in a 9 MiB workspace")
