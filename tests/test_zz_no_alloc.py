"""fr_decode_attn_noalloc, the entry point for callers that cannot allocate
device memory (their memory is planned up front by an allocator they do not
control, or they must not allocate once running). On two calls in a row it
must match the fp64 oracle and fr_decode_attn with a caller-owned workspace,
although every call reuses the library's one fixed scratch array.

This file is collected last on purpose, so that a run stopping at the first
failure has already run every other test; it also passes on its own."""
import numpy as np
import pytest
import torch

from gen import RopeParams, Workload, named_config
import gqa_kv_head_gb300 as fr
from fr_harness import assert_close, oracle_out, run_fused, to_device

pytestmark = pytest.mark.gpu


def _rows(out):
    return out.reshape(-1, out.shape[-1]).cpu().numpy().astype(np.float64)


@pytest.mark.parametrize("name", ["tiny", "pi05", "c3", "long_decode"])
def test_noalloc_matches_oracle_and_workspace_entry_on_two_calls(name):
    w = named_config(name)
    d = to_device(w)
    ref = oracle_out(w)
    ws_out = _rows(run_fused(w, d))                    # fr_decode_attn + its own workspace
    for call in range(2):
        out = fr.decode_attn_noalloc(d["k"], d["v"], w.n_tok, w.n_head, q=d["q"], pos=d["pos"],
                                     rope=w.rope, q_scale=w.q_scale, mask=d["mask"],
                                     kq_scale=w.kq_scale)
        torch.cuda.synchronize()
        got = _rows(out)
        assert_close(got, ref, f"{name} no-alloc call {call} vs oracle")
        assert_close(got, ws_out, f"{name} no-alloc call {call} vs fr_decode_attn")
    fr.decode_attn_noalloc_check()                     # no device wait gave up


def test_noalloc_given_f16_q_rows():
    w = named_config("c3")
    d = to_device(w)
    q16, _ = fr.qkv_post(d["q"], d["pos"], w.n_head, w.hd, w.rope, w.q_scale)
    ref = oracle_out(w)
    for call in range(2):
        out = fr.decode_attn_noalloc(d["k"], d["v"], w.n_tok, w.n_head, q16=q16, mask=d["mask"])
        torch.cuda.synchronize()
        assert_close(_rows(out), ref, f"q16 no-alloc call {call}")


def test_noalloc_prefill_window_within_its_scratch():
    """A longer query window whose smallest workspace fits the scratch (hd 256,
    80 tokens x 8 heads = 640 rows) runs and matches the oracle."""
    w = Workload("noalloc-prefill", n_head=8, n_tok=80, hd=256, n_kv=1024, n_kv_real=1000,
                 rope=RopeParams(n_dims=256), positions=tuple(range(920, 1000)), mask_kind="causal", seed=4)
    d = to_device(w)
    out = fr.decode_attn_noalloc(d["k"], d["v"], w.n_tok, w.n_head, q=d["q"], pos=d["pos"], rope=w.rope,
                                 mask=d["mask"])
    torch.cuda.synchronize()
    assert_close(_rows(out), oracle_out(w), "no-alloc prefill window")


@pytest.mark.parametrize("n_tok,n_head,hd,n_kv", [(16, 32, 256, 32768), (2048, 8, 128, 4096)])
def test_noalloc_rejects_shapes_beyond_its_scratch(n_tok, n_head, hd, n_kv):
    """Shapes whose smallest workspace exceeds the 9 MiB scratch: FR_ERR_WORKSPACE,
    nothing launched."""
    k = torch.zeros((n_kv, hd), dtype=torch.float16, device="cuda")
    q16 = torch.zeros((n_tok * n_head, hd), dtype=torch.float16, device="cuda")
    with pytest.raises(fr.FrError) as e:
        fr.decode_attn_noalloc(k, k, n_tok, n_head, q16=q16)
    assert e.value.status == 3                        # FR_ERR_WORKSPACE
