"""fr_decode_attn_noalloc, the entry point for callers that cannot allocate
device memory (their memory is planned up front by an allocator they do not
control, or they must not allocate once running). It must give the same result
as fr_decode_attn with a caller-owned workspace, call after call, although every
call reuses the library's one fixed scratch array.

This file is collected last on purpose, so that a run stopping at the first
failure has already run every other test; it also passes on its own."""
import ctypes

import numpy as np
import pytest
import torch

from gen import named_config
import gqa_kv_head_gb300 as fr
from fr_harness import assert_close, run_fused, to_device

pytestmark = pytest.mark.gpu


def _rows(out):
    return out.reshape(-1, out.shape[-1]).cpu().numpy().astype(np.float64)


@pytest.mark.parametrize("name", ["tiny", "pi05", "c3", "long_decode"])
def test_noalloc_matches_workspace_entry_on_two_calls(name):
    w = named_config(name)
    d = to_device(w)
    ref = _rows(run_fused(w, d))                       # fr_decode_attn + its own workspace
    for call in range(2):
        out = fr.decode_attn_noalloc(d["k"], d["v"], w.n_tok, w.n_head, q=d["q"], pos=d["pos"],
                                     rope=w.rope, q_scale=w.q_scale, mask=d["mask"],
                                     kq_scale=w.kq_scale)
        torch.cuda.synchronize()
        assert_close(_rows(out), ref, f"{name} no-alloc call {call}")


def test_noalloc_given_f16_q_rows():
    w = named_config("c3")
    d = to_device(w)
    q16, _ = fr.qkv_post(d["q"], d["pos"], w.n_head, w.hd, w.rope, w.q_scale)
    ref = _rows(fr.decode_attn(d["k"], d["v"], w.n_tok, w.n_head, q16=q16, mask=d["mask"]))
    for call in range(2):
        out = fr.decode_attn_noalloc(d["k"], d["v"], w.n_tok, w.n_head, q16=q16, mask=d["mask"])
        torch.cuda.synchronize()
        assert_close(_rows(out), ref, f"q16 no-alloc call {call}")


def test_noalloc_rejects_shapes_beyond_its_scratch():
    lib = fr.load()
    need = lib.fr_decode_attn_workspace_size(16, 32, 256, 32768)
    assert need > 9 * 2**20
    k = torch.zeros((32768, 256), dtype=torch.float16, device="cuda")
    q16 = torch.zeros((512, 256), dtype=torch.float16, device="cuda")
    with pytest.raises(fr.FrError) as e:
        fr.decode_attn_noalloc(k, k, 16, 32, q16=q16)
    assert e.value.status == 3                        # FR_ERR_WORKSPACE
