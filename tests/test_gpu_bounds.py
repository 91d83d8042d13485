"""Out-of-bounds write checks by guard canaries (no sanitizer on this pool):
every output buffer the library writes (out, the workspace, q16_out, the KV
cache) sits between two 4 KiB margins filled with a byte pattern; after a call
the margins must be byte-identical. Covers the named workloads, ragged row and
key counts, both split-merge strategies, forced clusters and split counts, the
keys-on-M kernel's row slices, prefill windows and fr_kv_append. Also: pointers that are not memory of the
current GPU are rejected on the host before any launch."""
import ctypes

import numpy as np
import pytest
import torch

from gen import RopeParams, Workload, make_workload, named_config
import gqa_kv_head_gb300 as fr
from fr_harness import assert_close, oracle_out, to_device

pytestmark = pytest.mark.gpu

GUARD = 4096
PATTERN = 0xA5


class Guarded:
    """A device byte buffer [GUARD | body | GUARD]; the margins hold PATTERN."""

    def __init__(self, nbytes, dev="cuda"):
        self.n = int(nbytes)
        body = (self.n + 255) // 256 * 256
        self.buf = torch.full((GUARD + body + GUARD,), PATTERN, dtype=torch.uint8, device=dev)
        self.body = self.buf[GUARD:GUARD + self.n]

    def view(self, dtype, shape):
        return self.body.view(dtype).view(shape)

    def assert_intact(self, what):
        torch.cuda.synchronize()
        lo = self.buf[:GUARD]
        hi = self.buf[GUARD + self.n:]
        assert bool(torch.all(lo == PATTERN)), f"{what}: write below the buffer"
        assert bool(torch.all(hi == PATTERN)), f"{what}: write past the end of the buffer"


def _guarded_call(w, d, **kw):
    out_g = Guarded(w.M * w.hd * 4)
    out = out_g.view(torch.float32, (w.n_tok, w.n_head, w.hd))
    nbytes = kw.pop("ws_bytes", None) or fr.workspace_size(w.n_tok, w.n_head, w.hd, w.n_kv)
    ws_g = Guarded(nbytes)
    ws_g.body.zero_()
    fr.decode_attn(d["k"], d["v"], w.n_tok, w.n_head, q=d["q"], pos=d["pos"], rope=w.rope, q_scale=w.q_scale,
                   mask=d["mask"], kq_scale=w.kq_scale, out=out, workspace=ws_g.body, **kw)
    out_g.assert_intact(f"{w.name} out {kw}")
    ws_g.assert_intact(f"{w.name} workspace {kw}")
    return out


def _rows(out):
    return out.reshape(-1, out.shape[-1]).cpu().numpy().astype(np.float64)


@pytest.mark.parametrize("name", ["tiny", "pi05", "c3", "long_decode", "sweep:256:1:65536", "sweep:128:2:4096",
                                  "sweep:256:8:16384", "sweep:128:16:1024"])
def test_guards_named_and_sweep(name):
    w = make_workload(name)
    d = to_device(w)
    out = _guarded_call(w, d)
    assert_close(_rows(out), oracle_out(w), name)


@pytest.mark.parametrize("hd", [128, 256])
@pytest.mark.parametrize("opts", [{"slice_rows": 16}, {"slice_rows": 32}, {"slice_rows": 64},
                                  {"slice_rows": 16, "splits": 1}, {"slice_rows": 32, "splits": 1000}])
def test_guards_keys_on_m_slices(hd, opts):
    """The keys-on-M kernel with ragged rows cut into slices (M = 35: slices
    end inside a token's heads and the last one is short), a one-key last
    tile, padded strides, one split (each slice normalises its own rows) and
    many."""
    w = Workload("ragged-slices", n_head=5, n_tok=7, hd=hd, n_kv=4097, rope=RopeParams(n_dims=hd),
                 positions=tuple(range(4090, 4097)), mask_kind="random5", seed=13)
    d = to_device(w, k_pad=16, mask_pad=8, q_extra_heads=2)
    out = _guarded_call(w, d, layout=2, **opts)
    assert_close(_rows(out), oracle_out(w), f"ragged slices hd {hd} {opts}")


@pytest.mark.parametrize("hd", [64, 128, 256])
@pytest.mark.parametrize("opts", [{}, {"merge_mode": 1}, {"merge_mode": 2}, {"splits": 3, "cluster": 2},
                                  {"splits": 1000, "cluster": 8}, {"splits": 5, "merge_mode": 2}])
def test_guards_ragged_every_plan(hd, opts):
    """Ragged rows (M = 35, not a multiple of any tile) and keys (4097: a
    one-key last tile), padded strides, every merge strategy."""
    w = Workload("ragged-guard", n_head=5, n_tok=7, hd=hd, n_kv=4097, rope=RopeParams(n_dims=hd),
                 positions=tuple(range(4090, 4097)), mask_kind="random5", seed=11)
    d = to_device(w, k_pad=16, mask_pad=8, q_extra_heads=2)
    out = _guarded_call(w, d, **opts)
    assert_close(_rows(out), oracle_out(w), f"ragged hd {hd} {opts}")


def test_guards_in_launch_merge_small_workspace():
    """The in-launch merge plan in a workspace that admits only it (cluster
    partials + arrival tickets), several clusters per row tile."""
    w = named_config("long_decode")
    d = to_device(w)
    out = _guarded_call(w, d, ws_bytes=9 << 20)
    assert_close(_rows(out), oracle_out(w), "long decode in a 9 MiB workspace")


@pytest.mark.parametrize("n_tok", [968, 203])
def test_guards_prefill_window(n_tok):
    w = named_config("pi05_prefill").with_(n_tok=n_tok, positions=tuple(range(n_tok)))
    d = to_device(w)
    out = _guarded_call(w, d)
    rows = np.unique(np.concatenate([np.arange(0, w.M, 97), [w.M - 1]]))
    assert_close(_rows(out)[rows], oracle_out(w, rows=rows), f"prefill {n_tok}")


def test_guards_qkv_post():
    for name in ("tiny", "pi05", "long_decode"):
        w = named_config(name)
        d = to_device(w)
        g16 = Guarded(w.M * w.hd * 2)
        g32 = Guarded(w.M * w.hd * 4)
        fr.qkv_post(d["q"], d["pos"], w.n_head, w.hd, w.rope, w.q_scale,
                    q16_out=g16.view(torch.float16, (w.M, w.hd)), q32_out=g32.view(torch.float32, (w.M, w.hd)))
        g16.assert_intact(f"{name} q16_out")
        g32.assert_intact(f"{name} q32_out")


def test_guards_kv_append():
    hd, n_ctx, n_tok = 256, 1024, 10
    rp = RopeParams(n_dims=hd)
    kg = Guarded(n_ctx * hd * 2)
    vg = Guarded(n_ctx * hd * 2)
    kc = kg.view(torch.float16, (n_ctx, hd))
    vc = vg.view(torch.float16, (n_ctx, hd))
    kc.fill_(1.0)
    vc.fill_(1.0)
    k_new = torch.randn((n_tok, hd), device="cuda")
    v_new = torch.randn((n_tok, hd), device="cuda")
    pos = torch.arange(958, 968, dtype=torch.int32, device="cuda")
    fr.kv_append(k_new, v_new, pos, rp, kc, vc, 958, pad=(968, 1024))
    kg.assert_intact("k_cache")
    vg.assert_intact("v_cache")
    assert bool(torch.all(kc[:958] == 1.0)) and bool(torch.all(vc[:958] == 1.0))
    assert bool(torch.all(kc[968:] == 0)) and bool(torch.all(vc[968:] == 0))


def test_pointers_not_on_this_gpu_are_rejected():
    """A host buffer passed where device memory is expected: FR_ERR_INVALID_ARG
    from the host-side check, nothing launched."""
    lib = fr.load()
    w = named_config("tiny")
    d = to_device(w)
    host = torch.zeros(w.M * w.hd * 4 + 256, dtype=torch.uint8)            # pageable host memory
    pinned = torch.zeros(w.M * w.hd * 4 + 256, dtype=torch.uint8).pin_memory()
    ws = fr.make_workspace(w.n_tok, w.n_head, w.hd, w.n_kv)
    rp = fr.rope_params(w.hd)
    for bad in (host, pinned):
        addr = (bad.data_ptr() + 255) // 256 * 256
        st = lib.fr_decode_attn(None, d["q"].data_ptr(), d["q"].stride(0), d["pos"].data_ptr(), ctypes.byref(rp),
                                0.0, d["k"].data_ptr(), w.hd, d["v"].data_ptr(), w.hd, None, 0, w.n_tok, w.n_head,
                                w.hd, w.n_kv, 1.0, addr, ws.data_ptr(), ws.numel(),
                                ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
        assert st == 1
        st = lib.fr_qkv_post(d["q"].data_ptr(), d["q"].stride(0), d["pos"].data_ptr(), w.n_tok, w.n_head, w.hd,
                             ctypes.byref(rp), 0.0, addr, None,
                             ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
        assert st == 1
    torch.cuda.synchronize()
