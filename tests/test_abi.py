"""The C-ABI library without a GPU: it builds, loads, exports every function
include/fr_kernels.h declares, and rejects invalid arguments on the host
before any CUDA call is made."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from gqa_kv_head_gb300 import build
    build.build()
    import gqa_kv_head_gb300 as fr
    return fr.load()


def _declared():
    names = set()
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if fn.endswith(".h"):
            src = open(os.path.join(ROOT, "include", fn)).read()
            src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
            names |= set(re.findall(r"\b(fr_[a-z0-9_]+)\s*\(", src))
    return names


def test_exports_every_declared_symbol(lib):
    names = _declared()
    assert {"fr_qkv_post", "fr_decode_attn", "fr_decode_attn_workspace_size"} <= names
    for n in sorted(names):
        assert hasattr(lib, n), f"{n} declared in include/ but not exported"


def test_library_is_in_tree(lib):
    import gqa_kv_head_gb300 as fr
    assert os.path.realpath(fr.library_path()).startswith(os.path.realpath(ROOT))


def test_status_strings_and_version(lib):
    assert lib.fr_status_string(0) == b"FR_OK"
    for s in range(1, 6):
        assert lib.fr_status_string(s).startswith(b"FR_ERR_")
    assert lib.fr_abi_version() >> 16 == 4


def test_workspace_size_host_logic(lib):
    ws = lib.fr_decode_attn_workspace_size
    assert ws(10, 8, 256, 1024) > 0
    assert ws(17, 1, 128, 64) == 0          # > 16 tokens with < 8 heads: no 16-token mask window
    assert ws(17, 8, 128, 64) > 0           # prefill window, 8 heads
    assert ws(16, 4097, 128, 64) == 0       # M > 65536
    assert ws(8193, 8, 128, 64) == 0        # n_tok > 8192
    assert ws(1, 1, 96, 64) == 0            # unsupported hd
    assert ws(1, 1, 128, 0) == 0
    assert ws(16, 8, 128, 65536) >= ws(16, 8, 128, 4096) >= ws(16, 8, 128, 64)


FAKE = 0x10000            # aligned, never dereferenced: validation fails first
MIS = 0x10004


def _rope(lib):
    from gqa_kv_head_gb300 import rope_params
    return rope_params(128)


def _attn(lib, q16=FAKE, k=FAKE, v=FAKE, mask=None, k_rs=128, m_rs=0, n_tok=4, n_head=8,
          hd=128, n_kv=64, ws=FAKE, ws_bytes=0, rp=None):
    return lib.fr_decode_attn(q16, None, 0, None, rp, 0.0, k, k_rs, v, 128, mask, m_rs,
                              n_tok, n_head, hd, n_kv, 1.0, FAKE, ws, ws_bytes, None)


def test_decode_attn_validation(lib):
    assert _attn(lib, k=None) == 1
    assert _attn(lib, hd=96) == 2
    assert _attn(lib, n_tok=17, n_head=4) == 2
    assert _attn(lib, n_tok=16, n_head=4097) == 2
    assert _attn(lib, n_kv=0) == 1
    assert _attn(lib, k_rs=100) == 1                 # stride not a multiple of 8
    assert _attn(lib, k_rs=64) == 1                  # stride < hd
    assert _attn(lib, k=MIS) == 1                    # misaligned pointer
    assert _attn(lib, mask=FAKE, m_rs=32) == 1       # mask stride < n_kv
    assert _attn(lib, ws=None) == 1
    assert _attn(lib, ws_bytes=16) == 3              # workspace too small
    # fused path without q/pos/rope
    assert _attn(lib, q16=None) == 1
    from gqa_kv_head_gb300._abi import FrAttnOpts
    ws_ok = lib.fr_decode_attn_workspace_size(4, 8, 128, 64)
    for bad in (FrAttnOpts(7, 0, 0, 0, 0), FrAttnOpts(0, -1, 0, 0, 0), FrAttnOpts(0, 0, 3, 0, 0),
                FrAttnOpts(0, 0, 16, 0, 0), FrAttnOpts(0, 0, 0, -5, 0), FrAttnOpts(0, 0, 0, 0, 3),
                FrAttnOpts(0, 0, 0, 0, 0, 3), FrAttnOpts(0, 0, 0, 0, 0, 2, 24), FrAttnOpts(0, 0, 0, 0, 0, 2, -16)):
        assert lib.fr_decode_attn_ex(FAKE, None, 0, None, None, 0.0, FAKE, 128, FAKE, 128, None, 0,
                                     4, 8, 128, 64, 1.0, FAKE, FAKE, ws_ok, ctypes.byref(bad), None) == 1


def test_qkv_post_validation(lib):
    rp = _rope(lib)
    call = lambda **kw: lib.fr_qkv_post(kw.get("q", FAKE), kw.get("stride", 8 * 128),
                                        kw.get("pos", FAKE), kw.get("n_tok", 4), 8,
                                        kw.get("hd", 128), ctypes.byref(kw.get("rp", rp)),
                                        0.1, kw.get("out", FAKE), None, None)
    assert call(q=None) == 1
    assert call(out=None) == 1
    assert call(hd=80) == 2
    assert call(n_tok=8193) == 2
    assert call(stride=8 * 128 - 4) == 1
    assert call(stride=8 * 128 + 2) == 1
    assert call(q=MIS) == 1
    from gqa_kv_head_gb300 import rope_params
    assert call(rp=rope_params(127)) == 1            # odd n_dims
    assert call(rp=rope_params(256)) == 1            # n_dims > hd
    assert call(rp=rope_params(128, freq_base=-1.0)) == 1
    assert call(rp=rope_params(128, ext_factor=1.0, n_ctx_orig=0)) == 1
    assert call(rp=rope_params(128, mode=2)) == 1                       # unknown angle mode
    assert call(rp=rope_params(128, freq_factors=[1.0] * 63 + [0.0])) == 1   # a zero divisor
    assert call(rp=rope_params(128, mode=1, freq_factors=[1.0] * 63 + [float("nan")])) == 1


def test_plan_validation(lib):
    from gqa_kv_head_gb300._abi import FrAttnOpts, FrAttnPlan
    plan = FrAttnPlan()
    ws_ok = lib.fr_decode_attn_workspace_size(10, 8, 256, 1024)
    call = lambda n_tok=10, hd=256, ws=ws_ok, opts=None, out=ctypes.byref(plan): lib.fr_decode_attn_plan(
        n_tok, 8, hd, 1024, 1, ws, opts, out)
    assert call(out=None) == 1
    assert call(hd=96) == 2
    assert call(n_tok=8193) == 2
    assert call(ws=64) == 3
    assert call(opts=ctypes.byref(FrAttnOpts(0, 0, 0, 0, 5))) == 1
    assert call(opts=ctypes.byref(FrAttnOpts(0, 0, 3, 0, 0))) == 1


def test_workspace_size_covers_the_merge_kernel_plan(lib):
    # room for the most splits any plan uses: 160 over the row tiles, each split
    # 128 rows of hd fp32 plus an (m, l) pair per row
    ws = lib.fr_decode_attn_workspace_size
    for n_tok, n_head, hd in ((10, 8, 256), (16, 32, 128), (1, 4, 64)):
        rt = (n_tok * n_head + 127) // 128
        assert ws(n_tok, n_head, hd, 1024) >= (160 // rt) * rt * 128 * (hd * 4 + 8)


def test_prefill_shapes_host_logic(lib):
    """Longer query windows run on the tcgen05 engine only; the mma.sync
    engine keeps the decode bounds."""
    from gqa_kv_head_gb300._abi import FrAttnOpts, FrAttnPlan
    n_tok, n_head, hd, n_kv = 968, 8, 256, 1024
    ws = lib.fr_decode_attn_workspace_size(n_tok, n_head, hd, n_kv)
    assert ws > 0
    # no per-row-tile cluster partials beyond 4 row tiles: the workspace stays modest
    assert ws < 64 << 20
    plan = FrAttnPlan()
    assert lib.fr_decode_attn_plan(n_tok, n_head, hd, n_kv, 1, ws, ctypes.byref(FrAttnOpts(1, 0, 0, 0, 0)),
                                   ctypes.byref(plan)) == 2
    assert lib.fr_decode_attn_ex(FAKE, None, 0, None, None, 0.0, FAKE, hd, FAKE, hd, None, 0,
                                 n_tok, n_head, hd, n_kv, 1.0, FAKE, FAKE, ws,
                                 ctypes.byref(FrAttnOpts(1, 0, 0, 0, 0)), None) == 2


def test_kv_append_validation(lib):
    rp = _rope(lib)
    def call(k=FAKE, v=FAKE, pos=FAKE, n_tok=4, hd=128, ks=128, kr=128, n_ctx=64, row0=10, pb=40, pe=64,
             k32=None, rp_=rp):
        return lib.fr_kv_append(k, ks, v, 128, pos, n_tok, hd, ctypes.byref(rp_), FAKE, kr, FAKE, 128,
                                n_ctx, row0, pb, pe, k32, None, None)
    assert call(k=None) == 1
    assert call(pos=None) == 1
    assert call(hd=96) == 2
    assert call(n_tok=8193) == 2
    assert call(ks=100) == 1                 # f32 row stride not a multiple of 4
    assert call(ks=64) == 1                  # stride < hd
    assert call(kr=132) == 1                 # f16 row stride not a multiple of 8
    assert call(k=MIS) == 1                  # misaligned
    assert call(k32=MIS) == 1
    assert call(row0=62) == 1                # tail past n_ctx
    assert call(row0=-1) == 1
    assert call(pb=12, pe=20) == 1           # pad overlaps the tail rows
    assert call(pe=65) == 1                  # pad past n_ctx
    assert call(pb=30, pe=20) == 1
    from gqa_kv_head_gb300 import rope_params
    assert call(rp_=rope_params(127)) == 1   # odd n_dims


def test_workspace_init_rejects_null(lib):
    assert lib.fr_workspace_init(None, 4096, None) == 1
    assert lib.fr_workspace_check(None, None) == 1


def test_binding_has_no_cpu_path():
    """The Python layer is marshalling only: no numpy/oracle import, and it
    refuses CPU tensors instead of computing anything."""
    import gqa_kv_head_gb300 as fr
    pkg = os.path.dirname(fr.__file__)
    for fn in os.listdir(pkg):
        if fn.endswith(".py"):
            src = open(os.path.join(pkg, fn)).read()
            assert "import oracle" not in src and "from oracle" not in src, fn
    import torch
    with pytest.raises(ValueError):
        fr.decode_attn(torch.zeros(4, 64, dtype=torch.float16), torch.zeros(4, 64, dtype=torch.float16),
                       1, 1, q16=torch.zeros(1, 64, dtype=torch.float16))


def test_noalloc_size_limit_matches_the_documented_thresholds(lib):
    """The smallest workspace fr_decode_attn accepts, against the 9 MiB scratch
    of fr_decode_attn_noalloc: the thresholds include/fr_kernels.h states
    (host-side sizing only; without a GPU a fitting call stops at the device
    query, FR_ERR_CUDA, and one that does not fit at FR_ERR_WORKSPACE)."""
    from gqa_kv_head_gb300._abi import FrAttnPlan
    plan = FrAttnPlan()

    def fits(n_tok, n_head, hd, n_kv=4096):
        st = lib.fr_decode_attn_plan(n_tok, n_head, hd, n_kv, 1, 9 << 20, None, ctypes.byref(plan))
        assert st in (0, 3, 4), st
        return st != 3
    assert fits(16, 16, 256) and not fits(16, 17, 256)          # M 256 | 272
    assert not fits(16, 32, 256) and fits(80, 8, 256)           # M 512 | 640
    assert fits(755, 8, 256) and not fits(756, 8, 256)          # M 6040 | 6048
    assert fits(1520, 8, 128) and not fits(1521, 8, 128)        # M 12160 | 12168
    assert fits(3008, 8, 64) and not fits(3009, 8, 64)          # M 24064 | 24072
    assert fits(1, 8, 256, 65536) and fits(4, 8, 128, 65536)    # keys-on-M plans need only the Q slot


def test_trace_build_compiles_and_exports_the_same_abi():
    """The timeline-instrumented variant (FR_TRACE, used by
    `python -m gqa_kv_head_gb300.trace`) builds into its own directory,
    loads without a GPU and exports every declared function; the library
    itself stays uninstrumented."""
    from gqa_kv_head_gb300 import build
    path = build.build(trace=True)
    assert os.path.realpath(path) != os.path.realpath(build.library_path())
    tr = ctypes.CDLL(path)
    for n in sorted(_declared()):
        assert hasattr(tr, n), f"{n} missing from the FR_TRACE build"
