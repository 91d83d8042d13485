"""The sweep workload in full: n_head 8 over one KV head, hd in {128, 256},
n_tok in {1, 2, 4, 8, 16}, n_kv in {256, 1024, 4096, 16384, 65536}, causal
mask, NEOX RoPE base 10000, 20 seeds per point: 1000 (point, seed) cases,
each compared element by element over its whole output with the fp64 oracle
(max-abs <= 2e-3, rel-L2 <= 1e-3), through the C ABI, in the launch
configuration bench.py times (the fused call with library-chosen plans).

FlashRT PR #185, commit "FLASH_ATTN_EXT with q_tokens <= 16 over a single
padded f16 KV head": the decode shapes of this path."""
import numpy as np
import pytest
import torch

from gen import SWEEP_HD, SWEEP_NKV, SWEEP_NTOK, make_workload
import fr_harness
from fr_harness import assert_close, oracle_out, run_fused, to_device

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("seed", range(20))
def test_sweep_every_point(seed):
    for hd in SWEEP_HD:
        for n_kv in SWEEP_NKV:
            d_kv = None
            for n_tok in SWEEP_NTOK:
                w = make_workload(f"sweep:{hd}:{n_tok}:{n_kv}", seed=seed)
                if d_kv is None:                  # K/V depend on (hd, n_kv, seed) only
                    d_kv = to_device(w)
                d = dict(to_device_q(w), k=d_kv["k"], v=d_kv["v"])
                out = run_fused(w, d)
                torch.cuda.synchronize()
                got = out.reshape(w.M, w.hd).cpu().numpy().astype(np.float64)
                assert_close(got, oracle_out(w), f"{w.name} seed {seed}")
            del d_kv
            fr_harness._kv_cached.cache_clear()


def to_device_q(w, dev="cuda"):
    """Q, positions and mask of workload w on the device (K/V passed separately)."""
    m = w.mask()
    mask = None
    if m is not None:
        stride = ((w.n_kv + 7) // 8) * 8
        buf = torch.zeros((w.n_tok, stride), dtype=torch.float16, device=dev)
        buf[:, :w.n_kv] = torch.from_numpy(m)
        mask = buf[:, :w.n_kv]
    return {"q": torch.from_numpy(w.q().reshape(w.n_tok, -1)).to(dev),
            "pos": torch.from_numpy(w.pos()).to(dev), "mask": mask}
