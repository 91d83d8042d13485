"""Workload recipes: shapes, RoPE parameters, positions, masks and seeded tensors.

Shapes follow the decode windows the FlashRT ggml adapter targets (PR #185,
"FLASH_ATTN_EXT with q_tokens <= 16 over a single padded f16 KV head"): GQA
with n_head query heads sharing ONE f16 KV head, up to 16 query tokens.

Streams of the counter-based generator (gen.rng):
    1 = Q, 2 = K, 3 = V, 4 = random mask columns, 5 = K outliers, 6 = V outliers.

Tensors (numpy, logical layouts; the GPU harness may copy them into strided
device buffers):
    q    float32 [n_tok, n_head, hd]   N(0, 1) rounded to f32
    pos  int32   [n_tok]
    k, v float16 [n_kv, hd]            N(0, sigma) (x outlier_mult with prob.
                                       outlier_p), rounded to f16 once; rows
                                       >= n_kv_real are exact zeros (KV pad)
    mask float16 [n_tok, n_kv] or None additive: 0 = visible, -inf = excluded
"""
from dataclasses import dataclass, field, replace
import math
import numpy as np

from .rng import normal, uniform


@dataclass(frozen=True)
class RopeParams:
    """NEOX RoPE parameters with the YaRN terms, as ggml's rope_ext takes them.
    mode 0: angles exact modulo one turn; mode 1: ggml's fp32 angle evaluation.
    freq_factors: None, or n_dims/2 per-pair divisors of the angle (rope_ext's
    optional freq_factors input)."""
    n_dims: int
    freq_base: float = 10000.0
    freq_scale: float = 1.0
    ext_factor: float = 0.0
    attn_factor: float = 1.0
    beta_fast: float = 32.0
    beta_slow: float = 1.0
    n_ctx_orig: int = 4096
    mode: int = 0
    freq_factors: tuple = None


@dataclass
class Workload:
    name: str
    n_head: int
    n_tok: int
    hd: int
    n_kv: int
    rope: RopeParams
    positions: tuple
    mask_kind: str = "none"          # none | causal | random5
    n_kv_real: int = -1              # -1: equal to n_kv (no pad rows)
    kv_sigma: float = 1.0
    outlier_p: float = 0.0
    outlier_mult: float = 20.0
    seed: int = 0
    q_scale: float = -1.0            # -1: 1/sqrt(hd)
    kq_scale: float = 1.0
    _cache: dict = field(default_factory=dict, repr=False, compare=False)

    def __post_init__(self):
        if self.n_kv_real < 0:
            self.n_kv_real = self.n_kv
        if self.q_scale < 0:
            self.q_scale = 1.0 / math.sqrt(self.hd)

    @property
    def M(self):
        return self.n_head * self.n_tok

    # -- tensors ---------------------------------------------------------
    def q(self):
        if "q" not in self._cache:
            n = self.n_tok * self.n_head * self.hd
            self._cache["q"] = normal(self.seed, 1, n).astype(np.float32).reshape(
                self.n_tok, self.n_head, self.hd)
        return self._cache["q"]

    def pos(self):
        return np.asarray(self.positions, dtype=np.int32)

    def _kv(self, stream, outlier_stream):
        n = self.n_kv * self.hd
        x = normal(self.seed, stream, n, self.kv_sigma)
        if self.outlier_p > 0.0:
            u = uniform(self.seed, outlier_stream, n)
            x = np.where(u < self.outlier_p, x * self.outlier_mult, x)
        x = x.astype(np.float16).reshape(self.n_kv, self.hd)
        if self.n_kv_real < self.n_kv:
            x[self.n_kv_real:, :] = 0
        return x

    def k(self):
        if "k" not in self._cache:
            self._cache["k"] = self._kv(2, 5)
        return self._cache["k"]

    def v(self):
        if "v" not in self._cache:
            self._cache["v"] = self._kv(3, 6)
        return self._cache["v"]

    def mask(self):
        """Additive f16 mask [n_tok, n_kv] shared by all heads, or None."""
        if self.mask_kind == "none" and self.n_kv_real == self.n_kv:
            return None
        if "mask" in self._cache:
            return self._cache["mask"]
        m = np.zeros((self.n_tok, self.n_kv), dtype=np.float16)
        cols = np.arange(self.n_kv)
        pos = self.pos()
        for t in range(self.n_tok):
            if self.mask_kind == "causal":
                m[t, cols > pos[t]] = -np.inf
            elif self.mask_kind == "random5":
                n_off = int(math.floor(0.05 * self.n_kv))
                keys = uniform(self.seed, 4, self.n_kv, offset=t * self.n_kv)
                off = np.argsort(keys, kind="stable")[:n_off]
                m[t, off] = -np.inf
            elif self.mask_kind != "none":
                raise ValueError(self.mask_kind)
            m[t, self.n_kv_real:] = -np.inf
        self._cache["mask"] = m
        return m

    def with_(self, **kw):
        """A copy with fields replaced (and a fresh tensor cache)."""
        kw.setdefault("_cache", {})
        return replace(self, **kw)


def _tail_positions(n_kv_real, n_tok):
    """Query tokens are the last n_tok rows of the cache."""
    return tuple(range(n_kv_real - n_tok, n_kv_real))


def named_config(name, seed=0):
    """The five documented workloads (the sweep via sweep_config)."""
    if name == "tiny":
        return Workload("tiny", n_head=4, n_tok=1, hd=64, n_kv=128,
                        rope=RopeParams(n_dims=64, freq_base=10000.0),
                        positions=(128,), mask_kind="none", seed=seed)
    if name == "pi05":
        return Workload("pi05", n_head=8, n_tok=10, hd=256, n_kv=1024, n_kv_real=968,
                        rope=RopeParams(n_dims=256, freq_base=10000.0),
                        positions=_tail_positions(968, 10), mask_kind="causal",
                        kv_sigma=0.5, seed=seed)
    if name == "c3":
        return Workload("c3", n_head=8, n_tok=16, hd=256, n_kv=4096,
                        rope=RopeParams(n_dims=256, freq_base=10000.0),
                        positions=tuple(range(4096, 4112)), mask_kind="random5",
                        seed=seed)
    if name == "long_decode":
        return Workload("long_decode", n_head=32, n_tok=16, hd=128, n_kv=32768,
                        rope=RopeParams(n_dims=128, freq_base=1.0e6, freq_scale=1.0 / 8.0,
                                        ext_factor=1.0, attn_factor=1.0,
                                        beta_fast=32.0, beta_slow=1.0, n_ctx_orig=4096),
                        positions=_tail_positions(32768, 16), mask_kind="causal",
                        outlier_p=0.01, outlier_mult=20.0, seed=seed)
    if name == "pi05_prefill":
        # the prefix window: KV length = query count, pad-only (prefix-LM) mask
        return Workload("pi05_prefill", n_head=8, n_tok=968, hd=256, n_kv=1024, n_kv_real=968,
                        rope=RopeParams(n_dims=256, freq_base=10000.0),
                        positions=tuple(range(968)), mask_kind="none", kv_sigma=0.5, seed=seed)
    raise KeyError(name)


NAMED_CONFIGS = ("tiny", "pi05", "c3", "long_decode")
SWEEP_HD = (128, 256)
SWEEP_NTOK = (1, 2, 4, 8, 16)
SWEEP_NKV = (256, 1024, 4096, 16384, 65536)


def sweep_config(hd, n_tok, n_kv, seed=0):
    return Workload(f"sweep_hd{hd}_t{n_tok}_kv{n_kv}", n_head=8, n_tok=n_tok, hd=hd,
                    n_kv=n_kv, rope=RopeParams(n_dims=hd, freq_base=10000.0),
                    positions=_tail_positions(n_kv, n_tok), mask_kind="causal",
                    seed=seed)


def make_workload(name, seed=0, **overrides):
    """Named config (or 'sweep:hd:n_tok:n_kv') with optional field overrides."""
    if name.startswith("sweep:"):
        _, hd, nt, nkv = name.split(":")
        w = sweep_config(int(hd), int(nt), int(nkv), seed=seed)
    else:
        w = named_config(name, seed=seed)
    return w.with_(**overrides) if overrides else w
