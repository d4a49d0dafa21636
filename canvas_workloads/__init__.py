"""Seeded synthetic inputs for the canvas refinement step.

This module is the one piece shared by the fp64 oracle, the tests and the
benchmark.  It draws random numbers and lays them out; it holds none of the
method's arithmetic (no norm, no rotation, no softmax, no sampling rule).
The only numeric transforms here are the quantisation of the random draws to
the storage dtype (fp32 -> bf16 bit patterns, round to nearest even) and the
RoPE frequency table that a model configuration hands to the attention call as
data.

Shapes and distributions follow the five workloads of the canvas step:

* ``tiny``    -- 1 sequence, canvas 16, prefix 32, d_model 128, 2 query heads
  sharing 1 KV head, head_dim 64, fp32, vocab 512 (seed 0).
* ``sliding`` -- batch 1, canvas 256, prefix 4096, d_model 2816, 16/8 heads,
  head_dim 256, window 1024, bf16 (seed 2).
* ``global``  -- batch 1, canvas 256, prefix 32768, d_model 2816, 16/2 heads,
  head_dim 512, shared W_v = W_k, partial RoPE (theta 1e6, first 25% of the
  frequencies), bf16 (seed 3).
* ``sampler`` -- 256 positions x vocab 262144 bf16 logits, half peaked rows,
  half flat rows, E[262144 x 2816] ~ N(0, 0.02^2) (seed 7).
* ``loop``    -- 4 canvases x 256, 5 sliding + 1 global layers, prefix swept
  over 1K/8K/32K/128K, 48 steps (seed 11); a small loop of the same
  structure for step-by-step parity.
"""
from __future__ import annotations

from dataclasses import dataclass, field, replace
from typing import Optional

import numpy as np

# --------------------------------------------------------------------------
# storage helpers (quantisation of random draws; not part of the method)
# --------------------------------------------------------------------------


def f32_to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """fp32 array -> uint16 bf16 bit patterns, round to nearest, ties to even."""
    u = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32).astype(np.uint64)
    lsb = (u >> np.uint64(16)) & np.uint64(1)
    u = (u + np.uint64(0x7FFF) + lsb) >> np.uint64(16)
    return u.astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    """uint16 bf16 bit patterns -> exact fp32 values."""
    return (np.ascontiguousarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def as_f64(a: np.ndarray, dtype: str) -> np.ndarray:
    """Exact fp64 values of a stored array (bf16 bits or fp32)."""
    if dtype == "bf16":
        return bf16_bits_to_f32(a).astype(np.float64)
    return np.asarray(a, dtype=np.float32).astype(np.float64)


def _store(a32: np.ndarray, dtype: str) -> np.ndarray:
    return f32_to_bf16_bits(a32) if dtype == "bf16" else np.ascontiguousarray(a32, dtype=np.float32)


def rope_frequencies(d: int, theta: float, rotary_fraction: float = 1.0) -> np.ndarray:
    """RoPE frequency table handed to the attention call (fp32, length d/2).

    freq[t] = theta**(-2t/d) for t < floor(rotary_fraction * d/2), else 0.
    """
    half = d // 2
    t = np.arange(half, dtype=np.float64)
    f = theta ** (-2.0 * t / d)
    n_rot = int(np.floor(rotary_fraction * half + 1e-9))
    f[n_rot:] = 0.0
    return f.astype(np.float32)


# --------------------------------------------------------------------------
# attention workloads
# --------------------------------------------------------------------------


@dataclass(frozen=True)
class AttnConfig:
    name: str
    B: int
    C: int
    prefix: tuple          # committed prefix length per sequence
    D: int
    Hq: int
    Hkv: int
    d: int
    layer: str             # "sliding" (cache holds final K, V) or "global" (raw shared r)
    window: int            # prefix tokens visible back from each canvas position; <=0: all
    theta: float
    rotary_fraction: float
    dtype: str             # "fp32" or "bf16"
    seed: int
    gamma_q: Optional[float] = None   # fixed constant, or None: drawn U[0.5, 2]
    gamma_k: Optional[float] = None
    eps: float = 1e-6
    page_tokens: int = 64
    cache_std: float = 1.0

    @property
    def max_prefix(self) -> int:
        return int(max(self.prefix))

    @property
    def G(self) -> int:
        return self.Hq // self.Hkv


TINY = AttnConfig("tiny", B=1, C=16, prefix=(32,), D=128, Hq=2, Hkv=1, d=64, layer="sliding",
                  window=0, theta=1e4, rotary_fraction=1.0, dtype="fp32", seed=0,
                  gamma_q=1.3, gamma_k=0.8, page_tokens=16)
SLIDING = AttnConfig("sliding", B=1, C=256, prefix=(4096,), D=2816, Hq=16, Hkv=8, d=256,
                     layer="sliding", window=1024, theta=1e4, rotary_fraction=1.0,
                     dtype="bf16", seed=2)
GLOBAL = AttnConfig("global", B=1, C=256, prefix=(32768,), D=2816, Hq=16, Hkv=2, d=512,
                    layer="global", window=0, theta=1e6, rotary_fraction=0.25,
                    dtype="bf16", seed=3)


@dataclass
class AttnInputs:
    cfg: AttnConfig
    x: np.ndarray          # [B, C, D]
    W_q: np.ndarray        # [Hq*d, D]
    W_k: np.ndarray        # [Hkv*d, D]
    W_v: Optional[np.ndarray]  # [Hkv*d, D] or None (global: shared with W_k)
    gamma_q: np.ndarray    # fp32 [d]
    gamma_k: np.ndarray    # fp32 [d]
    freq: np.ndarray       # fp32 [d/2]
    cache_k: np.ndarray    # [B, Hkv, max_prefix, d]  (global: raw shared r)
    cache_v: Optional[np.ndarray]  # [B, Hkv, max_prefix, d] or None (global)
    prefix_len: np.ndarray  # int32 [B]


def make_attention_inputs(cfg: AttnConfig) -> AttnInputs:
    """Seeded draws for one attention call (dense caches, storage dtype)."""
    rng = np.random.default_rng(cfg.seed)
    dt = cfg.dtype
    wstd = 1.0 / np.sqrt(cfg.D)
    x = rng.standard_normal((cfg.B, cfg.C, cfg.D), dtype=np.float32)
    W_q = rng.standard_normal((cfg.Hq * cfg.d, cfg.D), dtype=np.float32) * np.float32(wstd)
    W_k = rng.standard_normal((cfg.Hkv * cfg.d, cfg.D), dtype=np.float32) * np.float32(wstd)
    W_v = None
    if cfg.layer == "sliding":
        W_v = rng.standard_normal((cfg.Hkv * cfg.d, cfg.D), dtype=np.float32) * np.float32(wstd)
    gq = cfg.gamma_q if cfg.gamma_q is not None else float(rng.uniform(0.5, 2.0))
    gk = cfg.gamma_k if cfg.gamma_k is not None else float(rng.uniform(0.5, 2.0))
    shape = (cfg.B, cfg.Hkv, cfg.max_prefix, cfg.d)
    ck = rng.standard_normal(shape, dtype=np.float32) * np.float32(cfg.cache_std)
    cv = None
    if cfg.layer == "sliding":
        cv = rng.standard_normal(shape, dtype=np.float32) * np.float32(cfg.cache_std)
    return AttnInputs(
        cfg=cfg,
        x=_store(x, dt),
        W_q=_store(W_q, dt),
        W_k=_store(W_k, dt),
        W_v=None if W_v is None else _store(W_v, dt),
        gamma_q=np.full(cfg.d, gq, dtype=np.float32),
        gamma_k=np.full(cfg.d, gk, dtype=np.float32),
        freq=rope_frequencies(cfg.d, cfg.theta, cfg.rotary_fraction),
        cache_k=_store(ck, dt),
        cache_v=None if cv is None else _store(cv, dt),
        prefix_len=np.asarray(cfg.prefix, dtype=np.int32),
    )


def page_layout(cfg: AttnConfig, seed: int = 1234, spare_pages: int = 3):
    """A shuffled block table for a paged cache.

    Returns (block_table [B, max_pages] int32, num_pages).  Physical pages are
    a seeded permutation, with a few spare pages so that ids are not dense.
    Entries past a sequence's last page are -1.
    """
    pt = cfg.page_tokens
    max_pages = (cfg.max_prefix + pt - 1) // pt
    used = [(int(p) + pt - 1) // pt for p in cfg.prefix]
    num_pages = sum(used) + spare_pages
    perm = np.random.default_rng(seed).permutation(num_pages)
    table = np.full((cfg.B, max(max_pages, 1)), -1, dtype=np.int32)
    k = 0
    for b in range(cfg.B):
        for i in range(used[b]):
            table[b, i] = perm[k]
            k += 1
    return table, num_pages


def scatter_pages(dense: np.ndarray, table: np.ndarray, num_pages: int, page_tokens: int,
                  fill: Optional[int] = None) -> np.ndarray:
    """Dense cache [B, Hkv, P, d] -> page pool [num_pages, Hkv, page_tokens, d].

    Pool slots that hold no token are filled with ``fill`` (a bit pattern /
    value of the storage dtype; default: NaN), so that a kernel that reads an
    unused slot without masking it shows up in the results.
    """
    B, Hkv, P, d = dense.shape
    if fill is None:
        fill = 0x7FC0 if dense.dtype == np.uint16 else np.float32(np.nan)
    pool = np.full((num_pages, Hkv, page_tokens, d), fill, dtype=dense.dtype)
    for b in range(B):
        for lp in range(table.shape[1]):
            pid = table[b, lp]
            if pid < 0:
                continue
            lo = lp * page_tokens
            hi = min(P, lo + page_tokens)
            if lo >= hi:
                continue
            pool[pid, :, : hi - lo, :] = dense[b, :, lo:hi, :]
    return pool


# --------------------------------------------------------------------------
# sampler workloads
# --------------------------------------------------------------------------


@dataclass(frozen=True)
class SampleConfig:
    name: str
    rows: int
    C: int                 # canvas length (rows = B*C)
    V: int
    D: int
    dtype: str
    seed: int
    step: int
    bound: float
    logits: str            # "normal" or "mixture"
    logit_std: float = 1.0
    peak: float = 12.0
    gen_temperature: float = 1.0
    E_std: float = 1.0


TINY_SAMPLE = SampleConfig("tiny", rows=16, C=16, V=512, D=128, dtype="fp32", seed=0, step=0,
                           bound=0.5, logits="normal", logit_std=2.0, E_std=1.0)
FULL_SAMPLE = SampleConfig("sampler", rows=256, C=256, V=262144, D=2816, dtype="bf16", seed=7,
                           step=0, bound=0.3, logits="mixture", peak=12.0, gen_temperature=0.5,
                           E_std=0.02)


@dataclass
class SampleInputs:
    cfg: SampleConfig
    logits: np.ndarray     # [rows, V]
    E: np.ndarray          # [V, D]
    peaked: np.ndarray     # bool [rows] (mixture workloads; all False otherwise)


def make_logits(cfg: SampleConfig, rng) -> tuple:
    rows, V = cfg.rows, cfg.V
    z = rng.standard_normal((rows, V), dtype=np.float32)
    peaked = np.zeros(rows, dtype=bool)
    if cfg.logits == "normal":
        z *= np.float32(cfg.logit_std)
    elif cfg.logits == "mixture":
        peaked = rng.random(rows) < 0.5
        hot = rng.integers(0, V, size=rows)
        for r in np.nonzero(peaked)[0]:
            z[r, hot[r]] += np.float32(cfg.peak)
        z *= np.float32(1.0 / cfg.gen_temperature)
    else:
        raise ValueError(cfg.logits)
    return z, peaked


def make_sample_inputs(cfg: SampleConfig, with_E: bool = True) -> SampleInputs:
    rng = np.random.default_rng(cfg.seed)
    z, peaked = make_logits(cfg, rng)
    E = None
    if with_E:
        E = rng.standard_normal((cfg.V, cfg.D), dtype=np.float32) * np.float32(cfg.E_std)
        E = _store(E, cfg.dtype)
    return SampleInputs(cfg=cfg, logits=_store(z, cfg.dtype), E=E, peaked=peaked)


# --------------------------------------------------------------------------
# multi-layer loop workload
# --------------------------------------------------------------------------


@dataclass(frozen=True)
class LoopConfig:
    """A batch of canvases denoised for ``steps`` steps through a stack of
    ``n_sliding`` sliding-window layers (shapes of ``sliding``) followed by
    ``n_global`` global layers (shapes of ``global_``), a tied LM head and the
    sampler.  Each layer draws its own weights, QK-norm constants and cache."""
    name: str
    B: int
    C: int
    prefix: int
    steps: int
    V: int
    D: int
    seed: int
    sliding: AttnConfig
    global_: AttnConfig
    n_sliding: int = 5
    n_global: int = 1
    bound: float = 0.3
    E_std: float = 0.02
    selfcond_hidden: int = 0   # > 0: the self-conditioning MLP's hidden width (0: P.E enters as it is)

    def layer_cfgs(self):
        out = []
        for k in range(self.n_sliding + self.n_global):
            t = self.sliding if k < self.n_sliding else self.global_
            out.append(replace(t, name=f"{self.name}-L{k}", B=self.B, C=self.C, prefix=(self.prefix,) * self.B,
                               D=self.D, seed=self.seed * 1000 + k))
        return out


def loop_config(prefix: int, B: int = 4, steps: int = 48, selfcond_hidden: int = 0) -> LoopConfig:
    """The batched loop: 4 canvases of 256, 5 sliding layers (the sliding-layer
    shapes) and 1 global layer (the global-layer shapes), vocab 262144."""
    return LoopConfig(f"loop_p{prefix}", B=B, C=256, prefix=prefix, steps=steps, V=262144, D=2816, seed=11,
                      sliding=SLIDING, global_=GLOBAL, selfcond_hidden=selfcond_hidden)


def mini_loop_config(steps: int = 4, selfcond_hidden: int = 0) -> LoopConfig:
    """A small loop of the same structure for step-by-step parity."""
    sl = AttnConfig("mini-sliding", B=2, C=32, prefix=(160,), D=256, Hq=4, Hkv=2, d=64, layer="sliding",
                    window=48, theta=1e4, rotary_fraction=1.0, dtype="bf16", seed=0)
    gl = AttnConfig("mini-global", B=2, C=32, prefix=(160,), D=256, Hq=4, Hkv=1, d=128, layer="global",
                    window=0, theta=1e6, rotary_fraction=0.25, dtype="bf16", seed=0)
    return LoopConfig("mini_loop", B=2, C=32, prefix=160, steps=steps, V=4096, D=256, seed=21, sliding=sl,
                      global_=gl, bound=0.3, E_std=0.3, selfcond_hidden=selfcond_hidden)


@dataclass
class LoopLayer:
    cfg: AttnConfig
    W_q: np.ndarray
    W_k: np.ndarray
    W_v: Optional[np.ndarray]
    W_o: np.ndarray          # [D, Hq*d]
    gamma_q: np.ndarray
    gamma_k: np.ndarray
    freq: np.ndarray
    cache_lo: int            # first cached position (64-aligned); earlier pages are not allocated
    cache_k: np.ndarray      # [B, Hkv, prefix - cache_lo, d]
    cache_v: Optional[np.ndarray]


@dataclass
class LoopInputs:
    cfg: LoopConfig
    layers: list
    E: np.ndarray            # [V, D]
    tokens0: np.ndarray      # int32 [B*C]
    sc_W1: Optional[np.ndarray] = None   # [H, D] self-conditioning MLP (bf16 bits), or None
    sc_W2: Optional[np.ndarray] = None   # [D, H]


def make_loop_inputs(cfg: LoopConfig) -> LoopInputs:
    """Seeded draws for the loop: per layer W ~ N(0, 1/D), W_o ~ N(0, 1/(Hq d)),
    constant QK-norm vectors drawn U[0.5, 2], cache rows ~ N(0, 1) (sliding
    layers keep only the pages a canvas row can see); E ~ N(0, E_std^2);
    initial tokens uniform."""
    layers = []
    for lc in cfg.layer_cfgs():
        rng = np.random.default_rng(lc.seed)
        wstd = np.float32(1.0 / np.sqrt(lc.D))
        W_q = rng.standard_normal((lc.Hq * lc.d, lc.D), dtype=np.float32) * wstd
        W_k = rng.standard_normal((lc.Hkv * lc.d, lc.D), dtype=np.float32) * wstd
        W_v = None
        if lc.layer == "sliding":
            W_v = rng.standard_normal((lc.Hkv * lc.d, lc.D), dtype=np.float32) * wstd
        W_o = rng.standard_normal((lc.D, lc.Hq * lc.d), dtype=np.float32) * np.float32(1.0 / np.sqrt(lc.Hq * lc.d))
        gq, gk = float(rng.uniform(0.5, 2.0)), float(rng.uniform(0.5, 2.0))
        P = cfg.prefix
        lo = 0
        if lc.layer == "sliding" and lc.window > 0:
            lo = max(0, P - lc.window) // 64 * 64
        shape = (cfg.B, lc.Hkv, P - lo, lc.d)
        ck = rng.standard_normal(shape, dtype=np.float32)
        cv = rng.standard_normal(shape, dtype=np.float32) if lc.layer == "sliding" else None
        layers.append(LoopLayer(cfg=lc, W_q=_store(W_q, "bf16"), W_k=_store(W_k, "bf16"),
                                W_v=None if W_v is None else _store(W_v, "bf16"), W_o=_store(W_o, "bf16"),
                                gamma_q=np.full(lc.d, gq, np.float32), gamma_k=np.full(lc.d, gk, np.float32),
                                freq=rope_frequencies(lc.d, lc.theta, lc.rotary_fraction), cache_lo=lo,
                                cache_k=_store(ck, "bf16"), cache_v=None if cv is None else _store(cv, "bf16")))
    rng = np.random.default_rng(cfg.seed)
    E = rng.standard_normal((cfg.V, cfg.D), dtype=np.float32) * np.float32(cfg.E_std)
    tokens0 = rng.integers(0, cfg.V, size=cfg.B * cfg.C).astype(np.int32)
    W1 = W2 = None
    if cfg.selfcond_hidden > 0:
        # a separate stream, so the other draws do not depend on it
        r2 = np.random.default_rng(cfg.seed + 7919)
        H = cfg.selfcond_hidden
        W1 = _store(r2.standard_normal((H, cfg.D), dtype=np.float32) * np.float32(1.0 / np.sqrt(cfg.D)), "bf16")
        W2 = _store(r2.standard_normal((cfg.D, H), dtype=np.float32) * np.float32(1.0 / np.sqrt(H)), "bf16")
    return LoopInputs(cfg=cfg, layers=layers, E=_store(E, "bf16"), tokens0=tokens0, sc_W1=W1, sc_W2=W2)


def page_layout_range(B: int, lo: int, hi: int, page_tokens: int, seed: int = 1234, spare_pages: int = 2):
    """Block table for caches that hold positions [lo, hi) of each sequence
    (lo a multiple of page_tokens): logical pages below lo are -1, the others
    a seeded permutation of physical pages.  Returns (table, num_pages)."""
    first = lo // page_tokens
    last = (hi + page_tokens - 1) // page_tokens
    per = last - first
    num_pages = B * per + spare_pages
    perm = np.random.default_rng(seed).permutation(num_pages)
    table = np.full((B, max(last, 1)), -1, dtype=np.int32)
    k = 0
    for b in range(B):
        for lp in range(first, last):
            table[b, lp] = perm[k]
            k += 1
    return table, num_pages


def scatter_pages_range(rows: np.ndarray, lo: int, table: np.ndarray, num_pages: int, page_tokens: int,
                        fill: Optional[int] = None) -> np.ndarray:
    """Rows [B, Hkv, n, d] holding positions lo .. lo+n-1 -> page pool."""
    B, Hkv, n, d = rows.shape
    if fill is None:
        fill = 0x7FC0 if rows.dtype == np.uint16 else np.float32(np.nan)
    pool = np.full((num_pages, Hkv, page_tokens, d), fill, dtype=rows.dtype)
    for b in range(B):
        for lp in range(table.shape[1]):
            pid = table[b, lp]
            if pid < 0:
                continue
            p0 = lp * page_tokens
            a, z = max(p0, lo), min(p0 + page_tokens, lo + n)
            if a >= z:
                continue
            pool[pid, :, a - p0:z - p0, :] = rows[b, :, a - lo:z - lo, :]
    return pool


__all__ = [
    "AttnConfig", "AttnInputs", "SampleConfig", "SampleInputs", "LoopConfig",
    "TINY", "SLIDING", "GLOBAL", "TINY_SAMPLE", "FULL_SAMPLE",
    "make_attention_inputs", "make_sample_inputs", "make_logits", "page_layout",
    "scatter_pages", "rope_frequencies", "f32_to_bf16_bits", "bf16_bits_to_f32",
    "as_f64", "loop_config", "mini_loop_config", "make_loop_inputs", "LoopInputs", "LoopLayer",
    "page_layout_range", "scatter_pages_range", "replace",
]
