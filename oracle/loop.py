"""One step of the batched multi-layer denoising loop, fp64 -- TEST
INFRASTRUCTURE ONLY (see the package docstring).

The step chains the attention layer and the sampler the way a caller does
([AIT] §섹션별 상세, the sampling-loop paragraph; glossary, self-conditioning):

1. canvas input: v = E[tokens] + soft_emb of the previous step (0 at step 0);
   the attention layers read bf16(v);
2. for each layer: out = canvas_attention(bf16(x)), stored in bf16; the
   residual stream x (fp64 here, fp32 on the device) gains out W_o^T;
3. tied LM head: logits = bf16(x) E^T, stored in bf16;
4. the sampler with the step's seed and index; committed positions of earlier
   steps are frozen with their tokens.

Storage model: every tensor the device keeps in bf16 is rounded to bf16 here
at the same point (``oracle.attention`` rounds its own internals); all other
arithmetic is exact fp64.  The output projection W_o, the residual add and
the tied head are the loop's glue: the pages do not print them, and no MLP /
MoE block or final norm is applied (they need trained weights).
"""
from __future__ import annotations

from typing import Iterable, Optional

import numpy as np

from .attention import canvas_attention
from .numerics import bf16_round, gelu_tanh
from .sampler import canvas_sample


def selfcond_mlp(soft: np.ndarray, W1: np.ndarray, W2: np.ndarray) -> np.ndarray:
    """The self-conditioning MLP on the previous step's soft embedding ([AIT]
    glossary, self-conditioning: P.E passes through a small MLP, which maps
    zero to zero, before it is added to the canvas input):
    W2 bf16(gelu(W1 bf16(soft))), no biases, the rounding points of the path
    (bf16 GEMM operands) mirrored; W1 [H, D], W2 [D, H] exact values."""
    h = bf16_round(soft) @ np.asarray(W1, np.float64).T
    return bf16_round(gelu_tanh(h)) @ np.asarray(W2, np.float64).T


def dense_cache(rows: np.ndarray, lo: int, prefix: int) -> np.ndarray:
    """Cache rows [B, Hkv, prefix - lo, d] at positions lo.. -> [B, Hkv, prefix, d]
    indexed by absolute position (NaN below lo: never visible)."""
    B, Hkv, n, d = rows.shape
    out = np.full((B, Hkv, prefix, d), np.nan)
    out[:, :, lo:lo + n, :] = rows
    return out


def loop_step(layers, E: np.ndarray, tokens: np.ndarray, soft_prev: Optional[np.ndarray], step: int, B: int,
              C: int, seed: int, bound: float, frozen=None, frozen_tokens=None,
              sample_rows: Optional[Iterable[int]] = None, slack_eps: Optional[float] = None,
              selfcond=None):
    """One step.  ``layers``: dicts of exact fp64 layer inputs (keys W_q, W_k,
    W_v, W_o, gamma_q, gamma_k, freq, eps, Hq, Hkv, d, layer, window,
    cache_k, cache_v [dense by position], prefix).  Returns a dict with the
    residual stream before every layer and after the last (``xs``, fp64
    [rows, D]), the per-layer attention outputs (``attn``: bf16-rounded as
    stored, ``attn_exact``: before that rounding; [B, C, Hq*d]) and, with
    ``slack_eps``, their rounding slack; the bf16 logits (all rows, or only
    ``sample_rows`` -- NaN elsewhere) and the sampler outputs of those rows
    (soft_emb for them).  ``selfcond`` = (W1, W2): the previous soft
    embedding enters through ``selfcond_mlp`` (default: as it is)."""
    rows = B * C
    D = E.shape[1]
    sel = np.arange(rows) if sample_rows is None else np.asarray(sorted(set(sample_rows)), np.int64)
    v = E[np.asarray(tokens, np.int64)]
    if soft_prev is not None:
        v = v + (soft_prev if selfcond is None else selfcond_mlp(soft_prev, *selfcond))
    x = v.copy()
    xs, outs, exact, slacks = [x.copy()], [], [], []
    for L in layers:
        xb = bf16_round(x).reshape(B, C, D)
        res = canvas_attention(xb, L["W_q"], L["W_k"], L["W_v"], L["Hq"], L["Hkv"], L["d"], L["gamma_q"],
                               L["gamma_k"], L["eps"], L["freq"], L["layer"], L["cache_k"], L["cache_v"],
                               np.full(B, L["prefix"]), L["window"], storage="bf16", slack_eps=slack_eps)
        out = res[0]
        if slack_eps is not None:
            slacks.append(res[2])
        exact.append(out)
        ob = bf16_round(out).reshape(rows, -1)
        outs.append(ob.reshape(B, C, -1))
        x = x + ob @ L["W_o"].T
        xs.append(x.copy())
    xb = bf16_round(x)
    logits = np.full((rows, E.shape[0]), np.nan)
    logits[sel] = bf16_round(xb[sel] @ E.T)
    # the sampler of the selected rows (each keeps its global row index for
    # the renoise key)
    fr = None if frozen is None else np.asarray(frozen)[sel]
    ft = None if frozen_tokens is None else np.asarray(frozen_tokens)[sel]
    res = _sample_rows(logits[sel], E, bound, seed, step, C, fr, ft, sel)
    return dict(attn=outs, attn_exact=exact, slack=slacks, logits=logits, xs=xs, x=xb, rows=sel, **res)


def _sample_rows(logits, E, bound, seed, step, C, frozen, frozen_tokens, rows):
    """The sampler on a subset of rows, each keeping its global row index (the
    renoise key uses it)."""
    from .splitmix import renoise_token
    full = canvas_sample(logits, E, bound, seed, step, canvas_len=C, frozen=frozen, frozen_tokens=frozen_tokens,
                         probs_storage="bf16")
    # canvas_sample numbers rows 0..n-1; re-key the renoised ones by their global row
    tok = full["tokens"].copy()
    V = logits.shape[1]
    for k, r in enumerate(rows):
        fr = frozen is not None and bool(frozen[k])
        if not fr and not full["commit_mask"][k]:
            tok[k] = renoise_token(seed, step, int(r), V)
    full["tokens"] = tok
    return full
