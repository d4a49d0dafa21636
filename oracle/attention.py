"""The canvas attention layer (decode mode), fp64, explicit loops.

Test infrastructure only (see the package docstring).

What is computed, in the order of [AIT] §섹션별 상세 (the attention-block
snippet and the paragraph on decode / encode modes):

1. projections q = x W_q^T, k = x W_k^T, v = x W_v^T; on global
   (full-attention) layers W_v = W_k, so v is the raw k projection;
2. split into heads, 'l (n h) -> n l h';
3. q, k <- rms(q, gamma_q), rms(k, gamma_k)   (v is left as it is);
4. q, k <- rotate(q), rotate(k) at the canvas positions start = prefix_len;
5. decode-mode attention: every canvas position attends, bidirectionally, to
   the committed prefix held in the KV cache and to the whole canvas.  On
   sliding-window layers only the prefix tokens within ``window`` positions
   back are visible ([AIT] glossary, sliding-window attention; [TC] §아키텍처:
   window 1,024); on global layers the whole prefix is visible.

Readings where the pages are silent (each is listed in the design notes):

* softmax scale 1: with constant QK-norm vectors the logit already equals
  d_h * gamma_q * gamma_k * cos(theta) ([AIT] §섹션별 상세 and the scalar
  QK-norm glossary entry), which sets the layer's temperature;
* window: canvas position p = P + i sees prefix keys j with j >= p - window,
  plus every canvas key;
* GQA: query head h reads KV head floor(h / (Hq / Hkv));
* the sliding cache holds final keys (normed, rotated) and values; the global
  cache holds the raw shared projection r, whose key is rotate(rms(r)) at the
  key's own position and whose value is r itself;
* ``v_unit_rms`` (off by default): the prose of [AIT] mentions a unit-RMS rule
  for V on shared layers that the printed code does not apply; when set, the
  value of a global key is sqrt(d) * r / (||r|| + eps).

Storage model (``storage='bf16'``).  The path keeps some tensors in bf16
memory; there the value is rounded to bf16 once, at the point it is stored,
and every other step is exact fp64.  The rounded tensors are:

* the canvas query after norm and rotation (the page's rotate() casts its
  result to the input dtype);
* on sliding layers the canvas key after norm and rotation, and the canvas
  value;
* on global layers the canvas's raw shared projection r (it becomes part of
  the key set exactly like a cached row) and, for every key row, the rotation
  rotate(r) of the raw row.  Because rms multiplies a row by the scalar
  sqrt(d) / (||r|| + eps) and the per-layer QK-norm vector is constant
  ([AIT] glossary, scalar QK norm), rotate(rms(r, gamma_k)) equals
  gamma_k * sqrt(d) / (||r|| + eps) * rotate(r); the path stores rotate(r) in
  bf16 and applies the scalar to the score.  This mode requires a constant
  gamma_k on global layers.

``storage='fp64'`` applies no rounding anywhere (the pages' formulas as
written, evaluated exactly).
"""
from __future__ import annotations

from typing import Iterable, Optional

import numpy as np

from .numerics import bf16_round, rms, rotate


def _maybe_round(a, storage):
    return bf16_round(a) if storage == "bf16" else a


def _global_keys(r: np.ndarray, pos0: int, gamma_k: np.ndarray, freq, eps: float, storage: str):
    """Keys of raw shared rows r [L, d] sitting at positions pos0 .. pos0+L-1."""
    d = r.shape[-1]
    if storage == "bf16":
        g = np.asarray(gamma_k, np.float64)
        if not np.all(g == g[0]):
            raise ValueError("bf16 storage model on global layers needs a constant gamma_k")
        s = np.sqrt(d) / (np.sqrt(np.sum(r * r, axis=-1, keepdims=True)) + eps)
        return g[0] * s * bf16_round(rotate(r, freq, pos0))
    return rotate(rms(r, gamma_k, eps), freq, pos0)


def visible_prefix(P: int, i: int, window: int, layer: str) -> range:
    """Prefix key positions visible from canvas row i (absolute position P+i)."""
    if layer == "global" or window <= 0:
        return range(0, P)
    return range(max(0, P + i - window), P)


def canvas_attention(x, W_q, W_k, W_v, Hq: int, Hkv: int, d: int, gamma_q, gamma_k,
                     eps: float, freq, layer: str, cache_k, cache_v, prefix_len, window: int,
                     scale: float = 1.0, v_unit_rms: bool = False, storage: str = "fp64",
                     rows: Optional[Iterable] = None):
    """Decode-mode canvas attention for one layer.

    Arguments are exact fp64 values (the stored inputs widened).  Shapes:
    x [B, C, D]; W_q [Hq*d, D]; W_k, W_v [Hkv*d, D] (W_v None on global
    layers); gamma_q, gamma_k [d]; freq [d/2]; cache_k (and cache_v on sliding
    layers) [B, Hkv, >=max(prefix_len), d]; prefix_len [B].

    Returns (out [B, C, Hq*d], lse [B, C, Hq]); lse is the natural-log
    normaliser of each softmax row.  ``rows`` optionally restricts the work to
    a list of (b, h, i) triples; the other entries are NaN.
    """
    x = np.asarray(x, np.float64)
    B, C, D = x.shape
    G = Hq // Hkv
    W_q = np.asarray(W_q, np.float64)
    W_k = np.asarray(W_k, np.float64)
    shared = W_v is None
    if layer == "global" and not shared:
        raise ValueError("global layers share W_v = W_k")
    if v_unit_rms and layer != "global":
        raise ValueError("v_unit_rms applies to global layers only")

    # 1-2: projections and head split: [B, H, C, d]
    def heads(z, H):
        return z.reshape(B, C, H, d).transpose(0, 2, 1, 3)

    q_raw = heads(x @ W_q.T, Hq)
    k_raw = heads(x @ W_k.T, Hkv)
    v_raw = k_raw if shared else heads(x @ np.asarray(W_v, np.float64).T, Hkv)

    out = np.full((B, C, Hq * d), np.nan)
    lse = np.full((B, C, Hq), np.nan)
    wanted = None if rows is None else {(int(b), int(h), int(i)) for (b, h, i) in rows}

    for b in range(B):
        P = int(prefix_len[b])
        # 3-4: queries of this sequence, [Hq, C, d]
        q = rotate(rms(q_raw[b], gamma_q, eps), freq, P)
        q = _maybe_round(q, storage)
        for hk in range(Hkv):
            # the key / value rows of this KV head: prefix then canvas
            if layer == "sliding":
                kp = np.asarray(cache_k[b, hk, :P], np.float64)
                vp = np.asarray(cache_v[b, hk, :P], np.float64)
                kc = _maybe_round(rotate(rms(k_raw[b, hk], gamma_k, eps), freq, P), storage)
                vc = _maybe_round(v_raw[b, hk], storage)
            else:
                rp = np.asarray(cache_k[b, hk, :P], np.float64)
                rc = _maybe_round(k_raw[b, hk], storage)
                kp = _global_keys(rp, 0, gamma_k, freq, eps, storage)
                kc = _global_keys(rc, P, gamma_k, freq, eps, storage)
                if v_unit_rms:
                    vp = np.sqrt(d) * rp / (np.sqrt(np.sum(rp * rp, -1, keepdims=True)) + eps)
                    vc = np.sqrt(d) * rc / (np.sqrt(np.sum(rc * rc, -1, keepdims=True)) + eps)
                else:
                    vp, vc = rp, rc
            for g in range(G):
                h = hk * G + g
                for i in range(C):
                    if wanted is not None and (b, h, i) not in wanted:
                        continue
                    vis = visible_prefix(P, i, window, layer)
                    keys = np.concatenate([kp[vis.start:vis.stop], kc], axis=0)
                    vals = np.concatenate([vp[vis.start:vis.stop], vc], axis=0)
                    s = scale * (keys @ q[h, i])
                    m = np.max(s)
                    e = np.exp(s - m)
                    Z = np.sum(e)
                    out[b, i, h * d:(h + 1) * d] = (e / Z) @ vals
                    lse[b, i, h] = m + np.log(Z)
    return out, lse


def visible_pairs(C: int, P: int, window: int, layer: str) -> int:
    """Number of (query, key) pairs one head scores: sum over canvas rows of
    (visible prefix keys + C)."""
    return sum(len(visible_prefix(P, i, window, layer)) + C for i in range(C))
