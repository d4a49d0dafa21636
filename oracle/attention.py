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
and every other step is exact fp64.  The page's rms() and rotate() snippets
cast their results back to the input dtype, so a normed, rotated row is a
stored row.  The rounded tensors are:

* the canvas query after norm and rotation;
* the canvas projections that become key / value rows: on sliding layers the
  canvas key after norm and rotation and the canvas value x W_v^T; on global
  layers the canvas's raw shared projection r = x W_k^T (it joins the key set
  exactly like a cached row);
* on global layers the key of every row, rotate(rms(r, gamma_k)) at the row's
  own position.  The unit-RMS value variant keeps the stored row r and its
  exact row scalar (no further rounding).

``storage='fp64'`` applies no rounding anywhere (the pages' formulas as
written, evaluated exactly).

Rounding slack.  A stored bf16 value is a decision taken in floating point:
when the exact value lies within the path's own arithmetic error of a bf16
rounding midpoint, both neighbours are correct stored values, and attention
with its sharp softmax can turn one such flip into a visible change of the
output.  With ``slack_eps`` set, the oracle also returns, per output element,
a bound on how far the output can move under every combination of such
flips: an element x is ambiguous when |x - midpoint| <= slack_eps * (|x| +
|partner| + rms(row)) (partner: the other element of its rotation pair), and
the bound propagates the one-ulp alternatives exactly through the softmax:
with logit moves |delta_j| <= D_j and Zmax = sum_j p_j exp(D_j), every
probability ratio p'_j / p_j lies within [exp(-D_j) / Zmax, Zmax exp(D_j)],
so |o' - o| <= sum_j p_j (Zmax e^{D_j} - 1) |v_j - o| + sum_j p_j Zmax e^{D_j}
|dv_j|.
"""
from __future__ import annotations

from typing import Iterable, Optional

import numpy as np

from .numerics import bf16_round, rms, rotate


def _step(r: np.ndarray, direction: int) -> np.ndarray:
    """The next bf16 value from bf16 value r towards +inf (1) or -inf (-1)."""
    r = np.asarray(r, np.float64)
    out = np.empty_like(r)
    bits = _bf16_bits(r)
    # bf16 values are ordered like sign-magnitude integers
    pos = r > 0
    neg = r < 0
    zero = r == 0
    up = direction > 0
    nb = np.where(pos, bits + (1 if up else -1), np.where(neg, bits - (1 if up else -1), 0))
    out = _from_bits(nb)
    if zero.any():
        tiny = np.ldexp(1.0, -133)      # smallest positive bf16 subnormal
        out = np.where(zero, tiny if up else -tiny, out)
    return out


def _bf16_bits(r):
    f = np.asarray(r, np.float64).astype(np.float32)
    return (f.view(np.uint32) >> np.uint32(16)).astype(np.int64)


def _from_bits(b):
    u = (np.asarray(b, np.int64).astype(np.uint32) << np.uint32(16))
    return u.view(np.float32).astype(np.float64)


def rounding_flips(x: np.ndarray, partner: np.ndarray, eps: float):
    """Stored bf16 value of x and the signed change to the other neighbour
    where the rounding is ambiguous (0 elsewhere).

    Ambiguous: |x - midpoint(lo, hi)| <= eps * (|x| + |partner| + rms of the
    row), i.e. within the arithmetic error a path that computes x in fp32
    makes before rounding.
    """
    x = np.asarray(x, np.float64)
    stored = bf16_round(x)
    lo = np.where(stored > x, _step(stored, -1), stored)
    hi = np.where(stored > x, stored, _step(stored, +1))
    exact = (stored == x)
    mid = 0.5 * (lo + hi)
    row_rms = np.sqrt(np.mean(x * x, axis=-1, keepdims=True))
    tol = eps * (np.abs(x) + np.abs(partner) + row_rms)
    amb = (np.abs(x - mid) <= tol) & ~exact
    alt = np.where(stored == lo, hi, lo)
    delta = np.where(amb, alt - stored, 0.0)
    return stored, delta


def _pair_partner(x: np.ndarray) -> np.ndarray:
    """The other element of each split-half rotation pair (t <-> t + d/2)."""
    h = x.shape[-1] // 2
    return np.concatenate([x[..., h:], x[..., :h]], axis=-1)


def _store(x, storage, slack_eps, partner=None):
    """(stored value, flip delta or None) of a tensor the path keeps in bf16."""
    if storage != "bf16":
        return x, None
    if slack_eps is None:
        return bf16_round(x), None
    return rounding_flips(x, _pair_partner(x) if partner is None else partner, slack_eps)


def visible_prefix(P: int, i: int, window: int, layer: str) -> range:
    """Prefix key positions visible from canvas row i (absolute position P+i)."""
    if layer == "global" or window <= 0:
        return range(0, P)
    return range(max(0, P + i - window), P)


def _row_slack(q, dq, abs_keys_hi, abs_dkeys, vals, abs_dvals, p, o, scale):
    """Bound on |o' - o| for one query row under every combination of flips.

    q, dq [d]; for the row's n visible keys: abs_keys_hi = |k_j| + |dk_j|,
    abs_dkeys = |dk_j|, vals = v_j, abs_dvals = |dv_j| (all [n, d]); p [n]
    softmax weights; o [d].
    Logit move bound D_j = scale * (|dq| . (|k_j| + |dk_j|) + |q| . |dk_j|).
    """
    aq, adq = np.abs(q), np.abs(dq)
    D = abs(scale) * (abs_keys_hi @ adq + abs_dkeys @ aq)
    ed = np.exp(D)
    zmax = float(p @ ed)
    w = p * (zmax * ed - 1.0)
    return w @ np.abs(vals - o) + (p * zmax * ed) @ abs_dvals


def canvas_attention(x, W_q, W_k, W_v, Hq: int, Hkv: int, d: int, gamma_q, gamma_k,
                     eps: float, freq, layer: str, cache_k, cache_v, prefix_len, window: int,
                     scale: float = 1.0, v_unit_rms: bool = False, storage: str = "fp64",
                     rows: Optional[Iterable] = None, slack_eps: Optional[float] = None,
                     causal: bool = False, cache_dk=None, cache_dv=None):
    """Canvas attention for one layer: decode mode, or encode mode with
    ``causal`` ([AIT] §섹션별 상세, the decode / encode paragraph: encoding the
    committed tokens is causal, like a prefill -- canvas row i sees the
    canvas keys j <= i, and the committed prefix as in decode mode).

    Arguments are exact fp64 values (the stored inputs widened).  Shapes:
    x [B, C, D]; W_q [Hq*d, D]; W_k, W_v [Hkv*d, D] (W_v None on global
    layers); gamma_q, gamma_k [d]; freq [d/2]; cache_k (and cache_v on sliding
    layers) [B, Hkv, >=max(prefix_len), d]; prefix_len [B].

    Returns (out [B, C, Hq*d], lse [B, C, Hq]); lse is the natural-log
    normaliser of each softmax row.  ``rows`` optionally restricts the work to
    a list of (b, h, i) triples; the other entries are NaN.  With
    ``slack_eps`` (bf16 storage only) a third array [B, C, Hq*d] holds the
    rounding slack of every output element (module docstring);
    ``cache_dk`` / ``cache_dv`` (same shapes as the caches, or None) then give
    the flip of every cached element that was itself a rounding tie when it
    was stored (rows appended by ``kv_append``), 0 elsewhere.
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
    want_slack = slack_eps is not None and storage == "bf16"

    # 1-2: projections and head split: [B, H, C, d]
    def heads(z, H):
        return z.reshape(B, C, H, d).transpose(0, 2, 1, 3)

    q_raw = heads(x @ W_q.T, Hq)
    k_raw = heads(x @ W_k.T, Hkv)
    v_raw = k_raw if shared else heads(x @ np.asarray(W_v, np.float64).T, Hkv)

    out = np.full((B, C, Hq * d), np.nan)
    lse = np.full((B, C, Hq), np.nan)
    slack = np.full((B, C, Hq * d), np.nan) if want_slack else None
    wanted = None if rows is None else {(int(b), int(h), int(i)) for (b, h, i) in rows}
    sl_eps = slack_eps if want_slack else None

    def zeros_like(a):
        return np.zeros_like(a)

    for b in range(B):
        P = int(prefix_len[b])
        if wanted is not None and not any(w[0] == b for w in wanted):
            continue
        # 3-4: queries of this sequence, [Hq, C, d]
        q, dq = _store(rotate(rms(q_raw[b], gamma_q, eps), freq, P), storage, sl_eps)
        for hk in range(Hkv):
            if wanted is not None and not any(w[0] == b and w[1] // G == hk for w in wanted):
                continue
            # the key / value rows of this KV head: prefix then canvas
            if layer == "sliding":
                kp = np.asarray(cache_k[b, hk, :P], np.float64)
                vp = np.asarray(cache_v[b, hk, :P], np.float64)
                kc, dkc = _store(rotate(rms(k_raw[b, hk], gamma_k, eps), freq, P), storage, sl_eps)
                vc, dvc = _store(v_raw[b, hk], storage, sl_eps)
                dkp = zeros_like(kp) if cache_dk is None else np.abs(np.asarray(cache_dk[b, hk, :P], np.float64))
                dvp = zeros_like(vp) if cache_dv is None else np.abs(np.asarray(cache_dv[b, hk, :P], np.float64))
            else:
                rp = np.asarray(cache_k[b, hk, :P], np.float64)
                rc, drc = _store(k_raw[b, hk], storage, sl_eps)
                r = np.concatenate([rp, rc], axis=0)
                kk, dkk = _store(rotate(rms(r, gamma_k, eps), freq, 0), storage, sl_eps)
                kp, kc = kk[:P], kk[P:]
                if v_unit_rms:
                    # the row scalar sqrt(d) / (|r| + eps) is applied in fp32 to
                    # the softmax weight of the row; the value row stays r
                    vv = np.sqrt(d) * r / (np.sqrt(np.sum(r * r, -1, keepdims=True)) + eps)
                else:
                    vv = r
                vp, vc = vv[:P], vv[P:]
                if want_slack:
                    # a flip of a stored r element (a canvas row, or a cached
                    # row that was a tie when appended) moves that row's key
                    # (through rms and rotate: at most |gamma_k| s (|dr_t| +
                    # |dr_pair|)) and its value (dr itself, or its unit-RMS image)
                    drp = np.zeros_like(rp) if cache_dk is None else np.asarray(cache_dk[b, hk, :P], np.float64)
                    dr = np.abs(np.concatenate([drp, drc], axis=0))
                    nr = np.sqrt(np.sum(r * r, -1, keepdims=True))
                    s_row = np.sqrt(d) / (nr + eps)
                    prop = np.max(np.abs(gamma_k)) * s_row * (dr + _pair_partner(dr))
                    dkk = np.abs(dkk) + prop * 1.01
                    dvv = dr * (s_row * 1.01 if v_unit_rms else 1.0)
                    dkp, dkc = dkk[:P], dkk[P:]
                    dvp, dvc = dvv[:P], dvv[P:]
            # the keys of this head in position order, from the first prefix
            # position any canvas row sees (row 0's) to the end of the canvas:
            # a canvas row sees a range of prefix positions that ends at P,
            # followed by the whole canvas -- rows vis.start - lo.. of these
            lo = visible_prefix(P, 0, window, layer).start
            keys_all = np.concatenate([kp[lo:], kc], axis=0)
            vals_all = np.concatenate([vp[lo:], vc], axis=0)
            if want_slack:
                abs_dk_all = np.abs(np.concatenate([dkp[lo:], dkc], axis=0))
                abs_k_hi_all = np.abs(keys_all) + abs_dk_all
                abs_dv_all = np.abs(np.concatenate([dvp[lo:], dvc], axis=0))
            for g in range(G):
                h = hk * G + g
                for i in range(C):
                    if wanted is not None and (b, h, i) not in wanted:
                        continue
                    vis = visible_prefix(P, i, window, layer)
                    assert vis.stop == P and vis.start >= lo
                    j0 = vis.start - lo
                    # canvas keys 0 .. C-1 (decode) or 0 .. i (encode)
                    j1 = (P - lo) + (i + 1 if causal else C)
                    keys = keys_all[j0:j1]
                    vals = vals_all[j0:j1]
                    s = scale * (keys @ q[h, i])
                    m = np.max(s)
                    e = np.exp(s - m)
                    Z = np.sum(e)
                    o = (e / Z) @ vals
                    out[b, i, h * d:(h + 1) * d] = o
                    lse[b, i, h] = m + np.log(Z)
                    if want_slack:
                        slack[b, i, h * d:(h + 1) * d] = _row_slack(q[h, i], dq[h, i], abs_k_hi_all[j0:j1],
                                                                    abs_dk_all[j0:j1], vals, abs_dv_all[j0:j1],
                                                                    e / Z, o, scale)
    if want_slack:
        return out, lse, slack
    return out, lse


def kv_append(x, W_k, W_v, Hkv: int, d: int, gamma_k, eps: float, freq, layer: str, prefix_len,
              storage: str = "bf16", slack_eps: Optional[float] = None):
    """The cache rows a committed block adds ([AIT] §섹션별 상세, the decode /
    encode paragraph and the attention-block snippet; [AB] §블록 자동 회귀
    노이즈 제거 및 자체 수정: the denoised block is committed to the KV cache).

    Block row i of sequence b sits at position prefix_len[b] + i.  Sliding
    layers keep final keys and values: k = rotate(rms(x W_k^T, gamma_k)) at
    that position, v = x W_v^T.  Global layers keep the raw shared projection
    r = x W_k^T (its key is formed from it at attention time).  Each row is
    rounded to bf16 where it is stored (``storage='bf16'``).

    Returns (k_rows, v_rows or None) [B, Hkv, C, d]; with ``slack_eps`` also
    the flip deltas of the rows (0 where the rounding is not a tie).
    """
    x = np.asarray(x, np.float64)
    B, C, D = x.shape

    def heads(z):
        return z.reshape(B, C, Hkv, d).transpose(0, 2, 1, 3)

    k_raw = heads(x @ np.asarray(W_k, np.float64).T)
    sl = slack_eps if storage == "bf16" else None
    if layer == "global":
        kr, dk = _store(k_raw, storage, sl)
        return (kr, None, dk, None) if sl is not None else (kr, None)
    v_raw = heads(x @ np.asarray(W_v, np.float64).T)
    ks, dks, vs, dvs = [], [], [], []
    for b in range(B):
        P = int(prefix_len[b])
        kb, dkb = _store(rotate(rms(k_raw[b], gamma_k, eps), freq, P), storage, sl)
        vb, dvb = _store(v_raw[b], storage, sl)
        ks.append(kb)
        vs.append(vb)
        dks.append(dkb)
        dvs.append(dvb)
    k, v = np.stack(ks), np.stack(vs)
    if sl is not None:
        return k, v, np.stack(dks), np.stack(dvs)
    return k, v


def visible_pairs(C: int, P: int, window: int, layer: str) -> int:
    """Number of (query, key) pairs one head scores: sum over canvas rows of
    (visible prefix keys + C)."""
    return sum(len(visible_prefix(P, i, window, layer)) + C for i in range(C))
