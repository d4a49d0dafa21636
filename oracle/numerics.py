"""Numeric building blocks of the canvas attention layer, in fp64.

Test infrastructure only (see the package docstring).
"""
from __future__ import annotations

import numpy as np


def bf16_round(x) -> np.ndarray:
    """Round fp64 values to the nearest bf16 value (ties to even), kept in fp64.

    bf16 keeps 8 significant bits (7 stored + the implicit one).  Used only by
    the storage model: a tensor that the path keeps in bf16 memory is rounded
    once, where it is stored.  Normal range only (|x| in [2^-126, 2^127]);
    zeros pass through, and the workloads never leave that range.
    """
    x = np.asarray(x, dtype=np.float64)
    m, e = np.frexp(x)                 # x = m * 2**e, 0.5 <= |m| < 1
    m = np.rint(m * 256.0) / 256.0     # 8 significant bits, half-to-even
    return np.ldexp(m, e)


def rms(x: np.ndarray, w, eps: float) -> np.ndarray:
    """Scalar QK RMSNorm, [AIT] §섹션별 상세, the rms() snippet.

    rms(x, w) = w * x * sqrt(d) / (||x||_2 + eps), the norm taken over the
    last axis (length d).  The page evaluates the norm in fp32 and casts the
    result back to x's dtype; here everything is fp64 and rounding, if any, is
    applied by the caller (storage model).
    """
    x = np.asarray(x, dtype=np.float64)
    d = x.shape[-1]
    nrm = np.sqrt(np.sum(x * x, axis=-1, keepdims=True))
    return np.asarray(w, dtype=np.float64) * x * np.sqrt(d) / (nrm + eps)


def rope_frequencies(d: int, theta: float, rotary_fraction: float = 1.0) -> np.ndarray:
    """RoPE spectrum for one layer type, length d/2, fp64.

    [AIT] §섹션별 상세 (rotate() takes ``freq[layer_type]``) and the glossary
    entry on partial RoPE: build the spectrum, then set all but the leading
    fraction to zero.  The spectrum itself is not printed on the pages; the
    reading taken is the standard one, freq[t] = theta^(-2t/d) for
    t in [0, d/2), and on global layers the first floor(0.25 * d/2) entries
    are kept and the rest zeroed.
    """
    half = d // 2
    t = np.arange(half, dtype=np.float64)
    f = np.power(float(theta), -2.0 * t / d)
    keep = int(np.floor(rotary_fraction * half + 1e-9))
    f[keep:] = 0.0
    return f


def rotate(x: np.ndarray, freq: np.ndarray, start) -> np.ndarray:
    """Split-half RoPE, [AIT] §섹션별 상세, the rotate() snippet.

    x has shape [..., L, d].  The "rotated" companion of x is the
    concatenation [-x[d/2:], x[:d/2]] (pairs t and t + d/2, not adjacent
    pairs), the angle of row l and channel t is (l + start) * freq[t mod d/2],
    and the result is cos(angle) * x + sin(angle) * companion.  ``start`` is a
    scalar or broadcasts against [..., L, 1].  Channels whose frequency is 0
    come back unchanged.
    """
    x = np.asarray(x, dtype=np.float64)
    L, d = x.shape[-2], x.shape[-1]
    h = d // 2
    companion = np.concatenate([-x[..., h:], x[..., :h]], axis=-1)
    f2 = np.concatenate([np.asarray(freq, np.float64), np.asarray(freq, np.float64)])
    pos = np.arange(L, dtype=np.float64)[:, None] + np.asarray(start, dtype=np.float64)
    ang = pos * f2
    return np.cos(ang) * x + np.sin(ang) * companion


def gelu_tanh(x) -> np.ndarray:
    """GELU in its tanh form, 0.5 x (1 + tanh(sqrt(2/pi) (x + 0.044715 x^3))),
    fp64 -- the activation taken for the self-conditioning MLP ([AIT]
    glossary, self-conditioning: "a small MLP" that maps zero to zero; the
    pages name no activation, and this is the Gemma family's)."""
    x = np.asarray(x, dtype=np.float64)
    u = np.sqrt(2.0 / np.pi) * (x + 0.044715 * x ** 3)
    # 0.5 (1 + tanh(u)) = 1 / (1 + exp(-2u)): the same function, without the
    # cancellation of 1 + tanh(u) for u << 0 (there tanh(u) rounds to -1 in
    # fp64 once x < -6.5 or so)
    with np.errstate(over="ignore"):
        return x / (1.0 + np.exp(-2.0 * u))
