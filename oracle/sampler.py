"""The per-position vocab sampler of one denoising step, fp64.

Test infrastructure only (see the package docstring).

What is computed ([AIT] §섹션별 상세, the sampling-loop paragraph; [AB]
§블록 자동 회귀 노이즈 제거 및 자체 수정; [AIT] glossary, self-conditioning):

1. z = logits / temperature; p = softmax(z) per position (row);
2. entropy H = -sum p ln p (0 ln 0 = 0), argmax (lowest index on ties),
   confidence = max p;
3. entropy-bound decision: a position whose entropy is below the bound is
   committed to its argmax token; the others are renoised to a uniformly
   random token (uniform-state renoise);
4. self-conditioning soft embedding: soft_emb = P E, the probability-weighted
   embedding of every position.

Variants ([AIT] §섹션별 상세, sampling-loop paragraph: the temperature falls
from t_max to t_min over max_denoising_steps; a committed token is drawn from
the tempered softmax; "[논문리뷰] DiffusionGemma Technical Report" §1: adaptive
stopping once every position is committed): ``temperature_schedule``,
``categorical=True`` and ``all_committed``.

Readings (listed in the design notes): the commit test is strict, H < bound,
per position (``commit_mode=0``); ``commit_mode=1`` instead commits the longest
run of qualifying positions from the left of each canvas (the page's "fix the
low-entropy prefix" wording).  Frozen positions keep their token, count as
committed and still contribute to the soft embedding.  The random token is
splitmix.renoise_token(seed, step, row), row = flattened position b*C + i.
With ``probs_storage='bf16'`` the probabilities are rounded to bf16 before the
product with E (they are stored in bf16 for that product).
"""
from __future__ import annotations

from typing import Iterable, Optional

import numpy as np

from .numerics import bf16_round
from .splitmix import key_uniform, renoise_key, renoise_token


def temperature_schedule(step: int, steps: int, t_max: float, t_min: float) -> float:
    """Temperature of denoising step ``step`` of ``steps``: linear from t_max
    (step 0) to t_min (step steps - 1); one step, or a step before 0, is t_max."""
    if steps <= 1 or step <= 0:
        return float(t_max)
    if step >= steps - 1:
        return float(t_min)
    return float(t_max) + (float(t_min) - float(t_max)) * step / (steps - 1)


def categorical_token(stored_row: np.ndarray, u: float) -> int:
    """The inverse-CDF draw from one row of stored probabilities: the
    smallest k with cumsum(p)[k] > u * sum(p) (cumulative sums in fp64, index
    order; the stored row need not sum to exactly 1)."""
    c = np.cumsum(np.asarray(stored_row, np.float64))
    target = u * c[-1]
    return int(np.searchsorted(c, target, side="right"))


def categorical_margin(stored_row: np.ndarray, u: float) -> float:
    """Distance of the draw's target from the nearest cumulative boundary,
    relative to the row total (a tie when it is tiny)."""
    c = np.cumsum(np.asarray(stored_row, np.float64))
    target = u * c[-1]
    return float(np.min(np.abs(c - target)) / c[-1])


def all_committed(commit_mask: np.ndarray, canvas_len: int) -> np.ndarray:
    """Adaptive stopping: per canvas, whether every position is committed."""
    m = np.asarray(commit_mask).reshape(-1, canvas_len)
    return np.all(m != 0, axis=1)


def row_statistics(logits_row: np.ndarray, temperature: float = 1.0):
    """Softmax, entropy, argmax and confidence of one row, exactly in fp64."""
    z = np.asarray(logits_row, np.float64) / temperature
    a = int(np.argmax(z))            # numpy returns the first (lowest) index of the max
    m = z[a]
    e = np.exp(z - m)
    Z = np.sum(e)
    p = e / Z
    with np.errstate(divide="ignore", invalid="ignore"):
        plogp = np.where(p > 0, p * np.log(np.where(p > 0, p, 1.0)), 0.0)
    H = -np.sum(plogp)
    return p, float(H), a, float(p[a])


def canvas_sample(logits, E, entropy_bound: float, seed: int, step: int,
                  temperature: float = 1.0, commit_mode: int = 0, canvas_len: Optional[int] = None,
                  frozen=None, frozen_tokens=None, probs_storage: str = "fp64",
                  soft_rows: Optional[Iterable[int]] = None, categorical: bool = False):
    """One sampler call over ``rows`` positions.

    logits [rows, V] and E [V, D] are exact fp64 values.  Returns a dict with
    tokens, commit_mask, entropy, confidence, argmax (per row), probs
    [rows, V] (as stored: fp64 or bf16-rounded) and soft_emb [rows, D]
    (NaN rows outside ``soft_rows`` when that is given).
    """
    logits = np.asarray(logits, np.float64)
    rows, V = logits.shape
    C = rows if canvas_len is None else int(canvas_len)
    probs = np.empty((rows, V))
    H = np.empty(rows)
    conf = np.empty(rows)
    amax = np.empty(rows, dtype=np.int64)
    for r in range(rows):
        p, h, a, c = row_statistics(logits[r], temperature)
        probs[r], H[r], amax[r], conf[r] = p, h, a, c
    frozen_m = np.zeros(rows, bool) if frozen is None else np.asarray(frozen).astype(bool)
    below = H < entropy_bound
    if commit_mode == 0:
        commit = frozen_m | below
    elif commit_mode == 1:
        commit = np.zeros(rows, bool)
        for r0 in range(0, rows, C):
            for r in range(r0, min(r0 + C, rows)):
                if frozen_m[r] or below[r]:
                    commit[r] = True
                else:
                    break
        commit |= frozen_m
    else:
        raise ValueError(commit_mode)
    stored = bf16_round(probs) if probs_storage == "bf16" else probs
    tokens = np.empty(rows, dtype=np.int64)
    for r in range(rows):
        if frozen_m[r]:
            tokens[r] = int(frozen_tokens[r])
        elif commit[r]:
            tokens[r] = categorical_token(stored[r], key_uniform(renoise_key(seed, step, r))) if categorical \
                else amax[r]
        else:
            tokens[r] = renoise_token(seed, step, r, V)
    soft = None
    if E is not None:
        E = np.asarray(E, np.float64)
        if soft_rows is None:
            soft = stored @ E
        else:
            soft = np.full((rows, E.shape[1]), np.nan)
            for r in soft_rows:
                soft[r] = stored[r] @ E
    return dict(tokens=tokens, commit_mask=commit.astype(np.uint8), entropy=H, confidence=conf,
                argmax=amax, probs=stored, soft_emb=soft)
