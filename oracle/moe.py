"""A mixture-of-experts MLP block, fp64 -- TEST INFRASTRUCTURE ONLY (see the
package docstring).

What is computed ([AIT] glossary "혼합 전문가(MoE)": every token is routed to
its top-k experts, which run in parallel and are summed with weights, plus a
shared expert; the routing score is the exponential of the router key's dot
product with the input, renormalised and scaled.  [TC] §아키텍처: 128
experts, 8 active + 1 shared), for each token t:

1. s_e = x_t . router_e for every expert e;
2. the k experts with the largest s (equal scores: the lower index first);
3. w_j = exp(s_j) / sum over the chosen exp(s_i), times the expert's scale
   (the renormalisation over the chosen experts; computed about the largest
   score, which leaves it unchanged);
4. expert e's MLP in the gated form of the Gemma family (the pages print
   none): y_e = W_down_e bf16(gelu(W_gate_e x_t) * (W_up_e x_t)), GELU in its
   tanh form; the activation is stored in bf16 before the down projection,
   mirrored here (storage model);
5. out_t = sum over the chosen, in order, of w_j y_{e_j}, plus the shared
   expert's y_shared(x_t) (same form).

Inputs are exact fp64 values: x [R, D], router [E, D], W_gate / W_up
[E*F, D] (expert e: rows e*F ..), W_down [E*D, F], shared weights [Fs, D],
[Fs, D], [D, Fs] or None.
"""
from __future__ import annotations

import numpy as np

from .numerics import bf16_round, gelu_tanh


def route(x, router, k, scale=None):
    """(chosen [R, k] expert ids, weights [R, k], margin [R]); margin is the
    gap between the k-th and (k+1)-th largest score (a tie when tiny)."""
    x = np.asarray(x, np.float64)
    s = x @ np.asarray(router, np.float64).T
    R, E = s.shape
    chosen = np.empty((R, k), np.int64)
    w = np.empty((R, k))
    margin = np.full(R, np.inf)
    for t in range(R):
        # largest first; equal scores: lower index first (a stable sort of -s)
        order = np.argsort(-s[t], kind="stable")
        chosen[t] = order[:k]
        top = s[t, order[:k]]
        p = np.exp(top - top[0])
        w[t] = p / p.sum()
        if scale is not None:
            w[t] *= np.asarray(scale, np.float64)[order[:k]]
        if k < E:
            margin[t] = s[t, order[k - 1]] - s[t, order[k]]
    return chosen, w, margin


def gated_mlp(x, W_gate, W_up, W_down):
    """W_down bf16(gelu(W_gate x) * (W_up x)) for the rows of x."""
    h_g = x @ np.asarray(W_gate, np.float64).T
    h_u = x @ np.asarray(W_up, np.float64).T
    return bf16_round(gelu_tanh(h_g) * h_u) @ np.asarray(W_down, np.float64).T


def moe(x, router, k, W_gate, W_up, W_down, shared=None, scale=None):
    """out [R, D] and the routing (chosen, weights, margin)."""
    x = np.asarray(x, np.float64)
    R, D = x.shape
    E = np.asarray(router).shape[0]
    F = np.asarray(W_gate).shape[0] // E
    chosen, w, margin = route(x, router, k, scale)
    out = np.zeros((R, D))
    for t in range(R):
        for j in range(k):
            e = int(chosen[t, j])
            y = gated_mlp(x[t:t + 1], W_gate[e * F:(e + 1) * F], W_up[e * F:(e + 1) * F], W_down[e * D:(e + 1) * D])
            out[t] += w[t, j] * y[0]
    if shared is not None:
        out += gated_mlp(x, *shared)
    return out, (chosen, w, margin)
