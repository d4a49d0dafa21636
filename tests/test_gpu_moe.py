"""canvas_moe through the C ABI against the fp64 oracle (oracle/moe.py).

Routing: the chosen experts bit-exact, in order, except for tokens whose k-th
and (k+1)-th router scores lie within the fp32 error of the scores (a tie:
logged and excluded, as for sampled tokens at an entropy tie); weights
within 1e-5 relative.  Output: every element within a bound computed from
the arithmetic -- the fp32 recursive-summation bound of each product
(gamma_K sum |terms|), the bf16 activation's rounding ties (an activation
value within its fp32 error of a bf16 midpoint may take either neighbour),
the weights' fp32 error -- and relative Frobenius error <= 5e-3.
"""
import numpy as np
import pytest
import torch

import canvas_workloads as wl
from oracle import moe as omoe
from oracle import numerics as onum

pytestmark = pytest.mark.gpu
U = 2.0 ** -24


def gam(K):
    return K * U / (1 - K * U)


@pytest.fixture(scope="module")
def cv():
    import __graft_entry__
    __graft_entry__.build()
    import canvas_denoising_step_03_b300 as cv
    return cv


def spacing(a):
    a = np.abs(np.asarray(a, np.float64))
    return np.ldexp(1.0, (np.floor(np.log2(np.where(a > 0, a, 1.0))) - 7).astype(int))


def act_bound(x, Wg, Wu, Wd):
    """Per output element of W_down bf16(gelu(W_gate x) * (W_up x)): the bound
    of the device's deviation from the oracle (fp32 products, activation
    ties), for the rows of x."""
    D = x.shape[1]
    hg, hu = x @ Wg.T, x @ Wu.T
    dh_g = gam(D) * (np.abs(x) @ np.abs(Wg).T)
    dh_u = gam(D) * (np.abs(x) @ np.abs(Wu).T)
    g = onum.gelu_tanh(hg)
    a = g * hu
    # |gelu'| <= 1.13 everywhere; the fp32 GELU's own relative error as in
    # test_gpu_selfcond.gelu_rel_err
    u2 = 2.0 * np.sqrt(2.0 / np.pi) * np.abs(hg + 0.044715 * hg ** 3)
    da = 1.13 * dh_g * np.abs(hu) + np.abs(g) * dh_u + ((3.0 * u2 + 12.0) * 2.0 ** -24) * np.abs(a) + 1e-30
    ab = onum.bf16_round(a)
    sp = spacing(ab)
    frac = np.abs((np.abs(a) / sp) % 1.0 - 0.5) * sp
    tie = frac <= da
    F = Wg.shape[0]
    flip = tie * sp
    return gam(F) * ((np.abs(ab) + flip) @ np.abs(Wd).T) + flip @ np.abs(Wd).T, int(tie.sum())


def run_case(cv, R, D, E, F, k, Fs, seed, scale=False):
    rng = np.random.default_rng(seed)

    def q(*shape, std=1.0):
        return wl.f32_to_bf16_bits((rng.standard_normal(shape) * std).astype(np.float32))

    x = q(R, D)
    router = q(E, D, std=1.0 / np.sqrt(D))
    Wg, Wu = q(E * F, D, std=1.0 / np.sqrt(D)), q(E * F, D, std=1.0 / np.sqrt(D))
    Wd = q(E * D, F, std=1.0 / np.sqrt(F))
    sh = (q(Fs, D, std=1.0 / np.sqrt(D)), q(Fs, D, std=1.0 / np.sqrt(D)), q(D, Fs, std=1.0 / np.sqrt(Fs))) if Fs else None
    sc = rng.uniform(0.5, 1.5, E).astype(np.float32) if scale else None
    d = lambda a: None if a is None else torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).cuda().view(torch.bfloat16)  # noqa: E731
    out = torch.full((R, D), float("nan"), device="cuda")
    idx = torch.full((R, k), -1, dtype=torch.int32, device="cuda")
    w = torch.full((R, k), float("nan"), device="cuda")
    ws = cv.workspace(cv.canvas_moe_workspace_size(R, D, E, F, k, Fs))
    cv.canvas_moe(d(x), d(router), k, None if sc is None else torch.from_numpy(sc).cuda(), d(Wg), d(Wu), d(Wd),
                  *(sh and [d(a) for a in sh] or [None, None, None]), out, idx, w, ws)
    assert cv.canvas_device_status() == cv.CANVAS_OK, cv.canvas_last_error()
    f = lambda a: None if a is None else wl.as_f64(a, "bf16")  # noqa: E731
    X, Rt, G, Uw, Dn = f(x), f(router), f(Wg), f(Wu), f(Wd)
    SH = None if sh is None else tuple(f(a) for a in sh)
    want, (chosen, wts, margin) = omoe.moe(X, Rt, k, G, Uw, Dn, shared=SH,
                                           scale=None if sc is None else sc.astype(np.float64))
    # routing
    s_err = 2 * gam(D) * (np.abs(X) @ np.abs(Rt).T).max(axis=1)
    tie = margin <= s_err
    got_idx, got_w = idx.cpu().numpy(), w.cpu().numpy().astype(np.float64)
    assert np.array_equal(got_idx[~tie], chosen[~tie])
    np.testing.assert_allclose(got_w[~tie], wts[~tie], rtol=1e-5, atol=1e-7)
    # output bound
    got = out.cpu().numpy().astype(np.float64)
    bound = np.zeros((R, D))
    n_ties = 0
    for t in np.nonzero(~tie)[0]:
        for j in range(k):
            e = int(chosen[t, j])
            b, nt = act_bound(X[t:t + 1], G[e * F:(e + 1) * F], Uw[e * F:(e + 1) * F], Dn[e * D:(e + 1) * D])
            y = omoe.gated_mlp(X[t:t + 1], G[e * F:(e + 1) * F], Uw[e * F:(e + 1) * F], Dn[e * D:(e + 1) * D])
            bound[t] += wts[t, j] * b[0] + 1e-5 * abs(wts[t, j]) * np.abs(y[0])
            n_ties += nt
    if SH is not None:
        b, nt = act_bound(X, *SH)
        bound += b
        n_ties += nt
    bound += gam(k + 1) * np.abs(want) * (k + 1) + U * np.abs(want)
    ok = ~tie
    err = np.abs(got - want)[ok]
    assert np.all(err <= bound[ok]), float(np.max(err - bound[ok]))
    rf = np.linalg.norm(got[ok] - want[ok]) / np.linalg.norm(want[ok])
    assert rf <= 5e-3, rf
    print(f"moe R={R} E={E} k={k}: {int(tie.sum())} routing ties excluded, {n_ties} activation ties, "
          f"max |err| {err.max():.3g}, rel-Fro {rf:.2e}")
    return got_idx


def test_moe_small(cv):
    run_case(cv, R=96, D=256, E=16, F=64, k=4, Fs=64, seed=1)


def test_moe_128_experts_top8_shared_and_scales(cv):
    """The pages' routing shape: 128 experts, 8 chosen + 1 shared; many experts
    get only a few tokens (rows padded to whole tiles)."""
    idx = run_case(cv, R=256, D=256, E=128, F=64, k=8, Fs=64, seed=2, scale=True)
    assert len(np.unique(idx)) > 100      # most experts are used


def test_moe_without_shared_expert_and_k1(cv):
    run_case(cv, R=40, D=128, E=8, F=32, k=1, Fs=0, seed=3)
