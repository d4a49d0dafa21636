"""The self-conditioning MLP through the C ABI against the fp64 oracle:
sc = W2 bf16(gelu(W1 bf16(soft))) (canvas_cast_bf16, canvas_gemm_bf16,
canvas_gelu_bf16, canvas_gemm_bf16), the loop's input assembly with it, and
the loop's invariants with it switched on.

Bars: bf16 values bit-exact except at rounding ties (a value within the
path's fp32 error of a bf16 midpoint), where either neighbour is correct; the
fp32 products within the recursive-summation bound gamma_K sum |terms| plus
the effect of the tie flips.
"""
import numpy as np
import pytest
import torch

import canvas_workloads as wl
from oracle import loop as oloop
from oracle import numerics as onum

pytestmark = pytest.mark.gpu
U = 2.0 ** -24


@pytest.fixture(scope="module")
def cv():
    import __graft_entry__
    __graft_entry__.build()
    import canvas_denoising_step_03_b300 as cv
    return cv


def spacing(a):
    a = np.abs(np.asarray(a, np.float64))
    return np.ldexp(1.0, (np.floor(np.log2(np.where(a > 0, a, 1.0))) - 7).astype(int))


def gelu_rel_err(x):
    """Relative error of the device's fp32 GELU, x / (1 + exp(-2u)): a few
    units of 2^-24 from the division and exp, plus the argument's own
    rounding (about 3 units of 2^-24 of |2u|) magnified by exp's condition
    number |2u| where exp(-2u) dominates."""
    u2 = 2.0 * np.sqrt(2.0 / np.pi) * np.abs(x + 0.044715 * x ** 3)
    return (3.0 * u2 + 8.0) * 2.0 ** -24


def tie_mask(y, rel):
    """Where bf16 rounding of y is ambiguous within a relative error ``rel``."""
    s = onum.bf16_round(y)
    sp = spacing(s)
    frac = np.abs((np.abs(y) / sp) % 1.0 - 0.5)     # distance to a midpoint, in spacings
    return frac * sp <= rel * np.abs(y) + 1e-30


def test_gelu_bf16_against_the_oracle(cv):
    rng = np.random.default_rng(3)
    x = np.concatenate([rng.standard_normal(1 << 16) * 2, rng.standard_normal(4096) * 30,
                        [0.0, 1e-30, -1e-30, 1e-8, -1e-8, 50.0, -50.0, 3.0, -3.0, 0.5]]).astype(np.float32)
    x = x[: len(x) // 8 * 8]
    xd = torch.from_numpy(x).cuda()
    out = torch.empty(len(x), dtype=torch.bfloat16, device="cuda")
    cv.canvas_gelu_bf16(xd, out)
    assert cv.canvas_device_status() == cv.CANVAS_OK
    got = out.float().cpu().numpy().astype(np.float64)
    g = onum.gelu_tanh(x.astype(np.float64))
    want = onum.bf16_round(g)
    rel = gelu_rel_err(x.astype(np.float64))
    tie = tie_mask(g, rel)
    bad = np.nonzero((got != want) & ~tie)[0]
    assert bad.size == 0, [(float(x[i]), got[i], want[i]) for i in bad[:8]]
    assert np.all(np.abs(got - g)[tie] <= 0.5 * spacing(got[tie]) + rel[tie] * np.abs(g[tie]) + 1e-30)
    print(f"gelu: {int(tie.sum())} of {len(x)} values within the fp32 error of a bf16 midpoint")


def test_selfcond_mlp_stage(cv):
    """The loop's self-conditioning stage on an oracle-provided soft
    embedding (fp32 values), the mini-loop shapes with hidden width 64."""
    from canvas_denoising_step_03_b300.loop import CanvasLoop
    cfg = wl.mini_loop_config(steps=1, selfcond_hidden=64)
    inp = wl.make_loop_inputs(cfg)
    run = CanvasLoop(inp)
    R, D, H = cfg.B * cfg.C, cfg.D, cfg.selfcond_hidden
    rng = np.random.default_rng(9)
    soft32 = (rng.standard_normal((R, D)) * 0.4).astype(np.float32)
    W1, W2 = wl.as_f64(inp.sc_W1, "bf16"), wl.as_f64(inp.sc_W2, "bf16")
    got = run.selfcond(torch.from_numpy(soft32).cuda()).cpu().numpy().astype(np.float64)
    assert cv.canvas_device_status() == cv.CANVAS_OK
    s = soft32.astype(np.float64)
    want = oloop.selfcond_mlp(s, W1, W2)
    # h = bf16(s) W1^T in fp32 (recursive-summation bound), gelu, bf16 rounding
    s16 = onum.bf16_round(s)
    h = s16 @ W1.T
    hb = D * U / (1 - D * U) * (np.abs(s16) @ np.abs(W1).T)
    g = onum.gelu_tanh(h)
    # a rounding of gelu(h) is a tie when h's fp32 error (times |gelu'| <= 1.13)
    # or gelu's own can reach the midpoint
    sp = spacing(onum.bf16_round(g))
    frac = np.abs((np.abs(g) / sp) % 1.0 - 0.5) * sp
    tie = frac <= 1.13 * hb + gelu_rel_err(h) * np.abs(g) + 1e-30
    gb = onum.bf16_round(g)
    bound = (H * U / (1 - H * U)) * ((np.abs(gb) + tie * sp) @ np.abs(W2).T) + (tie * sp) @ np.abs(W2).T
    err = np.abs(got - want)
    assert np.all(err <= bound + U * np.abs(want)), float(np.max(err - bound))
    print(f"self-conditioning MLP: max |err| {err.max():.3g}, {int(tie.sum())} tie elements of {tie.size}")


def test_mini_loop_with_selfcond_invariants(cv):
    """Free-running steps with the MLP on: the sampler's rules still hold
    exactly (the MLP changes the input, not the rules)."""
    from canvas_denoising_step_03_b300.loop import CanvasLoop
    from test_gpu_loop import _free_run_invariants
    cfg = wl.mini_loop_config(steps=6, selfcond_hidden=64)
    run = CanvasLoop(wl.make_loop_inputs(cfg))
    _free_run_invariants(cfg, run, cfg.steps)
    assert cv.canvas_device_status() == cv.CANVAS_OK, cv.canvas_last_error()
