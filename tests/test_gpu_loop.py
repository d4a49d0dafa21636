"""The batched multi-layer denoising loop (canvas_denoising_step_03_b300.loop)
against the fp64 oracle of the same loop (oracle/loop.py).

A stack of random attention layers with these logit scales is chaotic: two
runs whose first layer agrees to bf16 rounding part by orders of magnitude a
few layers later (measured: 0.016, 0.03, 0.3, 2.1, 5.3, 6.8 max |err| over
the six layers of the small loop).  So the loop is checked stage by stage:
every stage of every step runs on the device from the oracle's own input to
that stage (oracle values feed the device, never the reverse) and its output
is held to the bar of that stage --
  attention layer  the bar of test_gpu_attention.py
                   (canvas_harness.attention_bar) against the oracle's
                   output before its bf16 store: |err| <= max(2e-2, half a
                   bf16 spacing of the value) + rounding slack on at most
                   MAX_FRAC_OVER of the elements, rel-Fro <= 5e-3 (the
                   activations of deeper layers reach |o| >= 8, where bf16
                   values are 1/16 apart);
  residual add     the fp32 recursive-summation bound;
  LM head          bf16 logits within one bf16 ulp plus that bound;
  sampler          entropy within 1e-3 nats, tokens / commit masks bit-exact
                   away from ties, soft embedding rel-Fro <= 5e-3.
Free-running device trajectories are checked through what holds exactly:
tokens are the argmax or the SplitMix64 renoise draw of their own decisions,
committed positions stay committed.
"""
import numpy as np
import pytest
import torch

import canvas_workloads as wl
from canvas_harness import SLACK_EPS, attention_bar
from oracle import attention as oatt
from oracle import loop as oloop
from oracle import sampler as osamp
from oracle import splitmix

pytestmark = pytest.mark.gpu
TIE = 1e-6


@pytest.fixture(scope="module")
def cv():
    import __graft_entry__
    __graft_entry__.build()
    import canvas_denoising_step_03_b300 as cv
    return cv


def oracle_layers(inp):
    f = lambda a: wl.as_f64(a, "bf16")  # noqa: E731
    out = []
    for L in inp.layers:
        c = L.cfg
        out.append(dict(W_q=f(L.W_q), W_k=f(L.W_k), W_v=None if L.W_v is None else f(L.W_v), W_o=f(L.W_o),
                        gamma_q=L.gamma_q.astype(np.float64), gamma_k=L.gamma_k.astype(np.float64),
                        freq=L.freq.astype(np.float64), eps=c.eps, Hq=c.Hq, Hkv=c.Hkv, d=c.d, layer=c.layer,
                        window=c.window, prefix=inp.cfg.prefix,
                        cache_k=oloop.dense_cache(f(L.cache_k), L.cache_lo, inp.cfg.prefix),
                        cache_v=None if L.cache_v is None else oloop.dense_cache(f(L.cache_v), L.cache_lo,
                                                                                inp.cfg.prefix)))
    return out


def to_bf16(a64, shape):
    """Exact bf16 values (fp64) -> a device bf16 tensor."""
    bits = wl.f32_to_bf16_bits(np.asarray(a64, np.float32))
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16).reshape(shape)).cuda().view(torch.bfloat16)


def bf16_ulp(a):
    a = np.abs(np.asarray(a, np.float64))
    e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    return np.ldexp(1.0, (e - 7).astype(int))


U = 2.0 ** -24


def gamma(K):
    return K * U / (1 - K * U)


def _fp64_layer(layers, k, xk, B, C, rows=None):
    """Layer k of the oracle with no bf16 rounding at all, on input xk."""
    L = layers[k]
    out, _ = oatt.canvas_attention(xk, L["W_q"], L["W_k"], L["W_v"], L["Hq"], L["Hkv"], L["d"], L["gamma_q"],
                                   L["gamma_k"], L["eps"], L["freq"], L["layer"], L["cache_k"], L["cache_v"],
                                   np.full(B, L["prefix"]), L["window"], storage="fp64", rows=rows)
    return out


def check_step(cv, run, ref, cfg, step, frozen, ftok, rows, run_wo, E_exact, layers=None):
    """Every stage of one step from the oracle's inputs; ``rows``: sampler rows
    the oracle evaluated; run_wo / E_exact: exact W_o of each layer and E;
    ``layers`` (the oracle's layer dicts): also record the distance to the
    oracle without bf16 rounding."""
    B, C, D = cfg.B, cfg.C, cfg.D
    R = B * C
    report = []
    nl = len(run.layers)
    for k in range(nl):
        # attention of layer k on the oracle's canvas stream
        xin = oloop.bf16_round(ref["xs"][k])
        xk = to_bf16(xin, (B, C, D))
        got = run.attention(k, xk).float().cpu().numpy().astype(np.float64)
        assert cv.canvas_device_status() == cv.CANVAS_OK, cv.canvas_last_error()
        want, slack = ref["attn_exact"][k], ref["slack"][k]
        want64 = None
        if layers is not None:
            want64 = _fp64_layer(layers, k, xin.reshape(B, C, D), B, C)
        rec = attention_bar(f"{cfg.name} step {step} layer {k} ({layers[k]['layer'] if layers else ''})", got,
                              want, slack, want64)
        # residual add on the oracle's fp32 stream and its stored attention
        # output: fp32 accumulation over K terms is within gamma_K * sum |terms|
        # (recursive summation bound, gamma_K = K u / (1 - K u), u = 2^-24),
        # plus the fp32 roundings of the incoming stream and of the result
        stored = ref["attn"][k]
        x32 = torch.from_numpy(ref["xs"][k].astype(np.float32)).cuda()
        xb = torch.empty((B, C, D), dtype=torch.bfloat16, device="cuda")
        run.residual(k, to_bf16(stored, (B, C, -1)), x32, xb)
        nxt = ref["xs"][k + 1]
        o = stored.reshape(R, -1)
        Wo = run_wo[k]
        bound = gamma(o.shape[1]) * (np.abs(o) @ np.abs(Wo).T) + U * (np.abs(ref["xs"][k]) + np.abs(nxt))
        rerr = np.abs(x32.cpu().numpy().astype(np.float64) - nxt)
        assert np.all(rerr <= bound), (step, k, float(np.max(rerr - bound)))
        report.append((k, rec["max_abs_err"], rec["rel_fro"], rec["over_bar"]))
    # tied LM head on the oracle's final stream
    # (bf16 result: one ulp of rounding plus the fp32 accumulation bound,
    # which dominates where the terms cancel)
    logits = run.head(to_bf16(ref["x"], (B, C, D)))
    got = logits.float().cpu().numpy()[rows].astype(np.float64)
    want = ref["logits"][rows]
    bound = bf16_ulp(want) + gamma(D) * (np.abs(ref["x"][rows]) @ np.abs(E_exact).T)
    assert np.all(np.abs(got - want) <= bound), float(np.max(np.abs(got - want) - bound))
    # sampler on the head's logits
    dev = "cuda"
    fr = torch.from_numpy((np.zeros(R) if frozen is None else frozen).astype(np.uint8)).to(dev)
    ft = torch.from_numpy((np.zeros(R) if ftok is None else ftok).astype(np.int32)).to(dev)
    run.sample(logits, step, fr, ft)
    assert cv.canvas_device_status() == cv.CANVAS_OK, cv.canvas_last_error()
    H = ref["entropy"]
    ent = run.entropy.cpu().numpy().astype(np.float64)[rows]
    assert np.max(np.abs(ent - H)) <= 1e-3, (step, float(np.max(np.abs(ent - H))))
    ok = np.abs(H - cfg.bound) > TIE
    np.testing.assert_array_equal(run.mask.cpu().numpy()[rows][ok], ref["commit_mask"][ok])
    np.testing.assert_array_equal(run.next_tokens.cpu().numpy()[rows][ok], ref["tokens"][ok])
    soft = run.soft.cpu().numpy().astype(np.float64)[rows]
    rf = np.linalg.norm(soft - ref["soft_emb"]) / np.linalg.norm(ref["soft_emb"])
    assert rf <= 5e-3, (step, rf)
    print(f"step {step}: layers (k, max|err|, rel-Fro, elements over the bar) {report}; "
          f"max |dH| {np.max(np.abs(ent - H)):.2e}, soft rel-Fro {rf:.2e}, ties {int((~ok).sum())}")
    return int(ref["commit_mask"].sum())


def test_mini_loop_every_stage_every_step(cv):
    """2 canvases x 32, prefix 160, 5 sliding (window 48) + 1 global layers,
    vocab 4096, 4 steps: every stage of every step, all rows."""
    from canvas_denoising_step_03_b300.loop import CanvasLoop
    cfg = wl.mini_loop_config(steps=4)
    inp = wl.make_loop_inputs(cfg)
    run = CanvasLoop(inp)
    layers = oracle_layers(inp)
    E = wl.as_f64(inp.E, "bf16")
    tokens = inp.tokens0.astype(np.int64)
    soft, frozen, ftok = None, None, None
    R = cfg.B * cfg.C
    commits = []
    for s in range(cfg.steps):
        ref = oloop.loop_step(layers, E, tokens, soft, s, cfg.B, cfg.C, cfg.seed, cfg.bound, frozen, ftok,
                              slack_eps=SLACK_EPS)
        commits.append(check_step(cv, run, ref, cfg, s, frozen, ftok, np.arange(R), [L["W_o"] for L in layers], E,
                                  layers=layers))
        tokens, soft = ref["tokens"], ref["soft_emb"]
        frozen, ftok = ref["commit_mask"], ref["tokens"]
    assert 0 < commits[-1] < R     # both branches of the sampler are exercised
    assert commits == sorted(commits)


def test_loop_workload_first_step_every_stage(cv):
    """4 canvases x 256, prefix 1024, 5 sliding + 1 global layers (the sliding-
    and global-layer shapes), vocab 262144: every stage of step 0, all rows of
    every layer, a sample of sampler rows."""
    from canvas_denoising_step_03_b300.loop import CanvasLoop
    cfg = wl.loop_config(1024, steps=1)
    inp = wl.make_loop_inputs(cfg)
    run = CanvasLoop(inp)
    rows = np.array([0, 1, 255, 256, 600, 777, 1022, 1023])
    layers = oracle_layers(inp)
    E = wl.as_f64(inp.E, "bf16")
    ref = oloop.loop_step(layers, E, inp.tokens0, None, 0, cfg.B, cfg.C, cfg.seed, cfg.bound, sample_rows=rows,
                          slack_eps=SLACK_EPS)
    check_step(cv, run, ref, cfg, 0, None, None, rows, [L["W_o"] for L in layers], E, layers=layers)


@pytest.mark.slow
@pytest.mark.parametrize("prefix", [8192, 32768, 131072])
def test_loop_workload_long_prefix_layers(cv, prefix):
    """The loop at the longer prefixes of the sweep, step 0: each of the six
    attention layers (5 sliding, 1 global) at its full size -- the global layer
    attends over the whole prefix with RoPE positions up to prefix + 255 --
    checked at a seeded sample of canvas rows (16; 8 at prefix 131072; every
    head of each), all
    from the same oracle-provided input: the step's canvas input bf16(E[tokens])
    (the first layer's real input; stage-wise parity needs no chaining, and a
    layer's sampled rows need every canvas row only as keys, which the input
    gives).  The head, sampler and residual stages do not depend on the prefix
    and are checked on every row of the prefix-1024 loop."""
    from canvas_denoising_step_03_b300.loop import CanvasLoop
    cfg = wl.loop_config(prefix, steps=1)
    inp = wl.make_loop_inputs(cfg)
    run = CanvasLoop(inp)
    B, C, D = cfg.B, cfg.C, cfg.D
    R = B * C
    rng = np.random.default_rng(prefix)
    n = 16 if prefix <= 32768 else 8        # the oracle's global layer costs O(prefix) per row
    rows = np.sort(np.concatenate([[0, R - 1], rng.choice(np.arange(1, R - 1), n - 2, replace=False)]))
    E_rows = wl.as_f64(inp.E[inp.tokens0.astype(np.int64)], "bf16")        # E[tokens], exact
    x0 = oloop.bf16_round(E_rows).reshape(B, C, D)
    xk = to_bf16(x0, (B, C, D))
    layers = oracle_layers(inp)
    for k, L in enumerate(layers):
        sub = [(int(r) // C, h, int(r) % C) for r in rows for h in range(L["Hq"])]
        got = run.attention(k, xk).float().cpu().numpy().astype(np.float64)
        assert cv.canvas_device_status() == cv.CANVAS_OK, cv.canvas_last_error()
        args = (x0, L["W_q"], L["W_k"], L["W_v"], L["Hq"], L["Hkv"], L["d"], L["gamma_q"], L["gamma_k"], L["eps"],
                L["freq"], L["layer"], L["cache_k"], L["cache_v"], np.full(B, L["prefix"]), L["window"])
        want, _, slack = oatt.canvas_attention(*args, storage="bf16", rows=sub, slack_eps=SLACK_EPS)
        want64, _ = oatt.canvas_attention(*args, storage="fp64", rows=sub)
        attention_bar(f"{cfg.name} step 0 layer {k} ({L['layer']}, {n} sampled canvas rows)", got, want, slack,
                        want64)


def _free_run_invariants(cfg, run, steps):
    R = cfg.B * cfg.C
    prev_mask = np.zeros(R, np.uint8)
    prev_tok = None
    for s in range(steps):
        run.step()
        mask = run.mask.cpu().numpy()
        tok = run.tokens.cpu().numpy()
        H = run.entropy.cpu().numpy()
        amax = run.argmax.cpu().numpy()
        assert np.all(H >= -1e-6) and np.all(H <= np.log(cfg.V) + 1e-3)
        assert np.all(mask[prev_mask == 1] == 1)                      # committed positions stay committed
        if prev_tok is not None:
            np.testing.assert_array_equal(tok[prev_mask == 1], prev_tok[prev_mask == 1])
        new = (mask == 1) & (prev_mask == 0)
        np.testing.assert_array_equal(mask[prev_mask == 0], (H[prev_mask == 0] < cfg.bound).astype(np.uint8))
        np.testing.assert_array_equal(tok[new], amax[new])            # newly committed: the argmax
        ren = np.nonzero(mask == 0)[0]
        want = np.array([splitmix.renoise_token(cfg.seed, s, int(r), cfg.V) for r in ren], dtype=np.int64)
        np.testing.assert_array_equal(tok[ren], want)                 # the rest: the renoise draw
        prev_mask, prev_tok = mask, tok
    return int(prev_mask.sum())


def test_mini_loop_free_run_invariants(cv):
    from canvas_denoising_step_03_b300.loop import CanvasLoop
    cfg = wl.mini_loop_config(steps=8)
    run = CanvasLoop(wl.make_loop_inputs(cfg))
    committed = _free_run_invariants(cfg, run, cfg.steps)
    assert cv.canvas_device_status() == cv.CANVAS_OK, cv.canvas_last_error()
    assert committed > 0


def test_loop_workload_48_steps_invariants(cv):
    """48 steps at prefix 1024 on the full loop; with these weights the
    distributions stay near-uniform, so every position is renoised every step."""
    from canvas_denoising_step_03_b300.loop import CanvasLoop
    cfg = wl.loop_config(1024, steps=48)
    run = CanvasLoop(wl.make_loop_inputs(cfg))
    committed = _free_run_invariants(cfg, run, cfg.steps)
    assert cv.canvas_device_status() == cv.CANVAS_OK, cv.canvas_last_error()
    assert committed == 0


def test_mini_loop_schedule_categorical_and_adaptive_stop(cv):
    """The loop with the linear temperature schedule, categorical draws and
    adaptive stopping: every step follows the sampler's rule at its own
    temperature (checked against the oracle's sampler on the device's own
    logits), and the loop stops at the first step where every canvas is
    committed."""
    from canvas_denoising_step_03_b300.loop import CanvasLoop
    cfg = wl.mini_loop_config(steps=24)
    steps, t_max, t_min = 24, 1.0, 0.05
    run = CanvasLoop(wl.make_loop_inputs(cfg), schedule=(t_max, t_min, steps), categorical=True)
    R = cfg.B * cfg.C
    prev_mask = np.zeros(R, np.uint8)
    prev_tok = None
    stopped = None
    E = wl.as_f64(wl.make_loop_inputs(cfg).E, "bf16")
    for s in range(steps):
        run.step()
        logits = wl.as_f64(np.ascontiguousarray(run.logits.cpu().view(torch.int16).numpy()).view(np.uint16),
                           "bf16")
        tau = osamp.temperature_schedule(s, steps, t_max, t_min)
        assert abs(run.temperature(s) - tau) <= 1e-6 * tau
        ref = osamp.canvas_sample(logits, E, cfg.bound, cfg.seed, s, temperature=run.temperature(s),
                                  canvas_len=cfg.C, frozen=prev_mask, frozen_tokens=prev_tok if prev_tok is not None
                                  else np.zeros(R, np.int64), probs_storage="bf16", categorical=True)
        mask = run.mask.cpu().numpy()
        tok = run.tokens.cpu().numpy()
        ok = np.abs(ref["entropy"] - cfg.bound) > TIE
        np.testing.assert_array_equal(mask[ok], ref["commit_mask"][ok])
        # renoised rows take the draw of their own global row
        ren = np.nonzero((mask == 0) & ok)[0]
        np.testing.assert_array_equal(tok[ren], [splitmix.renoise_token(cfg.seed, s, int(r), cfg.V) for r in ren])
        newc = np.nonzero((mask == 1) & (prev_mask == 0) & ok)[0]
        for r in newc:
            u = splitmix.key_uniform(splitmix.renoise_key(cfg.seed, s, int(r)))
            if osamp.categorical_margin(ref["probs"][r], u) > 1e-9:
                assert tok[r] == osamp.categorical_token(ref["probs"][r], u)
        counts = run.committed_counts().cpu().numpy()
        np.testing.assert_array_equal(counts, mask.reshape(cfg.B, cfg.C).sum(axis=1))
        prev_mask, prev_tok = mask, tok
        if np.all(osamp.all_committed(mask, cfg.C)):
            stopped = s + 1
            break
    assert stopped is not None, "the schedule should commit every position within the step budget"
    # the driver's own stopping rule stops at the same step on a fresh run
    run2 = CanvasLoop(wl.make_loop_inputs(cfg), schedule=(t_max, t_min, steps), categorical=True)
    assert run2.run(steps) == stopped
    assert cv.canvas_device_status() == cv.CANVAS_OK
