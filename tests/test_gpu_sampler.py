"""canvas_sample through the C ABI against the fp64 oracle.

Bars: entropy within 1e-3 nats; argmax, commit mask and tokens bit-exact
except at positions whose oracle entropy lies within 1e-6 of the bound (they
are reported and excluded); soft embedding relative Frobenius error <= 5e-3.
"""
import numpy as np
import pytest
import torch

import canvas_workloads as wl
from canvas_harness import to_device
from oracle import numerics as onum
from oracle import sampler as osamp

pytestmark = pytest.mark.gpu
TIE = 1e-6


def onum_spacing(a):
    """Distance between consecutive bf16 values around |a| (8 significant bits;
    normal range)."""
    a = np.abs(np.asarray(a, np.float64))
    e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    return np.ldexp(1.0, (e - 7).astype(int))


@pytest.fixture(scope="module")
def cv():
    import __graft_entry__
    __graft_entry__.build()
    import canvas_denoising_step_03_b300 as cv
    return cv


class SampleRun:
    def __init__(self, cv, s: wl.SampleInputs, probs_dtype=None, temperature=1.0, commit_mode=0, frozen=None,
                 frozen_tokens=None, step=None, seed=None):
        c = s.cfg
        dev = "cuda"
        self.logits = to_device(s.logits, c.dtype)
        self.E = to_device(s.E, c.dtype)
        self.tokens = torch.full((c.rows,), -7, dtype=torch.int32, device=dev)
        self.mask = torch.full((c.rows,), 9, dtype=torch.uint8, device=dev)
        self.ent = torch.full((c.rows,), float("nan"), device=dev)
        self.conf = torch.full((c.rows,), float("nan"), device=dev)
        self.amax = torch.full((c.rows,), -1, dtype=torch.int32, device=dev)
        self.soft = torch.full((c.rows, c.D), float("nan"), device=dev)
        self.probs = None
        pd = cv.CANVAS_FP32
        if probs_dtype is not None:
            tdt = torch.bfloat16 if probs_dtype == "bf16" else torch.float32
            pd = cv.CANVAS_BF16 if probs_dtype == "bf16" else cv.CANVAS_FP32
            self.probs = torch.full((c.rows, c.V), float("nan"), dtype=tdt, device=dev)
        dcode = cv.CANVAS_BF16 if c.dtype == "bf16" else cv.CANVAS_FP32
        ws = cv.workspace(cv.canvas_sample_workspace_size(dcode, c.rows, c.V, c.D))
        fr = None if frozen is None else torch.from_numpy(frozen.astype(np.uint8)).to(dev)
        ft = None if frozen_tokens is None else torch.from_numpy(frozen_tokens.astype(np.int32)).to(dev)
        cv.canvas_sample(self.logits, self.E, c.bound, c.seed if seed is None else seed,
                         c.step if step is None else step, temperature, commit_mode, c.C, fr, ft, self.tokens,
                         self.mask, self.ent, self.conf, self.amax, self.probs, pd, self.soft, ws)
        assert cv.canvas_device_status() == cv.CANVAS_OK, cv.canvas_last_error()


def compare(cv, s, run, ref, soft_rows=None):
    c = s.cfg
    H = ref["entropy"]
    tie = np.abs(H - c.bound) <= TIE
    if tie.any():
        print("near-tie positions excluded:", np.nonzero(tie)[0].tolist())
    ent = run.ent.cpu().numpy().astype(np.float64)
    assert np.max(np.abs(ent - H)) <= 1e-3, np.max(np.abs(ent - H))
    np.testing.assert_array_equal(run.amax.cpu().numpy(), ref["argmax"])
    ok = ~tie
    np.testing.assert_array_equal(run.mask.cpu().numpy()[ok], ref["commit_mask"][ok])
    np.testing.assert_array_equal(run.tokens.cpu().numpy()[ok], ref["tokens"][ok])
    np.testing.assert_allclose(run.conf.cpu().numpy(), ref["confidence"], rtol=1e-4, atol=1e-7)
    soft = run.soft.cpu().numpy().astype(np.float64)
    want = ref["soft_emb"]
    if soft_rows is not None:
        soft, want = soft[soft_rows], want[soft_rows]
    rf = np.linalg.norm(soft - want) / np.linalg.norm(want)
    assert rf <= 5e-3, rf
    return rf


def test_tiny_fp32_workload(cv):
    s = wl.make_sample_inputs(wl.TINY_SAMPLE)
    run = SampleRun(cv, s, probs_dtype="fp32")
    ref = osamp.canvas_sample(wl.as_f64(s.logits, "fp32"), wl.as_f64(s.E, "fp32"), s.cfg.bound, s.cfg.seed,
                              s.cfg.step, canvas_len=s.cfg.C)
    compare(cv, s, run, ref)
    np.testing.assert_allclose(run.probs.cpu().numpy(), ref["probs"], rtol=1e-5, atol=1e-9)


def _peaked_small(dtype="bf16", rows=48, V=4096, seed=5):
    # half peaked (low entropy, commit), half flat (renoise): exercises both branches
    return wl.make_sample_inputs(wl.SampleConfig("peaked", rows=rows, C=16, V=V, D=136, dtype=dtype, seed=seed,
                                                 step=3, bound=0.3, logits="mixture", peak=12.0,
                                                 gen_temperature=0.5, E_std=0.02))


@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
def test_peaked_and_flat_rows(cv, dtype):
    s = _peaked_small(dtype)
    run = SampleRun(cv, s, probs_dtype=dtype)
    st = "bf16" if dtype == "bf16" else "fp64"
    ref = osamp.canvas_sample(wl.as_f64(s.logits, dtype), wl.as_f64(s.E, dtype), s.cfg.bound, s.cfg.seed,
                              s.cfg.step, canvas_len=s.cfg.C, probs_storage=st)
    assert 0 < ref["commit_mask"].sum() < s.cfg.rows
    compare(cv, s, run, ref)
    got = run.probs.float().cpu().numpy().astype(np.float64)
    if dtype == "bf16":
        # each stored bf16 probability is a correct rounding of a value within
        # the path's fp32 error (2^-17 relative: the exponential, its scaled
        # argument and the 1/Z product) of the exact probability
        exact = osamp.canvas_sample(wl.as_f64(s.logits, dtype), None, s.cfg.bound, s.cfg.seed, s.cfg.step,
                                    canvas_len=s.cfg.C)["probs"]
        bar = 0.5 * onum_spacing(exact) + 2.0 ** -17 * exact
        err = np.abs(got - exact)
        assert np.all(err <= bar), float(np.max(err - bar))
        # and equal to the oracle's own stored value away from rounding ties
        mid = np.abs(exact - ref["probs"]) < 0.5 * onum_spacing(exact) - 2.0 ** -17 * exact
        assert np.array_equal(got[mid], ref["probs"][mid])
        print(f"bf16 probabilities: {int((~mid).sum())} of {mid.size} within the fp32 error of a rounding tie")
    else:
        np.testing.assert_allclose(got, ref["probs"], rtol=1e-5, atol=1e-12)


def test_temperature_prefix_mode_and_frozen(cv):
    s = _peaked_small("bf16", rows=64, V=2048, seed=8)
    rng = np.random.default_rng(1)
    frozen = (rng.random(64) < 0.2).astype(np.uint8)
    ft = rng.integers(0, 2048, 64)
    for mode in (0, 1):
        run = SampleRun(cv, s, temperature=1.7, commit_mode=mode, frozen=frozen, frozen_tokens=ft, step=11, seed=99)
        ref = osamp.canvas_sample(wl.as_f64(s.logits, "bf16"), wl.as_f64(s.E, "bf16"), s.cfg.bound, 99, 11,
                                  temperature=1.7, commit_mode=mode, canvas_len=16, frozen=frozen,
                                  frozen_tokens=ft, probs_storage="bf16")
        compare(cv, s, run, ref)


@pytest.mark.parametrize("V", [4096, 262136])
def test_deferred_and_cluster_paths_agree(cv, V):
    """Without probs_out a bf16 call normalises each vocabulary range after the
    soft-embedding product; with probs_out the cluster kernel writes the
    probabilities first.  Both come from the same per-row state: entropy and
    confidence to fp32 merge-order rounding, argmax, mask and tokens exactly,
    the soft embeddings to the bf16 rounding of the probabilities."""
    s = _peaked_small("bf16", rows=48, V=V, seed=21)
    deferred = SampleRun(cv, s)
    cluster = SampleRun(cv, s, probs_dtype="bf16")
    np.testing.assert_array_equal(deferred.amax.cpu().numpy(), cluster.amax.cpu().numpy())
    np.testing.assert_array_equal(deferred.mask.cpu().numpy(), cluster.mask.cpu().numpy())
    np.testing.assert_array_equal(deferred.tokens.cpu().numpy(), cluster.tokens.cpu().numpy())
    np.testing.assert_allclose(deferred.ent.cpu().numpy(), cluster.ent.cpu().numpy(), rtol=1e-5, atol=1e-6)
    np.testing.assert_allclose(deferred.conf.cpu().numpy(), cluster.conf.cpu().numpy(), rtol=1e-5, atol=1e-9)
    a = deferred.soft.cpu().numpy().astype(np.float64)
    b = cluster.soft.cpu().numpy().astype(np.float64)
    assert np.isfinite(a).all()
    rf = np.linalg.norm(a - b) / np.linalg.norm(b)
    assert rf <= 2e-3, rf


def test_renoise_tokens_independent_of_launch_shape(cv):
    # the same rows sampled as part of a larger batch get the same renoise draws
    s = _peaked_small("bf16", rows=32, V=1024, seed=4)
    run = SampleRun(cv, s)
    s2 = wl.SampleInputs(cfg=wl.replace(s.cfg, rows=16), logits=s.logits[:16], E=s.E, peaked=s.peaked[:16])
    run2 = SampleRun(cv, s2)
    assert torch.equal(run.tokens[:16], run2.tokens)


def test_full_vocab_workload(cv):
    """256 positions x vocab 262144 bf16 (half peaked, half flat), E[262144 x 2816]."""
    s = wl.make_sample_inputs(wl.FULL_SAMPLE)
    c = s.cfg
    run = SampleRun(cv, s)
    runb = SampleRun(cv, s)  # repeat: bit-identical
    assert torch.equal(run.soft, runb.soft) and torch.equal(run.tokens, runb.tokens)
    logits = wl.as_f64(s.logits, "bf16")
    soft_rows = sorted(set([0, 1, 2, 100, 128, 200, 254, 255] +
                           list(np.random.default_rng(31).choice(256, 24, replace=False))))
    ref = osamp.canvas_sample(logits, None, c.bound, c.seed, c.step, canvas_len=c.C, probs_storage="bf16")
    # soft embedding of sampled rows, streaming E in fp64 chunks
    want = np.zeros((len(soft_rows), c.D))
    P = ref["probs"][soft_rows]
    for v0 in range(0, c.V, 16384):
        want += P[:, v0:v0 + 16384] @ wl.as_f64(s.E[v0:v0 + 16384], "bf16")
    soft_full = np.full((c.rows, c.D), np.nan)
    soft_full[soft_rows] = want
    ref["soft_emb"] = soft_full
    assert 0.3 < ref["commit_mask"].mean() < 0.7
    compare(cv, s, run, ref, soft_rows=soft_rows)
    # the bf16 probabilities of those rows element by element: each a correct
    # rounding of a value within the path's fp32 error of the exact one
    runp = SampleRun(cv, s, probs_dtype="bf16")
    got = runp.probs.float().cpu().numpy()[soft_rows].astype(np.float64)
    exact = osamp.canvas_sample(logits[soft_rows], None, c.bound, c.seed, c.step, canvas_len=c.C)["probs"]
    bar = 0.5 * onum_spacing(exact) + 2.0 ** -17 * exact
    assert np.all(np.abs(got - exact) <= bar), float(np.max(np.abs(got - exact) - bar))


@pytest.mark.parametrize("V", [262144, 262136])   # every slice full / a shorter last slice
def test_argmax_ties_take_the_lowest_index(cv, V):
    """Exact ties of the maximum inside one 8-logit group, across the threads
    of a CTA and across the CTAs of a row's cluster: the lowest index wins."""
    rows, D = 6, 8
    rng = np.random.default_rng(12)
    x = rng.standard_normal((rows, V)).astype(np.float32)
    ties = [[5, 3000, 70000, V - 1], [V - 9, V - 1], [17, 19, 16], [33000, 32768 + 8, 65536 * 3 + 1],
            [2048 * 3 + 7, 2048 * 3 + 6], [0, V - 1]]
    for r, idx in enumerate(ties):
        x[r, idx] = 9.0
    bits = wl.f32_to_bf16_bits(x)
    E = wl.f32_to_bf16_bits(rng.standard_normal((V, D)).astype(np.float32) * 0.02)
    cfg = wl.SampleConfig("ties", rows=rows, C=rows, V=V, D=D, dtype="bf16", seed=3, step=0, bound=0.3,
                          logits="normal", peak=0.0, gen_temperature=1.0, E_std=0.02)
    s = wl.SampleInputs(cfg=cfg, logits=bits, E=E, peaked=np.zeros(rows, bool))
    run = SampleRun(cv, s)
    got = run.amax.cpu().numpy()
    np.testing.assert_array_equal(got, [min(t) for t in ties])
    ref = osamp.canvas_sample(wl.as_f64(bits, "bf16"), wl.as_f64(E, "bf16"), 0.3, 3, 0, canvas_len=rows,
                              probs_storage="bf16")
    np.testing.assert_array_equal(got, ref["argmax"])


@pytest.mark.parametrize("mode", [2, 3])   # categorical, per position / left prefix
@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
def test_categorical_draws_match_the_oracle(cv, mode, dtype):
    """Committed positions take the inverse-CDF draw from their stored
    probabilities with the row's key uniform; bit-exact away from ties (a
    target within 1e-9 of a cumulative boundary, relative to the row total)."""
    s = _peaked_small(dtype, rows=64, V=4096, seed=23)
    if mode & 1:
        # left-prefix commits: put each canvas's peaked rows first, so the
        # qualifying runs from the left are long
        order = np.concatenate([np.argsort(~s.peaked[c:c + 16], kind="stable") + c for c in range(0, 64, 16)])
        s = wl.SampleInputs(cfg=s.cfg, logits=s.logits[order], E=s.E, peaked=s.peaked[order])
    rng = np.random.default_rng(2)
    frozen = (rng.random(64) < 0.15).astype(np.uint8)
    ft = rng.integers(0, 4096, 64)
    run = SampleRun(cv, s, probs_dtype=dtype, temperature=1.3, commit_mode=mode, frozen=frozen, frozen_tokens=ft,
                    step=5, seed=77)
    st = "bf16" if dtype == "bf16" else "fp64"
    ref = osamp.canvas_sample(wl.as_f64(s.logits, dtype), wl.as_f64(s.E, dtype), s.cfg.bound, 77, 5,
                              temperature=1.3, commit_mode=mode & 1, canvas_len=16, frozen=frozen, frozen_tokens=ft,
                              probs_storage=st, categorical=True)
    committed = (ref["commit_mask"] == 1) & (frozen == 0)
    assert committed.sum() >= 8
    from oracle import splitmix
    margins = np.array([osamp.categorical_margin(ref["probs"][r], splitmix.key_uniform(splitmix.renoise_key(77, 5, r)))
                        if committed[r] else 1.0 for r in range(64)])
    tie = margins < 1e-9
    print(f"categorical draws: {int(committed.sum())} committed rows, {int(tie.sum())} within 1e-9 of a boundary")
    ok = ~tie & (np.abs(ref["entropy"] - s.cfg.bound) > TIE)
    np.testing.assert_array_equal(run.tokens.cpu().numpy()[ok], ref["tokens"][ok])
    # the draws are not all the argmax: the categorical path really ran
    flat_committed = committed & (ref["tokens"] != ref["argmax"])
    assert flat_committed.sum() == (committed & (run.tokens.cpu().numpy() != ref["argmax"])).sum()


def test_count_committed_matches_the_mask(cv):
    rng = np.random.default_rng(8)
    for rows, C in ((1024, 256), (64, 16), (33, 33)):
        m = (rng.random(rows) < 0.6).astype(np.uint8)
        mask = torch.from_numpy(m).cuda()
        counts = torch.full((rows // C,), -1, dtype=torch.int32, device="cuda")
        cv.canvas_count_committed(mask, C, counts)
        assert cv.canvas_device_status() == cv.CANVAS_OK
        np.testing.assert_array_equal(counts.cpu().numpy(), m.reshape(-1, C).sum(axis=1))
