"""Pins of the fp64 oracle to facts outside itself (CPU only).

Each test ties one oracle function to something the pages or mathematics fix:
a hand expansion, a closed form, an invariant, a library routine, or a
published test vector.  A plausible mistake in the oracle (dropped term, sign,
index, transposed operand, off-by-one window) fails at least one of them.
"""
import math
import os

import numpy as np
import pytest
import torch

import canvas_workloads as wl
from oracle import attention as oatt
from oracle import numerics as onum
from oracle import sampler as osamp
from oracle import splitmix as osm

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ---------------------------------------------------------------- bf16 rounding
def test_bf16_round_matches_torch_and_workload_quantiser():
    rng = np.random.default_rng(5)
    a = (rng.standard_normal(20000) * np.exp(rng.uniform(-20, 20, 20000))).astype(np.float32)
    ours = onum.bf16_round(a.astype(np.float64))
    lib = torch.from_numpy(a).to(torch.bfloat16).to(torch.float64).numpy()
    np.testing.assert_array_equal(ours, lib)
    wl_vals = wl.bf16_bits_to_f32(wl.f32_to_bf16_bits(a)).astype(np.float64)
    np.testing.assert_array_equal(wl_vals, lib)


def test_bf16_round_ties_to_even():
    # 1 + 2^-8 lies halfway between 1 and 1 + 2^-7 -> the even neighbour 1
    assert onum.bf16_round(1.0 + 2.0 ** -8) == 1.0
    # 1 + 3*2^-8 lies halfway between 1 + 2^-7 (odd) and 1 + 2^-6 (even)
    assert onum.bf16_round(1.0 + 3 * 2.0 ** -8) == 1.0 + 2.0 ** -6
    assert onum.bf16_round(-3.0) == -3.0


# ---------------------------------------------------------------- rms
def test_rms_hand_case():
    # ||(3,4)|| = 5, sqrt(d) = sqrt(2)
    got = onum.rms(np.array([3.0, 4.0]), 1.0, 0.0)
    np.testing.assert_allclose(got, [3 * math.sqrt(2) / 5, 4 * math.sqrt(2) / 5], rtol=1e-15)
    got = onum.rms(np.array([3.0, 4.0]), np.array([2.0, 0.5]), 1.0)
    np.testing.assert_allclose(got, [2 * 3 * math.sqrt(2) / 6, 0.5 * 4 * math.sqrt(2) / 6], rtol=1e-15)


def test_rms_norm_identity():
    rng = np.random.default_rng(1)
    x = rng.standard_normal((7, 64)) * 3
    g, eps = 1.7, 1e-3
    y = onum.rms(x, np.full(64, g), eps)
    nx = np.linalg.norm(x, axis=-1)
    np.testing.assert_allclose(np.linalg.norm(y, axis=-1), math.sqrt(64) * g * nx / (nx + eps), rtol=1e-13)


# ---------------------------------------------------------------- RoPE
def test_rope_frequencies_closed_form():
    np.testing.assert_allclose(onum.rope_frequencies(8, 1e4), [1.0, 0.1, 0.01, 0.001], rtol=1e-15)
    f = onum.rope_frequencies(512, 1e6, 0.25)
    assert np.count_nonzero(f) == 64 and f.shape == (256,)
    assert f[63] == pytest.approx(1e6 ** (-126 / 512), rel=1e-14) and f[64] == 0.0
    # the workload's fp32 table is the same spectrum, rounded to fp32
    np.testing.assert_allclose(wl.rope_frequencies(512, 1e6, 0.25), f, rtol=1e-7)
    np.testing.assert_allclose(wl.rope_frequencies(256, 1e4), onum.rope_frequencies(256, 1e4), rtol=1e-7)


def test_rotate_equals_complex_rotation_of_split_half_pairs():
    # an independent formulation: channel pair (t, t + d/2) as the complex
    # number x_t + i x_{t+d/2}, multiplied by exp(i * angle)
    rng = np.random.default_rng(2)
    L, d, start = 5, 12, 7
    x = rng.standard_normal((3, L, d))
    freq = rng.uniform(0.0, 2.0, d // 2)
    h = d // 2
    z = (x[..., :h] + 1j * x[..., h:]) * np.exp(1j * (np.arange(L)[:, None] + start) * freq)
    want = np.concatenate([z.real, z.imag], axis=-1)
    np.testing.assert_allclose(onum.rotate(x, freq, start), want, rtol=1e-13, atol=1e-13)


def test_rotate_hand_case_d4():
    x = np.array([[1.0, 2.0, 3.0, 4.0]])
    f = np.array([0.5, 0.25])
    a0, a1 = 3 * 0.5, 3 * 0.25      # row 0 at position start=3
    want = [math.cos(a0) * 1 - math.sin(a0) * 3, math.cos(a1) * 2 - math.sin(a1) * 4,
            math.cos(a0) * 3 + math.sin(a0) * 1, math.cos(a1) * 4 + math.sin(a1) * 2]
    np.testing.assert_allclose(onum.rotate(x, f, 3)[0], want, rtol=1e-15)


def test_rotate_invariants():
    rng = np.random.default_rng(3)
    d = 16
    f = onum.rope_frequencies(d, 1e4, 0.25)   # only 2 of 8 frequencies nonzero
    x = rng.standard_normal((1, d))
    y = onum.rotate(x, f, 123)
    # zero-frequency channels come back unchanged
    zero = np.concatenate([f, f]) == 0
    np.testing.assert_array_equal(y[0, zero], x[0, zero])
    # each (t, t + d/2) pair keeps its length
    h = d // 2
    np.testing.assert_allclose(np.hypot(y[0, :h], y[0, h:]), np.hypot(x[0, :h], x[0, h:]), rtol=1e-14)
    # relative position: <rot(q, m), rot(k, n)> depends only on m - n
    f = onum.rope_frequencies(d, 1e4)
    q, k = rng.standard_normal((1, d)), rng.standard_normal((1, d))
    s1 = onum.rotate(q, f, 10) @ onum.rotate(k, f, 3).T
    s2 = onum.rotate(q, f, 1010) @ onum.rotate(k, f, 1003).T
    np.testing.assert_allclose(s1, s2, rtol=1e-10)


def test_logit_invariant_constant_gamma():
    # with constant gamma, q.k = d * gq * gk * cos(theta) * |a|/(|a|+eps) * |b|/(|b|+eps)
    rng = np.random.default_rng(4)
    d, gq, gk, eps = 64, 1.3, 0.8, 1e-6
    a, b = rng.standard_normal(d), rng.standard_normal(d)
    q, k = onum.rms(a, np.full(d, gq), eps), onum.rms(b, np.full(d, gk), eps)
    na, nb = np.linalg.norm(a), np.linalg.norm(b)
    cos = a @ b / (na * nb)
    want = d * gq * gk * cos * (na / (na + eps)) * (nb / (nb + eps))
    assert q @ k == pytest.approx(want, rel=1e-12)
    # rotating both at the same position leaves the logit unchanged
    f = onum.rope_frequencies(d, 1e4)
    assert (onum.rotate(q[None], f, 77) @ onum.rotate(k[None], f, 77).T)[0, 0] == pytest.approx(want, rel=1e-12)


# ---------------------------------------------------------------- attention
def _small_cfg(**kw):
    base = dict(name="t", B=2, C=8, prefix=(40, 29), D=24, Hq=4, Hkv=2, d=16, layer="sliding",
                window=16, theta=1e4, rotary_fraction=1.0, dtype="fp32", seed=9, gamma_q=1.1,
                gamma_k=0.9, page_tokens=16)
    base.update(kw)
    return wl.AttnConfig(**base)


def _f64(inp, name):
    a = getattr(inp, name)
    return None if a is None else wl.as_f64(a, inp.cfg.dtype)


def _run_oracle(inp, storage="fp64", **kw):
    c = inp.cfg
    return oatt.canvas_attention(_f64(inp, "x"), _f64(inp, "W_q"), _f64(inp, "W_k"), _f64(inp, "W_v"),
                                 c.Hq, c.Hkv, c.d, inp.gamma_q, inp.gamma_k, c.eps, inp.freq, c.layer,
                                 _f64(inp, "cache_k"), _f64(inp, "cache_v"), inp.prefix_len, c.window,
                                 storage=storage, **kw)


def test_visible_pair_counts_match_workload_closed_forms():
    # sliding workload: sum_i (1024 - i) + 256 * 256 = 295040 pairs per head
    assert oatt.visible_pairs(256, 4096, 1024, "sliding") == 295040
    assert oatt.visible_pairs(256, 32768, 0, "global") == 256 * 33024


@pytest.mark.parametrize("layer", ["sliding", "global"])
def test_uniform_attention_pins_the_visible_key_set(layer):
    # gamma_q -> 0 makes every score 0: each output is the plain mean of the
    # visible value rows.  Value rows carry (position, 1) in channels 0, 1 and
    # the canvas values are 0 (W_v = 0 / canvas r = 0), so channel 0 gives the
    # sum of visible prefix positions and channel 1 their count, over n + C.
    cfg = _small_cfg(layer=layer, gamma_q=1e-30, window=16 if layer == "sliding" else 0)
    inp = wl.make_attention_inputs(cfg)
    P = cfg.max_prefix
    ck = np.zeros((cfg.B, cfg.Hkv, P, cfg.d))
    ck[..., 0] = np.arange(P)
    ck[..., 1] = 1.0
    x = _f64(inp, "x")
    Wk = _f64(inp, "W_k")
    if layer == "global":
        Wk = np.zeros_like(Wk)      # canvas raw r = 0 -> canvas values 0
        cache_v, Wv = None, None
    else:
        cache_v, Wv = ck, np.zeros_like(_f64(inp, "W_v"))
        ck = np.random.default_rng(0).standard_normal(ck.shape)   # keys do not matter
    out, _ = oatt.canvas_attention(x, _f64(inp, "W_q"), Wk, Wv, cfg.Hq, cfg.Hkv, cfg.d, inp.gamma_q,
                                   inp.gamma_k, cfg.eps, inp.freq, layer, ck if layer == "global" else ck,
                                   cache_v, inp.prefix_len, cfg.window)
    if layer == "global":
        # global values are the raw rows: channel 0 = position, channel 1 = 1
        pass
    for b in range(cfg.B):
        Pb = int(inp.prefix_len[b])
        for i in range(cfg.C):
            lo = max(0, Pb + i - cfg.window) if (layer == "sliding" and cfg.window > 0) else 0
            n = Pb - lo
            for h in range(cfg.Hq):
                o = out[b, i, h * cfg.d:(h + 1) * cfg.d]
                assert o[1] == pytest.approx(n / (n + cfg.C), abs=1e-12)
                assert o[0] == pytest.approx(sum(range(lo, Pb)) / (n + cfg.C), rel=1e-12, abs=1e-12)


def test_single_key_returns_its_value_row_and_gqa_mapping():
    # empty prefix and a one-token canvas: each query head sees exactly one key,
    # so its output is the value row of KV head floor(h / G) -- the projection
    # x W_v^T sliced by head.
    cfg = _small_cfg(B=1, C=1, prefix=(0,), Hq=6, Hkv=2)
    inp = wl.make_attention_inputs(cfg)
    out, lse = _run_oracle(inp)
    v = _f64(inp, "x")[0, 0] @ _f64(inp, "W_v").T
    for h in range(6):
        hk = h // 3
        np.testing.assert_allclose(out[0, 0, h * 16:(h + 1) * 16], v[hk * 16:(hk + 1) * 16], rtol=1e-13)


def _sdpa_reference(inp, scale=1.0, v_unit_rms=False, with_lse=False, causal=False):
    """The attention core through torch's scaled_dot_product_attention (fp64)
    with an explicit boolean mask, fed with q/k/v assembled from the pinned
    rms / rotate building blocks; the natural-log softmax normaliser of each
    row from scipy's logsumexp over the same masked scores."""
    from scipy.special import logsumexp
    c = inp.cfg
    lses = []
    x, Wq, Wk = _f64(inp, "x"), _f64(inp, "W_q"), _f64(inp, "W_k")
    Wv = _f64(inp, "W_v")
    outs = []
    for b in range(c.B):
        P = int(inp.prefix_len[b])
        q = (x[b] @ Wq.T).reshape(c.C, c.Hq, c.d).transpose(1, 0, 2)
        k = (x[b] @ Wk.T).reshape(c.C, c.Hkv, c.d).transpose(1, 0, 2)
        v = k if Wv is None else (x[b] @ Wv.T).reshape(c.C, c.Hkv, c.d).transpose(1, 0, 2)
        q = onum.rotate(onum.rms(q, inp.gamma_q, c.eps), inp.freq, P)
        if c.layer == "sliding":
            K = np.concatenate([_f64(inp, "cache_k")[b, :, :P], onum.rotate(onum.rms(k, inp.gamma_k, c.eps), inp.freq, P)], 1)
            Vv = np.concatenate([_f64(inp, "cache_v")[b, :, :P], v], 1)
        else:
            r = np.concatenate([_f64(inp, "cache_k")[b, :, :P], k], 1)
            K = onum.rotate(onum.rms(r, inp.gamma_k, c.eps), inp.freq, 0)
            Vv = r
            if v_unit_rms:   # sqrt(d) r / (|r| + eps), no weight
                Vv = math.sqrt(c.d) * r / (np.linalg.norm(r, axis=-1, keepdims=True) + c.eps)
        mask = np.ones((c.C, P + c.C), bool)
        if c.layer == "sliding" and c.window > 0:
            for i in range(c.C):
                mask[i, :max(0, P + i - c.window)] = False
        if causal:   # encode mode: canvas row i sees canvas keys 0..i
            for i in range(c.C):
                mask[i, P + i + 1:] = False
        G = c.Hq // c.Hkv
        Kq = np.repeat(K, G, axis=0)
        Vq = np.repeat(Vv, G, axis=0)
        o = torch.nn.functional.scaled_dot_product_attention(
            torch.from_numpy(q), torch.from_numpy(Kq), torch.from_numpy(Vq),
            attn_mask=torch.from_numpy(mask), scale=scale).numpy()
        outs.append(o.transpose(1, 0, 2).reshape(c.C, c.Hq * c.d))
        sc = np.einsum("hid,hjd->hij", q, Kq) * scale
        lses.append(logsumexp(np.where(mask[None], sc, -np.inf), axis=-1).T)   # [C, Hq]
    if with_lse:
        return np.stack(outs), np.stack(lses)
    return np.stack(outs)


@pytest.mark.parametrize("layer,window,rot", [("sliding", 16, 1.0), ("sliding", 0, 1.0), ("global", 0, 0.25)])
def test_attention_matches_library_sdpa(layer, window, rot):
    cfg = _small_cfg(layer=layer, window=window, rotary_fraction=rot, gamma_q=None, gamma_k=None,
                     theta=1e6 if layer == "global" else 1e4)
    inp = wl.make_attention_inputs(cfg)
    out, _ = _run_oracle(inp)
    np.testing.assert_allclose(out, _sdpa_reference(inp), rtol=1e-10, atol=1e-12)


@pytest.mark.parametrize("layer,scale,unit", [("sliding", 0.37, False), ("global", 1.0, True), ("global", 2.5, True)])
def test_scale_unit_rms_values_and_lse_match_library_sdpa(layer, scale, unit):
    """The softmax scale argument, the unit-RMS value variant of global layers
    and the natural-log normaliser the oracle returns, against the library
    path (SDPA) and scipy's logsumexp."""
    cfg = _small_cfg(layer=layer, window=16 if layer == "sliding" else 0, gamma_q=None, gamma_k=None,
                     rotary_fraction=0.25 if layer == "global" else 1.0, theta=1e6 if layer == "global" else 1e4)
    inp = wl.make_attention_inputs(cfg)
    out, lse = _run_oracle(inp, scale=scale, v_unit_rms=unit)
    want, want_lse = _sdpa_reference(inp, scale=scale, v_unit_rms=unit, with_lse=True)
    np.testing.assert_allclose(out, want, rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(lse, want_lse, rtol=1e-12, atol=1e-12)
    if unit:   # the variant changes the result
        assert np.max(np.abs(out - _run_oracle(inp, scale=scale)[0])) > 1e-3


def test_global_storage_model_decomposition():
    # rotate(rms(r, g)) == g * sqrt(d)/(|r|+eps) * rotate(r) for constant g; the
    # bf16 storage model only inserts a rounding of rotate(r)
    rng = np.random.default_rng(6)
    d, eps, g = 32, 1e-6, 1.7
    r = rng.standard_normal((9, d))
    f = onum.rope_frequencies(d, 1e6, 0.25)
    lhs = onum.rotate(onum.rms(r, np.full(d, g), eps), f, 5)
    s = math.sqrt(d) / (np.linalg.norm(r, axis=-1, keepdims=True) + eps)
    np.testing.assert_allclose(lhs, g * s * onum.rotate(r, f, 5), rtol=1e-13)
    # and the two storage modes of the full layer agree to bf16 rounding level
    cfg = _small_cfg(layer="global", window=0, rotary_fraction=0.25, theta=1e6, dtype="bf16")
    inp = wl.make_attention_inputs(cfg)
    a, _ = _run_oracle(inp, "fp64")
    b, _ = _run_oracle(inp, "bf16")
    assert np.max(np.abs(a - b)) < 0.05 and np.max(np.abs(a - b)) > 0


def test_attention_row_subset_matches_full():
    cfg = _small_cfg()
    inp = wl.make_attention_inputs(cfg)
    full, lse = _run_oracle(inp)
    rows = [(0, 1, 3), (1, 3, 7)]
    part, lse_p = _run_oracle(inp, rows=rows)
    for (b, h, i) in rows:
        np.testing.assert_array_equal(part[b, i, h * 16:(h + 1) * 16], full[b, i, h * 16:(h + 1) * 16])
        assert lse_p[b, i, h] == lse[b, i, h]
    assert np.isnan(part[0, 0, 0])


# ---------------------------------------------------------------- sampler
def test_entropy_extremes_and_two_level_closed_form():
    V = 512
    p, H, a, c = osamp.row_statistics(np.zeros(V))
    assert H == pytest.approx(math.log(V), rel=1e-14) and a == 0 and c == pytest.approx(1 / V)
    row = np.full(V, -1000.0)
    row[17] = 0.0
    p, H, a, c = osamp.row_statistics(row)
    assert H == 0.0 and a == 17 and c == 1.0
    # one logit A, n = V-1 logits Bv
    A, Bv, n = 3.0, -0.5, V - 1
    row = np.full(V, Bv)
    row[100] = A
    p1 = math.exp(A) / (math.exp(A) + n * math.exp(Bv))
    q = math.exp(Bv) / (math.exp(A) + n * math.exp(Bv))
    p, H, a, c = osamp.row_statistics(row)
    assert H == pytest.approx(-p1 * math.log(p1) - n * q * math.log(q), rel=1e-13)
    assert a == 100 and c == pytest.approx(p1, rel=1e-14)
    # temperature 2 on logits 2*row is the same distribution
    _, H2, _, _ = osamp.row_statistics(2 * row, temperature=2.0)
    assert H2 == pytest.approx(H, rel=1e-13)


def test_argmax_lowest_index_on_ties():
    row = np.zeros(64)
    row[[5, 9, 40]] = 2.0
    assert osamp.row_statistics(row)[2] == 5


def test_commit_renoise_rule_and_soft_embedding_closed_forms():
    V, D, C = 64, 8, 4
    rng = np.random.default_rng(8)
    E = rng.standard_normal((V, D))
    logits = np.zeros((8, V))              # uniform rows: H = ln 64 = 4.16
    logits[1, 7] = 1e4                     # one-hot rows: H = 0
    logits[2, 3] = 1e4
    logits[6, 60] = 1e4
    res = osamp.canvas_sample(logits, E, entropy_bound=0.5, seed=42, step=3, canvas_len=C)
    np.testing.assert_array_equal(res["commit_mask"], [0, 1, 1, 0, 0, 0, 1, 0])
    for r in range(8):
        if res["commit_mask"][r]:
            assert res["tokens"][r] == res["argmax"][r]
        else:
            assert res["tokens"][r] == osm.renoise_key(42, 3, r) % V
    # one-hot P gives the E row exactly; uniform P gives the column means
    np.testing.assert_array_equal(res["soft_emb"][1], E[7])
    np.testing.assert_allclose(res["soft_emb"][0], E.mean(axis=0), rtol=1e-12, atol=1e-14)
    # left-prefix mode: canvas 0 = rows 0..3 -> row 0 fails -> nothing committed;
    # canvas 1 = rows 4..7 -> rows 4,5 fail -> nothing; make row 4 frozen
    frozen = np.zeros(8, np.uint8)
    frozen[4] = 1
    ft = np.full(8, -1)
    ft[4] = 11
    res = osamp.canvas_sample(logits, E, 0.5, 42, 3, commit_mode=1, canvas_len=C, frozen=frozen,
                              frozen_tokens=ft)
    np.testing.assert_array_equal(res["commit_mask"], [0, 0, 0, 0, 1, 0, 0, 0])
    assert res["tokens"][4] == 11
    logits[5, 1] = 1e4
    res = osamp.canvas_sample(logits, E, 0.5, 42, 3, commit_mode=1, canvas_len=C, frozen=frozen,
                              frozen_tokens=ft)
    np.testing.assert_array_equal(res["commit_mask"], [0, 0, 0, 0, 1, 1, 1, 0])
    # strict bound: H equal to the bound does not commit
    res = osamp.canvas_sample(np.zeros((1, V)), None, math.log(V), 0, 0)
    assert res["commit_mask"][0] == 0


# ---------------------------------------------------------------- splitmix64
def test_splitmix64_published_vectors():
    with open(os.path.join(GOLDEN, "splitmix64_vectors.txt")) as fh:
        lines = [ln.split() for ln in fh if ln.strip() and not ln.startswith("#")]
    for ln in lines:
        seed, kind, n = int(ln[1]), ln[2], int(ln[3].rstrip(":"))
        vals = [int(v) for v in ln[4:]]
        if kind == "first":
            assert osm.stream(seed, n) == vals
        else:
            bins = [0] * 5
            for z in osm.stream(seed, n):
                bins[(z * 5) >> 64] += 1
            assert bins == vals


def test_renoise_key_composition():
    # key = mix(mix(mix(seed) ^ step) ^ row), mix = one SplitMix64 output
    s0 = osm.stream(7, 1)[0]
    s1 = osm.stream(s0 ^ 3, 1)[0]
    s2 = osm.stream(s1 ^ 129, 1)[0]
    assert osm.renoise_key(7, 3, 129) == s2
    assert osm.renoise_token(7, 3, 129, 262144) == s2 & (262144 - 1)


# ---------------------------------------------------------------- bf16 rounding slack
def test_rounding_flips_hand_cases():
    # 1 + 2^-8 + tiny lies just above the midpoint of 1 and 1 + 2^-7: it rounds
    # up, and the other neighbour 1 is one ulp below
    x = np.array([[1.0 + 2.0 ** -8 + 2.0 ** -20, 1.0 + 2.0 ** -9, 1.5, -1.0 - 2.0 ** -8 - 2.0 ** -20]])
    partner = np.zeros_like(x)
    stored, delta = oatt.rounding_flips(x, partner, 2.0 ** -16)
    np.testing.assert_array_equal(stored, onum.bf16_round(x))
    assert stored[0, 0] == 1.0 + 2.0 ** -7 and delta[0, 0] == -(2.0 ** -7)
    assert delta[0, 1] == 0.0          # a quarter ulp from the nearest value: far from any midpoint
    assert delta[0, 2] == 0.0          # exactly representable
    assert stored[0, 3] == -1.0 - 2.0 ** -7 and delta[0, 3] == 2.0 ** -7
    # a window too small to reach the midpoint flags nothing
    _, d0 = oatt.rounding_flips(x, partner, 2.0 ** -30)
    assert not d0.any()


@pytest.mark.parametrize("layer", ["sliding", "global"])
def test_rounding_slack_bounds_every_flip_combination(layer):
    # Nudging the inputs by a relative 1e-5 moves every pre-rounding value far
    # less than the ambiguity window (2^-12 of the row scale), so each perturbed
    # run flips some subset of the flagged roundings and nothing else: its
    # output must stay within the slack of the nominal run (plus the ~1e-5
    # continuous change of the nudge).
    cfg = _small_cfg(B=1, C=24, prefix=(90,), D=48, Hq=4, Hkv=2, d=32, window=40, dtype="bf16", gamma_q=2.0,
                     gamma_k=2.0, seed=13, layer=layer, theta=1e4 if layer == "sliding" else 1e6,
                     rotary_fraction=1.0 if layer == "sliding" else 0.25)
    inp = wl.make_attention_inputs(cfg)
    ref, _, slack = _run_oracle(inp, "bf16", slack_eps=2.0 ** -12)
    assert np.all(slack >= 0) and slack.max() > 0
    rng = np.random.default_rng(0)
    moved = 0.0
    for _ in range(6):
        x = _f64(inp, "x") * (1.0 + 1e-5 * rng.standard_normal(_f64(inp, "x").shape))
        c = inp.cfg
        alt, _ = oatt.canvas_attention(x, _f64(inp, "W_q"), _f64(inp, "W_k"), _f64(inp, "W_v"), c.Hq, c.Hkv, c.d,
                                       inp.gamma_q, inp.gamma_k, c.eps, inp.freq, c.layer, _f64(inp, "cache_k"),
                                       _f64(inp, "cache_v"), inp.prefix_len, c.window, storage="bf16")
        d = np.abs(alt - ref)
        assert np.all(d <= slack + 1e-4), float(np.max(d - slack))
        moved = max(moved, float(d.max()))
    assert moved > 1e-3   # some ambiguous rounding did flip: the check is not vacuous


def test_rounding_slack_is_zero_without_bf16_storage():
    cfg = _small_cfg()
    inp = wl.make_attention_inputs(cfg)
    out = _run_oracle(inp, "fp64", slack_eps=2.0 ** -14)
    assert len(out) == 2   # fp64 storage has no rounding decisions to bound


@pytest.mark.parametrize("which", ["q", "k", "v"])
def test_row_slack_bounds_brute_force_flips(which):
    # One query row, 5 keys, d = 4; ambiguous elements only in q, only in the
    # keys, or only in the values.  Enumerate every combination of flips and
    # evaluate the softmax output exactly: the largest change must stay within
    # the bound, and the bound must not be vacuous (it moves when flips do).
    rng = np.random.default_rng(7)
    d, n = 4, 5
    q = rng.standard_normal(d) * 3
    keys = rng.standard_normal((n, d)) * 2
    vals = rng.standard_normal((n, d))
    dq, dk, dv = np.zeros(d), np.zeros((n, d)), np.zeros((n, d))
    flips = [(0,), (2,)] if which == "q" else [(1, 0), (3, 2), (4, 1)]
    target = {"q": dq, "k": dk, "v": dv}[which]
    for idx in flips:
        target[idx] = 0.05 * (1 if len(idx) % 2 else -1)

    def out(qq, kk, vv):
        s = kk @ qq
        e = np.exp(s - s.max())
        return (e / e.sum()) @ vv

    base = out(q, keys, vals)
    s = keys @ q
    p = np.exp(s - s.max())
    p /= p.sum()
    bound = oatt._row_slack(q, dq, np.abs(keys) + np.abs(dk), np.abs(dk), vals, np.abs(dv), p, base, 1.0)
    worst = np.zeros(d)
    import itertools
    for mask in itertools.product([0, 1], repeat=len(flips)):
        qq, kk, vv = q.copy(), keys.copy(), vals.copy()
        t = {"q": qq, "k": kk, "v": vv}[which]
        for m_, idx in zip(mask, flips):
            if m_:
                t[idx] += target[idx]
        worst = np.maximum(worst, np.abs(out(qq, kk, vv) - base))
    assert np.all(worst <= bound + 1e-15), (worst, bound)
    assert np.all(bound <= 50 * worst + 1e-12)


# ---------------------------------------------------------------- the loop step
def _tiny_loop(seed=5):
    """Two layers (sliding with a window, global with W_v = W_k), D != Hq*d
    so that a transposed W_o cannot pass."""
    rng = np.random.default_rng(seed)
    B, C, D, P, V = 2, 3, 6, 5, 16
    Hq, Hkv, d = 2, 1, 4
    layers = []
    for k, (kind, window) in enumerate((("sliding", 2), ("global", 0))):
        L = dict(W_q=onum.bf16_round(rng.normal(size=(Hq * d, D)) / 2),
                 W_k=onum.bf16_round(rng.normal(size=(Hkv * d, D)) / 2),
                 W_v=onum.bf16_round(rng.normal(size=(Hkv * d, D)) / 2) if kind == "sliding" else None,
                 W_o=onum.bf16_round(rng.normal(size=(D, Hq * d))),
                 gamma_q=np.full(d, 1.1), gamma_k=np.full(d, 0.7), freq=onum.rope_frequencies(d, 1e4),
                 eps=1e-6, Hq=Hq, Hkv=Hkv, d=d, layer=kind, window=window, prefix=P,
                 cache_k=onum.bf16_round(rng.normal(size=(B, Hkv, P, d))),
                 cache_v=onum.bf16_round(rng.normal(size=(B, Hkv, P, d))) if kind == "sliding" else None)
        layers.append(L)
    E = onum.bf16_round(rng.normal(size=(V, D)))
    tokens = rng.integers(0, V, size=B * C)
    soft_prev = rng.normal(size=(B * C, D)) * 0.1
    return layers, E, tokens, soft_prev, B, C, D, V


def test_loop_step_glue_brute_force():
    """oracle.loop.loop_step against the step written out element by element:
    input = E[token] + soft_emb of the previous step; per layer the residual
    gains bf16(attention) times W_o^T; logits = bf16(bf16(x) E^T); the
    sampler's commit / renoise rule with each row's own index; soft_emb =
    bf16(p) E.  The attention layer itself is the oracle's (pinned above)."""
    from oracle import loop as oloop
    layers, E, tokens, soft_prev, B, C, D, V = _tiny_loop()
    R = B * C
    step, seed = 3, 9
    # residual stream and logits by explicit loops
    x = np.zeros((R, D))
    for r in range(R):
        for j in range(D):
            x[r, j] = E[tokens[r], j] + soft_prev[r, j]
    xs = [x.copy()]
    attn = []
    for L in layers:
        out = oatt.canvas_attention(onum.bf16_round(x).reshape(B, C, D), L["W_q"], L["W_k"], L["W_v"], L["Hq"],
                                    L["Hkv"], L["d"], L["gamma_q"], L["gamma_k"], L["eps"], L["freq"], L["layer"],
                                    L["cache_k"], L["cache_v"], np.full(B, L["prefix"]), L["window"],
                                    storage="bf16")[0]
        ob = onum.bf16_round(out).reshape(R, -1)
        attn.append(ob)
        nxt = x.copy()
        for r in range(R):
            for j in range(D):
                nxt[r, j] += sum(ob[r, c] * L["W_o"][j, c] for c in range(ob.shape[1]))
        x = nxt
        xs.append(x.copy())
    xb = onum.bf16_round(x)
    logits = np.zeros((R, V))
    for r in range(R):
        for v in range(V):
            logits[r, v] = sum(xb[r, j] * E[v, j] for j in range(D))
    logits = onum.bf16_round(logits)
    H = np.array([-sum(p * math.log(p) for p in np.exp(lg - lg.max()) / np.exp(lg - lg.max()).sum() if p > 0)
                  for lg in logits])
    bound = float(np.median(H))   # both branches of the rule
    ref = oloop.loop_step(layers, E, tokens, soft_prev, step, B, C, seed, bound)
    for k in range(len(layers) + 1):
        np.testing.assert_allclose(ref["xs"][k], xs[k], rtol=1e-12, atol=1e-12)
    for k in range(len(layers)):
        np.testing.assert_array_equal(ref["attn"][k].reshape(R, -1), attn[k])
    np.testing.assert_array_equal(ref["logits"], logits)
    np.testing.assert_allclose(ref["entropy"], H, rtol=1e-10)
    committed = 0
    for r in range(R):
        if H[r] < bound:
            committed += 1
            assert ref["commit_mask"][r] == 1 and ref["tokens"][r] == int(np.argmax(logits[r]))
        else:
            assert ref["commit_mask"][r] == 0
            assert ref["tokens"][r] == osm.renoise_token(seed, step, r, V)
        p = onum.bf16_round(np.exp(logits[r] - logits[r].max()) / np.exp(logits[r] - logits[r].max()).sum())
        want = [sum(p[v] * E[v, j] for v in range(V)) for j in range(D)]
        np.testing.assert_allclose(ref["soft_emb"][r], want, rtol=1e-12, atol=1e-14)
    assert 0 < committed < R


def test_loop_step_row_subset_keeps_global_row_keys():
    """Evaluating the sampler on a subset of rows gives those rows' full-step
    results, including renoise draws keyed by the global row index; frozen rows
    keep their tokens."""
    from oracle import loop as oloop
    layers, E, tokens, soft_prev, B, C, D, V = _tiny_loop(seed=8)
    R = B * C
    frozen = np.zeros(R, np.uint8)
    frozen[[1, 4]] = 1
    ftok = np.arange(R) + 3
    full = oloop.loop_step(layers, E, tokens, soft_prev, 2, B, C, 11, 0.5, frozen, ftok)
    rows = [4, 1, 5]
    sub = oloop.loop_step(layers, E, tokens, soft_prev, 2, B, C, 11, 0.5, frozen, ftok, sample_rows=rows)
    sel = sorted(rows)
    np.testing.assert_array_equal(sub["rows"], sel)
    for key in ("tokens", "commit_mask"):
        np.testing.assert_array_equal(sub[key], full[key][sel])
    np.testing.assert_allclose(sub["entropy"], full["entropy"][sel], rtol=0, atol=0)
    np.testing.assert_allclose(sub["soft_emb"], full["soft_emb"][sel], rtol=1e-15, atol=0)
    assert full["tokens"][1] == 4 and full["tokens"][4] == 7 and full["commit_mask"][[1, 4]].all()


# ---------------------------------------------------------------- encode mode and block commit
@pytest.mark.parametrize("layer,window", [("sliding", 16), ("sliding", 0), ("global", 0)])
def test_encode_mode_matches_library_sdpa_with_a_causal_mask(layer, window):
    cfg = _small_cfg(layer=layer, window=window, rotary_fraction=1.0 if layer == "sliding" else 0.25,
                     gamma_q=None, gamma_k=None, theta=1e6 if layer == "global" else 1e4)
    inp = wl.make_attention_inputs(cfg)
    out, _ = _run_oracle(inp, causal=True)
    np.testing.assert_allclose(out, _sdpa_reference(inp, causal=True), rtol=1e-10, atol=1e-12)
    # the last canvas row sees the whole block in both modes
    dec, _ = _run_oracle(inp)
    np.testing.assert_allclose(out[:, -1], dec[:, -1], rtol=1e-12, atol=1e-14)
    assert not np.allclose(out[:, 0], dec[:, 0])


@pytest.mark.parametrize("layer", ["sliding", "global"])
def test_encode_row_equals_decode_of_the_truncated_block(layer):
    # row i of the causal pass = row i of a decode pass over rows 0..i only
    cfg = _small_cfg(layer=layer, window=16 if layer == "sliding" else 0, C=6,
                     rotary_fraction=1.0 if layer == "sliding" else 0.25, theta=1e6 if layer == "global" else 1e4)
    inp = wl.make_attention_inputs(cfg)
    enc, enc_lse = _run_oracle(inp, causal=True)
    c = cfg
    for i in (0, 2, 5):
        x = _f64(inp, "x")[:, :i + 1]
        dec, dec_lse = oatt.canvas_attention(x, _f64(inp, "W_q"), _f64(inp, "W_k"), _f64(inp, "W_v"), c.Hq, c.Hkv,
                                             c.d, inp.gamma_q, inp.gamma_k, c.eps, inp.freq, c.layer,
                                             _f64(inp, "cache_k"), _f64(inp, "cache_v"), inp.prefix_len, c.window)
        np.testing.assert_allclose(enc[:, i], dec[:, i], rtol=1e-12, atol=1e-14)
        np.testing.assert_allclose(enc_lse[:, i], dec_lse[:, i], rtol=1e-12)


def _appended_cache(inp, rows_k, rows_v):
    """Caches [B, Hkv, P+C, d] holding each sequence's prefix then its appended block."""
    c = inp.cfg
    B, Hkv, C, d = rows_k.shape
    P = inp.prefix_len
    ck = np.full((B, Hkv, int(P.max()) + C, d), np.nan)
    cv = None if rows_v is None else np.full_like(ck, np.nan)
    for b in range(B):
        ck[b, :, :P[b]] = _f64(inp, "cache_k")[b, :, :P[b]]
        ck[b, :, P[b]:P[b] + C] = rows_k[b]
        if cv is not None:
            cv[b, :, :P[b]] = _f64(inp, "cache_v")[b, :, :P[b]]
            cv[b, :, P[b]:P[b] + C] = rows_v[b]
    return ck, cv


@pytest.mark.parametrize("layer", ["sliding", "global"])
def test_appended_block_is_what_a_later_token_sees(layer):
    # commit a block of C rows, then decode one more token over prefix P + C:
    # the same as decoding a canvas of C + 1 rows (block + token) at its last
    # row, where the block rows are canvas keys at the same positions
    cfg = _small_cfg(layer=layer, window=0, C=7, rotary_fraction=1.0 if layer == "sliding" else 0.25,
                     theta=1e6 if layer == "global" else 1e4)
    inp = wl.make_attention_inputs(cfg)
    c = cfg
    x = _f64(inp, "x")
    blk, tok = x[:, :-1], x[:, -1:]
    res = oatt.kv_append(blk, _f64(inp, "W_k"), _f64(inp, "W_v"), c.Hkv, c.d, inp.gamma_k, c.eps, inp.freq, c.layer,
                         inp.prefix_len, storage="fp64")
    ck, cv = _appended_cache(inp, res[0], res[1])
    nxt, _ = oatt.canvas_attention(tok, _f64(inp, "W_q"), _f64(inp, "W_k"), _f64(inp, "W_v"), c.Hq, c.Hkv, c.d,
                                   inp.gamma_q, inp.gamma_k, c.eps, inp.freq, c.layer, ck, cv,
                                   inp.prefix_len + blk.shape[1], c.window)
    full, _ = _run_oracle(inp)
    np.testing.assert_allclose(nxt[:, 0], full[:, -1], rtol=1e-11, atol=1e-13)
    # bf16 storage rounds the rows once; the flags mark rounding ties only
    k16, v16, dk, dv = oatt.kv_append(blk, _f64(inp, "W_k"), _f64(inp, "W_v"), c.Hkv, c.d, inp.gamma_k, c.eps,
                                      inp.freq, c.layer, inp.prefix_len, storage="bf16", slack_eps=2.0 ** -12)
    np.testing.assert_array_equal(k16, onum.bf16_round(res[0]))
    assert np.all((dk == 0) | (np.abs(dk) <= np.abs(k16) * 2.0 ** -7 + 1e-300))


@pytest.mark.parametrize("layer", ["sliding", "global"])
def test_slack_of_tie_rounded_cache_rows_bounds_their_flips(layer):
    # rows appended with rounding ties: every subset of the alternative
    # roundings moves the next canvas's output within the slack the oracle
    # computes from cache_dk / cache_dv
    cfg = _small_cfg(B=1, C=10, prefix=(60,), D=48, Hq=4, Hkv=2, d=32, window=0, dtype="bf16", gamma_q=2.0,
                     gamma_k=2.0, seed=17, layer=layer, theta=1e4 if layer == "sliding" else 1e6,
                     rotary_fraction=1.0 if layer == "sliding" else 0.25)
    inp = wl.make_attention_inputs(cfg)
    c = cfg
    x = _f64(inp, "x")
    blk, nxt_x = x[:, :6], x[:, 6:]
    k16, v16, dk, dv = oatt.kv_append(blk, _f64(inp, "W_k"), _f64(inp, "W_v"), c.Hkv, c.d, inp.gamma_k, c.eps,
                                      inp.freq, c.layer, inp.prefix_len, storage="bf16", slack_eps=2.0 ** -10)
    assert np.count_nonzero(dk) > 0
    ck, cv = _appended_cache(inp, k16, v16)
    dck = np.zeros_like(ck)
    dck[:, :, 60:66] = dk
    dcv = None
    if cv is not None:
        dcv = np.zeros_like(cv)
        dcv[:, :, 60:66] = dv
    args = (nxt_x, _f64(inp, "W_q"), _f64(inp, "W_k"), _f64(inp, "W_v"), c.Hq, c.Hkv, c.d, inp.gamma_q, inp.gamma_k,
            c.eps, inp.freq, c.layer)
    P2 = inp.prefix_len + 6
    ref, _, slack = oatt.canvas_attention(*args, ck, cv, P2, c.window, storage="bf16", slack_eps=2.0 ** -30,
                                          cache_dk=dck, cache_dv=dcv)
    ref0, _, slack0 = oatt.canvas_attention(*args, ck, cv, P2, c.window, storage="bf16", slack_eps=2.0 ** -30)
    assert np.all(slack >= slack0) and np.max(slack - slack0) > 0
    rng = np.random.default_rng(3)
    worst = 0.0
    for _ in range(8):
        mk = rng.random(dck.shape) < 0.5
        ck2 = ck + np.where(mk, dck, 0.0)
        cv2 = None if cv is None else cv + np.where(rng.random(dcv.shape) < 0.5, dcv, 0.0)
        alt, _ = oatt.canvas_attention(*args, ck2, cv2, P2, c.window, storage="bf16")
        d = np.abs(alt - ref)
        assert np.all(d <= slack + 1e-12), float(np.max(d - slack))
        worst = max(worst, float(d.max()))
    assert worst > 0


# ---------------------------------------------------------------- sampler variants
def test_temperature_schedule_closed_form():
    S, hi, lo = 48, 1.5, 0.25
    ts = [osamp.temperature_schedule(s, S, hi, lo) for s in range(S)]
    assert ts[0] == hi and ts[-1] == lo
    assert all(a > b for a, b in zip(ts, ts[1:]))                       # strictly falling
    np.testing.assert_allclose(np.diff(ts), (lo - hi) / (S - 1), rtol=1e-12)   # equal steps
    assert osamp.temperature_schedule(0, 1, hi, lo) == hi
    assert osamp.temperature_schedule(2, 5, 2.0, 1.0) == 1.5             # midpoint by hand


def test_categorical_token_is_the_inverse_cdf_by_hand():
    p = np.array([0.0, 0.125, 0.375, 0.0, 0.5])
    # boundaries of the cumulative sums: 0.125, 0.5, 1.0
    assert osamp.categorical_token(p, 0.0) == 1            # the first index with mass
    assert osamp.categorical_token(p, 0.1249) == 1
    assert osamp.categorical_token(p, 0.125) == 2          # strict: the boundary moves on
    assert osamp.categorical_token(p, 0.4999) == 2
    assert osamp.categorical_token(p, 0.5) == 4            # index 3 has no mass
    assert osamp.categorical_token(p, 0.9999) == 4
    # an unnormalised row (stored probabilities) is scaled by its own total
    assert osamp.categorical_token(2.0 * p, 0.3) == osamp.categorical_token(p, 0.3)


def test_categorical_frequencies_follow_the_probabilities():
    from oracle import splitmix
    p = np.array([0.05, 0.15, 0.5, 0.3])
    n = 20000
    draws = np.array([osamp.categorical_token(p, splitmix.key_uniform(splitmix.renoise_key(9, 2, r)))
                      for r in range(n)])
    freq = np.bincount(draws, minlength=4) / n
    assert np.all(np.abs(freq - p) < 4 * np.sqrt(p * (1 - p) / n))   # within 4 sigma


def test_categorical_sampler_changes_only_committed_tokens():
    from oracle import splitmix
    rng = np.random.default_rng(4)
    rows, V = 12, 64
    logits = rng.standard_normal((rows, V)) * 3.0
    logits[:6, 5] += 25.0            # peaked rows: commit
    frozen = np.zeros(rows, np.uint8)
    frozen[0] = 1
    ft = np.full(rows, 7)
    base = osamp.canvas_sample(logits, None, 0.3, 1, 2, frozen=frozen, frozen_tokens=ft, probs_storage="bf16")
    cat = osamp.canvas_sample(logits, None, 0.3, 1, 2, frozen=frozen, frozen_tokens=ft, probs_storage="bf16",
                              categorical=True)
    np.testing.assert_array_equal(cat["commit_mask"], base["commit_mask"])
    for r in range(rows):
        if frozen[r] or not base["commit_mask"][r]:
            assert cat["tokens"][r] == base["tokens"][r]
        else:
            u = splitmix.key_uniform(splitmix.renoise_key(1, 2, r))
            assert cat["tokens"][r] == osamp.categorical_token(cat["probs"][r], u)
    assert 1 <= int(base["commit_mask"][1:].sum()) < rows - 1


def test_all_committed_per_canvas():
    m = np.array([1, 1, 1, 0, 1, 1, 1, 1], np.uint8)
    np.testing.assert_array_equal(osamp.all_committed(m, 4), [False, True])


# ---------------------------------------------------------------- self-conditioning MLP
def test_gelu_tanh_form_against_the_exact_gelu_and_its_symmetry():
    from scipy.special import ndtr
    x = np.linspace(-8, 8, 4001)
    g = onum.gelu_tanh(x)
    # the tanh form approximates x * Phi(x) (Phi: the normal CDF, a library
    # routine) to within 1e-3 everywhere
    assert np.max(np.abs(g - x * ndtr(x))) < 1e-3
    # gelu(x) - gelu(-x) = x exactly (tanh is odd), gelu(0) = 0
    np.testing.assert_allclose(g - onum.gelu_tanh(-x), x, rtol=1e-13, atol=1e-14)
    assert onum.gelu_tanh(0.0) == 0.0
    assert abs(onum.gelu_tanh(20.0) - 20.0) < 1e-12 and abs(onum.gelu_tanh(-20.0)) < 1e-12
    # far in the negative tail the value is x e^{2u} to leading order (not 0):
    # relative accuracy is kept where 1 + tanh(u) would cancel
    for xv in (-7.0, -9.0, -12.0):
        u = math.sqrt(2 / math.pi) * (xv + 0.044715 * xv ** 3)
        lead = xv * math.exp(2 * u)
        assert abs(onum.gelu_tanh(xv) - lead) <= 1e-6 * abs(lead)


def test_selfcond_mlp_maps_zero_to_zero_and_is_the_plain_composition():
    from oracle import loop as oloop
    rng = np.random.default_rng(5)
    D, H = 16, 8
    W1 = onum.bf16_round(rng.standard_normal((H, D)) / 4)
    W2 = onum.bf16_round(rng.standard_normal((D, H)) / 3)
    assert np.all(oloop.selfcond_mlp(np.zeros((3, D)), W1, W2) == 0.0)
    s = rng.standard_normal((5, D))
    # element by element: row r, output j = sum_k W2[j,k] bf16(gelu(sum_i W1[k,i] bf16(s[r,i])))
    want = np.zeros((5, D))
    for r in range(5):
        for j in range(D):
            acc = 0.0
            for k in range(H):
                h = sum(W1[k, i] * onum.bf16_round(s[r, i]) for i in range(D))
                acc += W2[j, k] * onum.bf16_round(onum.gelu_tanh(h))
            want[r, j] = acc
    np.testing.assert_allclose(oloop.selfcond_mlp(s, W1, W2), want, rtol=1e-12, atol=1e-14)


# ---------------------------------------------------------------- mixture of experts
def _tiny_moe(seed=3, R=5, D=8, E=6, F=4, Fs=3):
    rng = np.random.default_rng(seed)
    q = lambda *s: onum.bf16_round(rng.standard_normal(s) / 2)  # noqa: E731
    return dict(x=q(R, D), router=q(E, D), Wg=q(E * F, D), Wu=q(E * F, D), Wd=q(E * D, F),
                shared=(q(Fs, D), q(Fs, D), q(D, Fs)), E=E, F=F, D=D)


def test_moe_routing_by_hand():
    from oracle import moe as omoe
    x = np.array([[1.0, 0.0], [0.0, 1.0]])
    router = np.array([[3.0, 0.0], [1.0, 1.0], [0.0, 2.0], [1.0, 0.0]])   # scores: row0 3,1,0,1 ; row1 0,1,2,0
    chosen, w, margin = omoe.route(x, router, 2)
    np.testing.assert_array_equal(chosen, [[0, 1], [2, 1]])   # row 0: 1 and 3 tie at 1 -> lower index 1
    np.testing.assert_allclose(w[0], [np.e ** 3 / (np.e ** 3 + np.e), np.e / (np.e ** 3 + np.e)], rtol=1e-14)
    assert margin[0] == 0.0 and margin[1] == 1.0
    np.testing.assert_allclose(w.sum(axis=1), 1.0, rtol=1e-14)
    _, ws, _ = omoe.route(x, router, 2, scale=np.array([2.0, 0.5, 1.0, 1.0]))
    np.testing.assert_allclose(ws[0], w[0] * [2.0, 0.5], rtol=1e-14)


def test_moe_brute_force_and_special_cases():
    from oracle import moe as omoe
    m = _tiny_moe()
    x, D, F, E = m["x"], m["D"], m["F"], m["E"]
    out, (chosen, w, _) = omoe.moe(x, m["router"], 3, m["Wg"], m["Wu"], m["Wd"], shared=m["shared"])
    # element by element, straight from the definition
    want = np.zeros_like(out)
    for t in range(x.shape[0]):
        s = [sum(x[t, i] * m["router"][e, i] for i in range(D)) for e in range(E)]
        top = sorted(range(E), key=lambda e: (-s[e], e))[:3]
        z = sum(math.exp(s[e] - s[top[0]]) for e in top)
        for e in top:
            we = math.exp(s[e] - s[top[0]]) / z
            for o in range(D):
                acc = 0.0
                for f in range(F):
                    hg = sum(m["Wg"][e * F + f, i] * x[t, i] for i in range(D))
                    hu = sum(m["Wu"][e * F + f, i] * x[t, i] for i in range(D))
                    acc += m["Wd"][e * D + o, f] * onum.bf16_round(onum.gelu_tanh(hg) * hu)
                want[t, o] += we * acc
        Wsg, Wsu, Wsd = m["shared"]
        for o in range(D):
            want[t, o] += sum(Wsd[o, f] * onum.bf16_round(onum.gelu_tanh(sum(Wsg[f, i] * x[t, i] for i in range(D)))
                                                            * sum(Wsu[f, i] * x[t, i] for i in range(D)))
                              for f in range(Wsg.shape[0]))
    np.testing.assert_allclose(out, want, rtol=1e-10, atol=1e-12)
    # zero input -> zero output (no biases anywhere)
    z, _ = omoe.moe(np.zeros_like(x), m["router"], 3, m["Wg"], m["Wu"], m["Wd"], shared=m["shared"])
    assert np.all(z == 0.0)
    # k = E with one expert's weights doubled in W_down doubles only that expert's share
    o1, (c1, w1, _) = omoe.moe(x, m["router"], E, m["Wg"], m["Wu"], m["Wd"])
    Wd2 = m["Wd"].copy()
    Wd2[2 * D:3 * D] *= 2
    o2, _ = omoe.moe(x, m["router"], E, m["Wg"], m["Wu"], Wd2)
    y2 = omoe.gated_mlp(x, m["Wg"][2 * F:3 * F], m["Wu"][2 * F:3 * F], m["Wd"][2 * D:3 * D])
    share = np.array([w1[t, list(c1[t]).index(2)] for t in range(x.shape[0])])
    np.testing.assert_allclose(o2 - o1, share[:, None] * y2, rtol=1e-10, atol=1e-12)
