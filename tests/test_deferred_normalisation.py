"""The algebra behind the sampler's deferred normalisation (CPU only, fp64).

Without a probabilities output, canvas_sample cuts each row's vocabulary into
the K ranges of the soft-embedding GEMM's split (ranges of whole 64-entry
blocks, the first `rem` ranges one block longer), keeps per range only
(m_s, Z_s, T_s, argmax_s) and p~ = exp(z - m_s), and applies exp(m_s - m) / Z
to each range's partial product.  These tests check, on random rows and
against the oracle's direct softmax, that this factorisation reproduces the
soft embedding, the entropy, the confidence and the argmax (lowest index on
ties) exactly up to fp64 rounding, whatever the range count, including
ranges cut at the end of a vocabulary that is not a whole number of blocks.
"""
import numpy as np
import pytest

from oracle import sampler as osamp


def split_ranges(V, splits):
    """[(c0, c1)] of the split rule: kb = ceil(V / 64) blocks, kb // splits per
    range, the first kb % splits ranges one block more, clipped at V."""
    kb = (V + 63) // 64
    per, rem = kb // splits, kb % splits
    out = []
    for s in range(splits):
        b0 = s * per + min(s, rem)
        b1 = b0 + per + (1 if s < rem else 0)
        out.append((b0 * 64, min(V, b1 * 64)))
    return out


def range_state(z):
    """(m, Z, T, best index) of one range: Z = sum exp(z - m), T = sum (z - m) exp(z - m)."""
    a = int(np.argmax(z))
    m = z[a]
    e = np.exp(z - m)
    return m, e.sum(), ((z - m) * e).sum(), a


def merge(states):
    """Fold range states in order into the row's (m, Z, T, argmax)."""
    m, Z, T, a = states[0]
    for mb, Zb, Tb, ab in states[1:]:
        if mb > m:  # strictly larger: an equal maximum keeps the earlier (lower) index
            a = ab
        M = max(m, mb)
        sa, sb = np.exp(m - M), np.exp(mb - M)
        T = sa * (T + (m - M) * Z) + sb * (Tb + (mb - M) * Zb)
        Z = sa * Z + sb * Zb
        m = M
    return m, Z, T, a


@pytest.mark.parametrize("V,splits", [(4096, 4), (4096, 7), (262136, 13), (1000, 3), (64 * 40 + 8, 40)])
def test_ranges_reproduce_softmax_statistics_and_soft_embedding(V, splits):
    rng = np.random.default_rng(V + splits)
    D = 24
    z = rng.standard_normal(V) * 3.0
    z[rng.integers(0, V, 3)] = z.max() + 0.0  # exact ties of the maximum
    E = rng.standard_normal((V, D))
    p, H, amax, conf = osamp.row_statistics(z)
    ranges = split_ranges(V, splits)
    assert ranges[0][0] == 0 and ranges[-1][1] == V
    assert all(r0[1] == r1[0] for r0, r1 in zip(ranges, ranges[1:]))
    states, partial = [], []
    for c0, c1 in ranges:
        m, Zs, Ts, a = range_state(z[c0:c1])
        states.append((m, Zs, Ts, c0 + a))
        partial.append(np.exp(z[c0:c1] - m) @ E[c0:c1])  # p~ . E of the range
    m, Z, T, a = merge(states)
    # row statistics from the merged state
    assert a == amax
    assert np.isclose(1.0 / Z, conf, rtol=1e-12)
    assert np.isclose(np.log(Z) - T / Z, H, rtol=1e-10, atol=1e-12)
    # soft embedding: partial products scaled by exp(m_s - m) / Z
    soft = sum(np.exp(s[0] - m) / Z * part for s, part in zip(states, partial))
    np.testing.assert_allclose(soft, p @ E, rtol=1e-10, atol=1e-12)


def test_merge_order_does_not_change_the_result_beyond_rounding():
    # the kernel merges the range states with a warp butterfly, the test
    # above in range order: both give the row's statistics
    rng = np.random.default_rng(3)
    z = rng.standard_normal(64 * 148) * 5.0
    ranges = split_ranges(z.size, 148)
    states = [(*range_state(z[c0:c1])[:3], c0 + range_state(z[c0:c1])[3]) for c0, c1 in ranges]
    seq = merge(states)
    # pairwise tree in butterfly order (lane pairs, then pairs of pairs, ...)
    level = states[:]
    while len(level) > 1:
        nxt = [merge(level[i:i + 2]) for i in range(0, len(level) - 1, 2)]
        if len(level) % 2:
            nxt.append(level[-1])
        level = nxt
    tree = level[0]
    assert tree[3] == seq[3]
    np.testing.assert_allclose(tree[:3], seq[:3], rtol=1e-12)
