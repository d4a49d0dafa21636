"""SplitMix64 counter RNG in exact 64-bit integer arithmetic.

Test infrastructure only (see the package docstring).

SplitMix64 is the published generator of Steele, Lea and Flood, "Fast
splittable pseudorandom number generators" (OOPSLA 2014), in the form Vigna
released into the public domain: the state advances by the golden-ratio
increment 0x9E3779B97F4A7C15 and each output is the state passed through two
xor-shift-multiply rounds and a final xor-shift.  The pages name no RNG; the
renoise draw (uniform random token, [AB] §블록 자동 회귀 노이즈 제거 및 자체 수정)
needs one that both sides can evaluate bit-exactly, so the counter-based key
below is the reading taken:

    key(seed, step, row) = mix(mix(mix(seed) ^ step) ^ row)
    token = key mod V

where mix(z) is the output SplitMix64 produces from state z (one ``next``).
A committed position that takes a categorical draw instead of its argmax
uses the same key (a position either commits or renoises): its uniform is
the key's top 24 bits over 2^24, exact in fp32 and fp64.
"""
from __future__ import annotations

MASK64 = (1 << 64) - 1
GOLDEN = 0x9E3779B97F4A7C15


def mix(z: int) -> int:
    """The SplitMix64 output for state ``z``: advance once, then finalise."""
    z = (z + GOLDEN) & MASK64
    z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & MASK64
    z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & MASK64
    return z ^ (z >> 31)


def stream(seed: int, n: int) -> list:
    """The first ``n`` outputs of a SplitMix64 generator seeded with ``seed``."""
    out = []
    s = seed & MASK64
    for _ in range(n):
        out.append(mix(s))
        s = (s + GOLDEN) & MASK64
    return out


def renoise_key(seed: int, step: int, row: int) -> int:
    return mix(mix(mix(seed & MASK64) ^ (step & MASK64)) ^ (row & MASK64))


def renoise_token(seed: int, step: int, row: int, V: int) -> int:
    return renoise_key(seed, step, row) % V


def key_uniform(key: int) -> float:
    """u in [0, 1): the top 24 bits of a 64-bit key over 2^24."""
    return (key >> 40) / float(1 << 24)
