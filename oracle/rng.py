"""Random draws of the method: the rotation's sign vector D and the QJL Gaussian matrix S.

The pages call the rotation "seeded random orthogonal" ([Guide] §二 step 1) and the QJL projection
a random projection ([Guide] §二 step 3). They name no generator. Reading used here: one
counter-based generator, SplitMix64 (Steele, Lea & Flood, "Fast Splittable Pseudorandom Number
Generators", OOPSLA 2014), written from its published definition:

* the state after ``i`` steps is ``seed + i * 0x9E3779B97F4A7C15 (mod 2^64)``;
* output ``i`` is that state passed through the finaliser
  ``z ^= z >> 30; z *= 0xBF58476D1CE4E5B9; z ^= z >> 27; z *= 0x94D049BB133111EB; z ^= z >> 31``.

Streams: ``seed_D = out_1(seed)`` and ``seed_S = out_2(seed)``.
* ``D_i = +1`` if bit 63 of ``out_{i+1}(seed_D)`` is 0, else ``-1``.
* ``S`` (row-major, index ``k = i*d + j``) is drawn by Box-Muller from ``u1 = U(out_{2k+1}(seed_S))``
  and ``u2 = U(out_{2k+2}(seed_S))``, with ``U(x) = ((x >> 11) + 0.5) * 2^-53``. Then
  ``S_ij = sqrt(-2 ln u1) * cos(2 pi u2)`` is rounded to nearest-even **bf16**. S is therefore exact
  in bf16 on every implementation.
"""

import numpy as np

_GOLDEN = np.uint64(0x9E3779B97F4A7C15)
_MIX1 = np.uint64(0xBF58476D1CE4E5B9)
_MIX2 = np.uint64(0x94D049BB133111EB)
TWO_PI = 6.283185307179586476925286766559


def splitmix64(seed, counters):
    """Output number ``counters`` (1-based, array) of a SplitMix64 generator whose state starts at ``seed``."""
    c = np.asarray(counters, dtype=np.uint64)
    with np.errstate(over="ignore"):
        z = np.uint64(seed) + c * _GOLDEN
        z = (z ^ (z >> np.uint64(30))) * _MIX1
        z = (z ^ (z >> np.uint64(27))) * _MIX2
        return z ^ (z >> np.uint64(31))


def derive_seed(seed, stream):
    """Sub-seed of a stream: output ``stream`` of the generator at ``seed`` (stream 1 = D, 2 = S)."""
    return int(splitmix64(seed, [stream])[0])


def _uniform_open(x):
    """Map a 64-bit word to a double in (0, 1): ((x >> 11) + 0.5) * 2^-53."""
    return ((x >> np.uint64(11)).astype(np.float64) + 0.5) * 2.0 ** -53


def round_to_bf16(x):
    """Round fp64 values to nearest-even bf16 (8 significant bits); returns fp64 holding bf16 values."""
    m, e = np.frexp(np.asarray(x, dtype=np.float64))
    return np.ldexp(np.round(m * 256.0), e - 8)  # np.round rounds halves to even


def rademacher_signs(seed, d):
    """D in {-1, +1}^d for the randomised Hadamard rotation."""
    x = splitmix64(derive_seed(seed, 1), np.arange(1, d + 1, dtype=np.uint64))
    return np.where((x >> np.uint64(63)) == 0, 1.0, -1.0)


def gaussian_matrix_bf16(seed, d):
    """S in R^{d x d}, i.i.d. N(0,1) by Box-Muller from SplitMix64, each entry rounded to bf16."""
    k = np.arange(d * d, dtype=np.uint64)
    s_seed = derive_seed(seed, 2)
    u1 = _uniform_open(splitmix64(s_seed, 2 * k + 1))
    u2 = _uniform_open(splitmix64(s_seed, 2 * k + 2))
    g = np.sqrt(-2.0 * np.log(u1)) * np.cos(TWO_PI * u2)
    return round_to_bf16(g).reshape(d, d)
