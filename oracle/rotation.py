"""Randomised Hadamard rotation.

[Guide] §二 step 1 names a random orthogonal rotation that spreads information over all dimensions.
[Overview] §核心技术解析 calls it a Hadamard transform, orthogonal, which spreads outlier energy across
dimensions. Reading used here: Pi = (1/sqrt(d)) * H * diag(D). H is the Sylvester Hadamard matrix
of order d (a power of two), and D is the seeded sign vector from ``rng.rademacher_signs``. Pi is
orthogonal, so <Pi q, Pi k> = <q, k>.
"""

import functools

import numpy as np


def hadamard(d):
    """Sylvester Hadamard matrix: H[i, j] = (-1)^popcount(i & j), d a power of two."""
    if d < 1 or d & (d - 1):
        raise ValueError("d must be a power of two")
    return _hadamard_cached(int(d)).copy()


@functools.lru_cache(maxsize=None)
def _hadamard_cached(d):
    i = np.arange(d)
    parity = np.zeros((d, d), dtype=np.int64)
    and_ij = i[:, None] & i[None, :]
    while np.any(and_ij):
        parity ^= and_ij & 1
        and_ij >>= 1
    return np.where(parity == 0, 1.0, -1.0)


def rotation_matrix(D):
    """Pi = H diag(D) / sqrt(d) (fp64, orthogonal)."""
    D = np.asarray(D, dtype=np.float64)
    d = D.shape[0]
    return hadamard(d) * D[None, :] / np.sqrt(d)
