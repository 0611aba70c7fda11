"""Pins for the oracle's random draws (SplitMix64, Box-Muller, bf16 rounding) and rotation."""
import json
import os

import numpy as np
import pytest
import scipy.linalg
import scipy.stats
import torch

from oracle import gaussian_matrix_bf16, hadamard, rademacher_signs, rotation_matrix, round_to_bf16, splitmix64

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def test_splitmix64_published_vector():
    g = json.load(open(os.path.join(GOLDEN, "splitmix64_seed1234567.json")))
    out = splitmix64(g["seed"], np.arange(1, 6, dtype=np.uint64))
    assert [int(x) for x in out] == g["outputs"]


def test_round_to_bf16_matches_torch_rne():
    rng = np.random.default_rng(7)
    x = np.concatenate([rng.standard_normal(20000), rng.standard_normal(2000) * 1e-3, rng.standard_normal(2000) * 1e4])
    x32 = x.astype(np.float32)  # fp32-exact inputs: torch's fp32 -> bf16 cast is a single RNE rounding
    ours = round_to_bf16(x32.astype(np.float64))
    ref = torch.from_numpy(x32).to(torch.bfloat16).to(torch.float64).numpy()
    assert np.array_equal(ours, ref)


# ---- hand-derived pins of D and S from the published SplitMix64 vector ----
# SplitMix64's finaliser is a bijection of 64-bit words, so a seed whose stream-1 (or stream-2) sub-seed is
# exactly 1234567 exists: invert the finaliser at 1234567 and step the state back by one (two) golden
# increments. The D (S) stream of that seed is then the published generator started at 1234567, whose
# first outputs the golden file holds. The inverse below undoes each xorshift by iteration and each
# multiplication by its inverse modulo 2^64; it shares nothing with the oracle's forward code.
_M64 = 2 ** 64
_GAMMA, _MUL1, _MUL2 = 0x9E3779B97F4A7C15, 0xBF58476D1CE4E5B9, 0x94D049BB133111EB


def _undo_xorshift(z, s):
    x = z
    for _ in range(64 // s + 1):
        x = z ^ (x >> s)
    return x


def _unmix(z):
    z = _undo_xorshift(z, 31)
    z = z * pow(_MUL2, -1, _M64) % _M64
    z = _undo_xorshift(z, 27)
    z = z * pow(_MUL1, -1, _M64) % _M64
    return _undo_xorshift(z, 30)


def test_rademacher_signs_from_the_published_vector():
    """D_i = +1 when bit 63 of output i+1 of the D stream is 0. With the D stream started at 1234567, the
    published outputs 6457827717110365317, 3203168211198807973, 9817491932198370423, 4593380528125082431 and
    16408922859458223821 have bit 63 = 0, 0, 1, 0, 1 (the third and fifth are >= 2^63), so D = +1 +1 -1 +1 -1."""
    seed = (_unmix(1234567) - _GAMMA) % _M64
    assert seed == 11906536674387683726
    assert rademacher_signs(seed, 5).tolist() == [1.0, 1.0, -1.0, 1.0, -1.0]


def test_gaussian_entry_from_the_published_vector():
    """S_00 by Box-Muller from the first two outputs of the S stream started at 1234567:
    u1 = ((6457827717110365317 >> 11) + 0.5) 2^-53 = (3153236189995295 + 0.5) 2^-53 = 0.3500795420...,
    u2 = ((3203168211198807973 >> 11) + 0.5) 2^-53 = (1564046978124417 + 0.5) 2^-53 = 0.1736440966...,
    sqrt(-2 ln u1) cos(2 pi u2) = 1.44903... x 0.46151... = 0.6687418...; to bf16 (8 significant bits):
    0.6687418 x 256 = 171.198 -> 171 / 256 = 0.66796875."""
    seed = (_unmix(1234567) - 2 * _GAMMA) % _M64
    assert seed == 505821855064485241
    S = gaussian_matrix_bf16(seed, 1)
    assert S.shape == (1, 1) and S[0, 0] == 0.66796875


def test_rademacher_signs_balanced():
    D = rademacher_signs(11, 4096)
    assert set(np.unique(D)) == {-1.0, 1.0}
    # binomial(4096, 1/2): |sum| within 5 sigma
    assert abs(D.sum()) < 5 * np.sqrt(4096)


@pytest.mark.parametrize("d", [64, 128, 256])
def test_gaussian_matrix_is_standard_normal_in_bf16(d):
    S = gaussian_matrix_bf16(3, d)
    assert np.array_equal(round_to_bf16(S), S)
    n = S.size
    assert abs(S.mean()) < 5 / np.sqrt(n)
    assert abs(S.var() - 1.0) < 5 * np.sqrt(2.0 / n) + 2 ** -8
    assert scipy.stats.kstest(S.ravel(), "norm").pvalue > 1e-4


@pytest.mark.parametrize("d", [2, 4, 8, 64, 128, 256])
def test_hadamard_is_sylvester(d):
    H = hadamard(d)
    assert np.array_equal(H, scipy.linalg.hadamard(d).astype(np.float64))
    assert np.array_equal(H @ H.T, d * np.eye(d))


@pytest.mark.parametrize("d", [64, 128, 256])
def test_rotation_orthogonal_and_norm_preserving(d):
    Pi = rotation_matrix(rademacher_signs(5, d))
    assert np.max(np.abs(Pi @ Pi.T - np.eye(d))) < 1e-14
    x = np.random.default_rng(d).standard_normal((10, d))
    assert np.allclose(np.linalg.norm(x @ Pi.T, axis=1), np.linalg.norm(x, axis=1), rtol=1e-14)
    # Pi = H diag(D) / sqrt(d): column j of Pi is D_j * H[:, j] / sqrt(d)
    D = rademacher_signs(5, d)
    assert np.allclose(Pi * np.sqrt(d), scipy.linalg.hadamard(d) * D[None, :])
