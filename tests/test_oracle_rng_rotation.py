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
