"""Pins for the inner-product estimator (unbiasedness) and the hybrid decode attention."""
import json
import os

import numpy as np
import pytest
import torch

from oracle import (decode_attention, dequantize_keys, dequantize_values, gaussian_matrix_bf16,
                    kv_bytes_bits_per_element, kv_bytes_dense, kv_bytes_turboquant, lloyd_max_codebook,
                    qjl_inner_product_estimate, quantize_keys, quantize_values, rademacher_signs)

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


@pytest.mark.parametrize("d,mse_bits", [(64, 2), (128, 2), (256, 2), (128, 3)])
def test_qjl_estimator_unbiased_over_seeds(d, mse_bits):
    """Mean estimator error over 10^4 independent Gaussian S is 0 within 3 sigma (fixed q, k); also for the
    3-bit index of key_bits 4."""
    rng = np.random.default_rng(100 + d)
    q = rng.standard_normal(d)
    k = rng.standard_normal(d)
    k[1] *= 6.0
    D = rademacher_signs(4, d)
    c, t = lloyd_max_codebook(d, mse_bits)
    truth = float(q @ k)
    n_trials = 10000
    err = np.empty(n_trials)
    for i in range(n_trials):
        S = rng.standard_normal((d, d))
        keys = quantize_keys(k[None, :], D, S, c, t)
        err[i] = qjl_inner_product_estimate(q, keys, D, S, c)[0] - truth
    # the MSE part is fixed; only the QJL correction varies with S; fp16 storage of n and gamma adds a
    # deterministic bias of at most ~2^-11 relative, below the 3-sigma bound here
    sigma = err.std() / np.sqrt(n_trials)
    assert abs(err.mean()) < 3 * sigma + 2 ** -11 * abs(truth)


def test_qjl_term_is_needed_for_unbiasedness():
    d = 128
    rng = np.random.default_rng(3)
    D = rademacher_signs(4, d)
    c, t = lloyd_max_codebook(d, 2)
    q = rng.standard_normal(d)
    ks = rng.standard_normal((4000, d))
    S = gaussian_matrix_bf16(4, d)
    keys = quantize_keys(ks, D, S, c, t)
    est = qjl_inner_product_estimate(q, keys, D, S, c)
    truth = ks @ q
    mse_only = (dequantize_keys(keys, D, S, c, with_qjl=False) @ q)
    # the 2-bit Lloyd-Max part alone shrinks inner products (biased by ~ -D(b) relative)
    slope_mse = np.polyfit(truth, mse_only, 1)[0]
    slope_est = np.polyfit(truth, est, 1)[0]
    assert slope_mse < 0.95
    assert abs(slope_est - 1.0) < 0.03


def _sdpa(q, k, v, scale):
    qt = torch.from_numpy(q)[None, :, None, :]                 # [1, G, 1, d]
    kt = torch.from_numpy(k)[None, None].expand(1, q.shape[0], -1, -1)
    vt = torch.from_numpy(v)[None, None].expand(1, q.shape[0], -1, -1)
    return torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, scale=scale)[0, :, 0].numpy()


@pytest.mark.parametrize("d", [64, 128])
def test_all_ring_context_is_exact_attention(d):
    rng = np.random.default_rng(d)
    q = rng.standard_normal((4, d))
    rk, rv = rng.standard_normal((37, d)), rng.standard_normal((37, d))
    D, S = rademacher_signs(0, d), gaussian_matrix_bf16(0, d)
    c, _ = lloyd_max_codebook(d, 2)
    out = decode_attention(q, None, None, rk, rv, D, S, c)
    assert np.allclose(out, _sdpa(q, rk, rv, 1 / np.sqrt(d)), atol=1e-13)


@pytest.mark.parametrize("vbits,mse_bits", [(2, 2), (4, 2), (4, 3)])
def test_hybrid_attention_equals_attention_on_dequantised_cache(vbits, mse_bits):
    d = 128
    rng = np.random.default_rng(vbits)
    D, S = rademacher_signs(5, d), gaussian_matrix_bf16(5, d)
    c, t = lloyd_max_codebook(d, mse_bits)
    kp, vp = rng.standard_normal((200, d)), rng.standard_normal((200, d))
    rk, rv = rng.standard_normal((17, d)), rng.standard_normal((17, d))
    q = rng.standard_normal((4, d)) * 2.0
    keys, vals = quantize_keys(kp, D, S, c, t), quantize_values(vp, D, vbits)
    k_hat = dequantize_keys(keys, D, S, c, with_qjl=True)
    v_hat = dequantize_values(vals, D)
    for scale in (None, 0.05):
        out = decode_attention(q, keys, vals, rk, rv, D, S, c, softmax_scale=scale)
        sc = 1 / np.sqrt(d) if scale is None else scale
        ref = _sdpa(q, np.concatenate([k_hat, rk]), np.concatenate([v_hat, rv]), sc)
        assert np.allclose(out, ref, atol=1e-12)


def test_single_packed_token_returns_its_value():
    d = 64
    rng = np.random.default_rng(1)
    D, S = rademacher_signs(6, d), gaussian_matrix_bf16(6, d)
    c, t = lloyd_max_codebook(d, 2)
    v = rng.standard_normal((1, d))
    keys, vals = quantize_keys(rng.standard_normal((1, d)), D, S, c, t), quantize_values(v, D, 4)
    out = decode_attention(rng.standard_normal((2, d)), keys, vals, np.zeros((0, d)), np.zeros((0, d)), D, S, c)
    assert np.allclose(out, np.repeat(dequantize_values(vals, D), 2, axis=0), atol=1e-14)
    # 4-bit g32 reconstruction of a Gaussian vector is close
    assert np.linalg.norm(out[0] - v[0]) / np.linalg.norm(v[0]) < 0.15


def test_memory_arithmetic_matches_pages():
    g = json.load(open(os.path.join(GOLDEN, "memory_figures.json")))
    a = g["llama31_8b_32k"]
    sh = a["shape"]
    MiB = 1 << 20
    assert kv_bytes_dense(sh["layers"], sh["kv_heads"], sh["seq_len"], sh["head_dim"]) == a["fp16_MB"] * MiB
    # 4-bit elements + one fp16 per 128-element vector
    assert kv_bytes_bits_per_element(sh["layers"], sh["kv_heads"], sh["seq_len"], sh["head_dim"], 4, 128) \
        == a["turboquant_4bit_MB"] * MiB
    # 1-bit elements + one fp16 per group of 128
    assert kv_bytes_bits_per_element(sh["layers"], sh["kv_heads"], sh["seq_len"], sh["head_dim"], 1, 128) \
        == a["bonsai_1bit_g128_MB"] * MiB
    # this path: K3 (52 B) + V2 (40 B) per token-head = 736 MiB; K3 + V4 = 992 MiB
    assert kv_bytes_turboquant(32, 8, 32768, 128, 2) == 736 * MiB
    assert kv_bytes_turboquant(32, 8, 32768, 128, 4) == 992 * MiB
    b = g["llama2_7b"]
    sb = b["shape"]
    gb = kv_bytes_dense(sb["layers"], sb["kv_heads"], 2048, sb["head_dim"]) / 1e9
    assert abs(gb - b["seq_2048_GB"]) < 0.005
    assert abs(kv_bytes_dense(sb["layers"], sb["kv_heads"], 8192, sb["head_dim"]) / 1e9 - b["seq_8192_GB_approx"]) < 0.05
