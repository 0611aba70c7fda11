"""Pins for the oracle's key/value quantisers, canonical packing and ring split."""
import json
import os

import numpy as np
import pytest
import scipy.linalg

from oracle import (gaussian_matrix_bf16, history_split, key_record_bytes, lloyd_max_codebook,
                    pack_key_records, pack_value_records, quantize_keys, quantize_values, rademacher_signs,
                    unpack_key_records, unpack_value_records, value_record_bytes, dequantize_values)
from oracle.quant import _pack_bits, _unpack_bits

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rotate(x, D):
    """Pi x computed with scipy's Hadamard (independent of the oracle's construction)."""
    d = x.shape[-1]
    return (x * D[None, :]) @ scipy.linalg.hadamard(d).T / np.sqrt(d)


@pytest.mark.parametrize("bits", [1, 2, 4])
def test_pack_unpack_exhaustive(bits):
    per = 8 // bits
    allbytes = np.arange(256, dtype=np.uint8).reshape(1, 256)
    codes = _unpack_bits(allbytes, bits, 256 * per)
    assert np.array_equal(_pack_bits(codes, bits), allbytes)
    rnd = np.random.default_rng(bits).integers(0, 1 << bits, size=(7, 256), dtype=np.uint8)
    assert np.array_equal(_unpack_bits(_pack_bits(rnd, bits), bits, 256), rnd)


def test_pack_bit_order_little_endian():
    # 3-bit stream, worked by hand: element j at bits 3j..3j+2, bit i of the stream = bit i % 8 of byte i // 8
    # [1, 2, 7, 0, 5, 3, 6, 4] sets stream bits 0 | 4 | 6 7 8 | - | 12 14 | 15 16 | 19 20 | 23
    assert list(_pack_bits(np.array([[1, 2, 7, 0, 5, 3, 6, 4]], np.uint8), 3)[0]) == [0xD1, 0xD1, 0x99]
    rnd = np.random.default_rng(3).integers(0, 8, size=(5, 64), dtype=np.uint8)
    assert np.array_equal(_unpack_bits(_pack_bits(rnd, 3), 3, 64), rnd)
    assert _pack_bits(np.array([[0, 1, 2, 3]], np.uint8), 2)[0, 0] == 0b11100100
    assert _pack_bits(np.array([[1, 0, 0, 0, 0, 0, 0, 1]], np.uint8), 1)[0, 0] == 0b10000001
    assert _pack_bits(np.array([[0x3, 0xA]], np.uint8), 4)[0, 0] == 0xA3


def test_record_sizes_and_golden_constants():
    g = json.load(open(os.path.join(GOLDEN, "memory_figures.json")))["pipeline_constants"]
    assert g["key_bits"] == 2 + g["qjl_bits_per_dim"]
    assert g["values_per_byte_at_2bit"] == 8 // 2
    assert key_record_bytes(128) == 52 and key_record_bytes(256) == 100
    assert key_record_bytes(128, 4) == 68 and key_record_bytes(64, 4) == 36 and key_record_bytes(256, 4) == 132
    assert value_record_bytes(128, 2) == 40 and value_record_bytes(128, 4) == 72
    assert value_record_bytes(256, 2) == 80 and value_record_bytes(256, 4) == 144


@pytest.mark.parametrize("key_bits", [3, 4])
@pytest.mark.parametrize("d", [64, 128, 256])
def test_key_records(d, key_bits):
    rng = np.random.default_rng(d)
    k = rng.standard_normal((64, d))
    k[:, 3] *= 8.0
    k[5] = 0.0
    D, S = rademacher_signs(1, d), gaussian_matrix_bf16(1, d)
    c, t = lloyd_max_codebook(d, key_bits - 1)
    rec = quantize_keys(k, D, S, c, t)
    assert rec.mse_bits == key_bits - 1 and rec.idx.max() == 2 ** (key_bits - 1) - 1
    n = np.linalg.norm(k, axis=1)
    assert np.array_equal(rec.norm, n.astype(np.float32).astype(np.float16))
    y = _rotate(k, D) / np.where(n > 0, n, 1)[:, None]
    y[5] = 0
    # the boundary rule equals the nearest-centroid rule (midpoint boundaries)
    nearest = np.argmin(np.abs(y[:, :, None] - c[None, None, :]), axis=2)
    assert np.array_equal(rec.idx, nearest)
    r = y - c[rec.idx]
    assert np.allclose(rec.gamma.astype(np.float64), np.linalg.norm(r, axis=1), rtol=2 ** -10)
    z = r @ S.T
    pm = 2.0 * rec.sign - 1.0
    assert np.allclose(np.sum(pm * z, axis=1), np.sum(np.abs(z), axis=1), rtol=1e-12)
    # round trip through the canonical bytes
    buf = pack_key_records(rec)
    assert buf.shape == (64, key_record_bytes(d, key_bits))
    back = unpack_key_records(buf, d, key_bits)
    for f in ("idx", "sign", "norm", "gamma"):
        assert np.array_equal(getattr(back, f), getattr(rec, f))


@pytest.mark.parametrize("bits", [2, 4])
@pytest.mark.parametrize("d", [64, 128, 256])
def test_value_records(bits, d):
    rng = np.random.default_rng(bits * d)
    v = rng.standard_t(5, size=(50, d))
    v[7] = 0.0
    D = rademacher_signs(2, d)
    rec = quantize_values(v, D, bits)
    half = 1 << (bits - 1)
    vr = _rotate(v, D).reshape(50, d // 32, 32)
    s = rec.scales.astype(np.float64)[:, :, None]
    absmax = np.abs(vr).max(axis=2)
    assert np.allclose(rec.scales.astype(np.float64), absmax / (half - 0.5), rtol=2 ** -10)
    lev = (rec.codes.reshape(50, d // 32, 32).astype(np.float64) - half + 0.5) * s
    # mid-rise quantiser: error within half a step (plus the fp16 rounding of the scale at the top level)
    assert np.all(np.abs(vr - lev) <= 0.5 * s + absmax[:, :, None] * 2 ** -10 + 1e-12)
    assert np.all(rec.codes[7] == half) and np.all(rec.scales[7] == 0)
    # the group's absmax element is reproduced by a top level (up to fp16 rounding of the scale)
    top = np.abs(lev).max(axis=2)
    assert np.allclose(top, absmax, rtol=2 ** -10)
    # dequantisation rotates back with Pi^T
    back = dequantize_values(rec, D)
    assert np.allclose(_rotate(back, D), lev.reshape(50, d), atol=1e-12)
    buf = pack_value_records(rec)
    assert buf.shape == (50, value_record_bytes(d, bits))
    r2 = unpack_value_records(buf, d, bits)
    assert np.array_equal(r2.codes, rec.codes) and np.array_equal(r2.scales, rec.scales)


def test_values_on_the_grid_are_lossless():
    d, bits = 128, 2
    D = rademacher_signs(9, d)
    rng = np.random.default_rng(0)
    codes = rng.integers(0, 4, size=(10, d))
    codes[:, ::32] = 3  # make each group's absmax exactly 1.5 * s with s = 0.5 (exact in fp16)
    vr = (codes - 1.5) * 0.5
    v = vr.reshape(10, d) @ (scipy.linalg.hadamard(d) * D[None, :] / np.sqrt(d))  # Pi^T v'
    rec = quantize_values(v, D, bits)
    assert np.all(rec.scales == np.float16(0.5))
    assert np.array_equal(rec.codes, codes)
    assert np.allclose(dequantize_values(rec, D), v, atol=1e-12)


def test_history_split_ring_semantics():
    assert history_split(0) == (0, 0)
    assert history_split(1) == (0, 1)
    assert history_split(128) == (0, 128)
    assert history_split(129) == (128, 1)
    assert history_split(1152) == (1024, 128)  # 1024 packed + 128-token ring
    assert history_split(32768) == (32640, 128)
    # full_tq (ring 0): nothing stays exact
    assert history_split(0, 0) == (0, 0) and history_split(1, 0) == (1, 0) and history_split(385, 0) == (385, 0)


def test_cos_sim_report_pins():
    """Values on the quantiser grid reconstruct exactly (cos 1). For keys, the Lloyd-Max centroid
    condition gives E<y, c[idx]> = E||c[idx]||^2 = 1 - D, so the MSE-only cosine of rotated unit vectors
    tends to sqrt(1 - D), with D = d x the codebook's per-coordinate distortion. Adding the QJL term (unbiased, not
    MSE-optimal) lowers the cosine."""
    from oracle import cos_sim_report, lloyd_max_codebook, mse_distortion, gaussian_matrix_bf16
    d, bits = 128, 2
    D = rademacher_signs(9, d)
    rng = np.random.default_rng(0)
    codes = rng.integers(0, 4, size=(10, d))
    codes[:, ::32] = 3
    v = ((codes - 1.5) * 0.5) @ (scipy.linalg.hadamard(d) * D[None, :] / np.sqrt(d))
    vrec = quantize_values(v, D, bits)
    c, t = lloyd_max_codebook(d, 2)
    S = gaussian_matrix_bf16(9, d)
    k = rng.standard_normal((4000, d))
    krec = quantize_keys(k, D, S, c, t)
    rep = cos_sim_report(k, v, krec, vrec, D, S, c)
    assert abs(rep["value_cos"] - 1.0) < 1e-12
    expect = np.sqrt(1.0 - d * mse_distortion(d, c, t))  # per-coordinate distortion x d = unit-vector D
    assert abs(rep["key_cos_mse"] - expect) < 3e-3, (rep, expect)
    assert rep["key_cos_qjl"] < rep["key_cos_mse"]


@pytest.mark.parametrize("d", [64, 128])
def test_dequantized_key_inner_product_is_unbiased(d):
    """The QJL term makes the key estimate unbiased ([Guide] §二 step 3): for a unit vector y and
    y_hat = c[idx] + sqrt(pi/2)/d * gamma * S^T sign(S r), E_S <y, y_hat> = <y, c> + <c, r> + gamma^2 =
    ||c + r||^2 = 1, since E[sign(s.r) s] = sqrt(2/pi) r / ||r|| for s ~ N(0, I). Over 2000 independent S
    (one unit key each, through dequantize_keys with n = 1) the mean of <k, k_hat> must be 1 within 3
    standard errors. A wrong constant in the QJL term (e.g. sqrt(2/pi)/d: mean ~0.96) or a flipped sign
    (mean ~0.77) fails, and so does leaving the term out (mean 1 - D ~ 0.88)."""
    from oracle import dequantize_keys, gaussian_matrix_bf16, lloyd_max_codebook
    c, t = lloyd_max_codebook(d, 2)
    D = rademacher_signs(3, d)
    rng = np.random.default_rng(d)
    vals = []
    for seed in range(2000):
        S = gaussian_matrix_bf16(10_000 + seed, d)
        k = rng.standard_normal((1, d))
        k /= np.linalg.norm(k)
        rec = quantize_keys(k, D, S, c, t)
        rec.norm[:] = np.float16(1.0)  # exact unit norm, so <k, k_hat> = <y, y_hat>
        vals.append(float(np.sum(k * dequantize_keys(rec, D, S, c, with_qjl=True))))
    vals = np.asarray(vals)
    se = vals.std(ddof=1) / np.sqrt(len(vals))
    assert abs(vals.mean() - 1.0) <= 3 * se + 2e-3, (vals.mean(), se)  # 2e-3: fp16 gamma and bf16 S
    assert se < 0.01
