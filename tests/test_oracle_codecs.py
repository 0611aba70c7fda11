"""Pins for the comparison codecs of the oracle (KIVI 2-bit, Bonsai 1-bit; [Overview] §核心技术解析
and the KV size table of §性能表现与实测数据)."""
import json
import os

import numpy as np
import pytest

from oracle import bonsai1_dequantize, bonsai1_quantize, kivi2_dequantize, kivi2_quantize

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _bytes_per_element(arrays, n_elems, code_bits):
    """Stored bytes per element: packed codes plus every parameter array at its own dtype."""
    return (n_elems * code_bits / 8 + sum(a.nbytes for a in arrays)) / n_elems


def test_table_sizes_from_codec_layout():
    """The codecs' own output sizes, scaled to Llama-3.1-8B at 32K tokens, give the table's rows."""
    g = json.load(open(os.path.join(GOLDEN, "memory_figures.json")))["llama31_8b_32k"]
    sh = g["shape"]
    elems = 2 * sh["layers"] * sh["kv_heads"] * sh["seq_len"] * sh["head_dim"]  # K and V
    x = np.random.default_rng(0).standard_normal((64, sh["head_dim"]))
    _, ks, kz = kivi2_quantize(x, 0)
    _, vs, vz = kivi2_quantize(x, 1)
    kivi = (_bytes_per_element([ks, kz], x.size, 2) + _bytes_per_element([vs, vz], x.size, 2)) / 2
    _, bs = bonsai1_quantize(x)
    bonsai = _bytes_per_element([bs], x.size, 1)
    MiB = 1 << 20
    assert kivi * elems == g["kivi_2bit_MB"] * MiB
    assert bonsai * elems == g["bonsai_1bit_g128_MB"] * MiB
    assert 2 * elems == g["fp16_MB"] * MiB


@pytest.mark.parametrize("axis", [0, 1])
def test_kivi_exact_level_grid(axis):
    """A group whose values sit on z + k s (fp16-exact z, s) is reproduced exactly with those codes."""
    rng = np.random.default_rng(axis)
    T, d = 32, 48
    codes = rng.integers(0, 4, size=(T, d)).astype(np.uint8)
    ng = (T // 16, d) if axis == 0 else (T, d // 16)
    z = (rng.integers(-64, 64, size=ng) / 16.0).astype(np.float16)
    s = (rng.integers(1, 32, size=ng) / 64.0).astype(np.float16)
    # force every group to contain both its end levels so that min = z and max = z + 3 s
    if axis == 0:
        codes[0::16, :] = 0
        codes[1::16, :] = 3
    else:
        codes[:, 0::16] = 0
        codes[:, 1::16] = 3
    x = kivi2_dequantize(codes, s, z, axis)
    c2, s2, z2 = kivi2_quantize(x, axis)
    assert np.array_equal(s2, s) and np.array_equal(z2, z)
    assert np.array_equal(c2, codes)
    assert np.array_equal(kivi2_dequantize(c2, s2, z2, axis), x)


def test_kivi_constant_group_and_extremes():
    x = np.full((16, 16), 1.25)
    c, s, z = kivi2_quantize(x, 0)
    assert np.all(s == 0) and np.all(z == np.float16(1.25)) and np.all(c == 0)
    assert np.array_equal(kivi2_dequantize(c, s, z, 0), x)
    y = np.random.default_rng(3).standard_normal((32, 64)) * 4
    for axis in (0, 1):
        c, s, z = kivi2_quantize(y, axis)
        g = y.reshape(2, 16, 64) if axis == 0 else y.reshape(32, 4, 16)
        red = 1 if axis == 0 else 2
        cg = c.reshape(g.shape)
        # the group minimum takes code 0 and the maximum code 3 (both fp16 parameters round to nearest)
        assert np.all(np.take_along_axis(cg, np.expand_dims(np.argmin(g, red), red), red) == 0)
        assert np.all(np.take_along_axis(cg, np.expand_dims(np.argmax(g, red), red), red) == 3)


@pytest.mark.parametrize("axis", [0, 1])
def test_kivi_brute_force_nearest_level(axis):
    """Each code names the nearest of the four levels z + k s (fp64 brute force), except within a
    rounding margin of a midpoint; the reconstruction error is at most half a step there."""
    x = np.random.default_rng(10 + axis).standard_normal((64, 32))
    c, s, z = kivi2_quantize(x, axis)
    g, red = (x.reshape(4, 16, 32), 1) if axis == 0 else (x.reshape(64, 2, 16), 2)
    sg = np.expand_dims(s.astype(np.float64), red)
    zg = np.expand_dims(z.astype(np.float64), red)
    levels = zg[..., None] + sg[..., None] * np.arange(4.0)
    dist = np.abs(g[..., None] - levels)
    best = np.argmin(dist, axis=-1)
    dsort = np.sort(dist, axis=-1)
    clear = (dsort[..., 1] - dsort[..., 0]) > 1e-5 * np.maximum(sg, 1e-30)
    cg = c.reshape(g.shape)
    assert np.array_equal(cg[clear], best[clear])
    assert clear.mean() > 0.99
    err = np.abs(kivi2_dequantize(c, s, z, axis) - x).reshape(g.shape)
    # half a step, plus the fp16 rounding of the zero point and of the step at code 3
    bound = 0.5 * sg + np.abs(zg - np.expand_dims(g.min(axis=red), red)) + 3 * 2.0 ** -11 * sg + 1e-12
    assert np.all(err <= bound)


def test_kivi_key_grouping_is_value_grouping_transposed():
    """Per-channel groups of 16 tokens of x are per-token groups of 16 channels of x^T."""
    x = np.random.default_rng(4).standard_normal((48, 32))
    ck, sk, zk = kivi2_quantize(x, 0)
    cv, sv, zv = kivi2_quantize(x.T, 1)
    assert np.array_equal(ck, cv.T) and np.array_equal(sk, sv.T) and np.array_equal(zk, zv.T)


def test_kivi_channel_outlier_rationale():
    """Keys whose large magnitudes sit in a few fixed channels lose less with per-channel groups than
    with per-token groups (the motivation given in §KIVI非对称量化)."""
    rng = np.random.default_rng(5)
    k = rng.standard_normal((256, 128))
    k[:, [7, 40, 99]] += np.array([25.0, -30.0, 20.0])
    per_channel = np.mean((kivi2_dequantize(*kivi2_quantize(k, 0), 0) - k) ** 2)
    per_token = np.mean((kivi2_dequantize(*kivi2_quantize(k, 1), 1) - k) ** 2)
    assert per_channel < 0.5 * per_token


def test_bonsai_bits_scale_and_least_squares():
    rng = np.random.default_rng(6)
    x = rng.standard_normal((8, 256))
    x[0, :5] = 0.0  # zero maps to bit 1
    bits, s = bonsai1_quantize(x)
    assert np.array_equal(bits, (x >= 0).astype(np.uint8)) and bits[0, 0] == 1
    assert s.shape == (8, 2)
    assert np.allclose(s.astype(np.float64), np.abs(x).reshape(8, 2, 128).mean(axis=2), rtol=2 ** -11)
    xh = bonsai1_dequantize(bits, s)
    assert np.array_equal(np.abs(xh).reshape(8, 2, 128), np.broadcast_to(s.astype(np.float64)[..., None], (8, 2, 128)))
    # mean |x| minimises sum (x - t sign)^2 over t: a nearby scale never does better
    e0 = np.sum((xh - x) ** 2)
    for f in (0.97, 1.03):
        assert np.sum((bonsai1_dequantize(bits, (s.astype(np.float64) * f)) - x) ** 2) > e0


def test_bonsai_constant_magnitude_is_exact():
    x = np.where(np.random.default_rng(7).random((4, 128)) < 0.5, -0.75, 0.75)
    bits, s = bonsai1_quantize(x)
    assert np.all(s == np.float16(0.75))
    assert np.array_equal(bonsai1_dequantize(bits, s), x)
