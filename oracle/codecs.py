"""Comparison KV codecs of [Overview]: KIVI 2-bit and Bonsai 1-bit (test infrastructure: a plain CPU
reference; only tests, smoke() and the bench's CPU baseline use it).

[Overview] §核心技术解析 names the two schemes and their granularity; it does not fix group sizes,
parameter types or rounding. The readings below are the plainest ones that reproduce the KV sizes of
its table in §性能表现与实测数据 for Llama-3.1-8B at 32K context (KIVI 2-bit 1,024 MB, Bonsai 1-bit
288 MB):

* KIVI 2-bit (§KIVI非对称量化): keys per channel, values per token, both asymmetric (scale and zero
  point). A group is 16 elements: 16 consecutive tokens of one key channel, or 16 consecutive
  channels of one value token. Per group: zero z = fp16(min), scale s = fp16((max - min) / 3) with
  the difference and quotient in fp32. Code = clamp(rint((x - z) * r), 0, 3) where r = 1 / s, both
  the subtraction, the reciprocal and the product in fp32 (IEEE round to nearest even); code 0 when
  s = 0. Reconstruction x_hat = z + code * s. 2 code bits + 2 * 16 parameter bits per 16 elements =
  4 bits per element.
* Bonsai 1-bit (§Bonsai 1-bit, named Q1_0_g128 in §TurboQuant-vLLM项目概览): groups of 128
  consecutive channels of one token; bit = 1 where x >= 0; scale s = fp16(mean |x|), the
  least-squares scale for a fixed sign pattern; x_hat = +s or -s. 1 + 16 / 128 bits per element. The
  page's fp16 residual cache of recent tokens is the same kind of ring as the hybrid mode's and is not
  part of the codec.

Inputs are values representable in fp32 (the kernels read bf16); |x| must stay below the fp16 range.
Parity status: pinned by tests/test_oracle_codecs.py (table sizes, exact level grids, brute-force
nearest level, the transpose relation between key and value grouping, least-squares optimality).
"""
import numpy as np

KIVI_GROUP = 16
KIVI_LEVELS = 4
BONSAI_GROUP = 128


def _to_f16(x32):
    return np.asarray(x32, dtype=np.float32).astype(np.float16)


def _kivi_groups(x, axis):
    """View x [T, d] as groups of 16 along `axis` (0: tokens of one channel, 1: channels of one token).
    Returns (grouped array, reduction axis)."""
    T, d = x.shape
    if axis == 0:
        assert T % KIVI_GROUP == 0, "per-channel key groups need a multiple of 16 tokens"
        return x.reshape(T // KIVI_GROUP, KIVI_GROUP, d), 1
    assert d % KIVI_GROUP == 0, "per-token value groups need a multiple of 16 channels"
    return x.reshape(T, d // KIVI_GROUP, KIVI_GROUP), 2


def kivi2_quantize(x, axis):
    """x [T, d] (one KV head). axis 0 = per-channel key quantisation, axis 1 = per-token value
    quantisation. Returns (codes uint8 [T, d] in 0..3, scale fp16, zero fp16); the parameters have
    shape [T/16, d] for axis 0 and [T, d/16] for axis 1."""
    x32 = np.asarray(x, dtype=np.float32)
    g, red = _kivi_groups(x32, axis)
    lo = np.min(g, axis=red)
    hi = np.max(g, axis=red)
    scale = _to_f16((hi - lo) / np.float32(KIVI_LEVELS - 1))
    zero = _to_f16(lo)
    s = np.expand_dims(scale.astype(np.float32), red)
    z = np.expand_dims(zero.astype(np.float32), red)
    with np.errstate(divide="ignore", invalid="ignore"):
        r = np.float32(1.0) / s
        v = np.rint((g - z) * r)
    codes = np.where(s == 0, 0, np.clip(v, 0, KIVI_LEVELS - 1)).astype(np.uint8)
    return codes.reshape(x32.shape), scale, zero


def kivi2_dequantize(codes, scale, zero, axis):
    """x_hat = zero + code * scale (fp64) for the grouping of kivi2_quantize."""
    c = np.asarray(codes, dtype=np.float64)
    g, red = _kivi_groups(c, axis)
    s = np.expand_dims(scale.astype(np.float64), red)
    z = np.expand_dims(zero.astype(np.float64), red)
    return (z + g * s).reshape(c.shape)


def bonsai1_quantize(x):
    """x [T, d] with d a multiple of 128 -> (bits uint8 [T, d], 1 where x >= 0; scale fp16 [T, d/128]
    = mean |x| of each group)."""
    x64 = np.asarray(x, dtype=np.float64)
    T, d = x64.shape
    assert d % BONSAI_GROUP == 0, "Bonsai groups are 128 channels of one token"
    g = x64.reshape(T, d // BONSAI_GROUP, BONSAI_GROUP)
    scale = np.mean(np.abs(g), axis=2).astype(np.float16)
    return (x64 >= 0).astype(np.uint8), scale


def bonsai1_dequantize(bits, scale):
    """x_hat = (2 bit - 1) * scale (fp64)."""
    T, d = bits.shape
    pm = 2.0 * np.asarray(bits, dtype=np.float64).reshape(T, d // BONSAI_GROUP, BONSAI_GROUP) - 1.0
    return (pm * scale.astype(np.float64)[:, :, None]).reshape(T, d)
