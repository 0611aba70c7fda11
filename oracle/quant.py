"""Quantize-on-append for one KV head: key and value records, and their canonical byte packing.

Steps, following [Guide] §二 (rotate -> Lloyd-Max -> QJL residual sign -> value group quantisation
-> bit packing). The magnitude/direction split follows [Overview] §核心技术解析 (PolarQuant).

Key k in R^d (key_bits per coordinate = (key_bits - 1)-bit Lloyd-Max + 1-bit QJL, [Guide] §二 and §五:
key_bits=3 is the configuration the guide runs; key_bits=4 is the 4-bit TurboQuant row of [Overview]
§性能表现与实测数据, read as a 3-bit Lloyd-Max index plus the QJL sign):
  n = ||k||_2;  y = Pi (k / n)  (y = 0 when n = 0);
  idx_j = #{ i : t_i < y_j }  (t = Lloyd-Max boundaries; the comparison is taken in fp32);
  r = y - c[idx];  gamma = ||r||_2;  z = S r;  sign_j = 1 if fp32(z_j) >= 0 else 0;
  stored: idx, sign bits, fp16(n), fp16(gamma)  (each fp16 rounded via fp32).

Value v in R^d (symmetric b-bit, groups of 32, fp16 scale per group, [Guide] §二 step 4):
  v' = Pi v;  per group G: s = fp16( fp32(max_G |v'|) / (2^(b-1) - 1/2) );
  code = clamp(floor(fp32(v') / s), -2^(b-1), 2^(b-1) - 1) + 2^(b-1)  (code = 2^(b-1) when s = 0);
  level = (code - 2^(b-1) + 1/2) * s  (mid-rise: +-absmax is a level up to the fp16 rounding of s).

Readings (the pages are silent; the plainest reading is used):
* values are rotated with the same Pi as keys;
* the fp16 scale is clamped to 65504;
* fp16 rounding goes through fp32, matching a kernel that computes in fp32;
* decisions (code index, sign, floor) are taken in fp32, the kernel's precision.

Canonical record bytes (bit packing, [Guide] §二 step 5: four 2-bit values per byte):
  a b-bit array is a little-endian bit stream: element j holds bits b*j .. b*j + b - 1, bit i of the
  stream is bit i mod 8 of byte floor(i/8) (for b = 1, 2, 4: bit b*(j mod 8/b) of byte floor(j*b/8));
  key record   = idx (key_bits-1 bits) | sign (1 bit) | n (fp16 LE) | gamma (fp16 LE)
                 -> d*(key_bits-1)/8 + d/8 + 4 bytes (52 B at d=128, key_bits 3; 68 B at key_bits 4);
  value record = codes (b bits) | scales (fp16 LE, d/32 of them)            -> d*b/8 + d/16 bytes.
"""

from dataclasses import dataclass

import numpy as np

from .rotation import rotation_matrix

KEY_MSE_BITS = 2
VALUE_GROUP = 32
RING = 128


@dataclass
class KeyRecords:
    idx: np.ndarray    # uint8 [T, d]
    sign: np.ndarray   # uint8 [T, d], 1 = projection >= 0
    norm: np.ndarray   # float16 [T]
    gamma: np.ndarray  # float16 [T]
    mse_bits: int = KEY_MSE_BITS  # bits of idx (key_bits - 1)


@dataclass
class ValueRecords:
    codes: np.ndarray   # uint8 [T, d]
    scales: np.ndarray  # float16 [T, d / 32]
    bits: int


def _fp16_via_fp32(x):
    return np.asarray(x, dtype=np.float64).astype(np.float32).astype(np.float16)


def quantize_keys(k, D, S, centroids, boundaries):
    """Key records for k [T, d] (fp64 values). S is the QJL matrix [d, d], D the rotation signs. The
    index width follows the codebook: 4 centroids -> 2 bits (key_bits 3), 8 -> 3 bits (key_bits 4)."""
    k = np.atleast_2d(np.asarray(k, dtype=np.float64))
    Pi = rotation_matrix(D)
    n = np.sqrt(np.sum(k * k, axis=1))
    y = (k @ Pi.T) / np.where(n > 0, n, 1.0)[:, None]
    y[n == 0] = 0.0
    y32 = y.astype(np.float32)
    t32 = np.asarray(boundaries, dtype=np.float64).astype(np.float32)
    idx = np.sum(y32[:, :, None] > t32[None, None, :], axis=2).astype(np.uint8)
    r = y - np.asarray(centroids, dtype=np.float64)[idx]
    gamma = np.sqrt(np.sum(r * r, axis=1))
    z = r @ np.asarray(S, dtype=np.float64).T
    sign = (z.astype(np.float32) >= 0).astype(np.uint8)
    mse_bits = int(np.log2(len(centroids)))
    assert 1 << mse_bits == len(centroids)
    return KeyRecords(idx=idx, sign=sign, norm=_fp16_via_fp32(n), gamma=_fp16_via_fp32(gamma), mse_bits=mse_bits)


def quantize_values(v, D, bits, group=VALUE_GROUP):
    """Value records for v [T, d] (fp64 values) at `bits` in {2, 4}."""
    v = np.atleast_2d(np.asarray(v, dtype=np.float64))
    T, d = v.shape
    half = 1 << (bits - 1)
    vr = (v @ rotation_matrix(D).T).reshape(T, d // group, group)
    absmax = np.max(np.abs(vr), axis=2)
    s32 = absmax.astype(np.float32) / np.float32(half - 0.5)
    s16 = np.minimum(s32, np.float32(65504.0)).astype(np.float16)
    s = s16.astype(np.float32)[:, :, None]
    with np.errstate(divide="ignore", invalid="ignore"):
        q = np.floor(vr.astype(np.float32) / s)
    code = np.clip(q, -half, half - 1) + half
    code = np.where(s == 0, half, code)
    return ValueRecords(codes=code.reshape(T, d).astype(np.uint8), scales=s16, bits=bits)


def dequantize_values(rec, D, rotated=False):
    """v_hat = Pi^T (level * s) per token; `rotated=True` returns the rotated-basis levels."""
    half = 1 << (rec.bits - 1)
    T, d = rec.codes.shape
    groups = rec.scales.shape[1]
    lev = (rec.codes.astype(np.float64) - half + 0.5).reshape(T, groups, d // groups)
    vr = (lev * rec.scales.astype(np.float64)[:, :, None]).reshape(T, d)
    if rotated:
        return vr
    return vr @ rotation_matrix(D)  # row form of Pi^T v'


def dequantize_keys(rec, D, S, centroids, with_qjl=True):
    """k_hat = n * Pi^T (c[idx] + sqrt(pi/2)/d * gamma * S^T (2 sign - 1)) (QJL term optional)."""
    T, d = rec.idx.shape
    y = np.asarray(centroids, dtype=np.float64)[rec.idx]
    if with_qjl:
        kappa = np.sqrt(np.pi / 2.0) / d
        pm = 2.0 * rec.sign.astype(np.float64) - 1.0
        y = y + kappa * rec.gamma.astype(np.float64)[:, None] * (pm @ np.asarray(S, dtype=np.float64))
    return rec.norm.astype(np.float64)[:, None] * (y @ rotation_matrix(D))


def _mean_cos(a, b):
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    na, nb = np.linalg.norm(a, axis=1), np.linalg.norm(b, axis=1)
    ok = (na > 0) & (nb > 0)
    return float(np.mean(np.sum(a[ok] * b[ok], axis=1) / (na[ok] * nb[ok])))


def cos_sim_report(k, v, key_rec, val_rec, D, S, centroids):
    """Mean per-vector cosine similarity of the dequantised keys and values against the originals.

    [Guide] §六 quotes cos_sim for 3-bit keys (about 1.000000) and for 2-/4-bit values (0.940 / 0.997) at
    head_dim 256, without defining the quantity. This is the plain per-vector cosine, for keys both
    without the QJL term (MSE codebook only) and with it. It is a report: the key figure is
    parity unpinned, and the value figures are quoted from real model activations, not synthetic data.
    """
    return {
        "key_cos_mse": _mean_cos(dequantize_keys(key_rec, D, S, centroids, with_qjl=False), k),
        "key_cos_qjl": _mean_cos(dequantize_keys(key_rec, D, S, centroids, with_qjl=True), k),
        "value_cos": _mean_cos(dequantize_values(val_rec, D), v),
    }


def history_split(L, ring=RING):
    """(packed, ring) token counts of a sequence of length L: whole ring blocks are flushed when full.

    ring = 0 is the full_tq mode of [Guide] §三 (read as: no exact recent buffer, every token is
    quantised as it arrives), so all L tokens are packed.
    """
    if L <= 0:
        return 0, 0
    if ring == 0:
        return L, 0
    packed = ring * ((L - 1) // ring)
    return packed, L - packed


def _pack_bits(a, bits):
    """[T, d] values of `bits` bits -> [T, d*bits/8] bytes, as a little-endian bit stream."""
    a = np.asarray(a, dtype=np.uint8)
    T, d = a.shape
    assert (d * bits) % 8 == 0
    stream = (a[:, :, None] >> np.arange(bits, dtype=np.uint8)) & 1  # [T, d, bits]: bit i of element j
    return np.packbits(stream.reshape(T, d * bits), axis=1, bitorder="little")


def _unpack_bits(b, bits, d):
    b = np.asarray(b, dtype=np.uint8)
    stream = np.unpackbits(b, axis=1, bitorder="little")[:, :d * bits].reshape(b.shape[0], d, bits)
    return np.sum(stream.astype(np.uint16) << np.arange(bits, dtype=np.uint16), axis=2).astype(np.uint8)


def key_record_bytes(d, key_bits=KEY_MSE_BITS + 1):
    return d * (key_bits - 1) // 8 + d // 8 + 4


def value_record_bytes(d, bits, group=VALUE_GROUP):
    return d * bits // 8 + 2 * (d // group)


def pack_key_records(rec):
    T, d = rec.idx.shape
    return np.concatenate([
        _pack_bits(rec.idx, rec.mse_bits), _pack_bits(rec.sign, 1),
        rec.norm.astype("<f2").view(np.uint8).reshape(T, 2),
        rec.gamma.astype("<f2").view(np.uint8).reshape(T, 2)], axis=1)


def unpack_key_records(buf, d, key_bits=KEY_MSE_BITS + 1):
    buf = np.asarray(buf, dtype=np.uint8)
    T = buf.shape[0]
    mb = key_bits - 1
    o1 = d * mb // 8
    o2 = o1 + d // 8
    return KeyRecords(
        mse_bits=mb,
        idx=_unpack_bits(buf[:, :o1], mb, d),
        sign=_unpack_bits(buf[:, o1:o2], 1, d),
        norm=np.ascontiguousarray(buf[:, o2:o2 + 2]).view("<f2").reshape(T).astype(np.float16),
        gamma=np.ascontiguousarray(buf[:, o2 + 2:o2 + 4]).view("<f2").reshape(T).astype(np.float16))


def pack_value_records(rec, group=VALUE_GROUP):
    T, d = rec.codes.shape
    return np.concatenate([
        _pack_bits(rec.codes, rec.bits),
        rec.scales.astype("<f2").view(np.uint8).reshape(T, 2 * (d // group))], axis=1)


def unpack_value_records(buf, d, bits, group=VALUE_GROUP):
    buf = np.asarray(buf, dtype=np.uint8)
    T = buf.shape[0]
    o1 = d * bits // 8
    scales = np.ascontiguousarray(buf[:, o1:o1 + 2 * (d // group)]).view("<f2").reshape(T, d // group)
    return ValueRecords(codes=_unpack_bits(buf[:, :o1], bits, d), scales=scales.astype(np.float16), bits=bits)
