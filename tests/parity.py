"""Comparison rules between the CUDA path's packed records and the oracle (test infrastructure).

Rules:
* Integer results (codes, sign bits) must match bit for bit. A mismatch is allowed only where the
  oracle's exact decision quantity lies within a stated distance of the decision boundary, and only
  for a bounded fraction.
* fp16-stored scalars (n, gamma, value scale) must match exactly, or differ by one fp16 ulp where
  the exact value sits next to an fp16 rounding midpoint.

Tolerances:
* Lloyd-Max code: |y - t_i| <= 1e-6 (unit-norm coordinates), with at most 1e-4 of the coordinates
  differing, each by one code.
* QJL sign: |z_i| <= 1e-5 * ||S_i|| * ||r||. That is above the fp32 accumulation error of a
  d-term dot product and the 2^-17 relative error of a bf16 hi/lo split. At most 1e-4 of the signs
  may differ.
* Value code: |v'/s - integer| <= 1e-5 (fp32 rotation and division). At most 1e-4 may differ.
"""
import numpy as np

import oracle


def f16_near_midpoint(exact, got16, rel=2e-6):
    """True where `got16` is one fp16 ulp from the nearest fp16 of `exact` and `exact` is near the midpoint."""
    exact = np.asarray(exact, np.float64)
    ref = exact.astype(np.float32).astype(np.float16)
    g = np.asarray(got16, np.float16)
    same = g.view(np.uint16) == ref.view(np.uint16)
    one_ulp = np.abs(g.view(np.uint16).astype(np.int32) - ref.view(np.uint16).astype(np.int32)) == 1
    mid = (g.astype(np.float64) + ref.astype(np.float64)) / 2
    near = np.abs(exact - mid) <= rel * np.maximum(np.abs(exact), 1e-30)
    return same | (one_ulp & near)


def check_key_records(gpu, k, D, S, cent, bnd, sign_tol=1e-5, max_frac=1e-4):
    """gpu: oracle.KeyRecords from the device; k: fp64 inputs [T, d]. Returns a dict of counts."""
    k = np.asarray(k, np.float64)
    T, d = k.shape
    ref = oracle.quantize_keys(k, D, S, cent, bnd)
    Pi = oracle.rotation_matrix(D)
    n = np.sqrt(np.sum(k * k, axis=1))
    y = (k @ Pi.T) / np.where(n > 0, n, 1)[:, None]
    y[n == 0] = 0
    # norms
    ok_n = f16_near_midpoint(n, gpu.norm)
    assert ok_n.all(), f"norm mismatch at tokens {np.nonzero(~ok_n)[0][:10]}"
    # codes
    diff = gpu.idx != ref.idx
    if diff.any():
        tt, jj = np.nonzero(diff)
        lo = np.minimum(gpu.idx[tt, jj], ref.idx[tt, jj]).astype(int)
        assert np.all(np.abs(gpu.idx[tt, jj].astype(int) - ref.idx[tt, jj].astype(int)) == 1), "code off by >1"
        dist = np.abs(y[tt, jj] - bnd[lo])
        assert np.all(dist <= 1e-6), f"code mismatch away from a boundary: max dist {dist.max()}"
        assert diff.mean() <= max_frac, f"too many boundary code flips: {diff.mean()}"
    # residual and signs recomputed from the device's own codes (same r when codes agree)
    r = y - np.asarray(cent)[gpu.idx]
    gamma = np.linalg.norm(r, axis=1)
    ok_g = f16_near_midpoint(gamma, gpu.gamma)
    assert ok_g.all(), f"gamma mismatch at tokens {np.nonzero(~ok_g)[0][:10]}"
    z = r @ np.asarray(S, np.float64).T
    ref_sign = (z.astype(np.float32) >= 0).astype(np.uint8)
    sd = gpu.sign != ref_sign
    if sd.any():
        rownorm = np.linalg.norm(np.asarray(S, np.float64), axis=1)
        tt, ii = np.nonzero(sd)
        bound = sign_tol * rownorm[ii] * np.maximum(gamma[tt], 1e-30)
        assert np.all(np.abs(z[tt, ii]) <= bound), f"sign flip away from 0: {np.abs(z[tt, ii]).max()}"
        assert sd.mean() <= max_frac, f"too many sign flips {sd.mean()}"
    return {"code_flips": int(diff.sum()), "sign_flips": int(sd.sum())}


def check_value_records(gpu, v, D, bits, max_frac=1e-4):
    v = np.asarray(v, np.float64)
    T, d = v.shape
    half = 1 << (bits - 1)
    vr = (v @ oracle.rotation_matrix(D).T).reshape(T, d // 32, 32)
    absmax = np.abs(vr).max(axis=2)
    ok_s = f16_near_midpoint(absmax / (half - 0.5), gpu.scales)
    assert ok_s.all(), f"scale mismatch at {np.argwhere(~ok_s)[:5]}"
    s = gpu.scales.astype(np.float64)[:, :, None]
    with np.errstate(divide="ignore", invalid="ignore"):
        ratio = vr / s
    q = np.floor(ratio.astype(np.float32))
    ref = np.where(s == 0, half, np.clip(q, -half, half - 1) + half).reshape(T, d).astype(np.uint8)
    diff = gpu.codes != ref
    if diff.any():
        rr = ratio.reshape(T, d)[diff]
        near = np.abs(rr - np.round(rr)) <= 1e-5
        assert np.all(near), f"value code mismatch away from a boundary: {rr[~near][:5]}"
        assert np.all(np.abs(gpu.codes[diff].astype(int) - ref[diff].astype(int)) == 1)
        assert diff.mean() <= max_frac
    return {"value_code_flips": int(diff.sum())}


def rel_l2(a, b):
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    return float(np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-30))
