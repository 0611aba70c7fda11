"""CPU check of the rule the CUDA coders use for 2-bit value codes (host logic, no GPU).

The mid-rise code is clamp(floor(fl(x / s)), -2, 1) + 2, decided on the fp32 quotient rounded to
nearest. The kernels decide it without a division, by three comparisons: [x + s >= -s 2^-24] +
[x >= 0] + [x - s >= -s 2^-25]. This test restates both in numpy float32 and compares them where a
slip would show: x within a few ulps of -2 s, -s, 0, s and 2 s for fp16 scales s spread over the whole
positive fp16 range, plus ordinary values.
"""
import numpy as np

F32 = np.float32


def _by_division(x, s):
    with np.errstate(all="ignore"):
        q = np.floor(x / s)  # float32 / float32: the IEEE quotient rounded to nearest
    return (np.clip(q, -2, 1) + 2).astype(np.int64)


def _by_comparisons(x, s):
    lo = (x + s) >= (-s * F32(2.0 ** -24))
    mid = x >= F32(0)
    hi = (x - s) >= (-s * F32(2.0 ** -25))
    return lo.astype(np.int64) + mid + hi


def test_two_bit_value_code_comparisons_equal_the_rounded_division():
    rng = np.random.default_rng(0)
    s16 = np.arange(1, 0x7C00, dtype=np.uint16).view(np.float16).astype(F32)  # every positive finite fp16
    checked = 0
    for _ in range(6):
        s = s16[rng.integers(0, len(s16), 200_000)]
        k = rng.choice(np.array([-2, -1, 0, 1, 2], F32), len(s))
        base = (k * s).astype(F32)
        x = (base.view(np.int32) + rng.integers(-8, 9, len(s)).astype(np.int32)).view(F32)  # ulp neighbours
        x = np.where(base == 0, (rng.standard_normal(len(s)) * s * 1e-6).astype(F32), x)
        x = np.concatenate([x, (rng.standard_normal(len(s)) * s * 2).astype(F32)])
        ss = np.concatenate([s, s])
        ok = np.isfinite(x)
        a, b = _by_division(x[ok], ss[ok]), _by_comparisons(x[ok], ss[ok])
        assert np.array_equal(a, b), np.nonzero(a != b)[0][:5]
        checked += int(ok.sum())
    assert checked > 2_000_000
