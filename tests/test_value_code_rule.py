"""CPU check of the rule the CUDA coders use for 2-bit value codes (host logic, no GPU).

The mid-rise code is clamp(floor(fl(x / s)), -2, 1) + 2, decided on the fp32 quotient rounded to
nearest. The kernels decide it without a division, by three comparisons: [x >= -s] + [x >= 0] + [x >= s].
The rounded quotient reaches -1 from x / s >= -(1 + 2^-24) and 1 from x / s >= 1 - 2^-25; neither
threshold times s has an fp32 strictly between it and -s / s, so for fp32 x the comparisons are exact.
This test restates both rules in numpy float32 and compares them where a slip would show: every positive
finite fp16 scale with x within 64 ulps of -2 s, -s, s and 2 s, random scales with x a few ulps from those
points or near 0, and ordinary values.
"""
import numpy as np

F32 = np.float32
S16 = np.arange(1, 0x7C00, dtype=np.uint16).view(np.float16).astype(F32)  # every positive finite fp16


def _by_division(x, s):
    with np.errstate(all="ignore"):
        q = np.floor(x / s)  # float32 / float32: the IEEE quotient rounded to nearest
    return (np.clip(q, -2, 1) + 2).astype(np.int64)


def _by_comparisons(x, s):
    return (x >= -s).astype(np.int64) + (x >= F32(0)) + (x >= s)


def test_two_bit_value_code_comparisons_equal_the_rounded_division_near_every_threshold():
    n = len(S16)
    s = np.repeat(S16, 4 * 129)
    k = np.tile(np.repeat(np.array([-2, -1, 1, 2], F32), 129), n)
    d = np.tile(np.arange(-64, 65, dtype=np.int32), 4 * n)
    x = ((k * s).astype(F32).view(np.int32) + d).view(F32)  # the 129 fp32 values around k s
    ok = np.isfinite(x)
    a, b = _by_division(x[ok], s[ok]), _by_comparisons(x[ok], s[ok])
    assert np.array_equal(a, b), np.nonzero(a != b)[0][:5]
    assert ok.sum() > 15_000_000


def test_two_bit_value_code_comparisons_equal_the_rounded_division_random():
    rng = np.random.default_rng(0)
    checked = 0
    for _ in range(6):
        s = S16[rng.integers(0, len(S16), 200_000)]
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
