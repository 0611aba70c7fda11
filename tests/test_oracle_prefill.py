"""Pins of the oracle's causal prefill attention against its decode attention.

prefill_attention builds one masked score matrix per head; decode_attention concatenates the packed and
exact parts of one query without a mask. They share the estimator, so these pins check the masking:
the position of each query, which packed and which exact tokens it sees, and the padding-free shape.
"""
import numpy as np
import pytest

import oracle


def _cache(d, P, R, seed):
    rng = np.random.default_rng(seed)
    D = oracle.rademacher_signs(seed, d)
    S = oracle.gaussian_matrix_bf16(seed, d)
    c, t = oracle.lloyd_max_codebook(d, 2)
    k = rng.standard_normal((P + R, d))
    v = rng.standard_normal((P + R, d))
    keys = oracle.quantize_keys(k[:P], D, S, c, t)
    vals = oracle.quantize_values(v[:P], D, 2)
    return D, S, c, keys, vals, k[P:], v[P:]


def _slice(rec, n):
    return type(rec)(**{f: (getattr(rec, f)[:n] if isinstance(getattr(rec, f), np.ndarray) else getattr(rec, f))
                        for f in rec.__dataclass_fields__})


@pytest.mark.parametrize("P,R", [(256, 40), (128, 128), (0, 9)])
def test_single_query_chunk_is_decode(P, R):
    d, G = 64, 4
    D, S, c, keys, vals, rk, rv = _cache(d, P, R, seed=P + R)
    q = np.random.default_rng(1).standard_normal((1, G, d))
    got = oracle.prefill_attention(q, keys if P else None, vals if P else None, rk, rv, P + R, D, S, c)
    ref = oracle.decode_attention(q[0], keys if P else None, vals if P else None, rk, rv, D, S, c)
    assert np.allclose(got[0], ref, rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("P,R,n_q", [(256, 40, 60), (128, 20, 148), (256, 128, 129)])
def test_each_query_sees_exactly_its_prefix(P, R, n_q):
    """Query i (position L - n_q + i) equals decode over the cache cut at its own position: the packed
    records up to it, and the exact tokens from P up to it."""
    d, G = 64, 2
    L = P + R
    D, S, c, keys, vals, rk, rv = _cache(d, P, R, seed=7 * n_q)
    q = np.random.default_rng(2).standard_normal((n_q, G, d))
    got = oracle.prefill_attention(q, keys, vals, rk, rv, L, D, S, c)
    for i in range(n_q):
        p = L - n_q + i
        np_ = min(P, p + 1)
        nr = max(0, p + 1 - P)
        ref = oracle.decode_attention(q[i], _slice(keys, np_) if np_ else None, _slice(vals, np_) if np_ else None,
                                      rk[:nr], rv[:nr], D, S, c)
        assert np.allclose(got[i], ref, rtol=1e-11, atol=1e-12), i
