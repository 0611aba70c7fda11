"""tq_dequantize_tokens against the oracle's dequantisers (test infrastructure).

The device reconstructs packed tokens from its own pages; the oracle reconstructs the same tokens from the
canonical records of those pages (fp64, its own rotation matrix and matrix products):
  k_hat = n Pi^T (c[idx] + sqrt(pi/2)/d gamma S^T sigma), with and without the QJL term,
  v_hat = Pi^T ((code - 2^(b-1) + 1/2) s_g).
The two must agree to fp32 rounding (the device sums in fp32). The per-vector cosine against the inputs,
the fidelity figure that the guide's §六 quotes, is computed from both and compared.
"""
import numpy as np
import pytest
import torch

import oracle
from kv_cache_quantization_quantize_gb300 import TurboQuantCache, config, synth
from tests.gpu_helpers import f64, i32, oracle_tables

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _cos(a, b):
    return float(np.mean(np.sum(a * b, axis=1) / (np.linalg.norm(a, axis=1) * np.linalg.norm(b, axis=1))))


@pytest.mark.parametrize("d,vb,kb,dist", [(64, 2, 3, "normal"), (128, 4, 3, "normal"), (256, 2, 3, "student_t5"),
                                          (256, 4, 3, "student_t5"), (128, 4, 4, "normal")])
def test_dequantize_tokens_matches_the_oracle(d, vb, kb, dist):
    Hkv, T = 2, 300  # two complete pages (256 packed tokens) and 44 ring tokens per head
    cfg = config(head_dim=d, value_bits=vb, key_bits=kb, n_layers=1, n_kv_heads=Hkv, n_q_heads=4 * Hkv, max_seqs=2,
                 max_ctx=512, seed=51)
    cache = TurboQuantCache(cfg)
    D, S, c, _ = oracle_tables(cache)
    k, v = synth.kv_tokens(T, Hkv, d, seed=5100 + d, dist=dist, outliers=("random", 4, 10.0))
    cache.append(0, k[None].contiguous().to(DEV), v[None].contiguous().to(DEV), i32([1]), i32([T]))
    torch.cuda.synchronize()
    assert cache.check_status() == 0
    P = 256
    for h in range(Hkv):
        kr, vr = cache.records(0, 1, h, P)
        krec = oracle.unpack_key_records(kr, d, kb)
        vrec = oracle.unpack_value_records(vr, d, vb)
        v_ref = oracle.dequantize_values(vrec, D)
        for with_qjl in (False, True):
            k_ref = oracle.dequantize_keys(krec, D, S, c, with_qjl=with_qjl)
            k_hat, v_hat = cache.dequantize(0, 1, h, 0, P, with_qjl=with_qjl)
            kg, vg = f64(k_hat), f64(v_hat)
            assert np.abs(kg - k_ref).max() <= 2e-5 * np.abs(k_ref).max(), (h, with_qjl)
            assert np.abs(vg - v_ref).max() <= 2e-5 * np.abs(v_ref).max(), h
            ko = f64(k[:P, h])
            assert abs(_cos(kg, ko) - _cos(k_ref, ko)) <= 1e-6
            # a sub-range gives the same rows
            ks, vs = cache.dequantize(0, 1, h, 37, 101, with_qjl=with_qjl)
            assert torch.equal(ks, k_hat[37:138]) and torch.equal(vs, v_hat[37:138])
        assert abs(_cos(vg, f64(v[:P, h])) - _cos(v_ref, f64(v[:P, h]))) <= 1e-6
    assert cache.check_status() == 0
    # the oracle's own report on the same records agrees with the figures above
    rep = oracle.cos_sim_report(f64(k[:P, Hkv - 1]), f64(v[:P, Hkv - 1]), krec, vrec, D, S, c)
    kq, _ = cache.dequantize(0, 1, Hkv - 1, 0, P, with_qjl=True)
    assert abs(rep["key_cos_qjl"] - _cos(f64(kq), f64(k[:P, Hkv - 1]))) <= 1e-6
    assert abs(rep["value_cos"] - _cos(vg, f64(v[:P, Hkv - 1]))) <= 1e-6
    # zero tokens is a no-op; tokens past the sequence's pages are refused on the host
    e0, _ = cache.dequantize(0, 1, 0, 5, 0)
    assert e0.shape == (0, d)
    with pytest.raises(Exception):
        cache.dequantize(0, 1, 0, 500, 20)
