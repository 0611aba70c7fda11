"""GPU parity at the full sizes of the batched, head_dim-256 and long-context workloads.

Outputs are sampled, and each workload runs in the launch configuration of its full-batch decode
call. The head_dim-256 workload also reports the cos_sim figures of [Guide] §六.
"""
import numpy as np
import pytest
import torch

import oracle
from kv_cache_quantization_quantize_gb300 import TurboQuantCache, config, synth
from tests.gpu_helpers import check_sequence, f64, i32, oracle_decode, oracle_tables
from tests.parity import rel_l2

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def built():
    from kv_cache_quantization_quantize_gb300 import build
    build.build()


def _prefill_and_step(cache, seqs, extra):
    """Batched prefill of every sequence's first L tokens, then one single-token append per row."""
    B = len(seqs)
    Hkv, d = seqs[0][0].shape[1], seqs[0][0].shape[2]
    lens = [k.shape[0] - extra for k, _ in seqs]
    kb = torch.zeros(B, max(lens), Hkv, d, dtype=torch.bfloat16, device=DEV)
    vb = torch.zeros_like(kb)
    for i, (k, v) in enumerate(seqs):
        kb[i, :lens[i]] = k[:lens[i]]
        vb[i, :lens[i]] = v[:lens[i]]
    ids = i32(list(range(B)))
    cache.append(0, kb, vb, ids, i32(lens))
    del kb, vb
    for s in range(extra):
        kd = torch.stack([k[lens[i] + s] for i, (k, _) in enumerate(seqs)])[:, None].contiguous()
        vd = torch.stack([v[lens[i] + s] for i, (_, v) in enumerate(seqs)])[:, None].contiguous()
        cache.append(0, kd, vd, ids, i32([1] * B))
    torch.cuda.synchronize()
    assert cache.check_status() == 0
    return ids


def test_batched_ragged_decode_v4_sampled():
    """Llama-3.1-8B shapes (32 q heads, 8 KV heads, d=128), batch 16, ragged lengths uniform in [4096, 8192]
    (seed 2), 3-bit keys, 4-bit values, bf16 N(0,1): batched prefill, one decode append, batched decode."""
    d, Hkv, Hq, B = 128, 8, 32, 16
    lens = synth.ragged_lengths(B, 4096, 8192, seed=2)
    cfg = config(head_dim=d, value_bits=4, n_layers=1, n_kv_heads=Hkv, n_q_heads=Hq, max_seqs=B, max_ctx=8192,
                 seed=2)
    cache = TurboQuantCache(cfg)
    tables = oracle_tables(cache)
    seqs = [synth.kv_tokens(L, Hkv, d, seed=2000 + i, device=DEV) for i, L in enumerate(lens)]
    ids = _prefill_and_step(cache, seqs, extra=1)
    q = synth.queries(B, Hq, d, seed=2)
    out = cache.decode(0, q.to(DEV), ids, max_ctx_hint=8192).cpu().numpy()
    assert cache.check_status() == 0
    G = Hq // Hkv
    for i in sorted({0, int(np.argmin(lens)), int(np.argmax(lens)), B - 1}):
        k, v = seqs[i]
        check_sequence(cache, 0, i, k, v, tables, heads=[0, Hkv - 1])
        ref = oracle_decode(cache, 0, i, q[i], tables)
        for hq in range(Hq):
            assert rel_l2(out[i, hq], ref[hq]) <= 2e-3, (i, hq, rel_l2(out[i, hq], ref[hq]))
    assert G == 4


@pytest.mark.parametrize("vb", [2, 4])
def test_head_dim_256_student_t_sampled_and_cos_sim(vb, capsys):
    """head_dim 256, 32 q heads, 8 KV heads, batch 4, context 16384, bf16 Student-t (nu=5) at unit variance
    (seed 3), 3-bit keys with 2- and 4-bit values; the cos_sim report of the dequantised K and V."""
    d, Hkv, Hq, B, L = 256, 8, 32, 4, 16384
    cfg = config(head_dim=d, value_bits=vb, n_layers=1, n_kv_heads=Hkv, n_q_heads=Hq, max_seqs=B, max_ctx=L, seed=3)
    cache = TurboQuantCache(cfg)
    tables = oracle_tables(cache)
    seqs = [synth.kv_tokens(L, Hkv, d, seed=3000 + i, dist="student_t5", device=DEV) for i in range(B)]
    ids = _prefill_and_step(cache, seqs, extra=1)
    q = synth.queries(B, Hq, d, seed=3)
    out = cache.decode(0, q.to(DEV), ids, max_ctx_hint=L).cpu().numpy()
    assert cache.check_status() == 0
    for i in (0, B - 1):
        k, v = seqs[i]
        check_sequence(cache, 0, i, k, v, tables, heads=[0, Hkv - 1])
        ref = oracle_decode(cache, 0, i, q[i], tables)
        for hq in range(Hq):
            assert rel_l2(out[i, hq], ref[hq]) <= 2e-3, (i, hq, rel_l2(out[i, hq], ref[hq]))
    # cos_sim of the device's packed records against the original vectors (sequence 0, KV heads 0 and 7)
    D, S, c, _ = tables
    Np, _ = oracle.history_split(L)
    reps = []
    for h in (0, Hkv - 1):
        kr, vr = cache.records(0, 0, h, Np)
        keys = oracle.unpack_key_records(kr, d)
        vals = oracle.unpack_value_records(vr, d, vb)
        reps.append(oracle.cos_sim_report(f64(seqs[0][0][:Np, h]), f64(seqs[0][1][:Np, h]), keys, vals, D, S, c))
    rep = {key: float(np.mean([r[key] for r in reps])) for key in reps[0]}
    with capsys.disabled():
        print(f"\ncos_sim head_dim 256, K3/V{vb}, Student-t: {rep}")
    assert 0.90 < rep["key_cos_mse"] < 0.97 and rep["key_cos_qjl"] < rep["key_cos_mse"]
    if vb == 2:
        assert 0.85 < rep["value_cos"] < 0.95
    else:
        assert rep["value_cos"] > 0.99


def test_long_context_batch32_decode_sampled():
    """Decode at batch 32 with context 131072 against the resident packed cache (d=128, 8 KV heads,
    32 q heads, K3/V2, bf16 N(0,1) seed 4 with 4 random K channels x10), after per-sequence bulk appends."""
    d, Hkv, Hq, B, L = 128, 8, 32, 32, 131072
    cfg = config(head_dim=d, value_bits=2, n_layers=1, n_kv_heads=Hkv, n_q_heads=Hq, max_seqs=B, max_ctx=L, seed=4)
    cache = TurboQuantCache(cfg)
    tables = oracle_tables(cache)
    sampled = {}
    for i in range(B):
        k, v = synth.kv_tokens(L, Hkv, d, seed=4000 + i, outliers=("random", 4, 10.0), device=DEV)
        cache.append(0, k[None].contiguous(), v[None].contiguous(), i32([i]), i32([L]))
        if i in (0, B - 1):
            sampled[i] = (k[:, 3].cpu(), v[:, 3].cpu())
        del k, v
    torch.cuda.synchronize()
    assert cache.check_status() == 0
    q = synth.queries(B, Hq, d, seed=4)
    out = cache.decode(0, q.to(DEV), i32(list(range(B))), max_ctx_hint=L).cpu().numpy()
    assert cache.check_status() == 0
    D, S, c, t = tables
    Np, R = oracle.history_split(L)
    G = Hq // Hkv
    h = 3
    for i, (k, v) in sampled.items():
        kr, vr = cache.records(0, i, h, Np)
        keys = oracle.unpack_key_records(kr, d)
        vals = oracle.unpack_value_records(vr, d, 2)
        from tests.parity import check_key_records, check_value_records
        check_key_records(keys, f64(k[:Np]), D, S, c, t)
        check_value_records(vals, f64(v[:Np]), D, 2)
        rk, rv = cache.ring(0, i, h)
        assert torch.equal(rk[:R].cpu(), k[Np:]) and torch.equal(rv[:R].cpu(), v[Np:])
        ref = oracle.decode_attention(f64(q[i, h * G:(h + 1) * G]), keys, vals, f64(rk[:R]), f64(rv[:R]), D, S, c)
        for g in range(G):
            assert rel_l2(out[i, h * G + g], ref[g]) <= 2e-3
