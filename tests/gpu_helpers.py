"""Helpers of the GPU parity tests: oracle tables from the library, record and ring checks, and the
oracle's hybrid attention on the device's own packed records (test infrastructure)."""
import numpy as np
import torch

import oracle
from tests.parity import check_key_records, check_value_records

DEV = "cuda"


def f64(t):
    return t.detach().to("cpu", torch.float64).numpy()


def i32(x):
    return torch.tensor(x, dtype=torch.int32, device=DEV)


def oracle_tables(cache):
    D, S, c, t = cache.tables()
    S64 = (S.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    return D.astype(np.float64), S64, c, t


def check_sequence(cache, layer, slot, k_all, v_all, tables, heads=None):
    """k_all, v_all: [L, Hkv, d] torch (bf16/f32 on any device): check packed records and ring."""
    D, S, c, t = tables
    L = k_all.shape[0]
    Lg, F = cache.state(layer, slot)
    assert Lg == L
    Np, R = oracle.history_split(L)
    P = Np + F
    stats = []
    for h in (range(k_all.shape[1]) if heads is None else heads):
        kr, vr = cache.records(layer, slot, h, P)
        if P:
            kk = oracle.unpack_key_records(kr, cache.cfg.head_dim, cache.cfg.key_bits)
            vv = oracle.unpack_value_records(vr, cache.cfg.head_dim, cache.cfg.value_bits)
            stats.append(check_key_records(kk, f64(k_all[:P, h]), D, S, c, t))
            stats.append(check_value_records(vv, f64(v_all[:P, h]), D, cache.cfg.value_bits))
        rk, rv = cache.ring(layer, slot, h)
        assert torch.equal(rk[:R].cpu(), k_all[Np:L, h].to(torch.bfloat16).cpu())
        assert torch.equal(rv[:R].cpu(), v_all[Np:L, h].to(torch.bfloat16).cpu())
    return stats


def oracle_decode(cache, layer, slot, q_row, tables, scale=None):
    """Oracle hybrid attention for one sequence on the device's own packed records and ring."""
    D, S, c, t = tables
    cfg = cache.cfg
    G = cfg.n_q_heads // cfg.n_kv_heads
    L, F = cache.state(layer, slot)
    Np, R = oracle.history_split(L)
    P = Np + F
    out = np.zeros((cfg.n_q_heads, cfg.head_dim))
    for h in range(cfg.n_kv_heads):
        kr, vr = cache.records(layer, slot, h, P)
        keys = oracle.unpack_key_records(kr, cfg.head_dim, cfg.key_bits) if P else None
        vals = oracle.unpack_value_records(vr, cfg.head_dim, cfg.value_bits) if P else None
        rk, rv = cache.ring(layer, slot, h)
        out[h * G:(h + 1) * G] = oracle.decode_attention(
            f64(q_row[h * G:(h + 1) * G]), keys, vals, f64(rk[F:R]), f64(rv[F:R]), D, S, c, softmax_scale=scale)
    return out
