"""GPU test of tq_decode_attention_noalloc, the decode entry point that takes no caller scratch.

It exists for callers that cannot allocate device memory when they decode. Such a caller passes
only q, out and the sequence ids; the library uses a fixed 4 MiB device array of its own as
scratch. This file is collected last, so a run that stops at the first failure has already run
every other test.
"""
import ctypes

import numpy as np
import pytest
import torch

from kv_cache_quantization_quantize_gb300 import TurboQuantCache, _abi, config, synth

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def built():
    from kv_cache_quantization_quantize_gb300 import build
    build.build()


def _noalloc(cache, layer, q, out, ids, scale=0.0, hint=0):
    lib = _abi.load()
    return lib.tq_decode_attention_noalloc(cache.ctx, layer, ctypes.c_void_p(q.data_ptr()),
                                           ctypes.c_void_p(out.data_ptr()), ctypes.c_void_p(ids.data_ptr()),
                                           q.shape[0], float(scale), hint,
                                           ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


def _rel_l2(a, b):
    a, b = a.double(), b.double()
    return float(torch.linalg.norm(a - b) / torch.linalg.norm(b))


def test_noalloc_matches_workspace_decode_on_two_calls():
    d, Hkv, G = 128, 2, 4
    lens = [5, 200, 1000, 129]
    cfg = config(head_dim=d, value_bits=2, n_layers=1, n_kv_heads=Hkv, n_q_heads=Hkv * G, max_seqs=4, max_ctx=1200,
                 seed=21)
    cache = TurboQuantCache(cfg)
    B = len(lens)
    k = torch.zeros(B, max(lens), Hkv, d, dtype=torch.bfloat16)
    v = torch.zeros_like(k)
    for i, L in enumerate(lens):
        kk, vv = synth.kv_tokens(L, Hkv, d, seed=40 + i, outliers=("random", 4, 10.0))
        k[i, :L], v[i, :L] = kk, vv
    ids = torch.arange(B, dtype=torch.int32, device=DEV)
    cache.append(0, k.to(DEV), v.to(DEV), ids, torch.tensor(lens, dtype=torch.int32, device=DEV))
    q = synth.queries(B, Hkv * G, d, seed=8).to(DEV)
    ref = cache.decode(0, q, ids)
    torch.cuda.synchronize()
    for _ in range(2):  # the scratch keeps the previous call's contents; results must not depend on it
        out = torch.full_like(ref, float("nan"))
        assert _noalloc(cache, 0, q, out, ids) == _abi.TQ_OK, _abi.load().tq_last_error()
        torch.cuda.synchronize()
        assert torch.isfinite(out).all()
        for i in range(B):
            for h in range(Hkv * G):
                assert _rel_l2(out[i, h], ref[i, h]) <= 2e-3
    assert cache.check_status() == 0


def test_noalloc_rejects_scratch_above_its_limit():
    # batch 64 x 8 KV heads at head_dim 256 needs more than the built-in 4 MiB of scratch: every plan has at
    # least 3 partials of 4128 bytes per (row, KV head)
    d, Hkv, G, B, L = 256, 8, 4, 64, 256
    cfg = config(head_dim=d, value_bits=2, n_layers=1, n_kv_heads=Hkv, n_q_heads=Hkv * G, max_seqs=B, max_ctx=L,
                 seed=2)
    cache = TurboQuantCache(cfg)
    assert cache.workspace_bytes(B, L) > (4 << 20)
    ids = torch.arange(B, dtype=torch.int32, device=DEV)
    q = torch.zeros(B, Hkv * G, d, dtype=torch.bfloat16, device=DEV)
    out = torch.full((B, Hkv * G, d), 7.0, dtype=torch.float32, device=DEV)
    st = _noalloc(cache, 0, q, out, ids, hint=L)
    assert st == _abi.TQ_ERR_CAPACITY
    msg = _abi.load().tq_last_error().decode()
    assert "exceeds" in msg and str(4 << 20) in msg
    torch.cuda.synchronize()
    assert torch.all(out == 7.0)  # nothing was launched


def _cache_with_history(max_seqs, lens, Hkv, d, seed):
    cfg = config(head_dim=d, value_bits=2, n_layers=1, n_kv_heads=Hkv, n_q_heads=Hkv * 4, max_seqs=max_seqs,
                 max_ctx=1200, seed=seed)
    cache = TurboQuantCache(cfg)
    B = len(lens)
    k = torch.zeros(B, max(lens), Hkv, d, dtype=torch.bfloat16)
    v = torch.zeros_like(k)
    for i, L in enumerate(lens):
        kk, vv = synth.kv_tokens(L, Hkv, d, seed=seed * 10 + i, outliers=("random", 4, 10.0))
        k[i, :L], v[i, :L] = kk, vv
    ids = torch.arange(B, dtype=torch.int32, device=DEV)
    cache.append(0, k.to(DEV), v.to(DEV), ids, torch.tensor(lens, dtype=torch.int32, device=DEV))
    q = synth.queries(B, Hkv * 4, d, seed=seed).to(DEV)
    return cache, ids, q


def test_noalloc_alternating_contexts_of_different_shapes():
    """The one scratch array serves every context. Calls alternate between a context with one sequence
    slot and one with sixteen (8 KV heads each): the small context's partials must never land on the
    large context's arrival counters. Both match the workspace decode on every call."""
    d, Hkv = 128, 8
    big, ids_b, q_b = _cache_with_history(16, [300 + 37 * i for i in range(16)], Hkv, d, seed=5)
    small, ids_s, q_s = _cache_with_history(1, [900], Hkv, d, seed=6)
    ref_b = big.decode(0, q_b, ids_b)
    ref_s = small.decode(0, q_s, ids_s)
    torch.cuda.synchronize()
    for _ in range(2):
        for cache, q, ids, ref in ((big, q_b, ids_b, ref_b), (small, q_s, ids_s, ref_s), (big, q_b, ids_b, ref_b)):
            out = torch.full_like(ref, float("nan"))
            assert _noalloc(cache, 0, q, out, ids) == _abi.TQ_OK, _abi.load().tq_last_error()
            torch.cuda.synchronize()
            assert torch.isfinite(out).all()
            for i in range(q.shape[0]):
                for h in range(q.shape[1]):
                    assert _rel_l2(out[i, h], ref[i, h]) <= 2e-3
    assert big.check_status() == 0 and small.check_status() == 0
