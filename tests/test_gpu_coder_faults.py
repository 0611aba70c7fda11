"""Bounded waits of the tcgen05 bulk coders (head_dim 64, 128 and 256), tested without a GPU fault.

A host-set hook (tq_debug_append_wait_fault) makes one page task's TMA copy go unissued: no copy and no
expected-byte count, so nothing can land later. The wait on it gives up after a few polls, and the owning
CTA takes the error path: it sets TQ_DEV_ERR_TIMEOUT, waits (bounded) for the copies and MMA batches it did
issue, frees its tensor memory and returns. Every page of the other CTAs must be exact, and the next append
with the hook off must be exact everywhere.
"""
import numpy as np
import pytest
import torch

import oracle
from kv_cache_quantization_quantize_gb300 import TurboQuantCache, _abi, config, synth
from tests.gpu_helpers import check_sequence, f64, i32, oracle_tables
from tests.parity import check_key_records, check_value_records

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _check_pages(cache, slot, h, k_all, v_all, tables, pages):
    """Records of the listed 128-token pages of (slot, head h) against the oracle."""
    D, S, c, t = tables
    cfg = cache.cfg
    P = 128 * (max(pages) + 1)
    kr, vr = cache.records(0, slot, h, P)
    kk = oracle.unpack_key_records(kr, cfg.head_dim, cfg.key_bits)
    vv = oracle.unpack_value_records(vr, cfg.head_dim, cfg.value_bits)
    rows = np.concatenate([np.arange(128 * p, 128 * (p + 1)) for p in pages])
    ks = oracle.KeyRecords(idx=kk.idx[rows], sign=kk.sign[rows], norm=kk.norm[rows], gamma=kk.gamma[rows],
                           mse_bits=kk.mse_bits)
    vs = oracle.ValueRecords(codes=vv.codes[rows], scales=vv.scales[rows], bits=vv.bits)
    tr = torch.as_tensor(rows)
    check_key_records(ks, f64(k_all[tr, h]), D, S, c, t)
    check_value_records(vs, f64(v_all[tr, h]), D, cfg.value_bits)


@pytest.mark.parametrize("d", [64, 128, 256])
def test_bulk_coder_wait_timeout_is_reported_and_the_cache_stays_usable(d):
    lib = _abi.load()
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    ctas = sms * (2 if d == 64 else 1)  # persistent CTAs: two per SM at head_dim 64, else one
    Hkv, G, B = 8, 4, 2
    npg = -(-(ctas + 1) // (B * Hkv))  # complete pages per row: more page tasks than CTAs
    T = 128 * npg + 37                  # npg complete pages and a 37-token ring per row
    ppr = -(-T // 128)                  # page tasks per row as the append numbers them: ceil(max_new / 128)
    ntasks = B * Hkv * ppr
    grid = min(ntasks, ctas)            # CTA 0 owns tasks 0, grid, 2 grid, ...
    assert ntasks > grid
    cfg = config(head_dim=d, value_bits=2, n_layers=1, n_kv_heads=Hkv, n_q_heads=Hkv * G, max_seqs=B,
                 max_ctx=T + 128, seed=41)
    cache = TurboQuantCache(cfg)
    tables = oracle_tables(cache)
    seqs = [synth.kv_tokens(T, Hkv, d, seed=4100 + i) for i in range(B)]
    k = torch.stack([s[0] for s in seqs]).to(DEV)
    v = torch.stack([s[1] for s in seqs]).to(DEV)
    ids = i32(list(range(B)))
    nn = i32([T] * B)
    # task 0: CTA 0's first page copy (before its loop); task `grid`: its second, after a page in flight
    for task in (0, grid):
        cache.reset(ids)
        assert lib.tq_debug_append_wait_fault(task, 8) == _abi.TQ_OK
        try:
            cache.append(0, k, v, ids, nn)
            torch.cuda.synchronize()
        finally:
            assert lib.tq_debug_append_wait_fault(-1, 0) == _abi.TQ_OK
        assert cache.check_status() & _abi.TQ_DEV_ERR_TIMEOUT, task
        # the pages of CTA 0 (tasks 0, grid, 2 grid, ...) are unspecified; every other page is exact
        for b in range(B):
            for h in range(Hkv):
                pages = [j for j in range(npg) if ((b * Hkv + h) * ppr + j) % grid != 0]
                _check_pages(cache, b, h, seqs[b][0], seqs[b][1], tables, pages)
                rk, rv = cache.ring(0, b, h)
                assert torch.equal(rk[:37].cpu(), seqs[b][0][128 * npg:, h].to(torch.bfloat16).cpu())
        # the next append, hook off: exact everywhere, and the status clean
        cache.reset(ids)
        cache.append(0, k, v, ids, nn)
        torch.cuda.synchronize()
        assert cache.check_status() == 0, task
        for b in range(B):
            check_sequence(cache, 0, b, seqs[b][0], seqs[b][1], tables)
