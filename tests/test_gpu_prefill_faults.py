"""Bounded waits of the tcgen05 prefill kernel, tested without a GPU fault.

A host-set hook (tq_debug_prefill_wait_fault) makes CTA (0, 0, 0) of the launch (query tile 0, KV head 0,
batch row 0, history split 0) leave one page copy unissued: no copy and no expected-byte count, so nothing
can land later. Its wait gives up after a few polls, and that CTA takes the error path: it sets
TQ_DEV_ERR_TIMEOUT, waits (bounded) for the copies and MMA batches it did issue, frees its tensor memory and
writes an empty partial. Every other CTA is untouched, so every output outside that CTA's 32 queries x 4
query heads must equal, bit for bit, the output of the same call without the hook (the kernel's arithmetic
order is fixed). The next call with the hook off must equal the clean call everywhere.
"""
import pytest
import torch

from kv_cache_quantization_quantize_gb300 import TurboQuantCache, _abi, config, synth
from tests.gpu_helpers import i32

pytestmark = pytest.mark.gpu
DEV = "cuda"


def test_prefill_wait_timeout_is_reported_and_other_outputs_are_unchanged():
    lib = _abi.load()
    d, Hkv, G = 128, 8, 4
    hist, chunk = 1500, 256  # 8 query tiles x 8 KV heads: 64 CTAs per split, so 2 splits of about 7 pages
    T = hist + chunk
    cfg = config(head_dim=d, value_bits=2, n_layers=1, n_kv_heads=Hkv, n_q_heads=Hkv * G, max_seqs=1,
                 max_ctx=2048, seed=43)
    cache = TurboQuantCache(cfg)
    k, v = synth.kv_tokens(T, Hkv, d, seed=4300, outliers=("random", 4, 10.0))
    ids = i32([0])
    cache.append(0, k[None].contiguous().to(DEV), v[None].contiguous().to(DEV), ids, i32([T]))
    torch.cuda.synchronize()
    assert cache.check_status() == 0
    q = synth.queries(chunk, Hkv * G, d, seed=4301).view(1, chunk, Hkv * G, d).to(DEV)
    nq = i32([chunk])
    clean = cache.prefill(0, q, ids, nq).cpu()
    assert cache.check_status() == 0
    assert torch.isfinite(clean).all()
    mask = torch.ones_like(clean, dtype=torch.bool)  # outputs outside CTA (0, 0, 0)
    mask[0, :32, :G] = False
    # page 0 and 1: the copies before the loop; page 3: a copy issued inside the loop (after three pages)
    for page in (0, 1, 3):
        assert lib.tq_debug_prefill_wait_fault(page, 8) == _abi.TQ_OK
        try:
            out = cache.prefill(0, q, ids, nq).cpu()
            torch.cuda.synchronize()
        finally:
            assert lib.tq_debug_prefill_wait_fault(-1, 0) == _abi.TQ_OK
        assert cache.check_status() & _abi.TQ_DEV_ERR_TIMEOUT, page
        assert torch.equal(out[mask], clean[mask]), page
        again = cache.prefill(0, q, ids, nq).cpu()
        assert cache.check_status() == 0, page
        assert torch.equal(again, clean), page
