"""GPU parity: the CUDA path (through the C ABI) against the fp64 oracle on the same seeded inputs."""
import numpy as np
import pytest
import torch

import oracle
from kv_cache_quantization_quantize_gb300 import TurboQuantCache, config, synth
from tests.gpu_helpers import check_sequence as _check_sequence, f64 as _f64, i32 as _i32
from tests.gpu_helpers import oracle_decode as _oracle_decode, oracle_tables as _oracle_tables
from tests.parity import rel_l2

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def built():
    from kv_cache_quantization_quantize_gb300 import build
    build.build()


def test_tiny_single_head_config():
    """1 layer, 1 KV head, 1 query head, d=128: 1024 packed + 128 ring tokens, fp32 N(0,1), seed 0,
    K channels 3 and 77 scaled x8; 3-bit keys, 2-bit values (g32); one decode step."""
    cfg = config(head_dim=128, value_bits=2, n_layers=1, n_kv_heads=1, n_q_heads=1, max_seqs=1, max_ctx=1152, seed=0)
    cache = TurboQuantCache(cfg)
    k, v = synth.kv_tokens(1152, 1, 128, seed=0, outliers=("fixed", (3, 77), 8.0), dtype=torch.float32)
    cache.append(0, k[None].to(DEV).contiguous(), v[None].to(DEV).contiguous(), _i32([0]), _i32([1152]))
    torch.cuda.synchronize()
    tables = _oracle_tables(cache)
    assert cache.state(0, 0) == (1152, 0)
    _check_sequence(cache, 0, 0, k, v, tables)
    q = synth.queries(1, 1, 128, seed=0)
    out = cache.decode(0, q.to(DEV), _i32([0]))
    ref = _oracle_decode(cache, 0, 0, q[0], tables)
    assert rel_l2(out[0].cpu().numpy(), ref) <= 2e-3
    assert cache.check_status() == 0


@pytest.mark.parametrize("d,vb,G,kbits", [(128, 2, 4, 3), (128, 4, 4, 3), (256, 2, 4, 3), (256, 4, 2, 3), (128, 2, 1, 3),
                                          (64, 2, 4, 3), (64, 4, 2, 3), (128, 4, 4, 4), (64, 4, 2, 4), (256, 4, 4, 4)])
def test_ragged_batch_appends_and_decode(d, vb, G, kbits):
    """Ragged lengths across several tiles and a ragged tail: 1, 127, 128, 129, 300, 1000 tokens,
    built by a prefill append and then single-token decode appends (ring overflow and flush).
    kbits 4: 3-bit Lloyd-Max index + QJL sign."""
    Hkv = 2
    lens = [1, 127, 128, 129, 300, 1000]
    B = len(lens)
    cfg = config(head_dim=d, value_bits=vb, n_layers=2, n_kv_heads=Hkv, n_q_heads=Hkv * G, max_seqs=8,
                 max_ctx=1200, seed=11, key_bits=kbits)
    cache = TurboQuantCache(cfg)
    tables = _oracle_tables(cache)
    layer, decode_steps = 1, 3
    seqs = [synth.kv_tokens(L + decode_steps, Hkv, d, seed=100 + i, outliers=("random", 4, 10.0))
            for i, L in enumerate(lens)]
    slots = [7, 0, 3, 1, 5, 2]
    max_new = max(lens)
    kb = torch.zeros(B, max_new, Hkv, d, dtype=torch.bfloat16)
    vbuf = torch.zeros_like(kb)
    for i, L in enumerate(lens):
        kb[i, :L] = seqs[i][0][:L]
        vbuf[i, :L] = seqs[i][1][:L]
    cache.append(layer, kb.to(DEV), vbuf.to(DEV), _i32(slots), _i32(lens))
    for s in range(decode_steps):
        kd = torch.stack([seqs[i][0][L + s] for i, L in enumerate(lens)])[:, None].contiguous()
        vd = torch.stack([seqs[i][1][L + s] for i, L in enumerate(lens)])[:, None].contiguous()
        cache.append(layer, kd.to(DEV), vd.to(DEV), _i32(slots), _i32([1] * B))
    torch.cuda.synchronize()
    assert cache.check_status() == 0
    for i, L in enumerate(lens):
        _check_sequence(cache, layer, slots[i], seqs[i][0], seqs[i][1], tables)
    q = synth.queries(B, Hkv * G, d, seed=5)
    worst = 0.0
    for scale in (0.0, 0.05):
        out = cache.decode(layer, q.to(DEV), _i32(slots), softmax_scale=scale).cpu().numpy()
        for i in range(B):
            ref = _oracle_decode(cache, layer, slots[i], q[i], tables, scale=None if scale == 0 else scale)
            for hq in range(Hkv * G):
                err = rel_l2(out[i, hq], ref[hq])
                worst = max(worst, err)
                assert err <= 2e-3, (i, hq, err)
    print(f"decode d={d} V{vb} G{G} K{kbits}: worst rel-L2 {worst:.2e}")
    # other layer untouched: empty sequences attend to nothing
    out0 = cache.decode(0, q.to(DEV), _i32(slots)).cpu()
    assert torch.all(out0 == 0)


@pytest.mark.parametrize("d,vb", [(128, 2), (64, 4), (256, 2)])
def test_append_then_decode_back_to_back(d, vb):
    """The decode step as a server issues it: on every layer a one-token append is followed at once by
    the decode, with no synchronisation in between, while different rows cross a 128-token page
    boundary (a page is coded) on different steps. Every decode output is checked against the oracle
    on the cache as that decode saw it."""
    Hkv, G, n_layers, steps = 2, 4, 3, 4
    lens = [126, 127, 128, 255, 256, 383]
    B = len(lens)
    cfg = config(head_dim=d, value_bits=vb, n_layers=n_layers, n_kv_heads=Hkv, n_q_heads=Hkv * G, max_seqs=B,
                 max_ctx=400, seed=21)
    cache = TurboQuantCache(cfg)
    tables = _oracle_tables(cache)
    slots = list(range(B))
    max_new = max(lens)
    seqs = {}
    for layer in range(n_layers):
        kb = torch.zeros(B, max_new, Hkv, d, dtype=torch.bfloat16)
        vbuf = torch.zeros_like(kb)
        for i, L in enumerate(lens):
            k, v = synth.kv_tokens(L + steps, Hkv, d, seed=300 + 10 * layer + i)
            seqs[layer, i] = (k, v)
            kb[i, :L], vbuf[i, :L] = k[:L], v[:L]
        cache.append(layer, kb.to(DEV), vbuf.to(DEV), _i32(slots), _i32(lens))
    ones, ids = _i32([1] * B), _i32(slots)
    ws = cache.workspace(B)
    outs = torch.empty((n_layers, B, Hkv * G, d), dtype=torch.float32, device=DEV)
    torch.cuda.synchronize()
    worst = 0.0
    for s in range(steps):
        qs = [synth.queries(B, Hkv * G, d, seed=40 + 7 * s + layer) for layer in range(n_layers)]
        # every input of the step is on the device first, so that nothing but the library's own
        # kernels runs between an append and its decode
        kds = [torch.stack([seqs[layer, i][0][L + s] for i, L in enumerate(lens)])[:, None].contiguous().to(DEV)
               for layer in range(n_layers)]
        vds = [torch.stack([seqs[layer, i][1][L + s] for i, L in enumerate(lens)])[:, None].contiguous().to(DEV)
               for layer in range(n_layers)]
        qd = [q.to(DEV) for q in qs]
        torch.cuda.synchronize()
        for layer in range(n_layers):
            cache.append(layer, kds[layer], vds[layer], ids, ones)
            cache.decode(layer, qd[layer], ids, out=outs[layer], workspace=ws)
        torch.cuda.synchronize()
        assert cache.check_status() == 0
        for layer in range(n_layers):
            out = outs[layer].cpu().numpy()
            for i in range(B):
                assert cache.state(layer, i)[0] == lens[i] + s + 1
                ref = _oracle_decode(cache, layer, i, qs[layer][i], tables)
                for hq in range(Hkv * G):
                    err = rel_l2(out[i, hq], ref[hq])
                    worst = max(worst, err)
                    assert err <= 2e-3, (s, layer, i, hq, err)
    print(f"back-to-back append + decode d={d} V{vb}: worst rel-L2 {worst:.2e}")


@pytest.mark.parametrize("d,vb", [(128, 2), (64, 4), (256, 2)])
def test_prefill_right_after_a_small_append(d, vb):
    """A chunk of fewer than 128 tokens that codes no page (the small-append kernel releases the next
    launch as it starts), followed at once by its prefill attention: every query's causal length comes
    from the new sequence length, so query 0 of a 100-token chunk appended at 1025 tokens still sees all
    1024 packed tokens. Checked against the oracle on the device's own records and ring."""
    Hkv, G = 2, 4
    hist, nq = 1025, 100
    cfg = config(head_dim=d, value_bits=vb, n_layers=1, n_kv_heads=Hkv, n_q_heads=Hkv * G, max_seqs=1,
                 max_ctx=1152, seed=17)
    cache = TurboQuantCache(cfg)
    tables = _oracle_tables(cache)
    k, v = synth.kv_tokens(hist + nq, Hkv, d, seed=800, outliers=("random", 4, 10.0))
    ids = _i32([0])
    cache.append(0, k[None, :hist].to(DEV).contiguous(), v[None, :hist].to(DEV).contiguous(), ids, _i32([hist]))
    kc, vc = k[None, hist:].to(DEV).contiguous(), v[None, hist:].to(DEV).contiguous()
    q = synth.queries(nq, Hkv * G, d, seed=18).view(1, nq, Hkv * G, d).contiguous().to(DEV)
    n_q, ws = _i32([nq]), cache.prefill_workspace(1, nq)
    out = torch.empty((1, nq, Hkv * G, d), dtype=torch.float32, device=DEV)
    torch.cuda.synchronize()
    cache.append(0, kc, vc, ids, n_q)  # 100 tokens: 1125 <= 1152, no page is coded
    cache.prefill(0, q, ids, n_q, out=out, workspace=ws)
    torch.cuda.synchronize()
    assert cache.check_status() == 0
    L, F = cache.state(0, 0)
    assert L == hist + nq
    Np, R = oracle.history_split(L)
    assert Np == 1024
    D, S, c, t = tables
    outn = out.cpu().numpy()
    worst = 0.0
    for h in range(Hkv):
        kr, vr = cache.records(0, 0, h, Np + F)
        keys = oracle.unpack_key_records(kr, d, cache.cfg.key_bits)
        vals = oracle.unpack_value_records(vr, d, vb)
        rk, rv = cache.ring(0, 0, h)
        qh = _f64(q[0, :, h * G:(h + 1) * G])
        ref = oracle.prefill_attention(qh, keys, vals, _f64(rk[F:R]), _f64(rv[F:R]), L, D, S, c)
        for j in range(nq):
            for g in range(G):
                err = rel_l2(outn[0, j, h * G + g], ref[j, g])
                worst = max(worst, err)
                assert err <= 2e-3, (j, h, g, err)
    print(f"prefill right after a small append d={d} V{vb}: worst rel-L2 {worst:.2e}")


def test_ring_flush_then_decode_and_overflow():
    d, vb, G, Hkv = 128, 2, 4, 2
    cfg = config(head_dim=d, value_bits=vb, n_layers=1, n_kv_heads=Hkv, n_q_heads=Hkv * G, max_seqs=2,
                 max_ctx=600, seed=3)
    cache = TurboQuantCache(cfg)
    tables = _oracle_tables(cache)
    k, v = synth.kv_tokens(400, Hkv, d, seed=9)
    cache.append(0, k[None, :290].to(DEV).contiguous(), v[None, :290].to(DEV).contiguous(), _i32([1]), _i32([290]))
    cache.flush(0, _i32([1]))
    torch.cuda.synchronize()
    assert cache.state(0, 1) == (290, 34)  # 256 packed + 34-token ring, flushed in full
    _check_sequence(cache, 0, 1, k[:290], v[:290], tables)
    q = synth.queries(1, Hkv * G, d, seed=1)
    out = cache.decode(0, q.to(DEV), _i32([1])).cpu().numpy()
    ref = _oracle_decode(cache, 0, 1, q[0], tables)
    assert rel_l2(out[0], ref) <= 2e-3
    # continue appending past the block: the flushed block is re-quantised identically
    cache.append(0, k[None, 290:400].to(DEV).contiguous(), v[None, 290:400].to(DEV).contiguous(), _i32([1]), _i32([110]))
    torch.cuda.synchronize()
    assert cache.state(0, 1) == (400, 0)
    _check_sequence(cache, 0, 1, k[:400], v[:400], tables)
    # capacity overflow is reported on the device status word and leaves the row untouched
    big = torch.zeros(1, 300, Hkv, d, dtype=torch.bfloat16, device=DEV)
    cache.append(0, big, big, _i32([1]), _i32([300]))
    assert cache.check_status() & 0x1
    assert cache.state(0, 1) == (400, 0)
    # a bad sequence id is reported and skipped
    cache.append(0, big[:, :1].contiguous(), big[:, :1].contiguous(), _i32([5]), _i32([1]))
    assert cache.check_status() & 0x2


def test_full_size_llama_layer_sampled():
    """One layer at the Llama-3.1-8B decode shape (32 q heads, 8 KV heads, d=128, 32K context, K3/V2,
    bf16 N(0,1) seed 1 with 4 random K channels x10), in the bench's launch configuration; sampled heads
    are checked against the oracle."""
    d, Hkv, Hq, L = 128, 8, 32, 32768
    cfg = config(head_dim=d, value_bits=2, n_layers=1, n_kv_heads=Hkv, n_q_heads=Hq, max_seqs=1, max_ctx=L + 64, seed=1)
    cache = TurboQuantCache(cfg)
    tables = _oracle_tables(cache)
    k, v = synth.kv_tokens(L, Hkv, d, seed=1, outliers=("random", 4, 10.0), device=DEV)
    cache.append(0, k[None].contiguous(), v[None].contiguous(), _i32([0]), _i32([L]))
    q = synth.queries(1, Hq, d, seed=1)
    out = cache.decode(0, q.to(DEV), _i32([0]), max_ctx_hint=L).cpu().numpy()
    assert cache.check_status() == 0
    kc, vc = k.cpu(), v.cpu()
    for h in (0, 5):
        _check_sequence(cache, 0, 0, kc, vc, tables, heads=[h])
    G = Hq // Hkv
    D, S, c, t = tables
    Np, R = oracle.history_split(L)
    for h in (0, 5):
        kr, vr = cache.records(0, 0, h, Np)
        keys = oracle.unpack_key_records(kr, d, cache.cfg.key_bits)
        vals = oracle.unpack_value_records(vr, d, 2)
        rk, rv = cache.ring(0, 0, h)
        ref = oracle.decode_attention(_f64(q[0, h * G:(h + 1) * G]), keys, vals, _f64(rk[:R]), _f64(rv[:R]), D, S, c)
        for g in range(G):
            assert rel_l2(out[0, h * G + g], ref[g]) <= 2e-3


@pytest.mark.parametrize("d,vb,kbits", [(128, 2, 3), (128, 4, 3), (256, 2, 3), (64, 4, 3), (128, 4, 4)])
def test_bulk_append_onto_a_partial_ring(d, vb, kbits):
    """Bulk appends (>= 128 tokens) onto sequences whose ring is partly full: the first page written
    takes its leading tokens from the ring and the rest from the new input; later pages come from the
    input only. Rows: ring of 72, 1 and 128 tokens before the second append."""
    Hkv, G = 2, 4
    first, second = [200, 129, 128], [300, 260, 130]
    B = len(first)
    cfg = config(head_dim=d, value_bits=vb, n_layers=1, n_kv_heads=Hkv, n_q_heads=Hkv * G, max_seqs=B, max_ctx=600,
                 seed=17, key_bits=kbits)
    cache = TurboQuantCache(cfg)
    tables = _oracle_tables(cache)
    seqs = [synth.kv_tokens(f + s_, Hkv, d, seed=300 + i, outliers=("random", 4, 10.0))
            for i, (f, s_) in enumerate(zip(first, second))]
    ids = _i32(list(range(B)))
    for part, lens in ((0, first), (1, second)):
        n = max(lens)
        kb = torch.zeros(B, n, Hkv, d, dtype=torch.bfloat16)
        vbuf = torch.zeros_like(kb)
        for i in range(B):
            lo = 0 if part == 0 else first[i]
            kb[i, :lens[i]] = seqs[i][0][lo:lo + lens[i]]
            vbuf[i, :lens[i]] = seqs[i][1][lo:lo + lens[i]]
        cache.append(0, kb.to(DEV), vbuf.to(DEV), ids, _i32(lens))
    torch.cuda.synchronize()
    assert cache.check_status() == 0
    for i in range(B):
        _check_sequence(cache, 0, i, seqs[i][0], seqs[i][1], tables)
    q = synth.queries(B, Hkv * G, d, seed=17)
    out = cache.decode(0, q.to(DEV), ids).cpu().numpy()
    for i in range(B):
        ref = _oracle_decode(cache, 0, i, q[i], tables)
        for hq in range(Hkv * G):
            assert rel_l2(out[i, hq], ref[hq]) <= 2e-3


@pytest.mark.parametrize("d,vb,kbits", [(128, 2, 3), (256, 4, 3), (64, 2, 3), (128, 4, 4)])
def test_full_tq_mode_appends_and_decode(d, vb, kbits):
    """full_tq mode (ring_size 0, [Guide] §三): every appended token is quantised by its own append and
    decode reads packed tokens only. A bulk prefill of 300 tokens, three single-token appends, then an
    82-token append that completes a page and starts the next (303 -> 385). After every step all L
    tokens are packed, the records equal the oracle's codes of every token, and decode matches the
    oracle's attention over the packed tokens with no exact ring."""
    Hkv, G, slot = 2, 4, 1
    cfg = config(head_dim=d, value_bits=vb, n_layers=1, n_kv_heads=Hkv, n_q_heads=Hkv * G, max_seqs=2,
                 max_ctx=640, seed=21, mode="full_tq", key_bits=kbits)
    cache = TurboQuantCache(cfg)
    tables = _oracle_tables(cache)
    k, v = synth.kv_tokens(400, Hkv, d, seed=21, outliers=("random", 4, 10.0))
    q = synth.queries(1, Hkv * G, d, seed=21)
    L = 0
    for n in (300, 1, 1, 1, 82):
        cache.append(0, k[None, L:L + n].to(DEV).contiguous(), v[None, L:L + n].to(DEV).contiguous(),
                     _i32([slot]), _i32([n]))
        L += n
        torch.cuda.synchronize()
        assert cache.check_status() == 0
        Lg, F = cache.state(0, slot)
        Np, R = oracle.history_split(L)
        assert Lg == L and Np + F == L and oracle.history_split(L, 0) == (L, 0)
        _check_sequence(cache, 0, slot, k[:L], v[:L], tables)
        out = cache.decode(0, q.to(DEV), _i32([slot])).cpu().numpy()
        ref = _oracle_decode(cache, 0, slot, q[0], tables)  # packed records only: the ring part is empty
        for hq in range(Hkv * G):
            assert rel_l2(out[0, hq], ref[hq]) <= 2e-3, (L, hq, rel_l2(out[0, hq], ref[hq]))


@pytest.mark.parametrize("d,vb,kbits", [(128, 2, 3), (256, 4, 3), (64, 4, 3), (256, 4, 4)])
def test_paged_cache_scrambled_block_table(d, vb, kbits):
    """Paged cache (n_blocks > 0): three sequences (300, 129 and 1000 tokens, then two single-token
    appends) share one pool of 24 blocks through a scrambled block table. Their pages are byte-identical
    to those of the contiguous layout fed the same inputs, decode outputs are identical, and both match
    the oracle. A page with no block is reported on the status word without a fault."""
    Hkv, G, extra = 2, 4, 2
    lens, slots = [300, 129, 1000], [2, 0, 1]
    B, max_ctx = len(lens), 1100
    common = dict(head_dim=d, value_bits=vb, n_layers=2, n_kv_heads=Hkv, n_q_heads=Hkv * G, max_seqs=3,
                  max_ctx=max_ctx, seed=5, key_bits=kbits)
    paged = TurboQuantCache(config(n_blocks=24, **common))
    flat = TurboQuantCache(config(**common))
    perm = torch.randperm(24, generator=torch.Generator().manual_seed(3))
    bt, nxt = paged.block_table, 0
    for s_, L in zip(slots, lens):
        for pg in range((L + extra + 127) // 128):
            bt[s_, pg] = int(perm[nxt])
            nxt += 1
    tables = _oracle_tables(paged)
    seqs = [synth.kv_tokens(L + extra, Hkv, d, seed=500 + i, outliers=("random", 4, 10.0)) for i, L in enumerate(lens)]
    kb = torch.zeros(B, max(lens), Hkv, d, dtype=torch.bfloat16)
    vbuf = torch.zeros_like(kb)
    for i, L in enumerate(lens):
        kb[i, :L] = seqs[i][0][:L]
        vbuf[i, :L] = seqs[i][1][:L]
    layer = 1
    for cache in (paged, flat):
        cache.append(layer, kb.to(DEV), vbuf.to(DEV), _i32(slots), _i32(lens))
        for s in range(extra):
            kd = torch.stack([seqs[i][0][L + s] for i, L in enumerate(lens)])[:, None].contiguous()
            vd = torch.stack([seqs[i][1][L + s] for i, L in enumerate(lens)])[:, None].contiguous()
            cache.append(layer, kd.to(DEV), vd.to(DEV), _i32(slots), _i32([1] * B))
    torch.cuda.synchronize()
    assert paged.check_status() == 0 and flat.check_status() == 0
    for i, s_ in enumerate(slots):
        assert paged.state(layer, s_) == flat.state(layer, s_)
        Lt, F = paged.state(layer, s_)
        P = oracle.history_split(Lt)[0] + F
        for h in range(Hkv):
            for pg in range((P + 127) // 128):
                assert np.array_equal(paged.page(layer, s_, h, pg), flat.page(layer, s_, h, pg)), (i, h, pg)
        _check_sequence(paged, layer, s_, seqs[i][0], seqs[i][1], tables)
    q = synth.queries(B, Hkv * G, d, seed=6)
    out_p = paged.decode(layer, q.to(DEV), _i32(slots)).cpu().numpy()
    out_f = flat.decode(layer, q.to(DEV), _i32(slots)).cpu().numpy()
    assert np.array_equal(out_p, out_f)
    for i, s_ in enumerate(slots):
        ref = _oracle_decode(paged, layer, s_, q[i], tables)
        for hq in range(Hkv * G):
            assert rel_l2(out_p[i, hq], ref[hq]) <= 2e-3
    # a page whose block is missing: reported, no fault; the append that would write one skips it
    bt[slots[0], 0] = -1
    paged.decode(layer, q.to(DEV), _i32(slots))
    assert paged.check_status() & 0x10
    bt[slots[1], 2] = -1
    k1 = torch.zeros(1, 260, Hkv, d, dtype=torch.bfloat16, device=DEV)
    paged.append(layer, k1, k1, _i32([slots[1]]), _i32([260]))  # 131 -> 391 tokens: writes pages 1 and 2
    assert paged.check_status() & 0x10


@pytest.mark.parametrize("d,vb,kbits,chunk,G", [(128, 2, 3, (200, 37), 4), (64, 4, 3, (200, 37), 4),
                                                (256, 2, 3, (200, 37), 4), (128, 4, 4, (200, 37), 4),
                                                (128, 2, 3, (199, 36), 4), (128, 4, 3, (200, 37), 2),
                                                (256, 4, 4, (199, 36), 2)])
def test_prefill_chunk_attention(d, vb, kbits, chunk, G):
    """Chunked prefill: histories of 300 and 129 tokens, then chunks of chunk[0] and chunk[1] tokens
    appended in one call (the second row padded to chunk[0] queries). Every chunk query attends causally
    over the cache after the append (packed tokens through their codes, ring tokens exactly), as the
    oracle's masked prefill attention gives it on the device's own records and ring; padding queries
    output zeros. head_dim 128 with key_bits 3 and G 4 takes the tcgen05 path (tiles of 32 queries x 4
    heads); elsewhere an even number of query slots per row takes two query rows per CTA (their causal
    lengths differ inside a CTA, and a query next to a padding query shares its CTA), an odd number one."""
    _prefill_chunk_case(d, vb, kbits, chunk, G, [300, 129])


@pytest.fixture
def cuda_core_prefill():
    """Every prefill of the test takes the CUDA-core (decode kernel) path, also where tcgen05 applies."""
    from kv_cache_quantization_quantize_gb300 import _abi
    lib = _abi.load()
    assert lib.tq_debug_prefill_path(1) == _abi.TQ_OK
    yield
    assert lib.tq_debug_prefill_path(0) == _abi.TQ_OK


@pytest.mark.parametrize("vb,chunk", [(2, (200, 37)), (2, (199, 36)), (4, (200, 37))])
def test_prefill_chunk_attention_cuda_core_path(cuda_core_prefill, vb, chunk):
    """The shapes that take the tcgen05 prefill by default (head_dim 128, key_bits 3, G 4), forced onto the
    CUDA-core path: both paths stay covered."""
    _prefill_chunk_case(128, vb, 3, chunk, 4, [300, 129])


@pytest.mark.parametrize("vb,paged", [(2, False), (4, False), (2, True)])
def test_prefill_tcgen05_long_history(vb, paged):
    """The tcgen05 prefill over several pages per split and several tiles per row: histories of 1500 and
    700 tokens, chunks of 256 and 64 queries (8 tiles of 32 queries per row, the second row mostly
    padding), x10 key outliers; contiguous and paged caches. Checked against the oracle, and against
    the CUDA-core path on the same cache."""
    out_tc = _prefill_chunk_case(128, vb, 3, (256, 64), 4, [1500, 700], paged=paged, max_ctx=1792)
    from kv_cache_quantization_quantize_gb300 import _abi
    lib = _abi.load()
    assert lib.tq_debug_prefill_path(1) == _abi.TQ_OK
    try:
        out_cc = _prefill_chunk_case(128, vb, 3, (256, 64), 4, [1500, 700], paged=paged, max_ctx=1792)
    finally:
        assert lib.tq_debug_prefill_path(0) == _abi.TQ_OK
    diff = max(rel_l2(out_tc[i, j, hq], out_cc[i, j, hq]) for i in range(2) for j in range(64) for hq in range(8))
    assert diff <= 2e-3, diff
    print(f"tcgen05 against CUDA-core prefill: worst rel-L2 {diff:.2e}")



@pytest.mark.parametrize("hist,chunk,max_ctx", [(3000, 40, 4096), (8000, 32, 8192)])
def test_prefill_tcgen05_many_history_splits(hist, chunk, max_ctx):
    """Few query tiles over a long history give many history splits: 2 x 2 tiles of 32 pages take 32 splits
    of one page, and 1 x 2 tiles of 64 pages take 64 (the most the combine takes). The combine then merges
    more partials than it loads ahead, and (at 64) weights held in a second register per lane."""
    _prefill_chunk_case(128, 2, 3, (chunk,), 4, [hist], max_ctx=max_ctx)

def _prefill_chunk_case(d, vb, kbits, chunk, G, hist, paged=False, max_ctx=640):
    Hkv = 2
    hist, chunk = list(hist), list(chunk)
    slots = [1, 0][:len(hist)]
    B, Tq = len(hist), max(chunk)
    max_pages = (max_ctx + 127) // 128
    cfg = config(head_dim=d, value_bits=vb, n_layers=1, n_kv_heads=Hkv, n_q_heads=Hkv * G, max_seqs=2,
                 max_ctx=max_ctx, seed=13, key_bits=kbits, n_blocks=2 * max_pages if paged else 0)
    cache = TurboQuantCache(cfg)
    if paged:
        perm = torch.randperm(2 * max_pages, generator=torch.Generator().manual_seed(3)).to(torch.int32)
        cache.block_table.copy_(perm.view(2, max_pages).to(DEV))
    tables = _oracle_tables(cache)
    seqs = [synth.kv_tokens(h_ + c_, Hkv, d, seed=700 + i, outliers=("random", 4, 10.0))
            for i, (h_, c_) in enumerate(zip(hist, chunk))]
    ids = _i32(slots)
    for lo, lens in ((None, hist), (hist, chunk)):
        n = max(lens)
        kb = torch.zeros(B, n, Hkv, d, dtype=torch.bfloat16)
        vbuf = torch.zeros_like(kb)
        for i in range(B):
            o = 0 if lo is None else lo[i]
            kb[i, :lens[i]] = seqs[i][0][o:o + lens[i]]
            vbuf[i, :lens[i]] = seqs[i][1][o:o + lens[i]]
        cache.append(0, kb.to(DEV), vbuf.to(DEV), ids, _i32(lens))
    torch.cuda.synchronize()
    assert cache.check_status() == 0
    q = synth.queries(B * Tq, Hkv * G, d, seed=14).view(B, Tq, Hkv * G, d).contiguous()
    out = cache.prefill(0, q.to(DEV), ids, _i32(chunk)).cpu().numpy()
    assert cache.check_status() == 0
    D, S, c, t = tables
    worst = 0.0
    for i, s_ in enumerate(slots):
        L, F = cache.state(0, s_)
        assert L == hist[i] + chunk[i]
        Np, R = oracle.history_split(L)
        P = Np + F
        nq = chunk[i]
        assert np.all(out[i, nq:] == 0)
        for h in range(Hkv):
            kr, vr = cache.records(0, s_, h, P)
            keys = oracle.unpack_key_records(kr, d, cache.cfg.key_bits)
            vals = oracle.unpack_value_records(vr, d, vb)
            rk, rv = cache.ring(0, s_, h)
            qh = _f64(q[i, :nq, h * G:(h + 1) * G])
            ref = oracle.prefill_attention(qh, keys, vals, _f64(rk[F:R]), _f64(rv[F:R]), L, D, S, c)
            for j in range(nq):
                for g in range(G):
                    err = rel_l2(out[i, j, h * G + g], ref[j, g])
                    worst = max(worst, err)
                    assert err <= 2e-3, (i, j, h, g, err)
    print(f"prefill d={d} V{vb} K{kbits} q_per_row {Tq} G{G} paged={paged}: worst rel-L2 {worst:.2e}")
    return out


def test_decode_wait_timeout_is_reported_and_the_workspace_stays_usable():
    """Bounded waits: a test hook makes one page stage of the first split CTA of (row 0, KV head 0) get
    neither its copy nor its expected-byte count, and its wait give up after a few polls. The call returns,
    the status word carries TQ_DEV_ERR_TIMEOUT, every other (row, KV head) is exact, and the next decode on
    the same workspace (hook off) matches the oracle everywhere: the kernel waited for the copies it had
    issued and left its arrival counters at zero. Nothing faults or hangs: the abandoned stage has no copy
    in flight."""
    from kv_cache_quantization_quantize_gb300 import _abi
    d, vb, Hkv, G = 128, 2, 2, 4
    # 32 rows of 900-993 tokens (7 packed pages each): the decode plan then gives one split of 8 pages per
    # (row, KV head), so the first page stream of a split CTA reads pages 0, 3 and 6 through stages 0-2
    lens = [900 + 3 * i for i in range(32)]
    B = len(lens)
    cfg = config(head_dim=d, value_bits=vb, n_layers=1, n_kv_heads=Hkv, n_q_heads=Hkv * G, max_seqs=B, max_ctx=1024,
                 seed=31)
    cache = TurboQuantCache(cfg)
    tables = _oracle_tables(cache)
    kb = torch.zeros(B, max(lens), Hkv, d, dtype=torch.bfloat16)
    vbuf = torch.zeros_like(kb)
    for i, L in enumerate(lens):
        kk, vv = synth.kv_tokens(L, Hkv, d, seed=900 + i)
        kb[i, :L], vbuf[i, :L] = kk, vv
    ids = _i32(list(range(B)))
    cache.append(0, kb.to(DEV), vbuf.to(DEV), ids, _i32(lens))
    q = synth.queries(B, Hkv * G, d, seed=32)
    ws = cache.workspace(B)
    torch.cuda.synchronize()
    assert cache.check_status() == 0
    lib = _abi.load()
    refs = [_oracle_decode(cache, 0, i, q[i], tables) for i in range(B)]
    for stage in (0, 2):
        assert lib.tq_debug_decode_wait_fault(stage, 8) == _abi.TQ_OK
        try:
            out = cache.decode(0, q.to(DEV), ids, workspace=ws).cpu().numpy()
        finally:
            assert lib.tq_debug_decode_wait_fault(-1, 0) == _abi.TQ_OK
        assert cache.check_status() & _abi.TQ_DEV_ERR_TIMEOUT
        for i in range(B):
            for hq in range(Hkv * G):
                if i == 0 and hq < G:
                    continue  # the unit whose wait gave up: unspecified
                assert rel_l2(out[i, hq], refs[i][hq]) <= 2e-3, (stage, i, hq)
        out = cache.decode(0, q.to(DEV), ids, workspace=ws).cpu().numpy()
        assert cache.check_status() == 0
        for i in range(B):
            for hq in range(Hkv * G):
                assert rel_l2(out[i, hq], refs[i][hq]) <= 2e-3, ("after", stage, i, hq)
    assert lib.tq_debug_decode_wait_fault(7, 8) == _abi.TQ_ERR_INVALID_ARG
    assert lib.tq_debug_decode_wait_fault(0, 0) == _abi.TQ_ERR_INVALID_ARG


def test_prefill_tcgen05_after_a_ring_flush_and_an_invalid_row():
    """The tcgen05 prefill where the ring's first F tokens were coded by a flush: 300 tokens, a flush (256
    packed + a 44-token ring block coded in full, F = 44), then a 70-token chunk (L = 370, ring tokens
    [44, 114) exact). Chunk queries before position 300 see only packed tokens; the rest see a growing part
    of the ring, read from ring row F on. A second batch row names slot -1 (invalid): its outputs are zero,
    and the valid row's outputs agree with the ones of a call without it."""
    d, vb, Hkv, G, slot = 128, 2, 2, 4, 1
    cfg = config(head_dim=d, value_bits=vb, n_layers=1, n_kv_heads=Hkv, n_q_heads=Hkv * G, max_seqs=2,
                 max_ctx=640, seed=61)
    cache = TurboQuantCache(cfg)
    tables = _oracle_tables(cache)
    k, v = synth.kv_tokens(370, Hkv, d, seed=6100, outliers=("random", 4, 10.0))
    cache.append(0, k[None, :300].to(DEV).contiguous(), v[None, :300].to(DEV).contiguous(), _i32([slot]),
                 _i32([300]))
    cache.flush(0, _i32([slot]))
    cache.append(0, k[None, 300:].to(DEV).contiguous(), v[None, 300:].to(DEV).contiguous(), _i32([slot]),
                 _i32([70]))
    torch.cuda.synchronize()
    assert cache.check_status() == 0
    L, F = cache.state(0, slot)
    Np, R = oracle.history_split(L)
    assert (L, F, Np, R) == (370, 44, 256, 114)
    nq = 70
    q = synth.queries(2 * nq, Hkv * G, d, seed=6101).view(2, nq, Hkv * G, d).contiguous()
    out = cache.prefill(0, q.to(DEV), _i32([slot, -1]), _i32([nq, nq])).cpu().numpy()
    alone = cache.prefill(0, q[:1].contiguous().to(DEV), _i32([slot]), _i32([nq])).cpu().numpy()
    assert np.all(out[1] == 0)
    assert np.allclose(out[0], alone[0], rtol=1e-5, atol=1e-7)  # (the split count may differ with the batch)
    D, S, c, _ = tables
    P = Np + F
    worst = 0.0
    for h in range(Hkv):
        kr, vr = cache.records(0, slot, h, P)
        keys = oracle.unpack_key_records(kr, d, cfg.key_bits)
        vals = oracle.unpack_value_records(vr, d, vb)
        rk, rv = cache.ring(0, slot, h)
        ref = oracle.prefill_attention(_f64(q[0, :, h * G:(h + 1) * G]), keys, vals, _f64(rk[F:R]), _f64(rv[F:R]),
                                       L, D, S, c)
        for j in range(nq):
            for g in range(G):
                err = rel_l2(out[0, j, h * G + g], ref[j, g])
                worst = max(worst, err)
                assert err <= 2e-3, (j, h, g, err)
    print(f"tcgen05 prefill after a flush: worst rel-L2 {worst:.2e}")
