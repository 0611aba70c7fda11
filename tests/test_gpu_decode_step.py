"""GPU tests of tq_decode_step (one decode step of one layer in one launch: the one-token append and the
hybrid decode) and of the append rule it relies on: every 128-token block is coded into its packed page
as soon as it is complete, including the block that fills the ring."""
import numpy as np
import pytest
import torch

import oracle
from kv_cache_quantization_quantize_gb300 import TurboQuantCache, config, synth
from tests.gpu_helpers import check_sequence, f64, i32, oracle_decode, oracle_tables
from tests.parity import check_key_records, check_value_records, rel_l2

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def built():
    from kv_cache_quantization_quantize_gb300 import build
    build.build()


def _twin_caches(d, vb, kbits, Hkv, G, n_layers, max_seqs, max_ctx, paged, seed):
    caches = []
    for _ in range(2):
        max_pages = (max_ctx + 127) // 128
        cfg = config(head_dim=d, value_bits=vb, key_bits=kbits, n_layers=n_layers, n_kv_heads=Hkv, n_q_heads=Hkv * G,
                     max_seqs=max_seqs, max_ctx=max_ctx, seed=seed, n_blocks=max_seqs * max_pages if paged else 0)
        c = TurboQuantCache(cfg)
        if paged:
            perm = torch.randperm(max_seqs * max_pages, generator=torch.Generator().manual_seed(seed))
            c.block_table.copy_(perm.to(torch.int32).view(max_seqs, max_pages).to(DEV))
        caches.append(c)
    return caches


def _same_cache(a, b, n_layers, slots, Hkv):
    """The parts of two caches that appends and steps write: the state, the pages of every complete block
    (128 floor(L / 128) tokens) and the ring rows of the current ring block."""
    for l in range(n_layers):
        for slot in slots:
            assert a.state(l, slot) == b.state(l, slot), (l, slot)
            L = a.state(l, slot)[0]
            R = L - 128 * ((L - 1) // 128) if L else 0
            for h in range(Hkv):
                for pg in range(L // 128):
                    assert np.array_equal(a.page(l, slot, h, pg), b.page(l, slot, h, pg)), (l, slot, h, pg)
                for x, y in zip(a.ring(l, slot, h), b.ring(l, slot, h)):
                    assert torch.equal(x[:R], y[:R]), (l, slot, h)


def _histories(caches, n_layers, lens, slots, Hkv, d, steps, seed):
    """One bulk append per layer of every row's history (the same inputs into both caches); returns the
    full token streams [L + steps, Hkv, d] per (layer, row)."""
    B = len(lens)
    seqs = {}
    for layer in range(n_layers):
        kb = torch.zeros(B, max(lens), Hkv, d, dtype=torch.bfloat16)
        vbuf = torch.zeros_like(kb)
        for i, L in enumerate(lens):
            k, v = synth.kv_tokens(L + steps, Hkv, d, seed=seed + 100 * layer + i, outliers=("random", 4, 10.0))
            seqs[layer, i] = (k, v)
            kb[i, :L], vbuf[i, :L] = k[:L], v[:L]
        for c in caches:
            c.append(layer, kb.to(DEV), vbuf.to(DEV), i32(slots), i32(lens))
    return seqs


@pytest.mark.parametrize("d,vb,kbits,new_dtype,paged", [
    (128, 2, 3, torch.bfloat16, False), (128, 4, 3, torch.float32, False), (64, 4, 4, torch.bfloat16, False),
    (256, 2, 3, torch.bfloat16, True), (128, 2, 3, torch.bfloat16, True)])
def test_decode_step_equals_append_then_decode(d, vb, kbits, new_dtype, paged):
    """Two caches built alike; one runs tq_decode_step, the other the one-token append followed by the
    decode, on the same inputs: 140 steps over 2 layers, issued layer after layer with no synchronisation.
    The rows start around 128-token boundaries, so each one fills its ring (the step codes that block)
    and then starts a new ring block over the page it coded. The outputs must be bit-identical on every
    step, and so must the whole cache (pages, ring rows, sequence state) at the end. The step's outputs
    are also checked against the oracle on the steps where a row fills or rolls its ring."""
    Hkv, G, n_layers, steps = 2, 4, 2, 140
    lens = [1, 100, 126, 127, 128, 129, 250, 383]
    slots = [3, 0, 7, 1, 6, 2, 5, 4]
    B = len(lens)
    step_c, ref_c = _twin_caches(d, vb, kbits, Hkv, G, n_layers, 8, 540, paged, seed=31)
    tables = oracle_tables(step_c)
    seqs = _histories((step_c, ref_c), n_layers, lens, slots, Hkv, d, steps, seed=700)
    ids, ones = i32(slots), i32([1] * B)
    ws_s, ws_r = step_c.workspace(B, 540), ref_c.workspace(B, 540)
    torch.cuda.synchronize()
    worst, checked = 0.0, 0
    for s in range(steps):
        kn = [torch.stack([seqs[l, i][0][L + s] for i, L in enumerate(lens)]).to(DEV, new_dtype).contiguous()
              for l in range(n_layers)]
        vn = [torch.stack([seqs[l, i][1][L + s] for i, L in enumerate(lens)]).to(DEV, new_dtype).contiguous()
              for l in range(n_layers)]
        qs = [synth.queries(B, Hkv * G, d, seed=5000 + 13 * s + l) for l in range(n_layers)]
        qd = [q.to(DEV) for q in qs]
        out_s = torch.empty((n_layers, B, Hkv * G, d), dtype=torch.float32, device=DEV)
        out_r = torch.empty_like(out_s)
        torch.cuda.synchronize()
        for l in range(n_layers):
            step_c.decode_step(l, kn[l], vn[l], qd[l], ids, out=out_s[l], max_ctx_hint=540, workspace=ws_s)
            ref_c.append(l, kn[l][:, None].contiguous(), vn[l][:, None].contiguous(), ids, ones)
            ref_c.decode(l, qd[l], ids, out=out_r[l], max_ctx_hint=540, workspace=ws_r)
        torch.cuda.synchronize()
        assert torch.equal(out_s, out_r), (s, float((out_s - out_r).abs().max()))
        new_len = [L + s + 1 for L in lens]
        if any(n % 128 in (0, 1) for n in new_len) or s == steps - 1:
            for l in range(n_layers):
                for i in range(B):
                    if new_len[i] % 128 not in (0, 1) and s != steps - 1:
                        continue
                    assert step_c.state(l, slots[i]) == ref_c.state(l, slots[i])
                    assert step_c.state(l, slots[i])[0] == new_len[i]
                    ref = oracle_decode(step_c, l, slots[i], qs[l][i], tables)
                    for hq in range(Hkv * G):
                        err = rel_l2(out_s[l, i, hq].cpu().numpy(), ref[hq])
                        worst = max(worst, err)
                        checked += 1
                        assert err <= 2e-3, (s, l, i, hq, err)
    assert step_c.check_status() == 0 and ref_c.check_status() == 0
    _same_cache(step_c, ref_c, n_layers, slots, Hkv)
    for l in range(n_layers):
        for i in range(B):
            check_sequence(step_c, l, slots[i], seqs[l, i][0], seqs[l, i][1], tables)
    print(f"decode step d={d} V{vb} K{kbits} {new_dtype} paged={paged}: {checked} oracle checks, worst {worst:.2e}")


def test_decode_step_back_to_back_on_one_layer():
    """Steps of one layer follow each other on the stream (the next launch reads the state the previous
    one publishes at its end), with a plain decode and a one-token append in between at times; the rows
    fill and roll their rings on the way. Outputs and cache equal the append-then-decode twin's."""
    d, vb, Hkv, G, steps = 128, 2, 2, 4, 40
    lens = [100, 120, 127, 255, 256]
    slots = list(range(len(lens)))
    B = len(lens)
    step_c, ref_c = _twin_caches(d, vb, 3, Hkv, G, 1, B, 400, False, seed=41)
    seqs = _histories((step_c, ref_c), 1, lens, slots, Hkv, d, steps, seed=900)
    ids, ones = i32(slots), i32([1] * B)
    ws_s, ws_r = step_c.workspace(B, 400), ref_c.workspace(B, 400)
    kn = [torch.stack([seqs[0, i][0][L + s] for i, L in enumerate(lens)]).to(DEV).contiguous() for s in range(steps)]
    vn = [torch.stack([seqs[0, i][1][L + s] for i, L in enumerate(lens)]).to(DEV).contiguous() for s in range(steps)]
    qd = [synth.queries(B, Hkv * G, d, seed=77 + s).to(DEV) for s in range(steps)]
    out_s = torch.empty((steps, B, Hkv * G, d), dtype=torch.float32, device=DEV)
    out_r = torch.empty_like(out_s)
    plain_s = torch.empty((steps, B, Hkv * G, d), dtype=torch.float32, device=DEV)
    plain_r = torch.empty_like(plain_s)
    torch.cuda.synchronize()
    for s in range(steps):  # nothing synchronises inside the loop
        if s % 7 == 3:  # a plain one-token append instead of a step, on both
            for c in (step_c, ref_c):
                c.append(0, kn[s][:, None].contiguous(), vn[s][:, None].contiguous(), ids, ones)
            step_c.decode(0, qd[s], ids, out=out_s[s], max_ctx_hint=400, workspace=ws_s)
            ref_c.decode(0, qd[s], ids, out=out_r[s], max_ctx_hint=400, workspace=ws_r)
        else:
            step_c.decode_step(0, kn[s], vn[s], qd[s], ids, out=out_s[s], max_ctx_hint=400, workspace=ws_s)
            ref_c.append(0, kn[s][:, None].contiguous(), vn[s][:, None].contiguous(), ids, ones)
            ref_c.decode(0, qd[s], ids, out=out_r[s], max_ctx_hint=400, workspace=ws_r)
        if s % 5 == 1:  # a plain decode right after the step
            step_c.decode(0, qd[s], ids, out=plain_s[s], max_ctx_hint=400, workspace=ws_s)
            ref_c.decode(0, qd[s], ids, out=plain_r[s], max_ctx_hint=400, workspace=ws_r)
    torch.cuda.synchronize()
    for s in range(steps):
        assert torch.equal(out_s[s], out_r[s]), s
        if s % 5 == 1:
            assert torch.equal(plain_s[s], plain_r[s]), s
    assert step_c.check_status() == 0 and ref_c.check_status() == 0
    _same_cache(step_c, ref_c, 1, slots, Hkv)
    tables = oracle_tables(step_c)
    for i in range(B):
        assert step_c.state(0, i)[0] == lens[i] + steps
        check_sequence(step_c, 0, i, seqs[0, i][0], seqs[0, i][1], tables)


def test_decode_step_at_capacity_and_invalid_slot():
    """A row at max_ctx takes no token (TQ_DEV_ERR_CAPACITY) and is decoded as it stands, like the append
    path; the other rows step normally."""
    d, Hkv, G = 128, 2, 4
    lens = [255, 100]
    step_c, ref_c = _twin_caches(d, 2, 3, Hkv, G, 1, 2, 256, False, seed=43)
    seqs = _histories((step_c, ref_c), 1, lens, [0, 1], Hkv, d, 2, seed=950)
    ids, ones = i32([0, 1]), i32([1, 1])
    for s in range(2):  # step 0 fills row 0 to max_ctx = 256 (and codes its block); step 1 overflows it
        kn = torch.stack([seqs[0, i][0][L + s] for i, L in enumerate(lens)]).to(DEV).contiguous()
        vn = torch.stack([seqs[0, i][1][L + s] for i, L in enumerate(lens)]).to(DEV).contiguous()
        q = synth.queries(2, Hkv * G, d, seed=3 + s).to(DEV)
        a = step_c.decode_step(0, kn, vn, q, i32([0, 1]), max_ctx_hint=256)
        ref_c.append(0, kn[:, None].contiguous(), vn[:, None].contiguous(), ids, ones)
        r = ref_c.decode(0, q, ids, max_ctx_hint=256)
        torch.cuda.synchronize()
        assert torch.equal(a, r), s
        w_s, w_r = step_c.check_status(clear=True), ref_c.check_status(clear=True)
        assert w_s == w_r == (0 if s == 0 else 1), (s, w_s, w_r)  # TQ_DEV_ERR_CAPACITY on the second step
    assert step_c.state(0, 0) == ref_c.state(0, 0) == (256, 0)
    assert step_c.state(0, 1) == ref_c.state(0, 1) == (102, 0)
    _same_cache(step_c, ref_c, 1, [0, 1], Hkv)


@pytest.mark.parametrize("d,kbits,how", [(128, 3, "small"), (128, 3, "bulk_bf16"), (128, 4, "bulk_bf16"),
                                         (128, 3, "bulk_f32"), (256, 3, "bulk_bf16"), (64, 3, "partial_ring")])
def test_append_codes_the_block_that_fills_the_ring(d, kbits, how):
    """Appends that end exactly on a 128-token boundary code the last block into its page at once (the
    ring keeps it too): small appends (100 + 28), bulk bf16 appends (tcgen05 coder at head_dim 128, the
    CUDA-core coder elsewhere), a bulk f32 append, and a bulk append onto a partial ring (50 + 206). The
    records of all 128 floor(L / 128) tokens match the oracle and the ring holds the last 128 tokens."""
    Hkv, vb = 2, 4 if kbits == 4 else 2
    cfg = config(head_dim=d, value_bits=vb, key_bits=kbits, n_layers=1, n_kv_heads=Hkv, n_q_heads=Hkv * 4,
                 max_seqs=2, max_ctx=512, seed=51)
    cache = TurboQuantCache(cfg)
    tables = oracle_tables(cache)
    D, S, c, t = tables
    dt = torch.float32 if how == "bulk_f32" else torch.bfloat16
    parts = {"small": [100, 28], "bulk_bf16": [256], "bulk_f32": [128], "partial_ring": [50, 206]}[how]
    L = sum(parts)
    k, v = synth.kv_tokens(L, Hkv, d, seed=61, outliers=("random", 4, 10.0), dtype=dt)
    pos = 0
    for n in parts:
        cache.append(0, k[None, pos:pos + n].to(DEV).contiguous(), v[None, pos:pos + n].to(DEV).contiguous(),
                     i32([1]), i32([n]))
        pos += n
    torch.cuda.synchronize()
    assert cache.check_status() == 0
    assert cache.state(0, 1) == (L, 0)
    C = 128 * (L // 128)
    for h in range(Hkv):
        kr, vr = cache.records(0, 1, h, C)
        kk = oracle.unpack_key_records(kr, d, kbits)
        vv = oracle.unpack_value_records(vr, d, vb)
        check_key_records(kk, f64(k[:C, h]), D, S, c, t)
        check_value_records(vv, f64(v[:C, h]), D, vb)
    check_sequence(cache, 0, 1, k, v, tables)  # decode's view: the ring still holds the last block
