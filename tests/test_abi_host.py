"""CPU tests of libtq's C ABI: exports, argument validation, tables vs the oracle, page layout."""
import ctypes
import json
import os

import numpy as np
import pytest

import kv_cache_quantization_quantize_gb300 as tqm
from kv_cache_quantization_quantize_gb300 import _abi
from oracle import gaussian_matrix_bf16, rademacher_signs

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


@pytest.fixture(scope="module", autouse=True)
def built():
    from kv_cache_quantization_quantize_gb300 import build
    build.build()


def test_library_exports_every_header_function():
    lib = _abi.load()
    names = _abi.header_functions()
    assert len(names) >= 19
    for n in names:
        assert hasattr(lib, n), n
    assert set(names) == set(_abi._SIGS)


@pytest.mark.parametrize("field,value,status", [
    ("head_dim", 32, _abi.TQ_ERR_UNSUPPORTED), ("head_dim", 96, _abi.TQ_ERR_UNSUPPORTED),
    ("value_bits", 3, _abi.TQ_ERR_UNSUPPORTED), ("key_bits", 4, _abi.TQ_ERR_UNSUPPORTED),
    ("value_group", 64, _abi.TQ_ERR_UNSUPPORTED), ("ring_size", 64, _abi.TQ_ERR_UNSUPPORTED),
    ("ring_size", -1, _abi.TQ_ERR_UNSUPPORTED),
    ("n_layers", 0, _abi.TQ_ERR_INVALID_ARG), ("n_q_heads", 12, _abi.TQ_ERR_UNSUPPORTED),
    ("n_q_heads", 9, _abi.TQ_ERR_INVALID_ARG), ("max_ctx", 0, _abi.TQ_ERR_INVALID_ARG),
    ("key_bits", 5, _abi.TQ_ERR_UNSUPPORTED), ("key_bits", 2, _abi.TQ_ERR_UNSUPPORTED),
])
def test_invalid_configs_rejected(field, value, status):
    lib = _abi.load()
    cfg = tqm.config(n_kv_heads=2, n_q_heads=8)
    setattr(cfg, field, value)
    assert lib.tq_tables_bytes(ctypes.byref(cfg)) == 0
    ctx = ctypes.c_void_p()
    assert lib.tq_init_codebooks(ctypes.byref(cfg), None, 0, None, ctypes.byref(ctx)) == status
    assert not ctx.value
    assert lib.tq_last_error()


def test_key_bits_4_needs_value_bits_4():
    lib = _abi.load()
    ctx = ctypes.c_void_p()
    cfg = tqm.config(key_bits=4, value_bits=2)
    assert lib.tq_init_codebooks(ctypes.byref(cfg), None, 0, None, ctypes.byref(ctx)) == _abi.TQ_ERR_UNSUPPORTED
    cfg = tqm.config(key_bits=4, value_bits=4)
    assert lib.tq_init_codebooks(ctypes.byref(cfg), None, 0, None, ctypes.byref(ctx)) == _abi.TQ_OK
    lib.tq_destroy(ctx)


def test_full_tq_mode_config_is_accepted():
    """ring_size 0 selects full_tq mode; the cache keeps the same layout (the ring is a staging copy)."""
    lib = _abi.load()
    hyb, full = tqm.config(), tqm.config(mode="full_tq")
    assert full.ring_size == 0
    assert lib.tq_tables_bytes(ctypes.byref(full)) == lib.tq_tables_bytes(ctypes.byref(hyb)) > 0
    assert lib.tq_cache_bytes(ctypes.byref(full)) == lib.tq_cache_bytes(ctypes.byref(hyb)) > 0
    with pytest.raises(ValueError):
        tqm.config(mode="capture_only")


def test_paged_cache_layout():
    """n_blocks > 0: the pages section is a per-layer pool of n_blocks blocks (every KV head of a 128-token
    page), followed by the ring, the state and the int32 block table [max_seqs][max_pages]."""
    lib = _abi.load()
    flat = tqm.config(n_layers=2, n_kv_heads=2, n_q_heads=8, max_seqs=64, max_ctx=8192)
    paged = tqm.config(n_layers=2, n_kv_heads=2, n_q_heads=8, max_seqs=64, max_ctx=8192, n_blocks=100)
    page = lib.tq_page_bytes(ctypes.byref(flat))
    cf, cp = lib.tq_cache_bytes(ctypes.byref(flat)), lib.tq_cache_bytes(ctypes.byref(paged))
    pool_flat, pool_paged = 2 * 64 * 2 * 64 * page, 2 * 100 * 2 * page
    assert cf - cp >= pool_flat - pool_paged - 64 * 64 * 4 - 1024
    bad = tqm.config(n_blocks=-1)
    ctx = ctypes.c_void_p()
    assert lib.tq_init_codebooks(ctypes.byref(bad), None, 0, None, ctypes.byref(ctx)) == _abi.TQ_ERR_INVALID_ARG
    h = tqm.HostTables(paged)
    assert lib.tq_page_offset(h.ctx, 0, 0, 0, 0) == ctypes.c_size_t(-1).value
    assert lib.tq_block_page_offset(h.ctx, 1, 3, 1) == ((1 * 100 + 3) * 2 + 1) * page
    assert lib.tq_block_table_offset(h.ctx) < cp
    hf = tqm.HostTables(flat)
    assert lib.tq_block_table_offset(hf.ctx) == ctypes.c_size_t(-1).value


def test_null_and_host_only_misuse_is_rejected():
    lib = _abi.load()
    assert lib.tq_init_codebooks(None, None, 0, None, None) == _abi.TQ_ERR_INVALID_ARG
    h = tqm.HostTables(tqm.config())
    # device calls on a host-only context are refused before any launch
    assert lib.tq_cache_bind(h.ctx, ctypes.c_void_p(256), 1 << 30, None) == _abi.TQ_ERR_INVALID_ARG
    assert lib.tq_quantize_append(h.ctx, 0, None, None, 0, None, None, 1, 1, None) == _abi.TQ_ERR_INVALID_ARG
    assert lib.tq_decode_attention(h.ctx, 0, None, None, None, 1, 0.0, None, 0, 0, None) == _abi.TQ_ERR_INVALID_ARG
    assert lib.tq_ring_flush(h.ctx, 0, None, 1, None) == _abi.TQ_ERR_INVALID_ARG
    assert lib.tq_dequantize_tokens(h.ctx, 0, 0, 0, 0, 1, 1, None, None, None) == _abi.TQ_ERR_INVALID_ARG
    assert lib.tq_decode_step(h.ctx, 0, None, None, 0, None, None, None, 1, 0.0, None, 0, 0, None) \
        == _abi.TQ_ERR_INVALID_ARG
    # tq_decode_phase has two phases (0: zero the counters, 1: the decode launch); others are refused
    for phase in (-1, 2):
        assert lib.tq_decode_phase(h.ctx, phase, 0, None, None, None, 1, 0.0, None, 0, 0, None) == _abi.TQ_ERR_INVALID_ARG
        assert f"phase {phase} not in".encode() in lib.tq_last_error()


@pytest.mark.parametrize("d", [64, 128, 256])
@pytest.mark.parametrize("seed", [0, 1, 12345])
def test_tables_match_oracle_bitwise(d, seed):
    h = tqm.HostTables(tqm.config(head_dim=d, seed=seed))
    D, S, c, t = h.tables()
    assert np.array_equal(D.astype(np.float64), rademacher_signs(seed, d))
    S_lib = (S.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    assert np.array_equal(S_lib, gaussian_matrix_bf16(seed, d))
    g = json.load(open(os.path.join(GOLDEN, "codebooks.json")))["codebooks"][f"d{d}_b2"]
    assert np.allclose(c, g["centroids"], rtol=0, atol=1e-13)
    assert np.allclose(t, g["boundaries"], rtol=0, atol=1e-13)
    assert t[1] == 0.0 and np.array_equal(c, -c[::-1])
    # key_bits 4: the 3-bit codebook
    h4 = tqm.HostTables(tqm.config(head_dim=d, seed=seed, key_bits=4, value_bits=4))
    _, _, c4, t4 = h4.tables()
    g4 = json.load(open(os.path.join(GOLDEN, "codebooks.json")))["codebooks"][f"d{d}_b3"]
    assert c4.shape == (8,) and t4.shape == (7,)
    # both are Lloyd iterations stopped near the fixed point (8 cells converge more slowly than 4)
    assert np.allclose(c4, g4["centroids"], rtol=0, atol=5e-13)
    assert np.allclose(t4, g4["boundaries"], rtol=0, atol=5e-13)
    assert t4[3] == 0.0 and np.array_equal(c4, -c4[::-1])
    # the fp32 values the kernels use agree exactly
    assert np.array_equal(c4.astype(np.float32), np.array(g4["centroids"]).astype(np.float32))
    assert np.array_equal(t4.astype(np.float32), np.array(g4["boundaries"]).astype(np.float32))
    # the fp32 values the kernels use agree exactly
    assert np.array_equal(c.astype(np.float32), np.array(g["centroids"]).astype(np.float32))


@pytest.mark.parametrize("d,vb,kb,expect", [(64, 2, 3, 48), (64, 4, 3, 64), (128, 2, 3, 92), (128, 4, 3, 124),
                                            (256, 2, 3, 180), (256, 4, 3, 244), (64, 4, 4, 72), (128, 4, 4, 140),
                                            (256, 4, 4, 276)])
def test_page_bytes_equal_canonical_records(d, vb, kb, expect):
    h = tqm.HostTables(tqm.config(head_dim=d, value_bits=vb, key_bits=kb))
    assert h.key_record_bytes() + h.value_record_bytes() == expect
    assert h.page_bytes() == 128 * expect


def _random_records(h, n, rng):
    kr = rng.integers(0, 256, size=(n, h.key_record_bytes()), dtype=np.uint8)
    vr = rng.integers(0, 256, size=(n, h.value_record_bytes()), dtype=np.uint8)
    return kr, vr


@pytest.mark.parametrize("d,vb,kb", [(64, 2, 3), (64, 4, 3), (128, 2, 3), (128, 4, 3), (256, 2, 3), (256, 4, 3),
                                     (64, 4, 4), (128, 4, 4), (256, 4, 4)])
def test_records_page_round_trip(d, vb, kb):
    h = tqm.HostTables(tqm.config(head_dim=d, value_bits=vb, key_bits=kb))
    rng = np.random.default_rng(d + vb)
    kr, vr = _random_records(h, 128, rng)
    page = h.records_to_page(kr, vr)
    k2, v2 = h.page_to_records(page, 128)
    assert np.array_equal(k2, kr) and np.array_equal(v2, vr)
    # partial page: the unused tail is zero and the first tokens survive
    page = h.records_to_page(kr[:37], vr[:37])
    k3, v3 = h.page_to_records(page, 37)
    assert np.array_equal(k3, kr[:37]) and np.array_equal(v3, vr[:37])


def _unpack(rec, bits, d):
    per = 8 // bits
    b = rec[:, :d * bits // 8]
    sh = (np.arange(per) * bits).astype(np.uint8)
    return ((b[:, :, None] >> sh) & ((1 << bits) - 1)).reshape(rec.shape[0], d)


@pytest.mark.parametrize("d,vb,kb", [(64, 2, 3), (64, 4, 3), (128, 2, 3), (128, 4, 3), (256, 2, 3), (256, 4, 3),
                                     (64, 4, 4), (128, 4, 4), (256, 4, 4)])
def test_decoder_operand_extraction_matches_records(d, vb, kb):
    """Emulate, on the CPU, how the decode kernel cuts mma.sync operands out of a page.

    Key side (f16 m16n8k16, A operand, rows = tokens, k = coordinates): every f16 half must be 0, or
    2^(q-24) for the bit position q it was masked from, exactly when the bit-plane value is 1.
    Value side (f16 m16n8k16, A operand): every f16 half must equal code * 2^(pos - 24) for the
    position that the B operand is prescaled with.
    With a 3-bit index (key_bits 4) the decoder also forms the parity plane b2 ^ b1 ^ b0 by XOR of the
    three index-plane words before masking; that plane is checked as a fifth.
    """
    from oracle.quant import _unpack_bits
    h = tqm.HostTables(tqm.config(head_dim=d, value_bits=vb, key_bits=kb))
    rng = np.random.default_rng(7)
    kr, vr = _random_records(h, 128, rng)
    page = h.records_to_page(kr, vr)
    mb = kb - 1
    idx = _unpack_bits(kr[:, :d * mb // 8], mb, d)
    sign = _unpack(kr[:, d * mb // 8:], 1, d)
    codes = _unpack(vr, vb, d)
    planes = [(idx >> (mb - 1 - p)) & 1 for p in range(mb)] + [sign]
    if kb == 4:
        planes.append(((idx >> 2) ^ (idx >> 1) ^ idx) & 1)
    kw = page[:kb * 128 * d // 8].view(np.uint32)
    halves = max(1, d // 128)

    def word(tile, pi, hf, lane, row):
        if pi == kb:  # the parity plane: XOR of the index-plane words
            return word(tile, 0, hf, lane, row) ^ word(tile, 1, hf, lane, row) ^ word(tile, 2, hf, lane, row)
        if d == 64:  # both tiles of a 32-token group share a word; the odd one 8 positions up
            return int(kw[(((tile >> 1) * kb + pi) * 32 + lane) * 2 + row]) >> (8 * (tile & 1))
        return int(kw[(((tile * kb + pi) * halves + hf) * 32 + lane) * 2 + row])

    for tile in range(8):
        for pi in range(len(planes)):
            for hf in range(halves):
                for lane in range(32):
                    g, c = lane >> 2, lane & 3
                    w0, w1 = word(tile, pi, hf, lane, 0), word(tile, pi, hf, lane, 1)  # rows g and g + 8 of the tile
                    for s_ in range(min(8, d // 16)):
                        if s_ < 6:
                            x0, x1, q0 = w0, w1, 2 * s_
                        else:
                            x0, x1, q0 = w0 >> 4, w1 >> 4, 2 * s_ - 4
                        m0, m1 = 0x00010001 << q0, 0x00010001 << (q0 + 1)
                        regs = [x0 & m0, x1 & m0, x0 & m1, x1 & m1]  # a0..a3 of m16n8k16
                        for r, reg in enumerate(regs):
                            row, kofs = r & 1, 8 * (r >> 1)
                            t = 16 * tile + g + 8 * row
                            for e in (0, 1):
                                half = (reg >> (16 * e)) & 0xFFFF
                                val = np.array([half], np.uint16).view(np.float16).astype(np.float64)[0]
                                j = 128 * hf + 16 * s_ + kofs + 2 * c + e
                                qeff = q0 + (r >> 1)
                                expect = 2.0 ** (qeff - 24) if planes[pi][t, j] else 0.0
                                assert val == expect
    off = kb * 128 * d // 8 + 4 * 128
    vw = page[off:off + 128 * d * vb // 8].view(np.uint32)
    nmt = d // 16
    pos2 = {(0, 0): 0, (0, 1): 4, (1, 0): 6, (1, 1): 8}
    for blk in range(4):
        for mt in range(nmt):
            for lane in range(32):
                g, c = lane >> 2, lane & 3
                if vb == 2:
                    w = int(vw[(blk * nmt + mt) * 32 + lane])
                    w2, w6 = w >> 2, w >> 6
                    regs = {0: [w & 0x00030003, w2 & 0x00030003, w & 0x00300030, w6 & 0x00300030],
                            1: [w & 0x00C000C0, w6 & 0x00C000C0, w & 0x03000300, w6 & 0x03000300]}
                else:
                    x = int(vw[((blk * nmt + mt) * 32 + lane) * 2])
                    y = int(vw[((blk * nmt + mt) * 32 + lane) * 2 + 1])
                    regs = {0: [x & 0x000F000F, (x >> 8) & 0x000F000F, x & 0x00F000F0, (x >> 8) & 0x00F000F0],
                            1: [y & 0x000F000F, (y >> 8) & 0x000F000F, y & 0x00F000F0, (y >> 8) & 0x00F000F0]}
                for kap in (0, 1):
                    for r in range(4):
                        rowhi, hiT = r & 1, r >> 1
                        pos = pos2[(kap, hiT)] if vb == 2 else (4 if hiT else 0)
                        for e in (0, 1):
                            half = (regs[kap][r] >> (16 * e)) & 0xFFFF
                            val = np.array([half], np.uint16).view(np.float16).astype(np.float64)[0]
                            t = 32 * blk + 16 * kap + 8 * hiT + 2 * c + e
                            j = 16 * mt + 8 * rowhi + g
                            assert val == codes[t, j] * 2.0 ** (pos - 24)


def test_codec_kv_bytes_reproduce_the_overview_table():
    """tq_codec_kv_bytes against the KV sizes the overview prints for Llama-3.1-8B at 32K tokens."""
    from kv_cache_quantization_quantize_gb300 import codecs
    g = json.load(open(os.path.join(GOLDEN, "memory_figures.json")))["llama31_8b_32k"]
    sh = g["shape"]
    MiB = 1 << 20
    args = (sh["layers"], sh["kv_heads"], sh["head_dim"], sh["seq_len"])
    assert codecs.codec_kv_bytes("fp16", *args) == g["fp16_MB"] * MiB
    assert codecs.codec_kv_bytes("kivi2", *args) == g["kivi_2bit_MB"] * MiB
    assert codecs.codec_kv_bytes("bonsai1", *args) == g["bonsai_1bit_g128_MB"] * MiB
    # this library's records: key d/4 + d/8 + 4 bytes, value d/4 (2-bit) or d/2 (4-bit) + d/16 bytes
    h = tqm.HostTables(tqm.config(head_dim=128, value_bits=2))
    per = h.key_record_bytes() + h.value_record_bytes()
    assert codecs.codec_kv_bytes("turboquant_k3v2", *args) == per * 32 * 8 * 32768 == 736 * MiB
    assert codecs.codec_kv_bytes("turboquant_k3v4", *args) == 992 * MiB
    lib = _abi.load()
    assert lib.tq_codec_kv_bytes(_abi.TQ_CODEC_BONSAI1, 1, 1, 64, 16) == 0  # head_dim not a multiple of 128
    assert lib.tq_codec_kv_bytes(_abi.TQ_CODEC_KIVI2, 1, 1, 24, 16) == 0
    assert lib.tq_codec_kv_bytes(99, 1, 1, 128, 16) == 0
    assert lib.tq_codec_kv_bytes(_abi.TQ_CODEC_FP16, 0, 1, 128, 16) == 0


def test_codec_entry_points_validate_before_launching():
    """Bad sizes and misaligned pointers are rejected on the host (no device work is attempted);
    an empty input returns TQ_OK without a launch."""
    lib = _abi.load()
    P = ctypes.c_void_p
    a16, mis = P(1 << 20), P((1 << 20) + 2)
    outs = [a16] * 6
    assert lib.tq_kivi2_quantize(a16, a16, 32, 2, 24, *outs, None) == _abi.TQ_ERR_INVALID_ARG      # d % 16
    assert lib.tq_kivi2_quantize(a16, None, 40, 2, 64, *outs, None) == _abi.TQ_ERR_INVALID_ARG     # keys: T % 16
    assert lib.tq_kivi2_quantize(mis, None, 32, 2, 64, *outs, None) == _abi.TQ_ERR_INVALID_ARG     # k alignment
    assert lib.tq_kivi2_quantize(a16, None, 32, 2, 64, None, a16, a16, None, None, None, None) \
        == _abi.TQ_ERR_INVALID_ARG                                                                  # NULL output
    assert lib.tq_kivi2_quantize(a16, a16, 0, 2, 64, *outs, None) == _abi.TQ_OK                    # empty
    assert lib.tq_kivi2_dequantize(*outs, 32, 2, 64, mis, None, None) == _abi.TQ_ERR_INVALID_ARG
    assert lib.tq_bonsai1_quantize(a16, a16, 4, 64, a16, a16, a16, a16, None) == _abi.TQ_ERR_INVALID_ARG
    assert lib.tq_bonsai1_quantize(a16, mis, 4, 128, a16, a16, a16, a16, None) == _abi.TQ_ERR_INVALID_ARG
    assert lib.tq_bonsai1_quantize(a16, None, -1, 128, a16, a16, None, None, None) == _abi.TQ_ERR_INVALID_ARG
    assert lib.tq_bonsai1_quantize(a16, a16, 0, 128, a16, a16, a16, a16, None) == _abi.TQ_OK
    assert lib.tq_bonsai1_dequantize(a16, a16, a16, a16, 4, 128, mis, None, None) == _abi.TQ_ERR_INVALID_ARG


def test_debug_hooks_validate_their_arguments():
    """The wait-timeout test hooks only set process-wide knobs: their argument checks run on the host."""
    lib = _abi.load()
    assert lib.tq_debug_append_wait_fault(-2, 8) == _abi.TQ_ERR_INVALID_ARG
    assert lib.tq_debug_append_wait_fault(0, 0) == _abi.TQ_ERR_INVALID_ARG
    assert lib.tq_debug_append_wait_fault(0, (1 << 22) + 1) == _abi.TQ_ERR_INVALID_ARG
    assert lib.tq_debug_append_wait_fault(5, 8) == _abi.TQ_OK
    assert lib.tq_debug_append_wait_fault(-1, 0) == _abi.TQ_OK
    assert lib.tq_debug_prefill_wait_fault(-2, 8) == _abi.TQ_ERR_INVALID_ARG
    assert lib.tq_debug_prefill_wait_fault(1, 0) == _abi.TQ_ERR_INVALID_ARG
    assert lib.tq_debug_prefill_wait_fault(1, (1 << 22) + 1) == _abi.TQ_ERR_INVALID_ARG
    assert lib.tq_debug_prefill_wait_fault(3, 8) == _abi.TQ_OK
    assert lib.tq_debug_prefill_wait_fault(-1, 0) == _abi.TQ_OK
    assert lib.tq_debug_decode_wait_fault(4, 8) == _abi.TQ_ERR_INVALID_ARG
    assert lib.tq_debug_decode_wait_fault(-1, 0) == _abi.TQ_OK
