"""GPU parity of the comparison codecs (KIVI 2-bit, Bonsai 1-bit) against the oracle, through the C ABI.

Codes and KIVI parameters are integer/fp16 decisions taken in fp32 on both sides: bit-exact. The
Bonsai scale is an fp32 sum of 128 magnitudes in the kernel and an fp64 mean in the oracle: at most one
fp16 ulp apart. Reconstructions are compared bit-exactly against the oracle's reconstruction of the
device's own codes, rounded to bf16 through fp32 as the kernel does.
"""
import numpy as np
import pytest
import torch

import oracle
from kv_cache_quantization_quantize_gb300 import TQError, codecs, synth

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def built():
    from kv_cache_quantization_quantize_gb300 import build
    build.build()


def _u32(t):
    return t.cpu().numpy().view(np.uint32)


def _unpack2(words):
    """uint32 words of 16 two-bit codes -> codes along a new trailing axis of 16 (code i at bits 2i)."""
    return ((words[..., None] >> (2 * np.arange(16, dtype=np.uint32))) & 3).astype(np.uint8)


def kivi_device_codes(out, T, H, d):
    """Device KIVI output -> per-head (k codes [T, d], k scale, k zero, v codes [T, d], v scale, v zero)."""
    res = []
    kc = _u32(out["k_codes"]).reshape(T // 16, H, d)
    ks = out["k_scale"].cpu().numpy().reshape(T // 16, H, d)
    kz = out["k_zero"].cpu().numpy().reshape(T // 16, H, d)
    vc = _u32(out["v_codes"]).reshape(T, H, d // 16)
    vs = out["v_scale"].cpu().numpy().reshape(T, H, d // 16)
    vz = out["v_zero"].cpu().numpy().reshape(T, H, d // 16)
    for h in range(H):
        kcodes = _unpack2(kc[:, h, :]).transpose(0, 2, 1).reshape(T, d)  # [g, c, t] -> [g*16+t, c]
        vcodes = _unpack2(vc[:, h, :]).reshape(T, d)                      # [t, j, i] -> [t, 16j+i]
        res.append((kcodes, ks[:, h], kz[:, h], vcodes, vs[:, h], vz[:, h]))
    return res


def _bf16_of(x64):
    """fp64 -> fp32 -> bf16 (round to nearest even), as the kernels round their fp32 result."""
    return torch.from_numpy(np.asarray(x64, dtype=np.float64).astype(np.float32)).to(torch.bfloat16)


@pytest.mark.parametrize("T,H,d,dist", [(64, 2, 64, "normal"), (400, 3, 128, "student_t5"), (48, 8, 256, "normal")])
def test_kivi2_quantize_and_dequantize(T, H, d, dist):
    k, v = synth.kv_tokens(T, H, d, seed=T + d, dist=dist, outliers=("random", 4, 12.0))
    kd, vd = k.to(DEV), v.to(DEV)
    out = codecs.kivi2_quantize(kd, vd)
    kh, vh = codecs.kivi2_dequantize(out, T, H, d)
    torch.cuda.synchronize()
    dev = kivi_device_codes(out, T, H, d)
    k64, v64 = k.double().numpy(), v.double().numpy()
    for h in range(H):
        kc, ks, kz, vc, vs, vz = dev[h]
        okc, oks, okz = oracle.kivi2_quantize(k64[:, h], 0)
        ovc, ovs, ovz = oracle.kivi2_quantize(v64[:, h], 1)
        assert np.array_equal(ks.view(np.uint16), oks.view(np.uint16)) and np.array_equal(kz.view(np.uint16), okz.view(np.uint16))
        assert np.array_equal(kc, okc)
        assert np.array_equal(vs.view(np.uint16), ovs.view(np.uint16)) and np.array_equal(vz.view(np.uint16), ovz.view(np.uint16))
        assert np.array_equal(vc, ovc)
        # reconstruction of the device's own codes
        assert torch.equal(kh[:, h].cpu(), _bf16_of(oracle.kivi2_dequantize(kc, ks, kz, 0)))
        assert torch.equal(vh[:, h].cpu(), _bf16_of(oracle.kivi2_dequantize(vc, vs, vz, 1)))


@pytest.mark.parametrize("T,H,d", [(37, 4, 128), (37, 1, 16)])
def test_kivi2_values_ragged_tokens_and_single_tensor_calls(T, H, d):
    """Values alone take any token count (per-token groups; 37 x 1 x 16 is an odd group count);
    keys alone need a multiple of 16 tokens."""
    k, v = synth.kv_tokens(T, H, d, seed=5)
    out = codecs.kivi2_alloc(T, H, d)
    codecs.kivi2_quantize(None, v.to(DEV), out=out)
    _, vh = codecs.kivi2_dequantize(out, T, H, d, keys=False)
    torch.cuda.synchronize()
    vc = _u32(out["v_codes"]).reshape(T, H, d // 16)
    for h in range(H):
        ovc, ovs, ovz = oracle.kivi2_quantize(v[:, h].double().numpy(), 1)
        assert np.array_equal(_unpack2(vc[:, h]).reshape(T, d), ovc)
        assert np.array_equal(out["v_scale"].cpu().numpy().reshape(T, H, -1)[:, h].view(np.uint16), ovs.view(np.uint16))
        assert torch.equal(vh[:, h].cpu(), _bf16_of(oracle.kivi2_dequantize(ovc, ovs, ovz, 1)))
    with pytest.raises(TQError):
        codecs.kivi2_quantize(k.to(DEV), None)
    k2 = k[:32].to(DEV).contiguous()
    out2 = codecs.kivi2_quantize(k2, None)
    torch.cuda.synchronize()
    kc = kivi_device_codes({**out2, "v_codes": torch.zeros(32, H * d // 16, dtype=torch.int32),
                            "v_scale": torch.zeros(32, H * d // 16, dtype=torch.float16),
                            "v_zero": torch.zeros(32, H * d // 16, dtype=torch.float16)}, 32, H, d)
    for h in range(H):
        assert np.array_equal(kc[h][0], oracle.kivi2_quantize(k[:32, h].double().numpy(), 0)[0])


def test_kivi2_constant_groups_and_empty():
    """A constant group has scale 0, zero = fp16(value) and codes 0; n_tokens = 0 launches nothing."""
    k = torch.full((16, 1, 64), 0.3125, dtype=torch.bfloat16, device=DEV)
    v = torch.full((16, 1, 64), -2.5, dtype=torch.bfloat16, device=DEV)
    out = codecs.kivi2_quantize(k, v)
    kh, vh = codecs.kivi2_dequantize(out, 16, 1, 64)
    torch.cuda.synchronize()
    assert int(out["k_codes"].abs().sum()) == 0 and int(out["v_codes"].abs().sum()) == 0
    assert float(out["k_scale"].abs().max()) == 0 and float(out["v_scale"].abs().max()) == 0
    assert torch.equal(kh, k) and torch.equal(vh, v)
    e = torch.empty(0, 2, 64, dtype=torch.bfloat16, device=DEV)
    codecs.kivi2_quantize(e, e)
    torch.cuda.synchronize()


def _bonsai_check(x, bits, scale, xh):
    """x [R, d] bf16 (CPU); device bits [R, d/32] words, scale [R, d/128] fp16, xh [R, d] bf16."""
    R, d = x.shape
    x64 = x.double().numpy()
    ob, os_ = oracle.bonsai1_quantize(x64)
    b = ((_u32(bits)[..., None] >> np.arange(32, dtype=np.uint32)) & 1).astype(np.uint8).reshape(R, d)
    assert np.array_equal(b, ob)
    s = scale.cpu().numpy()
    ulp = np.abs(s.view(np.int16).astype(np.int32) - os_.view(np.int16).astype(np.int32))
    assert ulp.max() <= 1, "Bonsai scale more than one fp16 ulp from the oracle's mean |x|"
    assert np.mean(ulp == 0) > 0.9
    assert torch.equal(xh.cpu(), _bf16_of(oracle.bonsai1_dequantize(b, s)))


@pytest.mark.parametrize("T,H,d", [(37, 3, 128), (64, 8, 128), (20, 2, 256)])
def test_bonsai1_quantize_and_dequantize(T, H, d):
    """T*H rows; 37*3 = 111 rows of one group gives an odd group count (half of the last span)."""
    k, v = synth.kv_tokens(T, H, d, seed=T * H + d, dist="student_t5", outliers=("random", 2, 8.0))
    k[0, 0, :7] = 0.0
    k[0, 0, 7:9] = -0.0
    out = codecs.bonsai1_quantize(k.to(DEV), v.to(DEV))
    kh, vh = codecs.bonsai1_dequantize(out, T, H, d)
    torch.cuda.synchronize()
    _bonsai_check(k.reshape(T * H, d), out["k_bits"], out["k_scale"], kh.reshape(T * H, d))
    _bonsai_check(v.reshape(T * H, d), out["v_bits"], out["v_scale"], vh.reshape(T * H, d))


def test_bonsai1_single_tensor_and_empty():
    T, H, d = 9, 1, 128
    k, v = synth.kv_tokens(T, H, d, seed=3)
    out = codecs.bonsai1_alloc(T * H, d)
    out["k_bits"].fill_(-1)
    codecs.bonsai1_quantize(None, v.to(DEV), out=out)
    _, vh = codecs.bonsai1_dequantize(out, T, H, d, keys=False)
    torch.cuda.synchronize()
    assert int((out["k_bits"] != -1).sum()) == 0  # the key outputs were left alone
    _bonsai_check(v.reshape(T, d), out["v_bits"], out["v_scale"], vh.reshape(T, d))
    e = torch.empty(0, 1, 128, dtype=torch.bfloat16, device=DEV)
    codecs.bonsai1_quantize(e, e)
    torch.cuda.synchronize()


def test_codecs_full_layer_sampled():
    """One layer of the Llama-3.1-8B workload (32768 tokens x 8 KV heads x 128), in the launch shape the
    codec bench times: sampled groups against the oracle, and the stored sizes against the table."""
    T, H, d = 32768, 8, 128
    k, v = synth.kv_tokens(T, H, d, seed=11, outliers=("random", 4, 10.0), device=DEV)
    kv = codecs.kivi2_quantize(k, v)
    bo = codecs.bonsai1_quantize(k, v)
    torch.cuda.synchronize()
    g = torch.Generator().manual_seed(1)
    kc = _u32(kv["k_codes"]).reshape(T // 16, H, d)
    vc = _u32(kv["v_codes"]).reshape(T, H, d // 16)
    for _ in range(24):
        grp = int(torch.randint(0, T // 16, (1,), generator=g))
        h = int(torch.randint(0, H, (1,), generator=g))
        ks = k[16 * grp:16 * grp + 16, h].double().cpu().numpy()
        oc, osc, oz = oracle.kivi2_quantize(ks, 0)
        assert np.array_equal(_unpack2(kc[grp, h]).T, oc)
        assert np.array_equal(kv["k_scale"][grp].view(H, d)[h].cpu().numpy().view(np.uint16), osc[0].view(np.uint16))
        t = int(torch.randint(0, T, (1,), generator=g))
        vs = v[t:t + 1, h].double().cpu().numpy()
        ovc, ovs, _ = oracle.kivi2_quantize(vs, 1)
        assert np.array_equal(_unpack2(vc[t, h]).reshape(1, d), ovc)
        row = t * H + h
        xr = v[t, h].float().cpu()[None]
        b = ((_u32(bo["v_bits"][row])[..., None] >> np.arange(32, dtype=np.uint32)) & 1).astype(np.uint8).reshape(1, d)
        assert np.array_equal(b, oracle.bonsai1_quantize(xr.double().numpy())[0])
    MiB = 1 << 20
    kv_bytes = sum(t.numel() * t.element_size() for t in kv.values())
    bo_bytes = sum(t.numel() * t.element_size() for t in bo.values())
    assert kv_bytes * 32 == codecs.codec_kv_bytes("kivi2", 32, 8, 128, 32768) == 1024 * MiB
    assert bo_bytes * 32 == codecs.codec_kv_bytes("bonsai1", 32, 8, 128, 32768) == 288 * MiB
