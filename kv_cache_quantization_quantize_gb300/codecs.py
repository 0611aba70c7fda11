"""Python binding of libtq's comparison codecs (KIVI 2-bit, Bonsai 1-bit; TurboQuant-vLLM overview
§核心技术解析). Argument marshalling only: the coding runs in libtq's kernels; there is no fallback.

Tensors are bf16 [n_tokens, n_heads, head_dim] on the device. Outputs are allocated here unless the
caller passes them (dict of tensors with the shapes below).
"""
import ctypes

import torch

from ._abi import (TQ_CODEC_BONSAI1, TQ_CODEC_FP16, TQ_CODEC_KIVI2, TQ_CODEC_TQ_K3V2, TQ_CODEC_TQ_K3V4, check,
                   load)

__all__ = ["kivi2_quantize", "kivi2_dequantize", "bonsai1_quantize", "bonsai1_dequantize", "codec_kv_bytes",
           "TQ_CODEC_FP16", "TQ_CODEC_KIVI2", "TQ_CODEC_BONSAI1", "TQ_CODEC_TQ_K3V2", "TQ_CODEC_TQ_K3V4"]

_CODECS = {"fp16": TQ_CODEC_FP16, "kivi2": TQ_CODEC_KIVI2, "bonsai1": TQ_CODEC_BONSAI1,
           "turboquant_k3v2": TQ_CODEC_TQ_K3V2, "turboquant_k3v4": TQ_CODEC_TQ_K3V4}


def _p(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else None


def _s(stream):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _shape(x):
    if x.dtype != torch.bfloat16 or x.dim() != 3 or not x.is_contiguous() or not x.is_cuda:
        raise ValueError("expected a contiguous bf16 CUDA tensor [n_tokens, n_heads, head_dim]")
    return x.shape


def codec_kv_bytes(codec, n_layers, n_kv_heads, head_dim, n_tokens):
    """Stored K + V bytes under `codec` ("fp16", "kivi2", "bonsai1", "turboquant_k3v2", "turboquant_k3v4")."""
    return load().tq_codec_kv_bytes(_CODECS[codec], n_layers, n_kv_heads, head_dim, n_tokens)


def kivi2_alloc(n_tokens, n_heads, head_dim, device="cuda"):
    C = n_heads * head_dim
    u32 = dict(dtype=torch.int32, device=device)
    f16 = dict(dtype=torch.float16, device=device)
    return {"k_codes": torch.empty(n_tokens // 16, C, **u32), "k_scale": torch.empty(n_tokens // 16, C, **f16),
            "k_zero": torch.empty(n_tokens // 16, C, **f16), "v_codes": torch.empty(n_tokens, C // 16, **u32),
            "v_scale": torch.empty(n_tokens, C // 16, **f16), "v_zero": torch.empty(n_tokens, C // 16, **f16)}


def kivi2_quantize(k, v, out=None, stream=None):
    """k, v: bf16 [T, H, d] (either may be None). Returns the dict of kivi2_alloc (codes as int32 words)."""
    T, H, d = _shape(k if k is not None else v)
    if v is not None and _shape(v) != (T, H, d):
        raise ValueError("k and v shapes differ")
    out = out if out is not None else kivi2_alloc(T, H, d, (k if k is not None else v).device)
    check(load().tq_kivi2_quantize(_p(k), _p(v), T, H, d, _p(out["k_codes"]), _p(out["k_scale"]),
                                   _p(out["k_zero"]), _p(out["v_codes"]), _p(out["v_scale"]), _p(out["v_zero"]),
                                   _s(stream)))
    return out


def _deq_out(out, dev, n_tokens, n_heads, head_dim, keys, values):
    if out is not None:
        return out
    mk = lambda: torch.empty(n_tokens, n_heads, head_dim, dtype=torch.bfloat16, device=dev)
    return (mk() if keys else None), (mk() if values else None)


def kivi2_dequantize(codes, n_tokens, n_heads, head_dim, keys=True, values=True, out=None, stream=None):
    """Returns (k_hat, v_hat) bf16 [T, H, d] (None for a tensor not asked for); `out` = (k_hat, v_hat)."""
    kh, vh = _deq_out(out, codes["k_codes"].device, n_tokens, n_heads, head_dim, keys, values)
    check(load().tq_kivi2_dequantize(_p(codes["k_codes"]), _p(codes["k_scale"]), _p(codes["k_zero"]),
                                     _p(codes["v_codes"]), _p(codes["v_scale"]), _p(codes["v_zero"]), n_tokens,
                                     n_heads, head_dim, _p(kh), _p(vh), _s(stream)))
    return kh, vh


def bonsai1_alloc(n_rows, head_dim, device="cuda"):
    return {"k_bits": torch.empty(n_rows, head_dim // 32, dtype=torch.int32, device=device),
            "k_scale": torch.empty(n_rows, head_dim // 128, dtype=torch.float16, device=device),
            "v_bits": torch.empty(n_rows, head_dim // 32, dtype=torch.int32, device=device),
            "v_scale": torch.empty(n_rows, head_dim // 128, dtype=torch.float16, device=device)}


def bonsai1_quantize(k, v, out=None, stream=None):
    """k, v: bf16 [T, H, d] (either may be None); rows are the T*H head vectors."""
    T, H, d = _shape(k if k is not None else v)
    if v is not None and _shape(v) != (T, H, d):
        raise ValueError("k and v shapes differ")
    out = out if out is not None else bonsai1_alloc(T * H, d, (k if k is not None else v).device)
    check(load().tq_bonsai1_quantize(_p(k), _p(v), T * H, d, _p(out["k_bits"]), _p(out["k_scale"]),
                                     _p(out["v_bits"]), _p(out["v_scale"]), _s(stream)))
    return out


def bonsai1_dequantize(codes, n_tokens, n_heads, head_dim, keys=True, values=True, out=None, stream=None):
    """Returns (k_hat, v_hat) bf16 [T, H, d] (None for a tensor not asked for); `out` = (k_hat, v_hat)."""
    kh, vh = _deq_out(out, codes["k_bits"].device, n_tokens, n_heads, head_dim, keys, values)
    check(load().tq_bonsai1_dequantize(_p(codes["k_bits"]), _p(codes["k_scale"]), _p(codes["v_bits"]),
                                       _p(codes["v_scale"]), n_tokens * n_heads, head_dim, _p(kh), _p(vh),
                                       _s(stream)))
    return kh, vh
