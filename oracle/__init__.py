"""CPU oracle for TurboQuant's KV-cache hot path (quantize-on-append and hybrid decode attention).

TEST INFRASTRUCTURE, NOT PRODUCT CODE. This package is a plain, slow, fp64 restatement of what the
method computes. Only the tests under ``tests/``, ``__graft_entry__.smoke()`` and the ``cpu_baseline``
leg of ``bench.py`` may import it. The CUDA path never calls it and shares no code with it.

Sources, cited by page title and section throughout:

* [Guide]    hotelren.com/news/5528865, a TurboQuant-on-vLLM guide (page title
             "企业官网建设流程全解析"). §二 gives the five-step pipeline: rotate, Lloyd-Max, QJL residual
             sign, value group quantisation, bit packing. §五 gives ``key_bits=3, value_bits=2,
             buffer_size=128``. §六 gives cos_sim figures. §七 covers the hybrid decode.
* [Overview] zingnex.cn thread "TurboQuant-vLLM：大模型推理的KV缓存量化实战方案". §核心技术解析 covers
             Hadamard rotation and the PolarQuant magnitude/direction split. Its memory table is in
             §性能表现与实测数据.
* [Blog]     tqpw.cn/news/605998, §2.1: the KV-cache memory formula and its Llama-2-7B example.
* [News]     "TurboQuant 把 vLLM KV 快取壓成 3 位元": 3.8x smaller KV cache.

Readings of points the pages leave open are listed with each function.

Parity status:
* The comparison codecs (``codecs``: KIVI 2-bit, Bonsai 1-bit, [Overview] §核心技术解析) are pinned
  by ``tests/test_oracle_codecs.py``.
* Every function here is pinned by a ``-m "not gpu"`` test in ``tests/test_oracle_*.py``, except
  the key figure of ``cos_sim_report``. Its page figure (key cos_sim of about 1.000000, [Guide] §六) names no quantity
  that can be reproduced. It is **parity unpinned** and is only reported.
"""

from .rng import splitmix64, derive_seed, rademacher_signs, gaussian_matrix_bf16, round_to_bf16
from .rotation import hadamard, rotation_matrix
from .codebook import lloyd_max_codebook, beta_marginal_pdf, mse_distortion
from .quant import (
    KeyRecords, ValueRecords, quantize_keys, quantize_values, dequantize_keys, dequantize_values,
    pack_key_records, unpack_key_records, pack_value_records, unpack_value_records,
    key_record_bytes, value_record_bytes, history_split, cos_sim_report,
)
from .attention import decode_attention, estimated_scores, prefill_attention, qjl_inner_product_estimate
from .memory import kv_bytes_dense, kv_bytes_turboquant, kv_bytes_bits_per_element

from .codecs import bonsai1_dequantize, bonsai1_quantize, kivi2_dequantize, kivi2_quantize
__all__ = [n for n in dir() if not n.startswith("_")]
