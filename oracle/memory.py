"""KV-cache memory arithmetic.

[Blog] §2.1 gives the dense formula: 2 * batch * layers * heads * seq_len * head_dim * bytes. Its
example is Llama-2-7B (32 layers, 32 heads, head_dim 128, fp16): 1.07 GB at 2048 tokens, ~4.3 GB at
8192.

[Overview] §性能表现与实测数据 (table) gives Llama-3.1-8B at 32K context:
* fp16: 4,096 MB;
* TurboQuant 4-bit: 1,056 MB;
* KIVI 2-bit: 1,024 MB;
* Bonsai 1-bit: 288 MB.
"""

from .quant import key_record_bytes, value_record_bytes


def kv_bytes_dense(layers, kv_heads, seq_len, head_dim, batch=1, bytes_per_elem=2):
    """Dense K+V bytes: 2 * B * layers * heads * S * D * bytes."""
    return 2 * batch * layers * kv_heads * seq_len * head_dim * bytes_per_elem


def kv_bytes_bits_per_element(layers, kv_heads, seq_len, head_dim, bits, fp16_per_elems, batch=1):
    """K+V bytes at `bits` per element plus one fp16 per `fp16_per_elems` elements (per vector)."""
    per_vec = head_dim * bits // 8 + 2 * (head_dim // fp16_per_elems)
    return 2 * batch * layers * kv_heads * seq_len * per_vec


def kv_bytes_turboquant(layers, kv_heads, seq_len, head_dim, value_bits, batch=1):
    """Packed K3 (2-bit Lloyd-Max + QJL sign + fp16 n, gamma) + Vb (g32, fp16 scales) record bytes."""
    per_tok = key_record_bytes(head_dim) + value_record_bytes(head_dim, value_bits)
    return batch * layers * kv_heads * seq_len * per_tok
