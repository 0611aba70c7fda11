"""ctypes declarations of libtq's C ABI (include/tq.h). Loading fails loudly if the library is missing."""
import ctypes
import os
import re

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libtq.so")
HEADER = os.path.join(os.path.dirname(_PKG), "include", "tq.h")

TQ_OK, TQ_ERR_INVALID_ARG, TQ_ERR_UNSUPPORTED, TQ_ERR_CAPACITY, TQ_ERR_CUDA, TQ_ERR_DEVICE = range(6)
TQ_BF16, TQ_F32 = 0, 1
TQ_CODEC_FP16, TQ_CODEC_KIVI2, TQ_CODEC_BONSAI1, TQ_CODEC_TQ_K3V2, TQ_CODEC_TQ_K3V4 = range(5)
TQ_DEV_ERR_CAPACITY, TQ_DEV_ERR_SEQ_ID, TQ_DEV_ERR_SPLITS, TQ_DEV_ERR_TIMEOUT, TQ_DEV_ERR_BLOCK = 0x1, 0x2, 0x4, 0x8, 0x10

c_int, c_size_t, c_void_p, c_float = ctypes.c_int, ctypes.c_size_t, ctypes.c_void_p, ctypes.c_float


class TQConfig(ctypes.Structure):
    _fields_ = [
        ("head_dim", ctypes.c_int32), ("key_bits", ctypes.c_int32), ("value_bits", ctypes.c_int32),
        ("value_group", ctypes.c_int32), ("ring_size", ctypes.c_int32), ("n_layers", ctypes.c_int32),
        ("n_kv_heads", ctypes.c_int32), ("n_q_heads", ctypes.c_int32), ("max_seqs", ctypes.c_int32),
        ("max_ctx", ctypes.c_int32), ("seed", ctypes.c_uint64), ("n_blocks", ctypes.c_int32),
    ]


_P = ctypes.POINTER
_SIGS = {
    "tq_tables_bytes": (c_size_t, [_P(TQConfig)]),
    "tq_cache_bytes": (c_size_t, [_P(TQConfig)]),
    "tq_page_bytes": (c_size_t, [_P(TQConfig)]),
    "tq_init_codebooks": (c_int, [_P(TQConfig), c_void_p, c_size_t, c_void_p, _P(c_void_p)]),
    "tq_cache_bind": (c_int, [c_void_p, c_void_p, c_size_t, c_void_p]),
    "tq_reset_seqs": (c_int, [c_void_p, c_int, c_void_p, c_int, c_void_p]),
    "tq_quantize_append": (c_int, [c_void_p, c_int, c_void_p, c_void_p, c_int, c_void_p, c_void_p, c_int, c_int, c_void_p]),
    "tq_ring_flush": (c_int, [c_void_p, c_int, c_void_p, c_int, c_void_p]),
    "tq_dequantize_tokens": (c_int, [c_void_p, c_int, c_int, c_int, c_int, c_int, c_int, c_void_p, c_void_p,
                                     c_void_p]),
    "tq_workspace_bytes": (c_size_t, [c_void_p, c_int, c_int]),
    "tq_decode_attention": (c_int, [c_void_p, c_int, c_void_p, c_void_p, c_void_p, c_int, c_float, c_void_p, c_size_t,
                                    c_int, c_void_p]),
    "tq_decode_step": (c_int, [c_void_p, c_int, c_void_p, c_void_p, c_int, c_void_p, c_void_p, c_void_p, c_int, c_float,
                               c_void_p, c_size_t, c_int, c_void_p]),
    "tq_prefill_workspace_bytes": (c_size_t, [c_void_p, c_int, c_int, c_int]),
    "tq_prefill_attention": (c_int, [c_void_p, c_int, c_void_p, c_void_p, c_void_p, c_void_p, c_int, c_int, c_float,
                                     c_void_p, c_size_t, c_int, c_void_p]),
    "tq_decode_phase": (c_int, [c_void_p, c_int, c_int, c_void_p, c_void_p, c_void_p, c_int, c_float, c_void_p,
                                c_size_t, c_int, c_void_p]),
    "tq_decode_attention_noalloc": (c_int, [c_void_p, c_int, c_void_p, c_void_p, c_void_p, c_int, c_float, c_int,
                                            c_void_p]),
    "tq_debug_decode_wait_fault": (c_int, [c_int, c_int]),
    "tq_debug_append_wait_fault": (c_int, [c_int, c_int]),
    "tq_debug_prefill_wait_fault": (c_int, [c_int, c_int]),
    "tq_debug_prefill_path": (c_int, [c_int]),
    "tq_check_status": (c_int, [c_void_p, c_void_p, _P(ctypes.c_uint32), c_int]),
    "tq_destroy": (None, [c_void_p]),
    "tq_last_error": (ctypes.c_char_p, []),
    "tq_page_offset": (c_size_t, [c_void_p, c_int, c_int, c_int, c_int]),
    "tq_block_page_offset": (c_size_t, [c_void_p, c_int, c_int, c_int]),
    "tq_block_table_offset": (c_size_t, [c_void_p]),
    "tq_ring_offset": (c_size_t, [c_void_p, c_int, c_int, c_int, c_int]),
    "tq_state_offset": (c_size_t, [c_void_p, c_int, c_int]),
    "tq_status_offset": (c_size_t, [c_void_p]),
    "tq_page_to_records": (c_int, [c_void_p, c_void_p, c_int, c_void_p, c_void_p]),
    "tq_records_to_page": (c_int, [c_void_p, c_void_p, c_void_p, c_int, c_void_p]),
    "tq_get_tables": (c_int, [c_void_p, c_void_p, c_void_p, c_void_p, c_void_p]),
    "tq_kivi2_quantize": (c_int, [c_void_p, c_void_p, c_int, c_int, c_int] + [c_void_p] * 7),
    "tq_kivi2_dequantize": (c_int, [c_void_p] * 6 + [c_int, c_int, c_int, c_void_p, c_void_p, c_void_p]),
    "tq_bonsai1_quantize": (c_int, [c_void_p, c_void_p, ctypes.c_int64, c_int] + [c_void_p] * 5),
    "tq_bonsai1_dequantize": (c_int, [c_void_p] * 4 + [ctypes.c_int64, c_int, c_void_p, c_void_p, c_void_p]),
    "tq_codec_kv_bytes": (c_size_t, [c_int, c_int, c_int, c_int, ctypes.c_int64]),
}

_lib = None


def header_functions():
    """Names of the functions include/tq.h declares."""
    text = open(HEADER).read()
    return sorted(set(re.findall(r"^\s*(?:[\w\s\*]+?)\b(tq_\w+)\s*\(", text, re.M)))


def load():
    """Load libtq.so once. Raises if it has not been built (no fallback exists)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(f"libtq.so not found at {LIB_PATH}; build it with "
                           "`python -m kv_cache_quantization_quantize_gb300.build` (there is no CPU fallback)")
    lib = ctypes.CDLL(LIB_PATH)
    for name, (res, args) in _SIGS.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib


class TQError(RuntimeError):
    def __init__(self, status, msg):
        super().__init__(f"libtq status {status}: {msg}")
        self.status = status


def check(status):
    if status != TQ_OK:
        raise TQError(status, load().tq_last_error().decode(errors="replace"))
    return status
