"""TurboQuant KV-cache hot path on GB300: Python binding of libtq (C ABI + sm_103a CUDA kernels).

PyTorch only provides device memory and streams here. Every step of quantize-on-append and hybrid
decode attention runs in libtq's kernels; there is no CPU or PyTorch fallback.
"""
import ctypes

import numpy as np
import torch

from . import _abi
from ._abi import TQConfig, TQError, check, load, TQ_BF16, TQ_F32
from . import codecs

__all__ = ["TQConfig", "TQError", "TurboQuantCache", "HostTables", "load", "config", "codecs"]


def config(head_dim=128, value_bits=2, n_layers=1, n_kv_heads=1, n_q_heads=1, max_seqs=1, max_ctx=1152, seed=0,
           mode="hybrid", n_blocks=0, key_bits=3):
    """mode "hybrid": 128-token exact recent buffer; "full_tq": every token quantised (ring_size 0).
    n_blocks > 0: paged cache with a pool of n_blocks 128-token blocks per layer (see block_table).
    key_bits 3: 2-bit Lloyd-Max index + QJL sign; key_bits 4 (with value_bits 4): 3-bit index + sign."""
    if mode not in ("hybrid", "full_tq"):
        raise ValueError(f"mode {mode!r}: expected 'hybrid' or 'full_tq'")
    return TQConfig(head_dim=head_dim, key_bits=key_bits, value_bits=value_bits, value_group=32,
                    ring_size=128 if mode == "hybrid" else 0, n_layers=n_layers, n_kv_heads=n_kv_heads,
                    n_q_heads=n_q_heads, max_seqs=max_seqs, max_ctx=max_ctx, seed=seed, n_blocks=n_blocks)


def _stream(stream=None):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else None


class HostTables:
    """Host-only context: the library's tables and record conversions (no device work)."""

    def __init__(self, cfg):
        self.cfg = cfg
        self.lib = load()
        self.ctx = ctypes.c_void_p()
        check(self.lib.tq_init_codebooks(ctypes.byref(cfg), None, 0, None, ctypes.byref(self.ctx)))

    def __del__(self):
        if getattr(self, "ctx", None) and self.ctx.value:
            self.lib.tq_destroy(self.ctx)
            self.ctx = ctypes.c_void_p()

    def tables(self):
        d = self.cfg.head_dim
        D = np.zeros(d, np.float32)
        S = np.zeros(d * d, np.uint16)
        nlev = 1 << (self.cfg.key_bits - 1)
        c = np.zeros(nlev, np.float64)
        t = np.zeros(nlev - 1, np.float64)
        check(self.lib.tq_get_tables(self.ctx, D.ctypes.data, S.ctypes.data, c.ctypes.data, t.ctypes.data))
        return D, S.reshape(d, d), c, t

    def page_bytes(self):
        return self.lib.tq_page_bytes(ctypes.byref(self.cfg))

    def key_record_bytes(self):
        d = self.cfg.head_dim
        return d * (self.cfg.key_bits - 1) // 8 + d // 8 + 4

    def value_record_bytes(self):
        d = self.cfg.head_dim
        return d * self.cfg.value_bits // 8 + d // 16

    def page_to_records(self, page, n_tokens):
        """Canonical key/value record bytes [n, kb], [n, vb] from one packed page (uint8 numpy)."""
        page = np.ascontiguousarray(page, dtype=np.uint8)
        kr = np.zeros((n_tokens, self.key_record_bytes()), np.uint8)
        vr = np.zeros((n_tokens, self.value_record_bytes()), np.uint8)
        check(self.lib.tq_page_to_records(self.ctx, page.ctypes.data, n_tokens, kr.ctypes.data, vr.ctypes.data))
        return kr, vr

    def records_to_page(self, keys, values):
        keys = np.ascontiguousarray(keys, dtype=np.uint8)
        values = np.ascontiguousarray(values, dtype=np.uint8)
        page = np.zeros(self.page_bytes(), np.uint8)
        check(self.lib.tq_records_to_page(self.ctx, keys.ctypes.data, values.ctypes.data, keys.shape[0],
                                          page.ctypes.data))
        return page


class TurboQuantCache(HostTables):
    """Device-resident packed KV cache of one model (all layers) plus its tables.

    Memory (tables, cache, decode workspace) is allocated with torch on `device`; the library never
    allocates device memory itself.
    """

    def __init__(self, cfg, device="cuda"):
        self.cfg = cfg
        self.lib = load()
        self.device = torch.device(device)
        with torch.cuda.device(self.device):
            tb = self.lib.tq_tables_bytes(ctypes.byref(cfg))
            if tb == 0:
                raise TQError(_abi.TQ_ERR_INVALID_ARG, "invalid config")
            self.tables_buf = torch.empty(tb, dtype=torch.uint8, device=self.device)
            self.ctx = ctypes.c_void_p()
            check(self.lib.tq_init_codebooks(ctypes.byref(cfg), _ptr(self.tables_buf), tb, _stream(),
                                             ctypes.byref(self.ctx)))
            cb = self.lib.tq_cache_bytes(ctypes.byref(cfg))
            self.cache_buf = torch.empty(cb, dtype=torch.uint8, device=self.device)
            check(self.lib.tq_cache_bind(self.ctx, _ptr(self.cache_buf), cb, _stream()))
        self._ws = None

    # ---- hot path ----
    def append(self, layer, k, v, seq_ids, n_new, stream=None):
        """k, v: [batch, max_new, n_kv_heads, d] bf16/f32 CUDA tensors; seq_ids, n_new: int32 CUDA tensors."""
        assert k.is_cuda and k.is_contiguous() and v.is_contiguous() and k.shape == v.shape and k.dtype == v.dtype
        dt = TQ_BF16 if k.dtype == torch.bfloat16 else TQ_F32
        if dt == TQ_F32:
            assert k.dtype == torch.float32
        check(self.lib.tq_quantize_append(self.ctx, layer, _ptr(k), _ptr(v), dt, _ptr(seq_ids), _ptr(n_new),
                                          k.shape[0], k.shape[1], _stream(stream)))

    def flush(self, layer, seq_ids, stream=None):
        check(self.lib.tq_ring_flush(self.ctx, layer, _ptr(seq_ids), seq_ids.numel(), _stream(stream)))

    def reset(self, seq_ids, layer=-1, stream=None):
        check(self.lib.tq_reset_seqs(self.ctx, layer, _ptr(seq_ids), seq_ids.numel(), _stream(stream)))

    def dequantize(self, layer, slot, head, t0, count, with_qjl=True, stream=None):
        """Packed tokens [t0, t0 + count) of (layer, slot, KV head) reconstructed in the original basis:
        (k_hat, v_hat), fp32 [count, d] CUDA tensors (tq_dequantize_tokens)."""
        d = self.cfg.head_dim
        k_hat = torch.empty((count, d), dtype=torch.float32, device=self.device)
        v_hat = torch.empty((count, d), dtype=torch.float32, device=self.device)
        check(self.lib.tq_dequantize_tokens(self.ctx, layer, slot, head, t0, count, 1 if with_qjl else 0,
                                            _ptr(k_hat), _ptr(v_hat), _stream(stream)))
        return k_hat, v_hat

    def workspace_bytes(self, batch, max_ctx_hint=0):
        return self.lib.tq_workspace_bytes(self.ctx, batch, max_ctx_hint)

    def workspace(self, batch, max_ctx_hint=0):
        n = self.workspace_bytes(batch, max_ctx_hint)
        if self._ws is None or self._ws.numel() < n:
            self._ws = torch.zeros(n, dtype=torch.uint8, device=self.device)  # arrival counters start at 0
        return self._ws

    def decode(self, layer, q, seq_ids, softmax_scale=0.0, out=None, max_ctx_hint=0, workspace=None, stream=None):
        """q: [batch, n_q_heads, d] bf16 CUDA tensor -> out [batch, n_q_heads, d] f32."""
        assert q.is_cuda and q.dtype == torch.bfloat16 and q.is_contiguous()
        batch = q.shape[0]
        if out is None:
            out = torch.empty(q.shape, dtype=torch.float32, device=q.device)
        ws = workspace if workspace is not None else self.workspace(batch, max_ctx_hint)
        check(self.lib.tq_decode_attention(self.ctx, layer, _ptr(q), _ptr(out), _ptr(seq_ids), batch,
                                           float(softmax_scale), _ptr(ws), ws.numel(), max_ctx_hint, _stream(stream)))
        return out

    def decode_step(self, layer, k_new, v_new, q, seq_ids, softmax_scale=0.0, out=None, max_ctx_hint=0,
                    workspace=None, stream=None):
        """One decode step in one launch: appends k_new, v_new [batch, n_kv_heads, d] (bf16/f32, one token
        per row) and returns the attention of q [batch, n_q_heads, d] bf16 over the sequence with it (f32).
        Equal to append(..., n_new=1) followed by decode()."""
        assert q.is_cuda and q.dtype == torch.bfloat16 and q.is_contiguous()
        assert k_new.is_cuda and k_new.is_contiguous() and v_new.is_contiguous() and k_new.shape == v_new.shape
        assert k_new.dtype == v_new.dtype and k_new.dtype in (torch.bfloat16, torch.float32)
        dt = TQ_BF16 if k_new.dtype == torch.bfloat16 else TQ_F32
        batch = q.shape[0]
        if out is None:
            out = torch.empty(q.shape, dtype=torch.float32, device=q.device)
        ws = workspace if workspace is not None else self.workspace(batch, max_ctx_hint)
        check(self.lib.tq_decode_step(self.ctx, layer, _ptr(k_new), _ptr(v_new), dt, _ptr(q), _ptr(out), _ptr(seq_ids),
                                      batch, float(softmax_scale), _ptr(ws), ws.numel(), max_ctx_hint,
                                      _stream(stream)))
        return out

    def prefill_workspace(self, batch, q_per_row, max_ctx_hint=0):
        n = self.lib.tq_prefill_workspace_bytes(self.ctx, batch, q_per_row, max_ctx_hint)
        return torch.empty(max(n, 256), dtype=torch.uint8, device=self.device)

    def prefill(self, layer, q, seq_ids, n_q, softmax_scale=0.0, out=None, max_ctx_hint=0, workspace=None,
                stream=None):
        """Chunk attention after its append: q [batch, q_per_row, n_q_heads, d] bf16 (a row's last n_q[b]
        tokens; the rest padding) -> out [batch, q_per_row, n_q_heads, d] f32, causal over the cache."""
        assert q.is_cuda and q.dtype == torch.bfloat16 and q.is_contiguous() and q.dim() == 4
        batch, qpr = q.shape[0], q.shape[1]
        if out is None:
            out = torch.empty(q.shape, dtype=torch.float32, device=q.device)
        ws = workspace if workspace is not None else self.prefill_workspace(batch, qpr, max_ctx_hint)
        check(self.lib.tq_prefill_attention(self.ctx, layer, _ptr(q), _ptr(out), _ptr(seq_ids), _ptr(n_q), batch, qpr,
                                            float(softmax_scale), _ptr(ws), ws.numel(), max_ctx_hint,
                                            _stream(stream)))
        return out

    def decode_phase(self, phase, layer, q, seq_ids, out, softmax_scale=0.0, max_ctx_hint=0, workspace=None,
                     stream=None):
        """One phase of decode(): 0 zeroes the workspace's arrival counters, 1 runs the decode launch (its
        last CTA per (row, KV head) combines). 0 then 1 equals decode()."""
        batch = q.shape[0]
        ws = workspace if workspace is not None else self.workspace(batch, max_ctx_hint)
        check(self.lib.tq_decode_phase(self.ctx, phase, layer, _ptr(q), _ptr(out), _ptr(seq_ids), batch,
                                       float(softmax_scale), _ptr(ws), ws.numel(), max_ctx_hint, _stream(stream)))
        return out

    def check_status(self, clear=True, stream=None):
        """Device status word (0 = fine); raises TQError on a non-zero word unless clear-and-return is wanted."""
        w = ctypes.c_uint32(0)
        st = self.lib.tq_check_status(self.ctx, _stream(stream), ctypes.byref(w), 1 if clear else 0)
        if st not in (_abi.TQ_OK, _abi.TQ_ERR_DEVICE):
            check(st)
        return w.value

    # ---- inspection (tests, tools) ----
    def state(self, layer, slot):
        off = self.lib.tq_state_offset(self.ctx, layer, slot)
        return tuple(int(x) for x in self.cache_buf[off:off + 8].view(torch.int32).cpu())

    @property
    def block_table(self):
        """Paged cache: the int32 block table [max_seqs, max_pages] (a view of the cache buffer, -1 = no
        block). The caller maps every page an append or decode will touch, once for all layers."""
        if self.cfg.n_blocks <= 0:
            return None
        off = self.lib.tq_block_table_offset(self.ctx)
        max_pages = (self.cfg.max_ctx + 127) // 128
        n = self.cfg.max_seqs * max_pages
        return self.cache_buf[off:off + 4 * n].view(torch.int32).view(self.cfg.max_seqs, max_pages)

    def page(self, layer, slot, head, page):
        if self.cfg.n_blocks > 0:
            blk = int(self.block_table[slot, page])
            off = self.lib.tq_block_page_offset(self.ctx, layer, blk, head)
        else:
            off = self.lib.tq_page_offset(self.ctx, layer, slot, head, page)
        return self.cache_buf[off:off + self.page_bytes()].cpu().numpy()

    def ring(self, layer, slot, head):
        d = self.cfg.head_dim
        out = []
        for which in (0, 1):
            off = self.lib.tq_ring_offset(self.ctx, layer, slot, head, which)
            out.append(self.cache_buf[off:off + 128 * d * 2].view(torch.bfloat16).view(128, d))
        return out

    def records(self, layer, slot, head, n_tokens):
        """Canonical key/value records of the first n_tokens packed tokens (device -> host)."""
        ks, vs = [], []
        for pg in range((n_tokens + 127) // 128):
            cnt = min(128, n_tokens - 128 * pg)
            kr, vr = self.page_to_records(self.page(layer, slot, head, pg), cnt)
            ks.append(kr)
            vs.append(vr)
        if not ks:
            return (np.zeros((0, self.key_record_bytes()), np.uint8), np.zeros((0, self.value_record_bytes()), np.uint8))
        return np.concatenate(ks), np.concatenate(vs)
