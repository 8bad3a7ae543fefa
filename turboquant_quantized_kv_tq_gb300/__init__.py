"""Rotated-codebook quantized KV cache and fused decode attention for GB300 (sm_103a).

The C library (``include/tq.h``, built in-tree as ``_lib/libtq.so``) holds the codec tables,
the cache layout and the CUDA kernels.  ``binding`` exposes its entry points by name;
``QuantizedKVCache`` owns the device buffers (through torch) for one configuration and marshals
tensors to those entry points.  There is no CPU fallback: without the built library the import
fails.
"""

import numpy as np

from . import binding as _b
from .binding import TQError, check  # noqa: F401

__all__ = ["QuantizedKVCache", "PagedKVCache", "TQError", "binding"]

_DTYPES = None


def _dtype_code(t):
    global _DTYPES
    import torch
    if _DTYPES is None:
        _DTYPES = {torch.float32: _b.TQ_F32, torch.bfloat16: _b.TQ_BF16, torch.float16: _b.TQ_F16}
    return _DTYPES[t.dtype]


def _stream_handle(stream=None):
    import torch
    s = stream if stream is not None else torch.cuda.current_stream()
    return s.cuda_stream


class _Codec:
    """A library context for one configuration with its tables uploaded to ``device``."""

    def _setup(self, head_dim, num_q_heads, num_kv_heads, batch, capacity, scheme, n, seed, k_codec,
               v_codec, headq_rank, headq_bits, device):
        import torch
        cfg = _b.tq_config()
        cfg.head_dim, cfg.num_q_heads, cfg.num_kv_heads = head_dim, num_q_heads, num_kv_heads
        cfg.batch, cfg.capacity = batch, capacity
        cfg.qjl_m, cfg.headq_rank, cfg.headq_bits, cfg.seed = 0, headq_rank, headq_bits, seed
        if scheme is not None:
            check(_b.tq_config_from_scheme(_b.SCHEMES[scheme.lower()], n, cfg))
        if k_codec is not None:
            cfg.k = _b.tq_codec(*k_codec)
        if v_codec is not None:
            cfg.v = _b.tq_codec(*v_codec)
        self.cfg = cfg
        ctx = _b.c_void_p()
        check(_b.tq_context_create(cfg, ctx))
        self._ctx = ctx
        self.device = torch.device(device)
        self.head_dim, self.num_q_heads, self.num_kv_heads = head_dim, num_q_heads, num_kv_heads
        self.batch, self.capacity = batch, capacity
        self.tables = torch.empty(int(_b.tq_tables_bytes(ctx)), dtype=torch.uint8, device=self.device)
        check(_b.tq_tables_upload(ctx, self.tables.data_ptr(), _stream_handle()))
        self._ws = None

    def __del__(self):
        ctx = getattr(self, "_ctx", None)
        if ctx is not None and ctx.value:
            _b.tq_context_destroy(ctx)
            self._ctx = None

    def workspace(self, max_seq):
        import torch
        need = int(_b.tq_decode_workspace_bytes(self._ctx, int(max_seq)))
        if self._ws is None or self._ws.numel() < need:
            self._ws = torch.empty(need, dtype=torch.uint8, device=self.device)
        return self._ws

    def set_spectral_basis(self, side, E, s, stream=None):
        """SQU-KV: side 0 (K) or 1 (V); E float32 CUDA [num_kv_heads][d][d], column j = eigenvector j
        by descending eigenvalue; s float32 CUDA [num_kv_heads][d], s_j = sqrt(d lambda_j)."""
        E, s = E.contiguous(), s.contiguous()
        check(_b.tq_spectral_set_basis(self._ctx, int(side), E.data_ptr(), s.data_ptr(), _stream_handle(stream)))
        self._sq = getattr(self, "_sq", {})
        self._sq[side] = (E, s)  # keep alive until the kernel has run

    def device_error(self, stream=None):
        """(status, code) of the decode workspace's error word (waits for the stream)."""
        code = _b.c_int32(0)
        st = _b.tq_get_device_error(self.workspace(0).data_ptr(), code, _stream_handle(stream))
        return st, code.value


class QuantizedKVCache(_Codec):
    """One packed KV cache of shape [batch][num_kv_heads][capacity] tokens on a CUDA device.

    ``scheme``/``n`` pick the codecs as ``tq_config_from_scheme`` does; ``k_codec``/``v_codec``
    (tuples bits, rotate, qjl) override them.  ``headq_rank`` = 16 turns the HeadQ side code on.
    """

    def __init__(self, head_dim, num_q_heads, num_kv_heads, batch, capacity, scheme="tq", n=4,
                 seed=0, k_codec=None, v_codec=None, headq_rank=0, headq_bits=4, device="cuda"):
        import torch
        self._setup(head_dim, num_q_heads, num_kv_heads, batch, capacity, scheme, n, seed, k_codec,
                    v_codec, headq_rank, headq_bits, device)
        ctx = self._ctx
        lay = _b.tq_cache_layout()
        check(_b.tq_get_cache_layout(ctx, lay))
        self.layout = lay
        # field offsets inside a side's 16-token block, and bytes per token
        self.fields = {n: (getattr(lay, n).offset, getattr(lay, n).record_bytes) for n in _b.REGION_NAMES}
        self.cache = torch.zeros(int(lay.total_bytes), dtype=torch.uint8, device=self.device)

    # ---- host tables (no GPU work)
    def host_tables(self):
        n = int(_b.tq_tables_bytes(self._ctx))
        buf = np.zeros(n, dtype=np.uint8)
        check(_b.tq_tables_host(self._ctx, buf.ctypes.data, n))
        return buf

    # ---- device calls
    def set_headq_basis(self, U, stream=None):
        """U: float32 CUDA tensor [num_kv_heads][head_dim][rank]."""
        U = U.contiguous()
        check(_b.tq_headq_set_basis(self._ctx, U.data_ptr(), _stream_handle(stream)))
        self._U = U  # keep alive until the kernel has run

    def append(self, k, v, start, stream=None):
        """k, v: CUDA tensors [batch][num_kv_heads][n_new][head_dim] (fp32/bf16/fp16)."""
        k, v = k.contiguous(), v.contiguous()
        if k.shape != v.shape or k.dtype != v.dtype:
            raise ValueError("k and v must have the same shape and dtype")
        check(_b.tq_quantize_append(self._ctx, self.cache.data_ptr(), k.data_ptr(), v.data_ptr(),
                                    _dtype_code(k), int(k.shape[2]), _b.int_array(start),
                                    _stream_handle(stream)))

    def decode(self, q, seq_len, out=None, stream=None):
        """q: float32 CUDA tensor [batch][num_q_heads][head_dim] -> attention output (same shape)."""
        import torch
        q = q.contiguous()
        if out is None:
            out = torch.empty_like(q)
        ws = self.workspace(max(int(x) for x in seq_len))
        check(_b.tq_decode_attention(self._ctx, self.cache.data_ptr(), q.data_ptr(), _b.int_array(seq_len),
                                     out.data_ptr(), ws.data_ptr(), ws.numel(), _stream_handle(stream)))
        return out

    def append_decode(self, k, v, q, seq_len, out=None, stream=None):
        """One decode step: append k, v ([batch][num_kv_heads][n_new][head_dim]) as the last n_new
        tokens of each sequence (positions seq_len[b] - n_new ..), then decode q over the first
        seq_len[b] tokens.  The same cache and output as append then decode; the library overlaps
        the query preparation with the append."""
        import torch
        k, v, q = k.contiguous(), v.contiguous(), q.contiguous()
        if k.shape != v.shape or k.dtype != v.dtype:
            raise ValueError("k and v must have the same shape and dtype")
        if out is None:
            out = torch.empty_like(q)
        ws = self.workspace(max(int(x) for x in seq_len))
        check(_b.tq_append_decode_attention(self._ctx, self.cache.data_ptr(), k.data_ptr(), v.data_ptr(),
                                            _dtype_code(k), int(k.shape[2]), q.data_ptr(),
                                            _b.int_array(seq_len), out.data_ptr(), ws.data_ptr(), ws.numel(),
                                            _stream_handle(stream)))
        return out

    def decode_multi(self, q, seq_len, out=None, stream=None):
        """q: float32 CUDA tensor [batch][nq][num_q_heads][head_dim]: the last nq positions of each
        sequence, query i attending to the first seq_len[b] - nq + 1 + i tokens."""
        import torch
        q = q.contiguous()
        if out is None:
            out = torch.empty_like(q)
        ws = self.workspace(max(int(x) for x in seq_len))
        check(_b.tq_decode_attention_multi(self._ctx, self.cache.data_ptr(), q.data_ptr(), int(q.shape[1]),
                                           _b.int_array(seq_len), out.data_ptr(), ws.data_ptr(), ws.numel(),
                                           _stream_handle(stream)))
        return out

    def prefill(self, q, seq_len, out=None, ws=None, stream=None):
        """Chunked-prefill attention.  q: float32 CUDA tensor [batch][nq][num_q_heads][head_dim], the
        chunk's last nq positions (already appended); query i attends to the first
        seq_len[b] - nq + 1 + i tokens.  ``ws``: optional uint8 CUDA workspace of at least
        prefill_workspace_bytes(nq) bytes (allocated here otherwise)."""
        import torch
        q = q.contiguous()
        nq = int(q.shape[1])
        if out is None:
            out = torch.empty_like(q)
        need = self.prefill_workspace_bytes(nq)
        if ws is None:
            ws = torch.empty(need, dtype=torch.uint8, device=self.device)
        check(_b.tq_prefill_attention(self._ctx, self.cache.data_ptr(), q.data_ptr(), nq, _b.int_array(seq_len),
                                      out.data_ptr(), ws.data_ptr(), ws.numel(), _stream_handle(stream)))
        return out

    def prefill_workspace_bytes(self, nq):
        return int(_b.tq_prefill_workspace_bytes(self._ctx, int(nq)))

    def logits(self, q, seq_len, stride=None, stream=None):
        """Corrected scores [batch][num_q_heads][stride] (entries past seq_len[b] are untouched: 0)."""
        import torch
        q = q.contiguous()
        stride = stride or max(1, max(int(x) for x in seq_len))
        out = torch.zeros(q.shape[0], q.shape[1], stride, dtype=torch.float32, device=self.device)
        check(_b.tq_headq_correct(self._ctx, self.cache.data_ptr(), q.data_ptr(), _b.int_array(seq_len),
                                  out.data_ptr(), stride, _stream_handle(stream)))
        return out

    def dequantize(self, b, kvh, t0, t1, stream=None):
        import torch
        k = torch.empty(t1 - t0, self.head_dim, dtype=torch.float32, device=self.device)
        v = torch.empty_like(k)
        check(_b.tq_dequantize(self._ctx, self.cache.data_ptr(), b, kvh, t0, t1, k.data_ptr(), v.data_ptr(),
                               _stream_handle(stream)))
        return k, v


class PagedKVCache(_Codec):
    """A pool of ``num_pages`` pages on a CUDA device, each holding one 16-token block per KV head
    of both sides (``tq_get_paged_cache_layout``).  ``block_table`` is an int32 CUDA tensor
    [batch][max_blocks_per_seq] of page indices owned by the caller; start positions and sequence
    lengths are int32 CUDA tensors [batch].  All three are read on the device, so they may change
    between replays of a captured CUDA graph.  Head dim 128.
    """

    def __init__(self, head_dim, num_q_heads, num_kv_heads, batch, num_pages, max_blocks_per_seq,
                 scheme="tq", n=4, seed=0, k_codec=None, v_codec=None, device="cuda"):
        import torch
        # the context's contiguous capacity is not used by the pool: the smallest valid one
        self._setup(head_dim, num_q_heads, num_kv_heads, batch, 64, scheme, n, seed, k_codec, v_codec,
                    0, 4, device)
        self.num_pages, self.max_blocks_per_seq = int(num_pages), int(max_blocks_per_seq)
        lay = _b.tq_cache_layout()
        check(_b.tq_get_paged_cache_layout(self._ctx, self.num_pages, lay))
        self.layout = lay
        self.fields = {n: (getattr(lay, n).offset, getattr(lay, n).record_bytes) for n in _b.REGION_NAMES}
        self.pool = torch.zeros(int(lay.total_bytes), dtype=torch.uint8, device=self.device)

    def _pages(self, block_table):
        if block_table.dtype != _torch().int32 or not block_table.is_contiguous():
            raise ValueError("block_table must be a contiguous int32 tensor")
        if tuple(block_table.shape) != (self.batch, self.max_blocks_per_seq):
            raise ValueError("block_table must be [batch][max_blocks_per_seq]")
        return _b.tq_page_table(block_table.data_ptr(), self.max_blocks_per_seq, self.num_pages)

    def append(self, k, v, start, block_table, error=None, stream=None):
        """k, v: CUDA tensors [batch][num_kv_heads][n_new][head_dim]; start: int32 CUDA [batch];
        error: optional int32 CUDA tensor of one element that receives a TQ_DEVERR_* code."""
        k, v = k.contiguous(), v.contiguous()
        if k.shape != v.shape or k.dtype != v.dtype:
            raise ValueError("k and v must have the same shape and dtype")
        pt = self._pages(block_table)
        check(_b.tq_quantize_append_paged(self._ctx, self.pool.data_ptr(), pt, k.data_ptr(), v.data_ptr(),
                                          _dtype_code(k), int(k.shape[2]), start.data_ptr(),
                                          error.data_ptr() if error is not None else None,
                                          _stream_handle(stream)))

    def decode(self, q, seq_len, block_table, out=None, stream=None):
        """q: float32 CUDA tensor [batch][nq][num_q_heads][head_dim] (or [batch][num_q_heads][head_dim]
        for one query); seq_len: int32 CUDA [batch].  Query i of nq attends to the first
        seq_len[b] - nq + 1 + i tokens."""
        import torch
        q = q.contiguous()
        nq = int(q.shape[1]) if q.dim() == 4 else 1
        if out is None:
            out = torch.empty_like(q)
        pt = self._pages(block_table)
        ws = self.workspace(16 * self.max_blocks_per_seq)
        check(_b.tq_decode_attention_paged(self._ctx, self.pool.data_ptr(), pt, q.data_ptr(), nq,
                                           seq_len.data_ptr(), out.data_ptr(), ws.data_ptr(), ws.numel(),
                                           _stream_handle(stream)))
        return out


def _torch():
    import torch
    return torch
