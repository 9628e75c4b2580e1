"""GB300-native (sm_103a) paged decode attention.

The computation lives in the CUDA library ``lib/libpagedattn.so`` behind the
C ABI of ``include/pa.h``.  This module only marshals PyTorch tensors (device
memory and the current CUDA stream) into those calls; there is no CPU or
PyTorch fallback - a missing library raises.

    reshape_and_cache(key, value, k_cache, v_cache, slot_mapping)
    decode(out, query, k_cache, v_cache, block_tables, context_lens, scale, ...)
    prefill(out, query, k_cache, v_cache, block_tables, context_lens, cu_seqlens_q, scale, ...)
    copy_blocks(k_cache, v_cache, block_mapping)

Cache layout: ``[num_blocks, block_size, num_kv_heads, head_dim]`` per layer
for K and for V ("LLM推理优化：vLLM PagedAttention深度解析与工程实践", §4.1).
Caches are float16 / bfloat16, or FP8 e4m3 codes (``torch.float8_e4m3fn`` or
``torch.uint8``) with per-tensor ``k_scale`` / ``v_scale``.
"""
from __future__ import annotations

import ctypes

from . import _lib
from ._lib import (FLAG_BAD_BLOCK_ID, FLAG_BAD_CONTEXT_LEN, FLAG_BAD_COPY_PAIR, FLAG_BAD_SLOT,
                   FLAG_TIMEOUT, PA_BF16, PA_F16, PA_F32, PA_FP8_E4M3, PagedAttentionError)

__all__ = ["reshape_and_cache", "decode", "decode_append", "prefill", "copy_blocks", "copy_blocks_layers", "swap_blocks", "decode_workspace_size",
           "decode_partition_size", "DecodeWorkspace", "new_err_flag", "read_err_flag",
           "PagedAttentionError", "FLAG_BAD_SLOT", "FLAG_BAD_BLOCK_ID", "FLAG_BAD_CONTEXT_LEN",
           "FLAG_BAD_COPY_PAIR", "FLAG_TIMEOUT", "library_path", "StepGraph"]


def library_path() -> str:
    return _lib.lib_path()


def _torch():
    import torch
    return torch


def _dtype_code(t, allow_f32=False) -> int:
    torch = _torch()
    if t.dtype == torch.float16:
        return PA_F16
    if t.dtype == torch.bfloat16:
        return PA_BF16
    if allow_f32 and t.dtype == torch.float32:
        return PA_F32
    raise TypeError(f"unsupported dtype {t.dtype}")


def _cache_code(t) -> int:
    torch = _torch()
    if t.dtype in (torch.uint8, getattr(torch, "float8_e4m3fn", None)):
        return PA_FP8_E4M3
    return _dtype_code(t)


def _need(cond: bool, msg: str) -> None:
    if not cond:
        raise ValueError(msg)


def _cuda_contig(name, t):
    _need(t.is_cuda, f"{name} must be a CUDA tensor")
    _need(t.is_contiguous(), f"{name} must be contiguous")


def _stream(device) -> ctypes.c_void_p:
    torch = _torch()
    return ctypes.c_void_p(torch.cuda.current_stream(device).cuda_stream)


def _ptr(t) -> ctypes.c_void_p:
    return ctypes.c_void_p(t.data_ptr()) if t is not None else ctypes.c_void_p(0)


def new_err_flag(device=None):
    """A zeroed device int32 that kernels OR their PA_FLAG_* bits into."""
    torch = _torch()
    return torch.zeros(1, dtype=torch.int32, device=device or "cuda")


def read_err_flag(err_flag, clear: bool = True) -> int:
    """Synchronise the current stream and return (optionally clearing) the flag bits."""
    lib = _lib.load()
    out = ctypes.c_int(0)
    st = lib.pa_check_err_flag(_ptr(err_flag), int(clear), ctypes.byref(out), _stream(err_flag.device))
    if st not in (_lib.PA_OK, _lib.PA_ERR_DEVICE_BOUNDS):
        _lib.check(st, "pa_check_err_flag")
    return int(out.value)


def reshape_and_cache(key, value, k_cache, v_cache, slot_mapping, err_flag=None,
                      k_scale: float = 1.0, v_scale: float = 1.0) -> None:
    """Write key/value rows [T, Hkv, D] into cache slots (slot < 0: skip);
    an FP8 cache receives e4m3(x / scale)."""
    for n, t in (("key", key), ("value", value), ("k_cache", k_cache), ("v_cache", v_cache),
                 ("slot_mapping", slot_mapping)):
        _cuda_contig(n, t)
    torch = _torch()
    _need(key.dim() == 3 and value.shape == key.shape, "key/value must be [T, Hkv, D]")
    _need(k_cache.dim() == 4 and v_cache.shape == k_cache.shape, "caches must be [NB, bs, Hkv, D]")
    _need(k_cache.shape[2:] == key.shape[1:], "cache and key head shapes differ")
    _need(key.dtype == value.dtype and k_cache.dtype == v_cache.dtype, "dtype mismatch")
    _need(slot_mapping.dtype == torch.int64 and slot_mapping.numel() == key.shape[0],
          "slot_mapping must be int64 [T]")
    nb, bs, hkv, d = k_cache.shape
    st = _lib.load().pa_reshape_and_cache(_ptr(key), _ptr(value), _ptr(k_cache), _ptr(v_cache),
                                          _ptr(slot_mapping), key.shape[0], nb, bs, hkv, d,
                                          _dtype_code(key), _cache_code(k_cache), float(k_scale),
                                          float(v_scale), _ptr(err_flag), _stream(key.device))
    _lib.check(st, "pa_reshape_and_cache")


def copy_blocks(k_cache, v_cache, block_mapping, err_flag=None) -> None:
    """Copy whole blocks for each (src, dst) row of block_mapping [P, 2] int64."""
    for n, t in (("k_cache", k_cache), ("v_cache", v_cache), ("block_mapping", block_mapping)):
        _cuda_contig(n, t)
    torch = _torch()
    _need(block_mapping.dtype == torch.int64 and block_mapping.dim() == 2 and block_mapping.shape[1] == 2,
          "block_mapping must be int64 [P, 2]")
    _need(k_cache.shape == v_cache.shape and k_cache.dtype == v_cache.dtype, "cache mismatch")
    nb, bs, hkv, d = k_cache.shape
    st = _lib.load().pa_copy_blocks(_ptr(k_cache), _ptr(v_cache), _ptr(block_mapping),
                                    block_mapping.shape[0], nb, bs, hkv, d, _cache_code(k_cache),
                                    _ptr(err_flag), _stream(k_cache.device))
    _lib.check(st, "pa_copy_blocks")


def copy_blocks_layers(kv_cache, block_mapping, err_flag=None) -> None:
    """copy_blocks for every layer of a model's cache
    ``kv_cache`` [layers, 2, NB, bs, Hkv, D] (K at [l][0], V at [l][1]), one launch."""
    for n, t in (("kv_cache", kv_cache), ("block_mapping", block_mapping)):
        _cuda_contig(n, t)
    torch = _torch()
    _need(kv_cache.dim() == 6 and kv_cache.shape[1] == 2, "kv_cache must be [layers, 2, NB, bs, Hkv, D]")
    _need(block_mapping.dtype == torch.int64 and block_mapping.dim() == 2 and block_mapping.shape[1] == 2,
          "block_mapping must be int64 [P, 2]")
    layers, _, nb, bs, hkv, d = kv_cache.shape
    st = _lib.load().pa_copy_blocks_layers(_ptr(kv_cache), layers, _ptr(block_mapping), block_mapping.shape[0],
                                           nb, bs, hkv, d, _cache_code(kv_cache), _ptr(err_flag),
                                           _stream(kv_cache.device))
    _lib.check(st, "pa_copy_blocks_layers")


def swap_blocks(src_k, src_v, dst_k, dst_v, block_mapping, err_flag=None) -> None:
    """Copy whole blocks src -> dst between two caches (for swap-mode
    preemption); either cache may be a pinned host tensor (``pin_memory()``),
    the other a CUDA tensor.  ``block_mapping`` [P, 2] int64 on the GPU."""
    torch = _torch()
    for n, t in (("src_k", src_k), ("src_v", src_v), ("dst_k", dst_k), ("dst_v", dst_v)):
        _need(t.is_contiguous(), f"{n} must be contiguous")
        _need(t.is_cuda or t.is_pinned(), f"{n} must be a CUDA tensor or pinned host memory")
    _cuda_contig("block_mapping", block_mapping)
    _need(block_mapping.dtype == torch.int64 and block_mapping.dim() == 2 and block_mapping.shape[1] == 2,
          "block_mapping must be int64 [P, 2]")
    _need(src_k.shape[1:] == dst_k.shape[1:] and src_k.dtype == dst_k.dtype, "cache shapes differ")
    _need(src_v.shape == src_k.shape and dst_v.shape == dst_k.shape, "K and V caches differ")
    nb_src, bs, hkv, d = src_k.shape
    device = block_mapping.device
    st = _lib.load().pa_swap_blocks(_ptr(src_k), _ptr(src_v), _ptr(dst_k), _ptr(dst_v), _ptr(block_mapping),
                                    block_mapping.shape[0], nb_src, dst_k.shape[0], bs, hkv, d,
                                    _cache_code(src_k), _ptr(err_flag), _stream(device))
    _lib.check(st, "pa_swap_blocks")


def decode_workspace_size(num_seqs, num_heads, num_kv_heads, head_dim, block_size,
                          max_context_len, partition_size=0) -> int:
    n = _lib.load().pa_decode_workspace_size(num_seqs, num_heads, num_kv_heads, head_dim, block_size,
                                             max_context_len, partition_size)
    if n == ctypes.c_size_t(-1).value:
        raise ValueError("arguments rejected by pa_decode_workspace_size")
    return int(n)


def decode_partition_size(num_seqs, num_heads, num_kv_heads, head_dim, block_size,
                          max_context_len, partition_size=0) -> int:
    return int(_lib.load().pa_decode_partition_size(num_seqs, num_heads, num_kv_heads, head_dim,
                                                    block_size, max_context_len, partition_size))


class DecodeWorkspace:
    """A device workspace for pa_decode, grown on demand (no initial contents
    are needed).

    One instance must not serve two decode calls that can overlap on the GPU
    (the default per-(device, stream) instances used by :func:`decode` never do).
    """

    def __init__(self, device=None):
        self.device = device
        self.buf = None

    def get(self, nbytes: int, layout=None):
        """A buffer of at least ``nbytes`` bytes (None when nothing is needed)."""
        torch = _torch()
        if nbytes == 0:
            return None
        if self.buf is None or self.buf.numel() < nbytes:
            self.buf = torch.empty(nbytes, dtype=torch.uint8, device=self.device or "cuda")
        return self.buf


_default_ws: dict = {}


def decode(out, query, k_cache, v_cache, block_tables, context_lens, scale: float,
           max_context_len: int | None = None, partition_size: int = 0, workspace=None,
           err_flag=None, k_scale: float = 1.0, v_scale: float = 1.0) -> None:
    """Paged decode attention into ``out`` [B, Hq, D] (f16, bf16 or f32).

    ``max_context_len`` is a host-side bound on ``context_lens`` (defaults to
    the block-table width times the block size)."""
    torch = _torch()
    for n, t in (("out", out), ("query", query), ("k_cache", k_cache), ("v_cache", v_cache),
                 ("block_tables", block_tables), ("context_lens", context_lens)):
        _cuda_contig(n, t)
    _need(query.dim() == 3 and out.shape == query.shape, "query/out must be [B, Hq, D]")
    _need(k_cache.dim() == 4 and v_cache.shape == k_cache.shape, "caches must be [NB, bs, Hkv, D]")
    _need(k_cache.dtype == v_cache.dtype, "K and V caches must share a dtype")
    _need(block_tables.dtype == torch.int32 and block_tables.dim() == 2 and
          block_tables.shape[0] == query.shape[0], "block_tables must be int32 [B, maxNB]")
    _need(context_lens.dtype == torch.int32 and context_lens.numel() == query.shape[0],
          "context_lens must be int32 [B]")
    B, Hq, D = query.shape
    nb, bs, hkv, d2 = k_cache.shape
    _need(d2 == D, "head_dim mismatch")
    maxnb = block_tables.shape[1]
    if max_context_len is None:
        max_context_len = maxnb * bs
    ws_bytes = decode_workspace_size(B, Hq, hkv, D, bs, max_context_len, partition_size)
    if workspace is None:
        key = (query.device.index, torch.cuda.current_stream(query.device).cuda_stream)
        workspace = _default_ws.setdefault(key, DecodeWorkspace(query.device))
    layout = (B, Hq, hkv, D, bs, int(max_context_len), int(partition_size))
    buf = workspace.get(ws_bytes, layout) if isinstance(workspace, DecodeWorkspace) else workspace
    nbytes = 0 if buf is None else buf.numel() * buf.element_size()
    st = _lib.load().pa_decode(_ptr(out), _dtype_code(out, allow_f32=True), _ptr(query), _dtype_code(query),
                               _ptr(k_cache), _ptr(v_cache), _cache_code(k_cache), float(k_scale),
                               float(v_scale), _ptr(block_tables),
                               maxnb, _ptr(context_lens), int(max_context_len), B, Hq, hkv, D, bs, nb,
                               float(scale), int(partition_size), _ptr(buf), nbytes, _ptr(err_flag),
                               _stream(query.device))
    _lib.check(st, "pa_decode")


def decode_append(out, query, key, value, k_cache, v_cache, block_tables, context_lens, scale: float,
                  max_context_len: int | None = None, partition_size: int = 0, workspace=None,
                  err_flag=None, k_scale: float = 1.0, v_scale: float = 1.0) -> None:
    """reshape_and_cache of each sequence's new token (position context_lens[s] - 1,
    rows ``key``/``value`` [B, Hkv, D]) fused with :func:`decode`, one launch."""
    torch = _torch()
    for n, t in (("out", out), ("query", query), ("key", key), ("value", value), ("k_cache", k_cache),
                 ("v_cache", v_cache), ("block_tables", block_tables), ("context_lens", context_lens)):
        _cuda_contig(n, t)
    _need(query.dim() == 3 and out.shape == query.shape, "query/out must be [B, Hq, D]")
    _need(k_cache.dim() == 4 and v_cache.shape == k_cache.shape and k_cache.dtype == v_cache.dtype,
          "caches must be [NB, bs, Hkv, D] of one dtype")
    B, Hq, D = query.shape
    nb, bs, hkv, d2 = k_cache.shape
    _need(d2 == D and key.shape == (B, hkv, D) and value.shape == key.shape, "key/value must be [B, Hkv, D]")
    _need(key.dtype == value.dtype == query.dtype, "key/value must have the query's dtype")
    _need(block_tables.dtype == torch.int32 and block_tables.dim() == 2 and block_tables.shape[0] == B,
          "block_tables must be int32 [B, maxNB]")
    _need(context_lens.dtype == torch.int32 and context_lens.numel() == B, "context_lens must be int32 [B]")
    maxnb = block_tables.shape[1]
    if max_context_len is None:
        max_context_len = maxnb * bs
    ws_bytes = decode_workspace_size(B, Hq, hkv, D, bs, max_context_len, partition_size)
    if workspace is None:
        wkey = (query.device.index, torch.cuda.current_stream(query.device).cuda_stream)
        workspace = _default_ws.setdefault(wkey, DecodeWorkspace(query.device))
    buf = workspace.get(ws_bytes) if isinstance(workspace, DecodeWorkspace) else workspace
    nbytes = 0 if buf is None else buf.numel() * buf.element_size()
    st = _lib.load().pa_decode_append(_ptr(out), _dtype_code(out, allow_f32=True), _ptr(query),
                                      _dtype_code(query), _ptr(key), _ptr(value), _ptr(k_cache), _ptr(v_cache),
                                      _cache_code(k_cache), float(k_scale), float(v_scale), _ptr(block_tables),
                                      maxnb, _ptr(context_lens), int(max_context_len), B, Hq, hkv, D, bs, nb,
                                      float(scale), int(partition_size), _ptr(buf), nbytes, _ptr(err_flag),
                                      _stream(query.device))
    _lib.check(st, "pa_decode_append")


def prefill(out, query, k_cache, v_cache, block_tables, context_lens, cu_seqlens_q, scale: float,
            max_q_len: int, err_flag=None) -> None:
    """Causal attention of each sequence's newest tokens over its paged context
    into ``out`` [T, Hq, D] (f16, bf16 or f32).

    Sequence s owns query rows ``cu_seqlens_q[s] .. cu_seqlens_q[s+1]-1`` (int32
    [B+1] on the GPU); ``context_lens[s]`` counts all its tokens, new ones
    included (their K/V rows already written with :func:`reshape_and_cache`).
    ``max_q_len`` is a host-side bound on every sequence's new-token count."""
    torch = _torch()
    for n, t in (("out", out), ("query", query), ("k_cache", k_cache), ("v_cache", v_cache),
                 ("block_tables", block_tables), ("context_lens", context_lens),
                 ("cu_seqlens_q", cu_seqlens_q)):
        _cuda_contig(n, t)
    _need(query.dim() == 3 and out.shape == query.shape, "query/out must be [T, Hq, D]")
    _need(k_cache.dim() == 4 and v_cache.shape == k_cache.shape and k_cache.dtype == v_cache.dtype,
          "caches must be [NB, bs, Hkv, D] of one dtype")
    _need(k_cache.dtype == query.dtype, "caches must have the query's dtype")
    B = context_lens.numel()
    _need(context_lens.dtype == torch.int32, "context_lens must be int32 [B]")
    _need(cu_seqlens_q.dtype == torch.int32 and cu_seqlens_q.numel() == B + 1, "cu_seqlens_q must be int32 [B+1]")
    _need(block_tables.dtype == torch.int32 and block_tables.dim() == 2 and block_tables.shape[0] == B,
          "block_tables must be int32 [B, maxNB]")
    T, Hq, D = query.shape
    nb, bs, hkv, d2 = k_cache.shape
    _need(d2 == D, "head_dim mismatch")
    st = _lib.load().pa_prefill(_ptr(out), _dtype_code(out, allow_f32=True), _ptr(query), _ptr(k_cache),
                                _ptr(v_cache), _dtype_code(query), _ptr(block_tables), block_tables.shape[1],
                                _ptr(context_lens), _ptr(cu_seqlens_q), B, T, int(max_q_len), Hq, hkv, D, bs,
                                nb, float(scale), _ptr(err_flag), _stream(query.device))
    _lib.check(st, "pa_prefill")


class StepGraph:
    """A step of this library's calls captured once as a CUDA graph and then
    replayed with one launch, as a serving loop does for its decode step.

    ``fn()`` enqueues the step (e.g. :func:`reshape_and_cache` then
    :func:`decode`) on the current stream, on device buffers that stay
    allocated at the same addresses for the graph's lifetime; refill those
    buffers in place between replays.  Everything ``fn`` needs is allocated
    before capture: it is run ``warmup`` times first (so default workspaces
    exist), and workspaces passed to it must already be large enough.  The
    argument checks of each call run at capture; a replay launches the
    captured kernels (with their programmatic dependent launch edges) as they
    were.
    """

    def __init__(self, fn, warmup: int = 1):
        torch = _torch()
        self._fn = fn
        side = torch.cuda.Stream()
        side.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(side):
            for _ in range(max(1, warmup)):
                fn()
        torch.cuda.current_stream().wait_stream(side)
        torch.cuda.synchronize()
        self.graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(self.graph):
            fn()
        torch.cuda.synchronize()

    def replay(self) -> None:
        """Launch the captured step on the current stream."""
        self.graph.replay()
