"""CPU oracle for paged decode attention -- TEST INFRASTRUCTURE ONLY.

Only the tests, the package's ``smoke()`` check and the benchmark's CPU
baseline may import this package.  The product path (the CUDA library and its
Python binding) never imports, links or runs anything here, and nothing here
imports the product.

Contents:
  * ``pa_oracle.c`` -- fp64 C implementation of reshape_and_cache,
    copy_blocks, paged attention and the partition-then-merge variant, plus
    the FP8 (e4m3) cache codec, reshape and attention, loaded
    through ctypes (built with gcc on first use, or by ``build()``).
  * ``brute.py`` -- an independent NumPy brute force for tiny inputs.
  * ``accounting.py`` -- the pages' block-count and KV-size formulas.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "pa_oracle.c")
_LIB = os.path.join(_HERE, "_build", "liboracle.so")
_lib = None

DTYPE_CODE = {"f16": 0, "bf16": 1}


def build(force: bool = False) -> str:
    """Compile the C oracle with gcc (-O2 -fopenmp, no fast-math)."""
    os.makedirs(os.path.dirname(_LIB), exist_ok=True)
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".{os.getpid()}.tmp"
        subprocess.check_call(["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-std=c11",
                               _SRC, "-o", tmp, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(build())
        P = ctypes.c_void_p
        i32, i64, dbl = ctypes.c_int, ctypes.c_int64, ctypes.c_double
        lib.oracle_half_to_double.argtypes = [ctypes.c_uint16, i32]
        lib.oracle_half_to_double.restype = dbl
        lib.oracle_reshape_and_cache.argtypes = [P, P, P, P, P, i64, i64, i32, i32, i32]
        lib.oracle_reshape_and_cache.restype = i64
        lib.oracle_copy_blocks.argtypes = [P, P, P, i64, i64, i32, i32, i32]
        lib.oracle_copy_blocks.restype = i64
        lib.oracle_paged_attention.argtypes = [P, P, P, P, i32, P, i32, P, i32, i32, i32, i32, i32, dbl]
        lib.oracle_paged_attention.restype = None
        lib.oracle_paged_attention_partitioned.argtypes = [P, P, P, P, P, P, P, i32, P, i32, P,
                                                           i32, i32, i32, i32, i32, dbl, i32, i32]
        lib.oracle_paged_attention_partitioned.restype = None
        lib.oracle_e4m3_encode_array.argtypes = [P, P, i64]
        lib.oracle_e4m3_encode_array.restype = None
        lib.oracle_e4m3_decode_array.argtypes = [P, P, i64]
        lib.oracle_e4m3_decode_array.restype = None
        f32 = ctypes.c_float
        lib.oracle_reshape_and_cache_fp8.argtypes = [P, P, i32, P, P, P, i64, i64, i32, i32, i32, f32, f32]
        lib.oracle_reshape_and_cache_fp8.restype = i64
        lib.oracle_paged_attention_fp8.argtypes = [P, P, i32, P, P, dbl, dbl, P, i32, P, i32, i32, i32,
                                                   i32, i32, dbl]
        lib.oracle_paged_attention_fp8.restype = None
        lib.oracle_swap_blocks.argtypes = [P, P, P, P, P, i64, i64, i64, i64]
        lib.oracle_swap_blocks.restype = i64
        _lib = lib
    return _lib


def _ptr(a: np.ndarray):
    return ctypes.c_void_p(a.ctypes.data)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


def half_to_double(bits, dtype: str) -> np.ndarray:
    """Exact value of each 16-bit pattern (elementwise, slow, for pinning)."""
    lib = _load()
    flat = np.asarray(bits, dtype=np.uint16).reshape(-1)
    out = np.array([lib.oracle_half_to_double(int(b), DTYPE_CODE[dtype]) for b in flat])
    return out.reshape(np.shape(bits))


def reshape_and_cache(key, value, k_cache, v_cache, slot_mapping):
    """Scatter the step's K/V rows into (copies of) the caches.

    Returns (k_cache_after, v_cache_after, number_of_out_of_range_slots)."""
    lib = _load()
    kc = np.array(k_cache, dtype=np.uint16, copy=True, order="C")
    vc = np.array(v_cache, dtype=np.uint16, copy=True, order="C")
    key = _c(key, np.uint16)
    value = _c(value, np.uint16)
    sm = _c(slot_mapping, np.int64)
    nb, bs, hkv, d = kc.shape
    bad = lib.oracle_reshape_and_cache(_ptr(key), _ptr(value), _ptr(kc), _ptr(vc), _ptr(sm),
                                       len(sm), nb, bs, hkv, d)
    return kc, vc, int(bad)


def copy_blocks(k_cache, v_cache, block_mapping):
    """Copy whole blocks pair by pair (copy-on-write) on copies of the caches."""
    lib = _load()
    kc = np.array(k_cache, dtype=np.uint16, copy=True, order="C")
    vc = np.array(v_cache, dtype=np.uint16, copy=True, order="C")
    bm = _c(np.asarray(block_mapping).reshape(-1, 2), np.int64)
    nb, bs, hkv, d = kc.shape
    bad = lib.oracle_copy_blocks(_ptr(kc), _ptr(vc), _ptr(bm), len(bm), nb, bs, hkv, d)
    return kc, vc, int(bad)


def copy_blocks_layers(kv_cache, block_mapping):
    """copy_blocks applied to every layer of a per-model cache
    [layers, 2, NB, bs, Hkv, D] (layer l's K is [l][0], its V [l][1];
    nano-vllm walkthrough §2.2), on a copy.  Elements of any size are moved
    as 16-bit words."""
    kv = np.array(kv_cache, copy=True, order="C")
    L = kv.shape[0]
    words = kv.view(np.uint16).reshape(L, 2, kv.shape[2], kv.shape[3], kv.shape[4], -1)
    bad = 0
    for layer in range(L):
        k, v, b = copy_blocks(words[layer, 0], words[layer, 1], block_mapping)
        words[layer, 0], words[layer, 1] = k, v
        bad += b
    return kv, bad


def paged_attention(q, k_cache, v_cache, dtype: str, block_tables, context_lens, scale,
                    num_kv_heads: int | None = None) -> np.ndarray:
    """softmax(q K^T * scale) V over each sequence's paged context, in fp64.

    q: uint16 [B, Hq, D]; caches: uint16 [NB, bs, Hkv, D]; block_tables: int32
    [B, maxNB]; context_lens: int32 [B].  Returns float64 [B, Hq, D]."""
    lib = _load()
    q = _c(q, np.uint16)
    kc = _c(k_cache, np.uint16)
    vc = _c(v_cache, np.uint16)
    bt = _c(block_tables, np.int32)
    cl = _c(context_lens, np.int32)
    B, Hq, D = q.shape
    nb, bs, hkv, d2 = kc.shape
    assert d2 == D and (num_kv_heads is None or num_kv_heads == hkv)
    out = np.empty((B, Hq, D), dtype=np.float64)
    lib.oracle_paged_attention(_ptr(out), _ptr(q), _ptr(kc), _ptr(vc), DTYPE_CODE[dtype],
                               _ptr(bt), bt.shape[1], _ptr(cl), B, Hq, hkv, D, bs, float(scale))
    return out


def paged_attention_partitioned(q, k_cache, v_cache, dtype: str, block_tables, context_lens,
                                scale, partition_size: int):
    """Partition-then-merge attention.  Returns (out, part_max, part_sum, part_acc)."""
    lib = _load()
    q = _c(q, np.uint16)
    kc = _c(k_cache, np.uint16)
    vc = _c(v_cache, np.uint16)
    bt = _c(block_tables, np.int32)
    cl = _c(context_lens, np.int32)
    B, Hq, D = q.shape
    nb, bs, hkv, _ = kc.shape
    maxp = max(1, -(-int(cl.max(initial=0)) // int(partition_size)))
    out = np.empty((B, Hq, D), dtype=np.float64)
    pm = np.empty((B, Hq, maxp), dtype=np.float64)
    ps = np.empty((B, Hq, maxp), dtype=np.float64)
    pa = np.empty((B, Hq, maxp, D), dtype=np.float64)
    lib.oracle_paged_attention_partitioned(_ptr(out), _ptr(pm), _ptr(ps), _ptr(pa), _ptr(q), _ptr(kc),
                                           _ptr(vc), DTYPE_CODE[dtype], _ptr(bt), bt.shape[1], _ptr(cl),
                                           B, Hq, hkv, D, bs, float(scale), int(partition_size), maxp)
    return out, pm, ps, pa


def decode_step(batch):
    """The whole step on the CPU: copy_blocks, reshape_and_cache, attention.

    ``batch`` is a workloads.Batch (16-bit or e4m3 cache).  Returns
    (out fp64 [B,Hq,D], k_cache_after, v_cache_after)."""
    kc, vc = batch.k_cache, batch.v_cache
    fp8 = getattr(batch, "cache_dtype", batch.dtype) == "fp8"
    if len(batch.block_mapping):
        kc, vc, _ = (copy_blocks_bytes if fp8 else copy_blocks)(kc, vc, batch.block_mapping)
    if fp8:
        kc, vc, _ = reshape_and_cache_fp8(batch.key, batch.value, batch.dtype, kc, vc, batch.slot_mapping,
                                          batch.k_scale, batch.v_scale)
        out = paged_attention_fp8(batch.q, batch.dtype, kc, vc, batch.k_scale, batch.v_scale,
                                  batch.block_tables, batch.context_lens, batch.scale)
        return out, kc, vc
    kc, vc, _ = reshape_and_cache(batch.key, batch.value, kc, vc, batch.slot_mapping)
    out = paged_attention(batch.q, kc, vc, batch.dtype, batch.block_tables, batch.context_lens,
                          batch.scale)
    return out, kc, vc


# ------------------------------------------------------------ FP8 (e4m3) cache

def e4m3_encode(x) -> np.ndarray:
    """Nearest e4m3 codes (ties to even, finite values saturate at +-448)."""
    lib = _load()
    a = _c(x, np.float32)
    out = np.empty(a.shape, dtype=np.uint8)
    lib.oracle_e4m3_encode_array(_ptr(a), _ptr(out), a.size)
    return out


def e4m3_decode(codes) -> np.ndarray:
    lib = _load()
    c = _c(codes, np.uint8)
    out = np.empty(c.shape, dtype=np.float64)
    lib.oracle_e4m3_decode_array(_ptr(c), _ptr(out), c.size)
    return out


def reshape_and_cache_fp8(key, value, dtype: str, k_cache, v_cache, slot_mapping, k_scale, v_scale):
    """Quantise the step's rows (x / scale in fp32, e4m3) into copies of the caches."""
    lib = _load()
    kc = np.array(k_cache, dtype=np.uint8, copy=True, order="C")
    vc = np.array(v_cache, dtype=np.uint8, copy=True, order="C")
    key = _c(key, np.uint16)
    value = _c(value, np.uint16)
    sm = _c(slot_mapping, np.int64)
    nb, bs, hkv, d = kc.shape
    bad = lib.oracle_reshape_and_cache_fp8(_ptr(key), _ptr(value), DTYPE_CODE[dtype], _ptr(kc), _ptr(vc),
                                           _ptr(sm), len(sm), nb, bs, hkv, d, float(k_scale), float(v_scale))
    return kc, vc, int(bad)


def paged_attention_fp8(q, q_dtype: str, k_cache, v_cache, k_scale, v_scale, block_tables,
                        context_lens, scale) -> np.ndarray:
    """Paged attention over e4m3 caches (K = code value * k_scale, V alike), fp64."""
    lib = _load()
    q = _c(q, np.uint16)
    kc = _c(k_cache, np.uint8)
    vc = _c(v_cache, np.uint8)
    bt = _c(block_tables, np.int32)
    cl = _c(context_lens, np.int32)
    B, Hq, D = q.shape
    nb, bs, hkv, _ = kc.shape
    out = np.empty((B, Hq, D), dtype=np.float64)
    lib.oracle_paged_attention_fp8(_ptr(out), _ptr(q), DTYPE_CODE[q_dtype], _ptr(kc), _ptr(vc),
                                   float(k_scale), float(v_scale), _ptr(bt), bt.shape[1], _ptr(cl), B, Hq,
                                   hkv, D, bs, float(scale))
    return out


def copy_blocks_bytes(k_cache, v_cache, block_mapping):
    """copy_blocks for caches of any element size (viewed as 16-bit words)."""
    kc = np.ascontiguousarray(k_cache)
    shape = kc.shape
    k16 = kc.view(np.uint16).reshape(shape[0], shape[1], shape[2], -1)
    v16 = np.ascontiguousarray(v_cache).view(np.uint16).reshape(k16.shape)
    a, b, bad = copy_blocks(k16, v16, block_mapping)
    return a.view(kc.dtype).reshape(shape), b.view(kc.dtype).reshape(shape), bad


def swap_blocks(src_k, src_v, dst_k, dst_v, block_mapping):
    """Copy whole blocks src -> dst between two caches (copies of the destination
    are returned).  Returns (dst_k_after, dst_v_after, number_of_skipped_pairs)."""
    lib = _load()
    sk, sv = np.ascontiguousarray(src_k), np.ascontiguousarray(src_v)
    dk, dv = np.array(dst_k, copy=True, order="C"), np.array(dst_v, copy=True, order="C")
    assert sk.dtype == dk.dtype and sk.shape[1:] == dk.shape[1:]
    bm = _c(np.asarray(block_mapping).reshape(-1, 2), np.int64)
    block_bytes = int(np.prod(sk.shape[1:])) * sk.itemsize
    bad = lib.oracle_swap_blocks(_ptr(sk), _ptr(sv), _ptr(dk), _ptr(dv), _ptr(bm), len(bm), sk.shape[0],
                                 dk.shape[0], block_bytes)
    return dk, dv, int(bad)


# ------------------------------------------------------ prefill over paged KV

def prefill_attention(q, k_cache, v_cache, dtype: str, block_tables, context_lens, cu_seqlens_q, scale):
    """Causal attention of each sequence's new tokens over its paged context.

    Sequence s owns query rows cu_seqlens_q[s] .. cu_seqlens_q[s+1]-1 (its last
    q_len_s tokens); query token i sits at position ctx_s - q_len_s + i and
    attends positions 0 .. that position.  By that definition each query token
    is a decode query over a context of (position + 1) tokens, which is how it
    is evaluated here.  q: uint16 [Tq, Hq, D].  Returns float64 [Tq, Hq, D]."""
    bt = np.asarray(block_tables)
    ctx = np.asarray(context_lens, dtype=np.int64)
    cu = np.asarray(cu_seqlens_q, dtype=np.int64)
    rows, lens = [], []
    for s in range(len(ctx)):
        ql = int(cu[s + 1] - cu[s])
        for i in range(ql):
            rows.append(s)
            lens.append(int(ctx[s]) - ql + i + 1)
    if not rows:
        return np.zeros((0,) + tuple(np.shape(q)[1:]))
    return paged_attention(q, k_cache, v_cache, dtype, bt[rows], np.asarray(lens, dtype=np.int32), scale)


def prefill_step(batch):
    """The whole prefill step on the CPU: copy_blocks, reshape_and_cache of the
    new tokens, causal attention of their queries.  ``batch`` is a
    workloads.PrefillBatch.  Returns (out fp64 [T,Hq,D], k_cache, v_cache)."""
    kc, vc = batch.k_cache, batch.v_cache
    if len(batch.block_mapping):
        kc, vc, _ = copy_blocks(kc, vc, batch.block_mapping)
    kc, vc, _ = reshape_and_cache(batch.key, batch.value, kc, vc, batch.slot_mapping)
    out = prefill_attention(batch.q, kc, vc, batch.dtype, batch.block_tables, batch.context_lens,
                            batch.cu_seqlens_q, batch.scale)
    return out, kc, vc
