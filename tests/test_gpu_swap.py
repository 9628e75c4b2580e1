"""GPU parity of swap_blocks (swap-mode preemption: blocks to pinned host
memory and back, "vLLM 核心：PagedAttention 与 Continuous Batching", §5)."""
import numpy as np
import pytest

import oracle
from paged_kv_cache_140_gb300 import workloads as W

from pa_harness import cache_bits, run_step, to_device

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from paged_kv_cache_140_gb300 import _build
    _build.build()
    oracle.build()


def _preempt_and_resume(cache_dtype):
    """Swap two sequences' blocks out to a host pool, scribble over their GPU
    blocks, swap them back into other free GPU blocks, and decode again."""
    import torch
    import paged_kv_cache_140_gb300 as pa
    b = W.make_batch("7b", num_seqs=5, ctx_cap=600, cache_dtype=cache_dtype)
    out0, T, flag = run_step(b)
    assert flag == 0
    victims = [1, 3]
    bs = b.block_size
    blocks = [int(x) for s in victims for x in b.block_tables[s, : -(-int(b.context_lens[s]) // bs)]]
    n = len(blocks)
    host_k = torch.zeros((n,) + tuple(T["k_cache"].shape[1:]), dtype=T["k_cache"].dtype).pin_memory()
    host_v = torch.zeros_like(host_k).pin_memory()
    out_map = torch.tensor([[blk, i] for i, blk in enumerate(blocks)], dtype=torch.int64, device="cuda")
    err = pa.new_err_flag()
    pa.swap_blocks(T["k_cache"], T["v_cache"], host_k, host_v, out_map, err_flag=err)
    torch.cuda.synchronize()
    assert pa.read_err_flag(err) == 0
    gk, gv = cache_bits(T["k_cache"]), cache_bits(T["v_cache"])
    hk, hv, bad = oracle.swap_blocks(gk, gv, np.zeros_like(gk[:n]), np.zeros_like(gv[:n]),
                                     out_map.cpu().numpy())
    assert bad == 0
    assert np.array_equal(cache_bits(host_k), hk) and np.array_equal(cache_bits(host_v), hv)
    # The freed GPU blocks are reused by someone else.
    T["k_cache"][blocks] = 0
    T["v_cache"][blocks] = 0
    # Resume into other physical blocks: ids the pool never handed out, then the
    # victims' own (zeroed) blocks in reverse order.
    used = set(int(x) for x in b.block_tables[b.block_tables >= 0].ravel())
    free = ([i for i in range(b.num_blocks) if i not in used] + blocks[::-1])[:n]
    assert len(set(free)) == n and free != blocks
    in_map = torch.tensor([[i, free[i]] for i in range(n)], dtype=torch.int64, device="cuda")
    pa.swap_blocks(host_k, host_v, T["k_cache"], T["v_cache"], in_map, err_flag=err)
    torch.cuda.synchronize()
    assert pa.read_err_flag(err) == 0
    remap = dict(zip(blocks, free))
    tables = b.block_tables.copy()
    for s in victims:
        nb = -(-int(b.context_lens[s]) // bs)
        tables[s, :nb] = [remap[int(x)] for x in tables[s, :nb]]
    T["block_tables"] = torch.from_numpy(tables).cuda()
    out1 = torch.empty_like(out0)
    pa.decode(out1, T["q"], T["k_cache"], T["v_cache"], T["block_tables"], T["context_lens"], float(b.scale),
              max_context_len=b.max_context_len, err_flag=err, k_scale=b.k_scale, v_scale=b.v_scale)
    torch.cuda.synchronize()
    assert pa.read_err_flag(err) == 0
    assert torch.equal(out0, out1), "decode after swap-out / swap-in differs"


def test_swap_out_and_in_16bit():
    _preempt_and_resume("f16")


def test_swap_out_and_in_fp8():
    _preempt_and_resume("fp8")


def test_swap_between_two_device_caches_and_bad_pairs():
    import torch
    import paged_kv_cache_140_gb300 as pa
    b = W.make_batch("13b", num_seqs=3)
    T = to_device(b)
    dst_k = torch.zeros((7,) + tuple(T["k_cache"].shape[1:]), dtype=T["k_cache"].dtype, device="cuda")
    dst_v = torch.zeros_like(dst_k)
    m = np.array([[0, 6], [5, 0], [9, 3], [b.num_blocks, 1], [2, 7]], dtype=np.int64)  # last two bad
    err = pa.new_err_flag()
    pa.swap_blocks(T["k_cache"], T["v_cache"], dst_k, dst_v, torch.from_numpy(m).cuda(), err_flag=err)
    torch.cuda.synchronize()
    assert pa.read_err_flag(err) & pa.FLAG_BAD_COPY_PAIR
    wk, wv, bad = oracle.swap_blocks(b.k_cache, b.v_cache, np.zeros_like(b.k_cache[:7]),
                                     np.zeros_like(b.v_cache[:7]), m)
    assert bad == 2
    assert np.array_equal(cache_bits(dst_k), wk) and np.array_equal(cache_bits(dst_v), wv)


def test_pageable_host_memory_is_rejected_before_launch():
    import torch
    import paged_kv_cache_140_gb300 as pa
    b = W.make_batch("tiny")
    T = to_device(b)
    host_k = torch.zeros((2,) + tuple(T["k_cache"].shape[1:]), dtype=T["k_cache"].dtype)   # not pinned
    m = torch.tensor([[0, 0]], dtype=torch.int64, device="cuda")
    with pytest.raises(ValueError):
        pa.swap_blocks(T["k_cache"], T["v_cache"], host_k, host_k.clone(), m)
    # Through the C ABI directly, the library itself refuses the pageable pointer.
    import ctypes
    from paged_kv_cache_140_gb300 import _lib as L
    lib = L.load()
    P = ctypes.c_void_p
    st = lib.pa_swap_blocks(P(T["k_cache"].data_ptr()), P(T["v_cache"].data_ptr()), P(host_k.data_ptr()),
                            P(host_k.data_ptr()), P(m.data_ptr()), 1, b.num_blocks, 2, 16, 4, 64, 0, None,
                            P(torch.cuda.current_stream().cuda_stream))
    assert st == L.PA_ERR_INVALID_ARG
