"""pa_decode_noalloc, the decode entry point for callers that cannot allocate.

Some users of this library cannot allocate device memory while they run - for
example a plugin executing inside an inference engine that owns all device
memory, or a deployment with a device-memory budget fixed at load time - so
they cannot hand pa_decode a workspace.  pa_decode_noalloc keeps that
workspace in a fixed scratch array inside the library instead.  These tests
call it through the C ABI and check it against pa_decode on consecutive calls
(the array keeps the previous call's contents, so nothing in it may be assumed
to start clean), including calls whose workspace layouts differ.

This file is named to be collected last.
"""
import ctypes

import numpy as np
import pytest

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def env():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from paged_kv_cache_140_gb300 import _build, _lib
    _build.build()
    return torch, _lib.load()


def _dev_batch(torch, b):
    from pa_harness import to_device
    T = to_device(b)
    import paged_kv_cache_140_gb300 as pa
    pa.reshape_and_cache(T["key"], T["value"], T["k_cache"], T["v_cache"], T["slot_mapping"])
    torch.cuda.synchronize()
    return T


def _reference(torch, b, T):
    """Output of the existing entry point, pa_decode (caller-provided workspace)."""
    import paged_kv_cache_140_gb300 as pa
    out = torch.empty(T["q"].shape, dtype=torch.float32, device="cuda")
    err = pa.new_err_flag()
    pa.decode(out, T["q"], T["k_cache"], T["v_cache"], T["block_tables"], T["context_lens"],
              float(b.scale), max_context_len=b.max_context_len, partition_size=b.partition_size,
              workspace=pa.DecodeWorkspace("cuda"), err_flag=err)
    assert pa.read_err_flag(err) == 0
    return out


def _noalloc(torch, lib, b, T):
    import paged_kv_cache_140_gb300 as pa
    out = torch.full(T["q"].shape, float("nan"), dtype=torch.float32, device="cuda")
    err = pa.new_err_flag()
    P = ctypes.c_void_p
    dt = 1 if b.dtype == "bf16" else 0
    st = lib.pa_decode_noalloc(
        P(out.data_ptr()), 2, P(T["q"].data_ptr()), dt, P(T["k_cache"].data_ptr()), P(T["v_cache"].data_ptr()),
        dt, 1.0, 1.0, P(T["block_tables"].data_ptr()), T["block_tables"].shape[1],
        P(T["context_lens"].data_ptr()), b.max_context_len, b.num_seqs, b.num_heads, b.num_kv_heads,
        b.head_dim, b.block_size, b.num_blocks, float(b.scale), b.partition_size, P(err.data_ptr()),
        P(torch.cuda.current_stream().cuda_stream))
    assert st == 0, f"pa_decode_noalloc returned {st}"
    torch.cuda.synchronize()
    assert pa.read_err_flag(err) == 0
    return out


def _same(torch, a, b):
    """Bitwise equal: both calls run the same kernel with the same partition
    plan, so only the workspace's address differs."""
    assert torch.isfinite(a).all()
    assert torch.equal(a, b), f"max abs difference {(a - b).abs().max().item():.3e}"


def test_noalloc_matches_pa_decode_on_consecutive_calls(env):
    torch, lib = env
    from paged_kv_cache_140_gb300 import workloads as W
    b1 = W.make_batch("13b", num_seqs=24)                 # split sequences: scratch in use
    b2 = W.make_batch("gqa", num_seqs=2, ctx_cap=12000)   # another workspace layout
    T1, T2 = _dev_batch(torch, b1), _dev_batch(torch, b2)
    r1, r2 = _reference(torch, b1, T1), _reference(torch, b2, T2)
    for b, T, r in ((b1, T1, r1), (b1, T1, r1), (b2, T2, r2), (b1, T1, r1)):
        _same(torch, _noalloc(torch, lib, b, T), r)


def test_noalloc_matches_the_oracle(env):
    torch, lib = env
    import oracle
    from paged_kv_cache_140_gb300 import workloads as W
    from pa_harness import assert_attention_close
    oracle.build()
    b = W.make_batch("13b", num_seqs=24)
    ref, _, _ = oracle.decode_step(b)
    T = _dev_batch(torch, b)
    for _ in range(2):
        assert_attention_close(_noalloc(torch, lib, b, T), ref, "f32", "noalloc 13b")


def test_noalloc_per_warp_kernel_with_split_sequences(env):
    """head_dim 64 runs the per-warp kernel; 16-token partitions split every
    context above 16 tokens, so its partials and merge go through the array.
    A call with another layout runs in between."""
    torch, lib = env
    from paged_kv_cache_140_gb300 import workloads as W
    b = W.make_batch("tiny", partition_size=16)
    b2 = W.make_batch("7b", num_seqs=4, head_dim=64, partition_size=48)
    T, T2 = _dev_batch(torch, b), _dev_batch(torch, b2)
    r, r2 = _reference(torch, b, T), _reference(torch, b2, T2)
    _same(torch, _noalloc(torch, lib, b, T), r)
    _same(torch, _noalloc(torch, lib, b2, T2), r2)
    _same(torch, _noalloc(torch, lib, b, T), r)


def test_noalloc_without_split_sequences(env):
    torch, lib = env
    from paged_kv_cache_140_gb300 import workloads as W
    b = W.make_batch("tiny")
    T = _dev_batch(torch, b)
    r = _reference(torch, b, T)
    for _ in range(2):
        _same(torch, _noalloc(torch, lib, b, T), r)


def test_noalloc_rejects_requests_beyond_the_scratch_limit(env):
    """Valid arguments whose workspace would exceed the array: PA_ERR_WORKSPACE,
    nothing enqueued (the output keeps its contents).  Invalid arguments get
    pa_decode's own answer first."""
    torch, lib = env
    from paged_kv_cache_140_gb300 import _lib as L
    B, H, D, bs, ctx, P = 256, 40, 128, 16, 2048, 16
    need = lib.pa_decode_workspace_size(B, H, H, D, bs, ctx, P)
    assert need > 32 * 1024 * 1024
    nb = 64
    q = torch.zeros((B, H, D), dtype=torch.bfloat16, device="cuda")
    kc = torch.zeros((nb, bs, H, D), dtype=torch.bfloat16, device="cuda")
    vc = torch.zeros_like(kc)
    bt = torch.zeros((B, ctx // bs), dtype=torch.int32, device="cuda")
    cl = torch.ones((B,), dtype=torch.int32, device="cuda")
    out = torch.full((B, H, D), 7.0, dtype=torch.float32, device="cuda")
    Pv = ctypes.c_void_p
    stream = Pv(torch.cuda.current_stream().cuda_stream)

    def call(q_ptr, head_dim=D):
        return lib.pa_decode_noalloc(Pv(out.data_ptr()), 2, q_ptr, 1, Pv(kc.data_ptr()), Pv(vc.data_ptr()), 1,
                                     1.0, 1.0, Pv(bt.data_ptr()), ctx // bs, Pv(cl.data_ptr()), ctx, B, H, H,
                                     head_dim, bs, nb, 0.088, P, Pv(0), stream)

    assert call(Pv(q.data_ptr())) == L.PA_ERR_WORKSPACE
    assert call(Pv(0)) == L.PA_ERR_INVALID_ARG          # null query: pa_decode's answer
    assert call(Pv(q.data_ptr()), head_dim=96) == L.PA_ERR_UNSUPPORTED
    torch.cuda.synchronize()
    assert bool((out == 7.0).all())
