"""GPU parity of pa_decode_append (the step's reshape_and_cache fused into decode).

The new token of sequence s is position context_lens[s] - 1; the fused call must
leave the caches bit-identical to the oracle's reshape_and_cache at that slot,
match the oracle's attention within 2e-3, and equal the separate
reshape_and_cache + decode path bit for bit.
"""
import numpy as np
import pytest

import oracle
from paged_kv_cache_140_gb300 import workloads as W

from pa_harness import assert_attention_close, cache_bits, run_step, to_device, torch_dtype

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from paged_kv_cache_140_gb300 import _build
    _build.build()
    oracle.build()


def run_append(b, out_dtype="f32", partition_size=None):
    import torch
    import paged_kv_cache_140_gb300 as pa
    T = to_device(b)
    # one row per sequence; sequences without a new token keep a zero row
    has = np.nonzero(b.context_lens > 0)[0]
    kf = torch.zeros((b.num_seqs, b.num_kv_heads, b.head_dim), dtype=T["key"].dtype, device="cuda")
    vf = torch.zeros_like(kf)
    kf[torch.from_numpy(has).cuda()] = T["key"]
    vf[torch.from_numpy(has).cuda()] = T["value"]
    out = torch.empty(T["q"].shape, dtype=torch_dtype(out_dtype if out_dtype != "native" else b.dtype),
                      device="cuda")
    err = pa.new_err_flag()
    P = b.partition_size if partition_size is None else partition_size
    pa.decode_append(out, T["q"], kf, vf, T["k_cache"], T["v_cache"], T["block_tables"], T["context_lens"],
                     float(b.scale), max_context_len=b.max_context_len, partition_size=P, err_flag=err,
                     k_scale=b.k_scale, v_scale=b.v_scale)
    torch.cuda.synchronize()
    return out, T, pa.read_err_flag(err)


CASES = [
    ("tiny", dict(), None),
    ("7b", dict(num_seqs=6), None),
    ("13b", dict(num_seqs=24), None),
    ("13b", dict(num_seqs=12, cache_dtype="fp8"), None),
    ("gqa", dict(num_seqs=2, ctx_cap=12000), None),
    ("13b", dict(num_seqs=8, block_size=8), 64),
    ("7b", dict(context_lens=[0, 1, 16, 17, 255, 256, 257]), 64),
    ("tiny", dict(num_heads=8, num_kv_heads=2), None),
    ("7b", dict(num_seqs=6, block_size=32), None),
    ("gqa", dict(num_seqs=3, ctx_cap=3000, block_size=8), 128),
    ("gqa", dict(num_seqs=2, ctx_cap=9000, cache_dtype="fp8"), None),
    ("13b", dict(num_seqs=8, block_size=8, cache_dtype="fp8"), 64),
]


@pytest.mark.parametrize("name,kw,P", CASES, ids=[f"{c[0]}-{i}" for i, c in enumerate(CASES)])
def test_append_matches_oracle_and_separate_path(name, kw, P):
    b = W.make_batch(name, **kw)
    ref, kc, vc = oracle.decode_step(b)
    out, T, flag = run_append(b, partition_size=P)
    assert flag == 0
    assert_attention_close(out, ref, "f32", f"{name} append")
    assert np.array_equal(cache_bits(T["k_cache"]), kc)
    assert np.array_equal(cache_bits(T["v_cache"]), vc)
    sep, _, flag2 = run_step(b, partition_size=P)
    assert flag2 == 0
    assert np.array_equal(out.cpu().numpy(), sep.cpu().numpy())


@pytest.mark.parametrize("name", ["13b", "13b_fp8", "gqa"])
def test_append_native_output_full_size_every_row(name):
    """The benchmark's default step (pa_decode_append) at full size: every
    output element against the oracle, the caches bit-exact in full."""
    b = W.make_batch(name)
    ref, kc, vc = oracle.decode_step(b)
    out, T, flag = run_append(b, out_dtype="native")
    assert flag == 0
    assert_attention_close(out, ref, b.dtype, f"{name} append full size")
    assert np.array_equal(cache_bits(T["k_cache"]), kc)
    assert np.array_equal(cache_bits(T["v_cache"]), vc)