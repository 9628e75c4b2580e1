"""GPU parity: the CUDA path through the C ABI against the CPU oracle.

Bit-exact for reshape_and_cache and copy_blocks; attention within 2e-3
max-abs (fp32 output) or 2e-3 + 1 ulp (half outputs).  Sizes are chosen so
the oracle finishes in seconds yet every case spans several 16-token stages,
several partitions and a ragged tail; the full-size workloads run in the
launch configuration the benchmark times and are checked on every output
element too.
"""
import numpy as np
import pytest

import oracle
from paged_kv_cache_140_gb300 import workloads as W

from pa_harness import assert_attention_close, cache_bits, run_step, to_device

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from paged_kv_cache_140_gb300 import _build
    _build.build()
    oracle.build()


def check_step(b, out_dtype="f32", partition_size=None, caches=True):
    ref, kc, vc = oracle.decode_step(b)
    out, T, flag = run_step(b, out_dtype=out_dtype, partition_size=partition_size)
    assert flag == 0, f"err_flag {flag:#x}"
    err = assert_attention_close(out, ref, b.dtype if out_dtype == "native" else out_dtype, b.name)
    if caches:
        assert np.array_equal(cache_bits(T["k_cache"]), kc), "k_cache differs from oracle"
        assert np.array_equal(cache_bits(T["v_cache"]), vc), "v_cache differs from oracle"
    return err, out


# ------------------------------------------------------------- the workloads

@pytest.mark.parametrize("out_dtype", ["f32", "native"])
def test_tiny_step(out_dtype):
    check_step(W.make_batch("tiny"), out_dtype)


SCALED = [
    ("7b", dict(num_seqs=6)),
    ("13b", dict(num_seqs=24)),
    ("gqa", dict(num_seqs=2, ctx_cap=20000)),
    ("gqa32", dict(num_seqs=2, ctx_cap=20000)),
    ("prefix", dict(groups=3)),
]


@pytest.mark.parametrize("name,kw", SCALED, ids=[s[0] for s in SCALED])
@pytest.mark.parametrize("out_dtype", ["f32", "native"])
def test_scaled_workloads(name, kw, out_dtype):
    check_step(W.make_batch(name, **kw), out_dtype)


# ----------------------------------------------------- shapes and partitions

@pytest.mark.parametrize("P", [0, 16, 32, 48, 256, 512])
def test_partition_sizes(P):
    b = W.make_batch("7b", num_seqs=5, ctx_cap=1500)
    check_step(b, "f32", partition_size=P, caches=False)


@pytest.mark.parametrize("bs", [8, 16, 32, 64])
def test_block_sizes(bs):
    b = W.make_batch("13b", num_seqs=12, block_size=bs)
    check_step(b, "f32", partition_size=0 if bs != 8 else 128)


@pytest.mark.parametrize("hq,hkv", [(8, 8), (8, 4), (16, 4), (16, 2)])
@pytest.mark.parametrize("head_dim", [64, 128])
@pytest.mark.parametrize("dtype", ["f16", "bf16"])
def test_groups_head_dims_dtypes(hq, hkv, head_dim, dtype):
    b = W.make_batch("7b", num_seqs=4, ctx_cap=700, num_heads=hq, num_kv_heads=hkv,
                     head_dim=head_dim, dtype=dtype)
    check_step(b, "f32", partition_size=128)
    check_step(b, "native", partition_size=0, caches=False)


def test_single_partition_equals_partition_larger_than_context():
    b = W.make_batch("7b", num_seqs=4, ctx_cap=300)
    _, a = check_step(b, "f32", partition_size=512, caches=False)
    _, c = check_step(b, "f32", partition_size=320, caches=False)
    assert np.array_equal(a.cpu().numpy(), c.cpu().numpy())


# --------------------------------------------------------------- invariants

def test_physical_block_permutation_is_bitwise_invariant():
    b = W.make_batch("13b", num_seqs=16)
    out1, _, f1 = run_step(b)
    rng = np.random.default_rng(3)
    perm = rng.permutation(b.num_blocks)
    b2 = W.Batch(**{**b.__dict__})
    b2.k_cache = np.empty_like(b.k_cache)
    b2.v_cache = np.empty_like(b.v_cache)
    b2.k_cache[perm] = b.k_cache
    b2.v_cache[perm] = b.v_cache
    b2.block_tables = np.where(b.block_tables >= 0, perm[np.maximum(b.block_tables, 0)], -1).astype(np.int32)
    bs = b.block_size
    b2.slot_mapping = perm[b.slot_mapping // bs] * bs + b.slot_mapping % bs
    out2, _, f2 = run_step(b2)
    assert f1 == f2 == 0
    assert np.array_equal(out1.cpu().numpy(), out2.cpu().numpy())


def test_run_to_run_bitwise_determinism():
    b = W.make_batch("gqa", num_seqs=2, ctx_cap=9000)
    dev = to_device(b)
    o1, _, _ = run_step(b, dev=dev)
    o2, _, _ = run_step(b, dev=dev)
    assert np.array_equal(o1.cpu().numpy(), o2.cpu().numpy())


def test_stale_slots_hold_nan_and_do_not_leak():
    # Every unused slot is NaN by construction; check explicitly on a ragged case.
    b = W.make_batch("7b", num_seqs=6, ctx_cap=333)
    assert np.isnan(b.k_cache.view(np.float16)).any()
    check_step(b, "f32")


# ------------------------------------------------------------------ edges

def test_zero_and_one_token_contexts():
    b = W.make_batch("7b", context_lens=[0, 1, 16, 17, 0, 2048, 255, 256, 257])
    ref, _, _ = oracle.decode_step(b)
    assert np.all(ref[0] == 0) and np.all(ref[4] == 0)
    out, _, flag = run_step(b)
    assert flag == 0
    assert_attention_close(out, ref, "f32", "edge lengths")
    o = out.cpu().numpy()
    assert np.all(o[0] == 0) and np.all(o[4] == 0)


def test_bad_block_id_is_flagged_and_isolated():
    import paged_kv_cache_140_gb300 as pa
    b = W.make_batch("13b", num_seqs=8)
    s_bad = int(np.argmax(b.context_lens))
    b.block_tables[s_bad, 0] = b.num_blocks + 5
    out, _, flag = run_step(b)
    assert flag & pa.FLAG_BAD_BLOCK_ID
    ref, _, _ = oracle.decode_step(W.subset_batch(b, [s for s in range(8) if s != s_bad]))
    keep = [s for s in range(8) if s != s_bad]
    assert_attention_close(out[keep], ref, "f32", "unaffected sequences")
    assert np.all(np.isfinite(out[s_bad].float().cpu().numpy()))


def test_bad_context_length_is_flagged():
    import paged_kv_cache_140_gb300 as pa
    import torch
    b = W.make_batch("7b", num_seqs=4, ctx_cap=200)
    T = to_device(b)
    T["context_lens"][1] = b.max_context_len + 7
    out, _, flag = run_step(b, dev=T)
    assert flag & pa.FLAG_BAD_CONTEXT_LEN
    assert torch.all(out[1] == 0)


def test_bad_slot_and_copy_pair_are_flagged():
    import paged_kv_cache_140_gb300 as pa
    import torch
    b = W.make_batch("prefix", groups=2)
    T = to_device(b)
    T["slot_mapping"][3] = b.num_blocks * b.block_size + 1
    T["slot_mapping"][4] = -1
    T["block_mapping"][0, 1] = -3
    err = pa.new_err_flag()
    pa.copy_blocks(T["k_cache"], T["v_cache"], T["block_mapping"], err_flag=err)
    pa.reshape_and_cache(T["key"], T["value"], T["k_cache"], T["v_cache"], T["slot_mapping"], err_flag=err)
    torch.cuda.synchronize()
    flag = pa.read_err_flag(err)
    assert flag & pa.FLAG_BAD_SLOT and flag & pa.FLAG_BAD_COPY_PAIR
    sm = b.slot_mapping.copy()
    sm[3] = b.num_blocks * b.block_size + 1
    sm[4] = -1
    bm = b.block_mapping.copy()
    bm[0, 1] = -3
    kc, vc, _ = oracle.copy_blocks(b.k_cache, b.v_cache, bm)
    kc, vc, bad = oracle.reshape_and_cache(b.key, b.value, kc, vc, sm)
    assert bad == 1
    assert np.array_equal(cache_bits(T["k_cache"]), kc)
    assert np.array_equal(cache_bits(T["v_cache"]), vc)


def test_copy_on_write_keeps_shared_source_and_decode_before_divergence():
    """After copy_blocks the copies equal the shared block bit for bit, and
    attention over the copied table equals attention over the shared one for
    the tokens written before divergence."""
    import paged_kv_cache_140_gb300 as pa
    import torch
    b = W.make_batch("prefix", groups=2)
    T = to_device(b)
    pa.copy_blocks(T["k_cache"], T["v_cache"], T["block_mapping"])
    torch.cuda.synchronize()
    kc = cache_bits(T["k_cache"])
    for src, dst in b.block_mapping:
        assert np.array_equal(kc[dst], kc[src])
    assert np.array_equal(kc, oracle.copy_blocks(b.k_cache, b.v_cache, b.block_mapping)[0])
    # Decode the 1000-token prompt through sample 0's table (copy) and sample 3's (shared).
    b2 = W.subset_batch(b, [0, 3])
    b2.context_lens = np.array([1000, 1000], dtype=np.int32)
    T2 = to_device(b2)
    T2["k_cache"], T2["v_cache"] = T["k_cache"], T["v_cache"]
    T2["q"][1] = T2["q"][0]
    out = torch.empty(T2["q"].shape, dtype=torch.float32, device="cuda")
    pa.decode(out, T2["q"], T2["k_cache"], T2["v_cache"], T2["block_tables"], T2["context_lens"],
              float(b.scale), max_context_len=b.max_context_len)
    torch.cuda.synchronize()
    assert torch.equal(out[0], out[1])


# ------------------------------------------------ full sizes, every row

FULL = ["7b", "13b", "gqa", "gqa32", "prefix"]


@pytest.mark.parametrize("name", FULL)
def test_full_size_every_row(name):
    """The bench workloads at full size, in the launch configuration the
    benchmark times: every output element against the oracle, and the caches
    after the step's writes bit-exact in full."""
    b = W.make_batch(name)
    ref, kc, vc = oracle.decode_step(b)
    out, T, flag = run_step(b, out_dtype="native")
    assert flag == 0
    assert_attention_close(out, ref, b.dtype, f"{name} full size")
    assert np.array_equal(cache_bits(T["k_cache"]), kc), "k_cache differs from oracle"
    assert np.array_equal(cache_bits(T["v_cache"]), vc), "v_cache differs from oracle"
