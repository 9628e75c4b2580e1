"""GPU parity of pa_prefill (causal attention of each sequence's new tokens
over its paged context) against the fp64 CPU oracle.

Small cases are compared on every output element; the full-size workloads
on an evenly spaced sample of rows (every head of each), each computed by the
oracle on its own, with the caches compared in full.  Edge cases: empty
and one-token tails, tails with no cached prefix, lengths on and next to the
128-token tile boundary, every supported group size, head_dim 64, block
sizes 8/32/64, all output types, single-tile tails over contexts of many
K/V tiles, and bad block ids."""
import numpy as np
import pytest

import oracle
from pa_harness import assert_attention_close, cache_bits, half_tensor, to_device, torch_dtype

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def torch():
    t = pytest.importorskip("torch")
    if not t.cuda.is_available():
        pytest.skip("no CUDA device")
    import paged_kv_cache_140_gb300._build as b
    b.build()
    return t


def run_prefill(torch, b, out_dtype="f32", dev=None):
    """copy_blocks -> reshape_and_cache -> prefill on the GPU."""
    import paged_kv_cache_140_gb300 as pa
    T = dev if dev is not None else to_device(b)
    cu = torch.from_numpy(b.cu_seqlens_q).cuda()
    err = pa.new_err_flag()
    if len(b.block_mapping):
        pa.copy_blocks(T["k_cache"], T["v_cache"], T["block_mapping"], err_flag=err)
    if len(b.slot_mapping):
        pa.reshape_and_cache(T["key"], T["value"], T["k_cache"], T["v_cache"], T["slot_mapping"], err_flag=err)
    out = torch.full(T["q"].shape, float("nan"), dtype=torch_dtype(out_dtype), device="cuda")
    pa.prefill(out, T["q"], T["k_cache"], T["v_cache"], T["block_tables"], T["context_lens"], cu,
               float(b.scale), max_q_len=b.max_q_len, err_flag=err)
    torch.cuda.synchronize()
    return out, T, pa.read_err_flag(err)


def oracle_rows(b, kc, vc, rows):
    """Oracle output of selected query rows: row r of sequence s (token i of
    its tail) is the decode query of a context of ctx - q_len + i + 1 tokens."""
    rows = np.asarray(rows, dtype=np.int64)
    cu = b.cu_seqlens_q.astype(np.int64)
    seq = np.searchsorted(cu, rows, side="right") - 1
    pos = b.context_lens[seq].astype(np.int64) - (cu[seq + 1] - cu[seq]) + (rows - cu[seq])
    return oracle.paged_attention(b.q[rows], kc, vc, b.dtype, b.block_tables[seq],
                                  (pos + 1).astype(np.int32), b.scale)


def make(name, **kw):
    from paged_kv_cache_140_gb300 import workloads as W
    return W.make_prefill_batch(name, **kw)


SMALL = {
    "13b_bf16": ("prefill", dict(num_seqs=3, prefix_cap=300, q_len_cap=200)),
    "13b_f16": ("prefill", dict(num_seqs=3, prefix_cap=260, q_len_cap=150, dtype="f16")),
    "gqa_g4": ("prefill_gqa", dict(num_seqs=2, prefix_cap=500, q_len_cap=100)),
    "g2_bs32": ("prefill_gqa", dict(num_seqs=2, prefix_cap=400, q_len_cap=90, num_heads=16, block_size=32)),
    "g8_bs8": ("prefill_gqa", dict(num_seqs=2, prefix_cap=333, q_len_cap=77, num_heads=64, block_size=8)),
    "d64_f16_bs64": ("prefill", dict(num_seqs=3, prefix_cap=400, q_len_cap=140, head_dim=64, num_heads=8,
                                     num_kv_heads=8, dtype="f16", block_size=64)),
    "d64_g16_bs128": ("prefill_gqa", dict(num_seqs=2, prefix_cap=300, q_len_cap=40, head_dim=64, num_heads=32,
                                          num_kv_heads=2, block_size=128)),
}


@pytest.mark.parametrize("case", sorted(SMALL))
def test_prefill_matches_oracle(torch, case):
    name, kw = SMALL[case]
    b = make(name, **kw)
    ref, kc, vc = oracle.prefill_step(b)
    out, T, err = run_prefill(torch, b)
    assert err == 0
    assert_attention_close(out, ref, "f32", case)
    assert np.array_equal(cache_bits(T["k_cache"]), kc) and np.array_equal(cache_bits(T["v_cache"]), vc)


@pytest.mark.parametrize("out_dtype", ["bf16", "f16"])
def test_prefill_half_outputs(torch, out_dtype):
    b = make("prefill_gqa", num_seqs=2, prefix_cap=200, q_len_cap=70)
    ref, _, _ = oracle.prefill_step(b)
    out, _, err = run_prefill(torch, b, out_dtype)
    assert err == 0
    assert_attention_close(out, ref, out_dtype, out_dtype)


def test_prefill_edge_lengths(torch):
    """Empty tail, one-token tails, whole-prompt prefill (no cached prefix),
    and contexts on / next to the 128-token tile boundary."""
    prefix = [0, 127, 128, 5, 300, 0, 1, 255]
    qlen = [1, 1, 129, 0, 128, 130, 127, 1]
    b = make("prefill", prefix_lens=prefix, q_lens=qlen, num_heads=8, num_kv_heads=8)
    ref, _, _ = oracle.prefill_step(b)
    out, _, err = run_prefill(torch, b)
    assert err == 0
    assert_attention_close(out, ref, "f32", "edges")


def test_prefill_gqa_edge_lengths(torch):
    """G = 4: 32 tokens per query tile; tails of 31/32/33 tokens."""
    b = make("prefill_gqa", prefix_lens=[0, 96, 17, 4000], q_lens=[33, 32, 31, 65], num_heads=16, num_kv_heads=4)
    ref, _, _ = oracle.prefill_step(b)
    out, _, err = run_prefill(torch, b)
    assert err == 0
    assert_attention_close(out, ref, "f32", "gqa edges")


TAIL_CASES = {
    # name: (workload, prefix lengths, tail lengths, overrides)
    "mha_bf16": ("prefill", [128, 200, 383, 256, 700, 900, 1000, 0], [1, 128, 1, 128, 64, 17, 100, 128],
                 dict(num_heads=4, num_kv_heads=4)),
    "mha_f16": ("prefill", [129, 511, 384, 2000], [127, 1, 128, 3], dict(num_heads=4, num_kv_heads=4, dtype="f16")),
    "g4": ("prefill_gqa", [500, 97, 31, 4000], [32, 5, 1, 20], dict(num_heads=16, num_kv_heads=4)),
    "g8_bs8": ("prefill_gqa", [333, 250, 16], [16, 9, 1], dict(num_heads=64, num_kv_heads=8, block_size=8)),
    "d64_bs64": ("prefill", [600, 129, 64], [128, 1, 100], dict(num_heads=8, num_kv_heads=8, head_dim=64,
                                                                 dtype="f16", block_size=64)),
}


@pytest.mark.parametrize("out_dtype", ["f32", "bf16"])
@pytest.mark.parametrize("case", sorted(TAIL_CASES))
def test_prefill_single_tile_tails(torch, case, out_dtype):
    """Tails that fit one query tile (the CTA's second query tile is empty),
    over contexts of one to 32 K/V tiles: odd and even K/V tile counts,
    contexts on and off the 128-token boundary, full tiles (TMA-store
    epilogue for 16-bit outputs), one-row tiles, every group size class,
    head_dim 64 and block sizes 8 / 64."""
    name, prefix, qlen, kw = TAIL_CASES[case]
    kw = dict(kw)
    bs = kw.pop("block_size", None)
    b = make(name, prefix_lens=prefix, q_lens=qlen, block_size=bs, **kw)
    ref, _, _ = oracle.prefill_step(b)
    out, _, err = run_prefill(torch, b, out_dtype)
    assert err == 0
    assert_attention_close(out, ref, out_dtype, f"tails {case}")


def test_prefill_bad_block_late_in_context(torch):
    """A bad block id in a late K/V tile of a one-tile tail zeroes the whole
    query tile and sets PA_FLAG_BAD_BLOCK_ID; the other sequence is
    unaffected."""
    import paged_kv_cache_140_gb300 as pa
    b = make("prefill", prefix_lens=[600, 300], q_lens=[20, 50], num_heads=4, num_kv_heads=4)
    ref, _, _ = oracle.prefill_step(b)
    T = to_device(b)
    T["block_tables"][0, 25] = b.num_blocks + 3      # positions 400 .. 415: K/V tile 3 of 5
    out, _, err = run_prefill(torch, b, dev=T)
    assert err & pa.FLAG_BAD_BLOCK_ID
    assert float(out[:20].abs().max()) == 0.0
    assert_attention_close(out[20:], ref[20:], "f32", "good sequence")


def _ramp_keys(b, per_token):
    """The batch with every key row at position p scaled by 1 + p * per_token
    (the cached prefix rows and the step's new rows alike; other slots keep
    their bits), so that each later K/V tile's scores exceed the earlier
    ones' by far more than the lazy-rescale margin."""
    import dataclasses

    def dec(bits):
        if b.dtype == "f16":
            return bits.view(np.float16).astype(np.float32)
        return (bits.astype(np.uint32) << 16).view(np.float32)

    def enc(x):
        if b.dtype == "f16":
            return x.astype(np.float16).view(np.uint16)
        u = x.astype(np.float32).view(np.uint32)
        return ((u + 0x7FFF + ((u >> 16) & 1)) >> 16).astype(np.uint16)

    bs = b.block_size
    cu = b.cu_seqlens_q.astype(np.int64)
    prefix = b.context_lens.astype(np.int64) - np.diff(cu)
    kc = b.k_cache.copy()
    key = b.key.copy()
    for s in range(len(prefix)):
        for pos in range(int(prefix[s])):
            blk, off = b.block_tables[s, pos // bs], pos % bs
            kc[blk, off] = enc(dec(kc[blk, off]) * (1.0 + pos * per_token))
        for r in range(int(cu[s]), int(cu[s + 1])):
            key[r] = enc(dec(key[r]) * (1.0 + (prefix[s] + r - cu[s]) * per_token))
    return dataclasses.replace(b, k_cache=kc, key=key)


@pytest.mark.parametrize("dtype", ["bf16", "f16"])
@pytest.mark.parametrize("name,heads", [("prefill", (4, 4)), ("prefill_gqa", (16, 4))])
def test_prefill_rescales_at_every_tile(torch, name, heads, dtype):
    """Keys that grow with their position push every row's running max up by
    more than the lazy-rescale margin at each K/V tile, so the output is
    rescaled throughout: in two-tile units (the PV before each QK), and in
    single-tile units that double-buffer S (the rescale waits for the
    previous PV)."""
    prefix = [300, 700, 129, 900, 40, 0]
    qlen = [100, 128, 250, 20, 256, 200]
    b = _ramp_keys(make(name, prefix_lens=prefix, q_lens=qlen, num_heads=heads[0], num_kv_heads=heads[1],
                        dtype=dtype), 1.0 / 32)
    ref, _, _ = oracle.prefill_step(b)
    out, _, err = run_prefill(torch, b)
    assert err == 0
    assert_attention_close(out, ref, "f32", f"rescaled {name} {dtype}")


@pytest.mark.parametrize("num_seqs", [128, 130])
def test_prefill_many_sequences(torch, num_seqs):
    """CTAs take sequences longest context first for batches of up to 128
    sequences (ranked in every CTA) and in index order above that: both
    sides of the limit, with many equal context lengths (rank ties) and
    empty tails, give every row once."""
    rng = np.random.default_rng(num_seqs)
    qlen = rng.integers(0, 40, num_seqs)
    ctx = rng.choice([40, 90, 200, 333], num_seqs)       # few distinct lengths: ties
    b = make("prefill", prefix_lens=list(ctx - qlen), q_lens=list(qlen), num_heads=4, num_kv_heads=4,
             head_dim=64, block_size=16)
    ref, _, _ = oracle.prefill_step(b)
    out, _, err = run_prefill(torch, b)
    assert err == 0
    assert_attention_close(out, ref, "f32", f"{num_seqs} sequences")


def test_prefill_equal_contexts_every_order(torch):
    """Sequences of equal context length (rank ties broken by index) and of
    falling, rising and mixed lengths: each CTA still owns one distinct
    (sequence, tile pair, KV head)."""
    prefix = [300, 300, 300, 0, 600, 20, 300, 1000]
    qlen = [40, 40, 40, 340, 5, 320, 40, 1]
    b = make("prefill_gqa", prefix_lens=prefix, q_lens=qlen, num_heads=16, num_kv_heads=4)
    ref, _, _ = oracle.prefill_step(b)
    out, _, err = run_prefill(torch, b)
    assert err == 0
    assert_attention_close(out, ref, "f32", "ties")


def test_prefill_of_prefix_hit_tails(torch):
    """The prefix-sharing workload: every sample's private tail prefilled over
    the shared 1000-token prompt (after copy-on-write of the partial block)."""
    b = make("prefix", groups=2)
    out, T, err = run_prefill(torch, b)
    assert err == 0
    kc, vc = cache_bits(T["k_cache"]), cache_bits(T["v_cache"])
    rng = np.random.default_rng(5)
    rows = np.unique(np.concatenate([b.cu_seqlens_q[:-1], b.cu_seqlens_q[1:] - 1,
                                     rng.integers(0, b.num_tokens, 96)]))
    ref = oracle_rows(b, kc, vc, rows)
    assert_attention_close(out[torch.from_numpy(rows).cuda()], ref, "f32", "prefix tails")
    # caches: the whole step is bit-exact against the oracle's copy + scatter
    okc, ovc = _oracle_caches(b)
    assert np.array_equal(kc, okc) and np.array_equal(vc, ovc)


def _oracle_caches(b):
    kc, vc = b.k_cache, b.v_cache
    if len(b.block_mapping):
        kc, vc, _ = oracle.copy_blocks(kc, vc, b.block_mapping)
    kc, vc, _ = oracle.reshape_and_cache(b.key, b.value, kc, vc, b.slot_mapping)
    return kc, vc


# Evenly spaced row stride per full-size workload: the fp64 oracle costs
# about a second per 40 query rows of the 13B chunk on 16 host cores, so
# every row of every workload would take minutes; every 8th (16th for the
# longer GQA contexts) row plus each sequence's first and last row spans
# every sequence, query tile and causal offset class.
FULL_STRIDE = {"prefill": 8, "prefill_gqa": 16, "prefill_prefix": 8}


@pytest.mark.parametrize("name", sorted(FULL_STRIDE))
def test_prefill_full_size_rows(torch, name):
    """The bench workloads at full size, in the benchmark's launch
    configuration: an evenly spaced row sample against the oracle (every
    head of each row), the caches after the step's writes bit-exact in full."""
    if name == "prefill_prefix":
        b = make("prefix")
    else:
        b = make(name)
    out, T, err = run_prefill(torch, b)
    assert err == 0
    okc, ovc = _oracle_caches(b)
    assert np.array_equal(cache_bits(T["k_cache"]), okc)
    assert np.array_equal(cache_bits(T["v_cache"]), ovc)
    cu = b.cu_seqlens_q
    rows = np.unique(np.concatenate([np.arange(0, b.num_tokens, FULL_STRIDE[name]),
                                     cu[:-1][cu[1:] > cu[:-1]], (cu[1:] - 1)[cu[1:] > cu[:-1]]]))
    ref = oracle_rows(b, okc, ovc, rows)
    assert_attention_close(out[torch.from_numpy(rows).cuda()], ref, "f32", name)
    assert bool(torch.isfinite(out.float()).all())


def test_prefill_one_token_tails_equal_decode(torch):
    """A one-token tail is a decode step: pa_prefill and pa_decode agree."""
    import paged_kv_cache_140_gb300 as pa
    b = make("prefill_gqa", num_seqs=4, prefix_cap=3000, q_lens=[1, 1, 1, 1])
    out, T, err = run_prefill(torch, b)
    assert err == 0
    dec = torch.empty_like(out)
    pa.decode(dec, T["q"], T["k_cache"], T["v_cache"], T["block_tables"], T["context_lens"], float(b.scale),
              max_context_len=int(b.context_lens.max()))
    torch.cuda.synchronize()
    assert float((dec - out).abs().max()) <= 2e-3


def test_prefill_is_deterministic(torch):
    b = make("prefill_gqa", num_seqs=2, prefix_cap=700, q_len_cap=120)
    out1, T, _ = run_prefill(torch, b)
    out2, _, _ = run_prefill(torch, b, dev=T)
    assert torch.equal(out1, out2)


def test_prefill_bad_block_id_is_flagged(torch):
    """A block id outside the pool is not read: its query tiles give zero rows
    and PA_FLAG_BAD_BLOCK_ID; other sequences are unaffected."""
    import paged_kv_cache_140_gb300 as pa
    b = make("prefill", num_seqs=2, prefix_lens=[200, 150], q_lens=[40, 60], num_heads=4, num_kv_heads=4)
    ref, _, _ = oracle.prefill_step(b)
    T = to_device(b)
    T["block_tables"][0, 1] = b.num_blocks + 7
    out, _, err = run_prefill(torch, b, dev=T)
    assert err & pa.FLAG_BAD_BLOCK_ID
    assert float(out[:40].abs().max()) == 0.0
    assert_attention_close(out[40:], ref[40:], "f32", "good sequence")


def test_prefill_rejects_bad_arguments(torch):
    import paged_kv_cache_140_gb300 as pa
    b = make("prefill", num_seqs=1, prefix_lens=[10], q_lens=[5], num_heads=4, num_kv_heads=4)
    T = to_device(b)
    cu = torch.from_numpy(b.cu_seqlens_q).cuda()
    out = torch.empty(T["q"].shape, dtype=torch.float32, device="cuda")
    with pytest.raises(pa.PagedAttentionError):
        pa.prefill(out, T["q"], T["k_cache"], T["v_cache"], T["block_tables"], T["context_lens"], cu, -1.0,
                   max_q_len=5)
    q3 = half_tensor(np.zeros((5, 3, 128), np.uint16), "bf16")     # 3 heads over 4 KV heads
    with pytest.raises(pa.PagedAttentionError):
        pa.prefill(torch.empty(q3.shape, device="cuda"), q3, T["k_cache"], T["v_cache"], T["block_tables"],
                   T["context_lens"], cu, 0.1, max_q_len=5)


def test_prefill_bad_lengths_are_flagged(torch):
    """q_len > ctx gives zero rows and PA_FLAG_BAD_CONTEXT_LEN; a decreasing
    cu_seqlens_q or a q_len above max_q_len is flagged too; good sequences
    are unaffected."""
    import paged_kv_cache_140_gb300 as pa
    b = make("prefill", num_seqs=3, prefix_lens=[40, 60, 20], q_lens=[30, 50, 10], num_heads=4, num_kv_heads=4)
    ref, _, _ = oracle.prefill_step(b)
    # context shorter than the tail of sequence 1
    T = to_device(b)
    T["context_lens"][1] = 20
    out, _, err = run_prefill(torch, b, dev=T)
    assert err & pa.FLAG_BAD_CONTEXT_LEN
    assert float(out[30:80].abs().max()) == 0.0
    assert_attention_close(out[:30], ref[:30], "f32", "sequence 0")
    assert_attention_close(out[80:], ref[80:], "f32", "sequence 2")
    # q_len above the host's max_q_len bound
    out2, _, err2 = run_prefill(torch, b.__class__(**{**b.__dict__, "max_q_len": 16}))
    assert err2 & pa.FLAG_BAD_CONTEXT_LEN
    # cu_seqlens_q running backwards for sequence 2
    T3 = to_device(b)
    cu = torch.from_numpy(b.cu_seqlens_q).cuda()
    cu[3] = 70
    out3 = torch.zeros(T3["q"].shape, dtype=torch.float32, device="cuda")
    err3 = pa.new_err_flag()
    pa.reshape_and_cache(T3["key"], T3["value"], T3["k_cache"], T3["v_cache"], T3["slot_mapping"])
    pa.prefill(out3, T3["q"], T3["k_cache"], T3["v_cache"], T3["block_tables"], T3["context_lens"], cu,
               float(b.scale), max_q_len=b.max_q_len, err_flag=err3)
    torch.cuda.synchronize()
    assert pa.read_err_flag(err3) & pa.FLAG_BAD_CONTEXT_LEN
    assert_attention_close(out3[:80], ref[:80], "f32", "sequences 0-1")
