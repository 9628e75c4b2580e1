"""Pins of the oracle's FP8 (e4m3) cache path against torch's float8_e4m3fn,
closed forms and the 16-bit oracle.

Readings (the pages name FP8 among vLLM's quantisation options, "LLM推理优化：
vLLM PagedAttention深度解析与工程实践", §八, without detail): per-tensor K and V
scales; code = e4m3(fp32(x) / scale) rounded to nearest-even, finite values
saturating at +-448; attention reads code value * scale.
"""
import math

import numpy as np
import pytest

import oracle
from oracle import brute

torch = pytest.importorskip("torch")


def torch_codes(x):
    return torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(torch.float8_e4m3fn) \
        .view(torch.uint8).numpy()


def torch_values(codes):
    return torch.from_numpy(np.ascontiguousarray(codes, dtype=np.uint8)).view(torch.float8_e4m3fn) \
        .to(torch.float64).numpy()


def test_decode_all_codes():
    c = np.arange(256, dtype=np.int64).astype(np.uint8)
    got, want = oracle.e4m3_decode(c), torch_values(c)
    assert np.array_equal(np.isnan(got), np.isnan(want))
    ok = ~np.isnan(want)
    assert np.array_equal(got[ok], want[ok])
    assert got[0x7E] == 448.0 and got[0x01] == 2.0 ** -9 and got[0x08] == 2.0 ** -6


def test_encode_matches_torch_below_the_saturation_point():
    rng = np.random.default_rng(0)
    x = np.concatenate([rng.standard_normal(200000).astype(np.float32) * s for s in (0.003, 0.1, 1, 30, 150)])
    # every representable value and every midpoint between neighbours
    vals = torch_values(np.arange(0, 0x7F, dtype=np.uint8))
    mids = (vals[:-1] + vals[1:]) / 2
    x = np.concatenate([x, vals, mids, -vals, -mids]).astype(np.float32)
    x = x[np.abs(x) < 464]
    assert np.array_equal(oracle.e4m3_encode(x), torch_codes(x))


def test_encode_saturates_and_keeps_nan():
    x = np.array([448, 464, 500, 1e30, np.inf, -464, -np.inf, np.nan, 0.0, -0.0], dtype=np.float32)
    got = oracle.e4m3_encode(x)
    assert list(got) == [0x7E, 0x7E, 0x7E, 0x7E, 0x7E, 0xFE, 0xFE, 0x7F, 0x00, 0x80]


def test_round_trip_of_every_finite_code():
    c = np.array([i for i in range(256) if i not in (0x7F, 0xFF)], dtype=np.uint8)
    assert np.array_equal(oracle.e4m3_encode(oracle.e4m3_decode(c).astype(np.float32)), c)


def test_reshape_fp8_quantises_like_torch():
    rng = np.random.default_rng(1)
    NB, bs, Hkv, D, T = 6, 16, 2, 8, 7
    kc = np.full((NB, bs, Hkv, D), 0x7F, dtype=np.uint8)
    vc = kc.copy()
    xk = rng.standard_normal((T, Hkv, D)).astype(np.float32) * 3
    xv = rng.standard_normal((T, Hkv, D)).astype(np.float32) * 3
    key = torch.from_numpy(xk).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    val = torch.from_numpy(xv).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    slots = rng.permutation(NB * bs)[:T].astype(np.int64)
    ks, vs = np.float32(1 / 16), np.float32(0.03)
    k2, v2, bad = oracle.reshape_and_cache_fp8(key, val, "bf16", kc, vc, slots, ks, vs)
    assert bad == 0
    kx = torch.from_numpy(key.view(np.int16)).view(torch.bfloat16).float().numpy()
    vx = torch.from_numpy(val.view(np.int16)).view(torch.bfloat16).float().numpy()
    want_k, want_v = kc.reshape(NB * bs, Hkv, D).copy(), vc.reshape(NB * bs, Hkv, D).copy()
    want_k[slots] = torch_codes(kx / ks)
    want_v[slots] = torch_codes(vx / vs)
    assert np.array_equal(k2.reshape(NB * bs, Hkv, D), want_k)
    assert np.array_equal(v2.reshape(NB * bs, Hkv, D), want_v)


def _fp8_case(rng, B=3, Hq=4, Hkv=2, D=8, bs=4, ctx=(5, 13, 22)):
    ctx = np.asarray(ctx, dtype=np.int32)
    nblk = [-(-int(c) // bs) for c in ctx]
    NB = sum(nblk) + 3
    perm = rng.permutation(NB)
    tables = np.full((B, max(nblk)), -1, dtype=np.int32)
    i = 0
    for s in range(B):
        tables[s, :nblk[s]] = perm[i:i + nblk[s]]
        i += nblk[s]
    kc = torch_codes(rng.standard_normal((NB, bs, Hkv, D)) * 16)
    vc = torch_codes(rng.standard_normal((NB, bs, Hkv, D)) * 16)
    q = torch.from_numpy(rng.standard_normal((B, Hq, D)).astype(np.float32)).to(torch.bfloat16) \
        .view(torch.int16).numpy().view(np.uint16)
    return q, kc, vc, tables, ctx


def test_fp8_attention_equals_16bit_oracle_on_the_same_values():
    rng = np.random.default_rng(2)
    q, kc, vc, t, ctx = _fp8_case(rng)
    s = 1.0 / 16
    got = oracle.paged_attention_fp8(q, "bf16", kc, vc, s, s, t, ctx, 0.35)
    # e4m3 values times 2^-4 are exact in bfloat16: the 16-bit oracle on those
    # values must give the same doubles.
    k16 = torch.from_numpy(oracle.e4m3_decode(kc) * s).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    v16 = torch.from_numpy(oracle.e4m3_decode(vc) * s).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    want = oracle.paged_attention(q, k16, v16, "bf16", t, ctx, 0.35)
    assert np.array_equal(got, want)


def test_fp8_attention_matches_brute_force_with_torch_dequantisation():
    rng = np.random.default_rng(3)
    q, kc, vc, t, ctx = _fp8_case(rng, B=2, ctx=(9, 17))
    ks, vs = 0.07, 0.02
    got = oracle.paged_attention_fp8(q, "bf16", kc, vc, ks, vs, t, ctx, 0.3)
    K, V = torch_values(kc) * ks, torch_values(vc) * vs
    for s in range(2):
        for hq in range(4):
            n = int(ctx[s])
            Kr = np.array([K[t[s, p // 4], p % 4, hq // 2] for p in range(n)])
            Vr = np.array([V[t[s, p // 4], p % 4, hq // 2] for p in range(n)])
            want = brute.attention_contiguous(brute.widen(q[s, hq], "bf16"), Kr, Vr, 0.3)
            np.testing.assert_allclose(got[s, hq], want, rtol=1e-12, atol=1e-13)


def test_fp8_generator_batch_runs_through_the_oracle():
    from paged_kv_cache_140_gb300 import workloads as W
    b = W.make_batch("13b", num_seqs=3, cache_dtype="fp8")
    assert b.k_cache.dtype == np.uint8 and b.k_scale == 1 / 16
    out, kc, vc = oracle.decode_step(b)
    assert np.all(np.isfinite(out))
    # every new-token slot was written with codes of the step's rows
    assert not np.any(kc.reshape(-1, 40 * 128)[b.slot_mapping] == 0x7F)
