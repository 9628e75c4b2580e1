"""GPU checks of pa.StepGraph: a decode or prefill step captured once as a
CUDA graph and replayed on refilled input buffers gives, bit for bit, what the
same calls give when launched one by one, and matches the oracle."""
import numpy as np
import pytest

import oracle
from paged_kv_cache_140_gb300 import workloads as W

from pa_harness import assert_attention_close, cache_bits, to_device

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from paged_kv_cache_140_gb300 import _build
    _build.build()
    oracle.build()


def test_decode_step_graph_replays_refilled_inputs():
    import torch
    import paged_kv_cache_140_gb300 as pa
    b = W.make_batch("13b", num_seqs=16)
    T = to_device(b)
    # fixed buffers the graph reads: inputs, caches, output, workspace
    buf = {k: T[k].clone() for k in ("q", "key", "value", "slot_mapping", "block_tables", "context_lens")}
    kc, vc = T["k_cache"].clone(), T["v_cache"].clone()
    out = torch.empty(buf["q"].shape, dtype=torch.float32, device="cuda")
    ws = pa.DecodeWorkspace("cuda")

    def step():
        pa.reshape_and_cache(buf["key"], buf["value"], kc, vc, buf["slot_mapping"])
        pa.decode(out, buf["q"], kc, vc, buf["block_tables"], buf["context_lens"], float(b.scale),
                  max_context_len=b.max_context_len, workspace=ws)

    g = pa.StepGraph(step)
    gen = torch.Generator(device="cuda").manual_seed(5)
    for round_ in range(2):
        if round_ == 1:   # refill the query buffer in place with other values
            buf["q"].copy_(torch.randn(buf["q"].shape, generator=gen, device="cuda").to(buf["q"].dtype))
        kc.copy_(T["k_cache"])
        vc.copy_(T["v_cache"])
        g.replay()
        torch.cuda.synchronize()
        got, got_k = out.clone(), cache_bits(kc)
        # the same calls launched one by one
        kc.copy_(T["k_cache"])
        vc.copy_(T["v_cache"])
        step()
        torch.cuda.synchronize()
        assert np.array_equal(got.cpu().numpy(), out.cpu().numpy())
        assert np.array_equal(got_k, cache_bits(kc))
        if round_ == 0:
            ref, kref, _ = oracle.decode_step(b)
            assert_attention_close(got, ref, "f32", "graph replay")
            assert np.array_equal(got_k, kref)


def test_prefill_step_graph_matches_eager():
    import torch
    import paged_kv_cache_140_gb300 as pa
    b = W.make_prefill_batch("prefill", num_seqs=2, prefix_cap=300, q_len_cap=200, num_heads=8, num_kv_heads=8)
    T = to_device(b)
    cu = torch.from_numpy(b.cu_seqlens_q).cuda()
    out = torch.empty(T["q"].shape, dtype=torch.float32, device="cuda")

    def step():
        pa.reshape_and_cache(T["key"], T["value"], T["k_cache"], T["v_cache"], T["slot_mapping"])
        pa.prefill(out, T["q"], T["k_cache"], T["v_cache"], T["block_tables"], T["context_lens"], cu,
                   float(b.scale), max_q_len=b.max_q_len)

    g = pa.StepGraph(step)
    out.zero_()
    g.replay()
    torch.cuda.synchronize()
    got = out.clone()
    step()
    torch.cuda.synchronize()
    assert np.array_equal(got.cpu().numpy(), out.cpu().numpy())
