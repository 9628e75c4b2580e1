"""Host logic of bench.py that needs no GPU: the code-only kernel hash that
decides whether a committed ncu traffic figure still describes the kernels,
and which decode kernel a workload runs on."""
import glob
import json
import os

import pytest

import bench
from paged_kv_cache_140_gb300 import workloads as W

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_code_only_ignores_comments_and_layout():
    a = 'int f(int x) {  // add one\n    return x + 1; /* done */\n}\n'
    b = "int f(int x){return x+1;}"
    assert bench._code_only(a) == bench._code_only(b)


def test_code_only_keeps_code_and_literals():
    base = bench._code_only('int f() { return g("a // b", 1); }')
    assert "a // b" in base                      # a comment marker inside a string literal is code
    assert bench._code_only('int f() { return g("a // b", 2); }') != base
    assert bench._code_only("int f() { return h('/'); }") != bench._code_only("int f() { return h('*'); }")


def test_source_hash_covers_every_listed_file():
    for kind, names in bench.KERNEL_SOURCES.items():
        for name in names:
            assert os.path.isfile(os.path.join(ROOT, "paged_kv_cache_140_gb300", "csrc", name)), name
        h = bench.source_hash(kind)
        assert len(h) == 16 and h == bench.source_hash(kind)
    assert bench.source_hash("decode") != bench.source_hash("prefill")


@pytest.mark.parametrize("path", sorted(glob.glob(os.path.join(ROOT, "profiles", "traffic_*.json"))),
                         ids=lambda p: os.path.basename(p))
def test_committed_traffic_files(path):
    """A committed traffic figure is read + write and is reported exactly when
    it was taken on the kernel code as it is now (null otherwise)."""
    with open(path) as f:
        d = json.load(f)
    w = d["workload"]
    kind = "prefill" if w in bench.PREFILL_WORKLOADS else "decode"
    assert d["dram_bytes_per_launch"] == d["dram_bytes_read"] + d["dram_bytes_write"]
    fresh = d["kernel_source_hash"] == bench.source_hash(kind)
    assert bench.load_traffic(w, kind) == (d["dram_bytes_per_launch"] if fresh else None)


def test_traffic_of_other_kernel_code_is_not_reported(tmp_path, monkeypatch):
    (tmp_path / "profiles").mkdir()
    (tmp_path / "profiles" / "traffic_x.json").write_text(json.dumps(
        {"workload": "x", "kernel_source_hash": "abc", "dram_bytes_read": 1, "dram_bytes_write": 2,
         "dram_bytes_per_launch": 3}))
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    monkeypatch.setattr(bench, "source_hash", lambda kind="decode": "abc")
    assert bench.load_traffic("x") == 3
    monkeypatch.setattr(bench, "source_hash", lambda kind="decode": "abd")
    assert bench.load_traffic("x") is None
    assert bench.load_traffic("missing") is None


def test_decode_kernel_choice(monkeypatch):
    monkeypatch.delenv("PA_DECODE_COOP", raising=False)
    coop, warp = "paged_decode_coop_kernel", "paged_decode_kernel"
    assert bench.decode_kernel_name(W.make_batch("13b", num_seqs=4)) == coop
    assert bench.decode_kernel_name(W.make_batch("13b", num_seqs=4, cache_dtype="fp8")) == coop
    assert bench.decode_kernel_name(W.make_batch("gqa", num_seqs=1, ctx_cap=100)) == coop
    assert bench.decode_kernel_name(W.make_batch("tiny")) == warp                       # head_dim 64
    assert bench.decode_kernel_name(W.make_batch("13b", num_seqs=4, block_size=8)) == warp
    assert bench.decode_kernel_name(W.make_batch("tiny", num_heads=8, num_kv_heads=2)) == warp
    monkeypatch.setenv("PA_DECODE_COOP", "0")
    assert bench.decode_kernel_name(W.make_batch("13b", num_seqs=4)) == warp


def test_end_to_end_entries_report_their_own_time_and_bytes():
    """The direct-call and overlapped end-to-end entries: value = the units of
    one step over that step's own host time, with the step's copies declared."""
    d = bench.e2e_direct_entry(2.0, "GB/s", 0.5, 1, 8_000_000, 2_600_000)
    assert d["value"] == 4000.0 and d["unit"] == "GB/s" and d["ms_per_step"] == 0.5
    assert d["h2d_bytes_per_step"] == 8_000_000 and d["d2h_bytes_per_step"] == 2_600_000
    p = bench.e2e_pipelined_entry(2.0, "GB/s", 0.25, 1, 8_000_000, 2_600_000)
    assert p["value"] == 8000.0 and p["ms_per_step"] == 0.25
    assert p["h2d_bytes_per_step"] == 8_000_000 and p["d2h_bytes_per_step"] == 2_600_000
    assert "overlapping" in p["note"] and "graph" in d["note"]
    t = bench.e2e_pipelined_entry(0.2083835, "TFLOP/s", 0.3, 1, 0, 0)
    assert t["value"] == round(0.2083835 / 0.3e-3, 2)
