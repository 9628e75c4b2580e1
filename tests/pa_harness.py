"""Helpers shared by the GPU tests: move a workloads.Batch to the device, run
the decode step through the library, and compare with the CPU oracle."""
from __future__ import annotations

import numpy as np

import paged_kv_cache_140_gb300 as pa

OUT_F32 = "f32"
ATOL = 2e-3   # max-abs bound for attention outputs (fp32 accumulate, half inputs)


def torch_dtype(name):
    import torch
    return {"f16": torch.float16, "bf16": torch.bfloat16, "f32": torch.float32}[name]


def half_tensor(bits: np.ndarray, dtype: str, device="cuda"):
    import torch
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch_dtype(dtype)).to(device)


def cache_tensor(b, bits, device="cuda"):
    """The cache as a device tensor: 16-bit values, or e4m3 codes as uint8."""
    import torch
    if b.cache_dtype == "fp8":
        return torch.from_numpy(np.ascontiguousarray(bits)).to(device)
    return half_tensor(bits, b.cache_dtype, device)


def to_device(b, device="cuda"):
    import torch
    return dict(
        q=half_tensor(b.q, b.dtype, device),
        k_cache=cache_tensor(b, b.k_cache, device),
        v_cache=cache_tensor(b, b.v_cache, device),
        key=half_tensor(b.key, b.dtype, device),
        value=half_tensor(b.value, b.dtype, device),
        slot_mapping=torch.from_numpy(b.slot_mapping).to(device),
        block_tables=torch.from_numpy(b.block_tables).to(device),
        context_lens=torch.from_numpy(b.context_lens).to(device),
        block_mapping=torch.from_numpy(np.ascontiguousarray(b.block_mapping)).to(device),
    )


def run_step(b, out_dtype=OUT_F32, partition_size=None, dev=None, device="cuda"):
    """copy_blocks -> reshape_and_cache -> decode on the GPU.

    Returns (out tensor, device tensors dict, err_flag bits)."""
    import torch
    T = dev if dev is not None else to_device(b, device)
    err = pa.new_err_flag(device)
    if len(b.block_mapping):
        pa.copy_blocks(T["k_cache"], T["v_cache"], T["block_mapping"], err_flag=err)
    pa.reshape_and_cache(T["key"], T["value"], T["k_cache"], T["v_cache"], T["slot_mapping"], err_flag=err,
                         k_scale=b.k_scale, v_scale=b.v_scale)
    out = torch.empty(T["q"].shape, dtype=torch_dtype(out_dtype if out_dtype != "native" else b.dtype),
                      device=device)
    P = b.partition_size if partition_size is None else partition_size
    pa.decode(out, T["q"], T["k_cache"], T["v_cache"], T["block_tables"], T["context_lens"],
              float(b.scale), max_context_len=b.max_context_len, partition_size=P, err_flag=err,
              k_scale=b.k_scale, v_scale=b.v_scale)
    torch.cuda.synchronize()
    return out, T, pa.read_err_flag(err)


def ulp(x: np.ndarray, dtype: str) -> np.ndarray:
    """Spacing of the half format at |x| (normal range; subnormal floor)."""
    mant, emin = {"f16": (10, -14), "bf16": (7, -126)}[dtype]
    a = np.maximum(np.abs(x), 2.0 ** emin)
    e = np.floor(np.log2(a))
    return 2.0 ** (e - mant)


def assert_attention_close(out, ref: np.ndarray, out_dtype: str, what: str = "") -> float:
    """|gpu - oracle| <= 2e-3 (+1 ulp of the output format for half outputs)."""
    g = out.float().cpu().numpy().astype(np.float64)
    assert g.shape == ref.shape
    assert np.all(np.isfinite(g)), f"{what}: non-finite GPU output"
    err = np.abs(g - ref)
    tol = ATOL + (0.0 if out_dtype in ("f32", OUT_F32) else ulp(ref, out_dtype))
    bad = err > tol
    if bad.any():
        i = np.unravel_index(np.argmax(err - tol), err.shape)
        raise AssertionError(f"{what}: {int(bad.sum())} elements over tolerance; worst at {i}: "
                             f"gpu {g[i]!r} oracle {ref[i]!r} err {err[i]:.3e} tol {np.broadcast_to(tol, err.shape)[i]:.3e}")
    return float(err.max()) if err.size else 0.0


def cache_bits(t) -> np.ndarray:
    import torch
    if t.element_size() == 1:
        return t.cpu().view(torch.uint8).numpy()
    return t.cpu().view(torch.int16).numpy().view(np.uint16)


def share_prefixes(b, chains):
    """Make sequences read the physical blocks of another: for each
    (head, members, blocks) in ``chains``, every member's first ``blocks``
    table entries become the head's (at most the member's block count and the
    head's blocks before its last, which hold only the head's history rows).  A
    sequence whose new-token slot then lies in a block another sequence also
    reads gets slot -1 (no write), so that the step writes only private
    blocks.  Modifies ``b`` in place and returns it."""
    bs = b.block_size
    for head, members, nblk in chains:
        for s in members:
            # only the head's full history blocks (positions it has written)
            n = min(int(nblk), -(-int(b.context_lens[s]) // bs), (int(b.context_lens[head]) - 1) // bs)
            b.block_tables[s, :n] = b.block_tables[head, :n]
    readers = {}
    for s in range(b.num_seqs):
        for blk in b.block_tables[s, : -(-int(b.context_lens[s]) // bs)]:
            readers[int(blk)] = readers.get(int(blk), 0) + 1
    with_token = np.nonzero(b.context_lens > 0)[0]
    slots = []
    for s in with_token:
        last = int(b.context_lens[s]) - 1
        blk = int(b.block_tables[s, last // bs])
        slots.append(-1 if readers[blk] > 1 else blk * bs + last % bs)
    b.slot_mapping = np.asarray(slots, dtype=np.int64)
    return b


SHARED_CHAINS = [   # (head, members, shared blocks): chains of 4 and 6 (longer than one run), two
    # sequences equal but for their last block, members ending inside the shared blocks
    (0, [1, 2, 3], 40),
    (4, [5, 6, 7, 8, 9], 12),
    (10, [11], 124),
]


def shared_prefix_batch(name="7b", **kw):
    """A 14-sequence batch whose sequences share leading blocks in the
    chains of SHARED_CHAINS, with contexts that end before, inside and after
    the shared blocks."""
    from paged_kv_cache_140_gb300 import workloads as W
    ctx = [1500, 900, 1500, 700, 300, 250, 190, 192, 600, 193, 2000, 2000, 64, 0]
    b = W.make_batch(name, context_lens=ctx, **kw)
    return share_prefixes(b, SHARED_CHAINS)
