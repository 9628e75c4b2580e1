"""The pages' block-count and KV-size numbers, checked against the formulas."""
import numpy as np
import pytest

from conftest import read_golden
from oracle import accounting


@pytest.mark.parametrize("row", read_golden("block_counts.txt"), ids=lambda r: "-".join(r[0][:2]))
def test_block_counts(row):
    f, cite = row
    n, bs, blocks, empty, fill = map(int, f)
    assert accounting.blocks_needed(n, bs) == blocks, cite
    assert accounting.empty_slots(n, bs) == empty, cite
    assert accounting.last_block_fill(n, bs) == fill, cite


@pytest.mark.parametrize("row", read_golden("kv_bytes.txt"), ids=lambda r: r[0][0])
def test_kv_bytes(row):
    f, cite = row
    layers, hkv, d, nbytes, tokens, seqs = map(int, f[1:7])
    expected, tol = int(f[7]), float(f[8])
    got = accounting.kv_bytes(layers, hkv, d, tokens, nbytes, seqs)
    if tol == 0:
        assert got == expected, cite
    else:
        assert abs(got - expected) <= tol * expected, cite


def test_llama13b_d_model_form():
    # §二 writes the per-token size with d_model = 5120 = 40 heads x 128.
    assert 2 * 40 * 5120 * 2 == accounting.kv_bytes_per_token(40, 40, 128, 2) == 819200
    assert 819200 == 800 * 1024


@pytest.mark.parametrize("row", read_golden("contiguous_waste.txt"), ids=lambda r: r[0][0])
def test_contiguous_reservation(row):
    f, cite = row
    max_len = int(f[0])
    used = [int(x) for x in f[1].split(",")]
    reserved, used_sum, frac = accounting.contiguous_reservation(max_len, used)
    assert reserved == int(f[2]) and used_sum == int(f[3]), cite
    assert round(100 * frac) == int(f[4]), cite


def test_waste_is_below_one_block():
    # Only a sequence's last block may hold unused slots, at most block_size - 1.
    rng = np.random.default_rng(0)
    for bs in (1, 4, 8, 16, 32, 128):
        for n in rng.integers(1, 5000, size=200):
            e = accounting.empty_slots(int(n), bs)
            assert 0 <= e <= bs - 1
            assert accounting.blocks_needed(int(n), bs) * bs == n + e
