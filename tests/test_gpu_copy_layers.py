"""pa_copy_blocks_layers: copy-on-write pairs applied to every layer of a
per-model cache [layers, 2, NB, bs, Hkv, D] in one launch, bit-exact against
the oracle."""
import numpy as np
import pytest

import oracle

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def torch():
    t = pytest.importorskip("torch")
    if not t.cuda.is_available():
        pytest.skip("no CUDA device")
    import paged_kv_cache_140_gb300._build as b
    b.build()
    return t


@pytest.mark.parametrize("layers,dtype", [(1, "bf16"), (4, "f16"), (40, "bf16"), (3, "fp8")])
def test_copy_blocks_layers_bit_exact(torch, layers, dtype):
    import paged_kv_cache_140_gb300 as pa
    rng = np.random.default_rng(layers)
    NB, bs, Hkv, D = 64, 16, 8, 128
    if dtype == "fp8":
        host = rng.integers(0, 256, size=(layers, 2, NB, bs, Hkv, D), dtype=np.uint8)
        dev = torch.from_numpy(host).cuda()
    else:
        host = rng.integers(0, 2**16, size=(layers, 2, NB, bs, Hkv, D), dtype=np.uint16)
        tdt = torch.float16 if dtype == "f16" else torch.bfloat16
        dev = torch.from_numpy(host.view(np.int16)).view(tdt).cuda()
    perm = rng.permutation(NB)
    pairs = np.stack([perm[:12], perm[12:24]], 1).astype(np.int64)
    err = pa.new_err_flag()
    pa.copy_blocks_layers(dev, torch.from_numpy(pairs).cuda(), err_flag=err)
    torch.cuda.synchronize()
    assert pa.read_err_flag(err) == 0
    want, bad = oracle.copy_blocks_layers(host, pairs)
    assert bad == 0
    got = dev.cpu().view(torch.uint8).numpy() if dtype == "fp8" else dev.cpu().view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(got, want)


def test_copy_blocks_layers_bad_pair_is_flagged(torch):
    import paged_kv_cache_140_gb300 as pa
    rng = np.random.default_rng(7)
    host = rng.integers(0, 2**16, size=(2, 2, 16, 16, 4, 64), dtype=np.uint16)
    dev = torch.from_numpy(host.view(np.int16)).view(torch.bfloat16).cuda()
    pairs = np.array([[1, 2], [3, 99]], dtype=np.int64)
    err = pa.new_err_flag()
    pa.copy_blocks_layers(dev, torch.from_numpy(pairs).cuda(), err_flag=err)
    torch.cuda.synchronize()
    assert pa.read_err_flag(err) & pa.FLAG_BAD_COPY_PAIR
    want, _ = oracle.copy_blocks_layers(host, pairs)
    assert np.array_equal(dev.cpu().view(torch.int16).numpy().view(np.uint16), want)
