"""Child process for tests/test_gpu_coop.py: decodes a seeded batch with the
decode kernel chosen by the environment (PA_DECODE_COOP) and saves the
output's raw bits.  Arguments: workload (a workload name, "shared" for the
shared-prefix batch of pa_harness, "prefix" for three prompt groups), query
heads, KV heads, dtype, output path, optional partition size."""
import os
import sys

import numpy as np

sys.path.insert(0, os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))

from paged_kv_cache_140_gb300 import workloads as W  # noqa: E402
from pa_harness import run_step, shared_prefix_batch  # noqa: E402


def main():
    name, hq, hkv, dtype, out_path = sys.argv[1], int(sys.argv[2]), int(sys.argv[3]), sys.argv[4], sys.argv[5]
    P = int(sys.argv[6]) if len(sys.argv) > 6 else None
    if name == "shared":      # sequences sharing leading blocks (runs in the cooperative kernel)
        b = shared_prefix_batch(num_heads=hq, num_kv_heads=hkv, dtype=dtype)
    elif name == "prefix":
        b = W.make_batch("prefix", groups=3, num_heads=hq, num_kv_heads=hkv, dtype=dtype)
    else:
        b = W.make_batch(name, num_seqs=12, ctx_cap=3000, num_heads=hq, num_kv_heads=hkv, dtype=dtype)
    out, _, flag = run_step(b, partition_size=P)
    assert flag == 0
    np.save(out_path, out.cpu().numpy().view(np.uint32))


if __name__ == "__main__":
    main()
