"""Child process for tests/test_gpu_coop.py: decodes a seeded batch with the
decode kernel chosen by the environment (PA_DECODE_COOP) and saves the
output's raw bits."""
import os
import sys

import numpy as np

sys.path.insert(0, os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))

from paged_kv_cache_140_gb300 import workloads as W  # noqa: E402
from pa_harness import run_step  # noqa: E402


def main():
    name, hq, hkv, dtype, out_path = sys.argv[1], int(sys.argv[2]), int(sys.argv[3]), sys.argv[4], sys.argv[5]
    b = W.make_batch(name, num_seqs=12, ctx_cap=3000, num_heads=hq, num_kv_heads=hkv, dtype=dtype)
    out, _, flag = run_step(b)
    assert flag == 0
    np.save(out_path, out.cpu().numpy().view(np.uint32))


if __name__ == "__main__":
    main()
