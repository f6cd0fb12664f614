"""Writes tests/golden/tiny_oracle.json from the CPU oracle alone (no CUDA code is
imported). The values are a cross-machine regression record of the oracle on the
tiny case (batch 2, 4 heads, head_dim 64, block_size 16, contexts 37 / 100, a
32-block pool in seeded random order, then a 48-token causal chunk); they are
checked by tests/test_golden.py. Run: python tests/golden/make_golden.py"""
import json
import os
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))

import oracle  # noqa: E402
from paged_kv_flash_cache_gb300 import workloads as W  # noqa: E402


def main():
    dec, pre = W.tiny()
    cache_dec = oracle.build_cache(dec)
    out_d, lse_d = oracle.attention_of(dec, cache_dec, nthreads=1)
    cache_pre = oracle.build_cache(pre)
    rows = [0, 47, 48, 95]
    out_p, lse_p = oracle.attention_of(pre, cache_pre, rows=rows, nthreads=1)
    doc = {
        "what": "CPU oracle outputs for the tiny paged decode + causal prefill case",
        "source": "tests/golden/make_golden.py (calls oracle/ only); inputs from "
                  "paged_kv_flash_cache_gb300.workloads.tiny(seed=1235)",
        "decode_out": out_d.tolist(), "decode_lse": lse_d.tolist(),
        "prefill_rows": rows, "prefill_out": out_p.tolist(), "prefill_lse": lse_p.tolist(),
    }
    with open(os.path.join(HERE, "tiny_oracle.json"), "w") as f:
        json.dump(doc, f, separators=(",", ":"))


if __name__ == "__main__":
    main()
