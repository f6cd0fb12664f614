"""The oracle reproduces its recorded outputs on the tiny case (x86 and Arm builds agree)."""
import json
import os

import numpy as np

import oracle
from paged_kv_flash_cache_gb300 import workloads as W

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden", "tiny_oracle.json")


def test_tiny_oracle_matches_record():
    doc = json.load(open(GOLDEN))
    dec, pre = W.tiny()
    out_d, lse_d = oracle.attention_of(dec, oracle.build_cache(dec), nthreads=2)
    np.testing.assert_allclose(out_d, np.array(doc["decode_out"]), rtol=1e-13, atol=1e-15)
    np.testing.assert_allclose(lse_d, np.array(doc["decode_lse"]), rtol=1e-13)
    out_p, lse_p = oracle.attention_of(pre, oracle.build_cache(pre), rows=doc["prefill_rows"], nthreads=2)
    np.testing.assert_allclose(out_p, np.array(doc["prefill_out"]), rtol=1e-13, atol=1e-15)
    np.testing.assert_allclose(lse_p, np.array(doc["prefill_lse"]), rtol=1e-13)
