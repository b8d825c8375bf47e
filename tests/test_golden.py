"""The oracle still reproduces the stored tiny-decode values (written by tests/golden/make_golden.py)."""
import json
import os

import numpy as np

import oracle
from gqa_attention_learned_head_gb300 import workloads as W

HERE = os.path.dirname(os.path.abspath(__file__))


def test_oracle_matches_stored_tiny_decode():
    ref = json.load(open(os.path.join(HERE, "golden", "tiny_decode.json")))
    inp = W.tiny_decode()
    out, lse = oracle.decode(inp.q, inp.k_pages, inp.v_pages, inp.page_table, inp.kv_lens, inp.sinks, inp.scale)
    np.testing.assert_allclose(out, np.array(ref["out"]), rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse, np.array(ref["lse"]), rtol=0, atol=1e-12)
