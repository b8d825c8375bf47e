"""Writes tiny_decode.json from the fp64 oracle (the only code this script runs)."""
import json
import os
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))

import oracle  # noqa: E402
from gqa_attention_learned_head_gb300 import workloads as W  # noqa: E402

if __name__ == "__main__":
    inp = W.tiny_decode()
    out, lse = oracle.decode(inp.q, inp.k_pages, inp.v_pages, inp.page_table, inp.kv_lens, inp.sinks, inp.scale)
    with open(os.path.join(HERE, "tiny_decode.json"), "w") as f:
        json.dump({"workload": "tiny decode, seed 0", "out": [[[float(x) for x in r] for r in o] for o in out],
                   "lse": [[float(x) for x in r] for r in lse]}, f)
