"""The oracle's thread count changes its speed, never its results (each row is computed by one
thread in a fixed order)."""
import numpy as np

import oracle
from gqa_attention_learned_head_gb300 import workloads as W


def test_one_thread_equals_all_threads():
    inp = W.make_decode(3, 8, 2, [40, 1, 300], seed=5)
    n = oracle.num_threads()
    try:
        oracle.set_num_threads(1)
        assert oracle.num_threads() == 1 or n == 1
        o1, l1 = oracle.decode(inp.q, inp.k_pages, inp.v_pages, inp.page_table, inp.kv_lens, inp.sinks, inp.scale)
    finally:
        oracle.set_num_threads(n)
    assert oracle.num_threads() == n
    on, ln = oracle.decode(inp.q, inp.k_pages, inp.v_pages, inp.page_table, inp.kv_lens, inp.sinks, inp.scale)
    assert np.array_equal(o1, on) and np.array_equal(l1, ln)
