"""sinkattn_decode_noalloc: the decode for callers that cannot allocate.

Callers such as a framework that owns the whole device through its own
memory pool, a plugin interface that hands over only input and output
buffers, or a serving loop that must not pay cudaMalloc's device
synchronisation, use this entry point; it takes its split-KV scratch from a
fixed array inside the library instead of a caller workspace.  This test
calls it through the C ABI twice in a row, on two different problems (so the
second call runs on scratch the first one left behind), and checks each
result against the regular sinkattn_decode with the parity tolerances used
everywhere else.  The file is named to be collected last.
"""
import numpy as np
import pytest
import torch

from gqa_attention_learned_head_gb300 import workloads as W
from parity_utils import assert_parity

pytestmark = pytest.mark.gpu


def _regular(S, g):
    out, lse = S.sinkattn_decode(g.q, g.k_pages, g.v_pages, g.page_table, g.kv_lens, g.sinks, g.scale)
    return out, lse


def test_noalloc_decode_matches_regular_decode_on_two_calls_in_a_row():
    from gqa_attention_learned_head_gb300 import sinkattn as S

    problems = [W.make_decode(32, 64, 8, (512, 4096), seed=21).to("cuda"),
                W.make_decode(6, 16, 2, [0, 1, 17, 300, 5000, 20000], seed=22).to("cuda")]
    results = []
    for g in problems:  # two calls in a row on the shared scratch
        assert S.sinkattn_decode_workspace_size(g.q, g.k_pages, g.page_table) <= S.NOALLOC_SCRATCH_BYTES
        out = torch.empty_like(g.q)
        lse = torch.empty(g.q.shape[:2], dtype=torch.float32, device="cuda")
        S.sinkattn_decode_noalloc(g.q, g.k_pages, g.v_pages, g.page_table, g.kv_lens, g.sinks, g.scale, out, lse)
        results.append((out, lse))
    assert S.sinkattn_get_error() == 0
    for g, (out, lse) in zip(problems, results):
        ro, rl = _regular(S, g)
        assert S.sinkattn_get_error() == 0
        assert_parity(out.float().cpu().numpy(), lse.cpu().numpy(), ro.float().cpu().numpy(), rl.cpu().numpy(),
                      "no-alloc decode vs sinkattn_decode")


def test_noalloc_decode_allocates_nothing():
    """After a warm-up call (which loads the kernels and looks up the scratch array), a call through
    the binding and the C ABI changes neither the caching allocator's count of allocations nor the
    device's free memory."""
    from gqa_attention_learned_head_gb300 import sinkattn as S

    g = W.make_decode(16, 64, 8, (300, 3000), seed=24).to("cuda")
    out = torch.empty_like(g.q)
    lse = torch.empty(g.q.shape[:2], dtype=torch.float32, device="cuda")
    S.sinkattn_decode_noalloc(g.q, g.k_pages, g.v_pages, g.page_table, g.kv_lens, g.sinks, g.scale, out, lse)
    torch.cuda.synchronize()
    allocs = torch.cuda.memory_stats()["allocation.all.allocated"]
    free0, _ = torch.cuda.mem_get_info()
    for _ in range(3):
        S.sinkattn_decode_noalloc(g.q, g.k_pages, g.v_pages, g.page_table, g.kv_lens, g.sinks, g.scale, out, lse)
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    assert torch.cuda.memory_stats()["allocation.all.allocated"] == allocs
    assert free1 == free0
    assert S.sinkattn_get_error() == 0


def test_noalloc_decode_rejects_problems_above_the_scratch_limit():
    from gqa_attention_learned_head_gb300 import sinkattn as S

    g = W.make_decode(32768, 16, 1, [1] * 32768, seed=23).to("cuda")  # needs far more than 16 MiB
    assert S.sinkattn_decode_workspace_size(g.q, g.k_pages, g.page_table) > S.NOALLOC_SCRATCH_BYTES
    out = torch.full_like(g.q, 7.0)
    with pytest.raises(S.SinkAttnError) as e:
        S.sinkattn_decode_noalloc(g.q, g.k_pages, g.v_pages, g.page_table, g.kv_lens, g.sinks, g.scale, out)
    assert e.value.status == S.ERR_WORKSPACE
    torch.cuda.synchronize()
    assert bool((out == 7.0).all())  # nothing was launched
