"""A stalled pipeline stage is reported, not hung on: the bounded-wait failure path run on purpose
without a fault (one thread waiting on an mbarrier that nothing completes), after which the
context is still usable."""
import time

import pytest

import oracle
from gqa_attention_learned_head_gb300 import workloads as W
from parity_utils import assert_parity

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def S():
    from gqa_attention_learned_head_gb300 import sinkattn

    return sinkattn


def test_bounded_wait_reports_timeout_and_context_survives(S):
    assert S.sinkattn_get_error() == 0
    t0 = time.time()
    S.sinkattn_selftest_wait_timeout()
    assert S.sinkattn_get_error() == S.ERR_TIMEOUT  # synchronises: the wait gave up and the kernel returned
    waited = time.time() - t0
    assert waited < 60.0, f"the bounded wait took {waited:.1f} s"
    assert S.sinkattn_get_error() == 0  # read and cleared
    inp = W.tiny_decode()
    g = inp.to("cuda")
    out, lse = S.sinkattn_decode(g.q, g.k_pages, g.v_pages, g.page_table, g.kv_lens, g.sinks, g.scale)
    assert S.sinkattn_get_error() == 0
    ro, rl = oracle.decode(inp.q, inp.k_pages, inp.v_pages, inp.page_table, inp.kv_lens, inp.sinks, inp.scale)
    assert_parity(out.float().cpu().numpy(), lse.cpu().numpy(), ro, rl, "decode after a timed-out wait")
