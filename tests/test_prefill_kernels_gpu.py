"""Every prefill kernel the library can select, against the fp64 oracle.

The library picks its prefill kernel once per process: the two-head tcgen05
kernel when the query-head group size is even, the one-head tcgen05 kernel
otherwise; SINKATTN_PREFILL_KERNEL=tc forces the one-head kernel and =mma the
warp-level mma.sync kernel.  The default choice is covered by
test_prefill_gpu.py; here each forced choice runs in a child process of its
own, on even and odd groups, causal and not, with ragged lengths.
"""
import os
import subprocess
import sys
from pathlib import Path

import pytest

pytestmark = pytest.mark.gpu

ROOT = Path(__file__).resolve().parents[1]

CHILD = r"""
import sys
sys.path.insert(0, sys.argv[1]); sys.path.insert(0, sys.argv[1] + "/tests")
import oracle
from gqa_attention_learned_head_gb300 import sinkattn as S, workloads as W
from parity_utils import assert_parity
cases = [(8, 1, [1, 127, 300, 129], True), (16, 2, [200, 5, 1000], False), (6, 2, [64, 513], True),
         (64, 8, [777], True)]
for Hq, Hkv, lens, causal in cases:
    inp = W.make_prefill(Hq, Hkv, lens, seed=Hq + len(lens), causal=causal)
    g = inp.to("cuda")
    out, lse = S.sinkattn_prefill(g.q, g.k, g.v, g.cu_seqlens, g.sinks, g.scale, g.causal, max_seqlen=inp.max_seqlen)
    assert S.sinkattn_get_error() == 0
    ro, rl = oracle.prefill(inp.q, inp.k, inp.v, inp.cu_seqlens, inp.sinks, inp.scale, inp.causal)
    assert_parity(out.float().cpu().numpy(), lse.cpu().numpy(), ro, rl, f"Hq={Hq} Hkv={Hkv} lens={lens} causal={causal}")
# the chunked prefill over pages (the mma.sync choice falls back to the one-head tcgen05 kernel there)
for Hq, Hkv in ((64, 8), (6, 2)):
    inp = W.make_paged_prefill(Hq, Hkv, [0, 300, 1000], [40, 129, 300], seed=Hq)
    g = inp.to("cuda")
    S.sinkattn_kv_append(g.k_new, g.v_new, g.cu_seqlens, g.start_pos, g.page_table, g.k_pages, g.v_pages)
    out, lse = S.sinkattn_prefill_paged(g.q, g.k_pages, g.v_pages, g.page_table, g.cu_seqlens, g.start_pos, g.sinks,
                                        g.scale, max_seqlen=inp.max_seqlen)
    assert S.sinkattn_get_error() == 0
    kb, vb = oracle.kv_append(inp.k_new, inp.v_new, inp.cu_seqlens, inp.start_pos, inp.page_table, inp.k_pages,
                              inp.v_pages)
    ro, rl = oracle.prefill_paged(inp.q, kb, vb, inp.page_table, inp.cu_seqlens, inp.start_pos, inp.sinks, inp.scale)
    assert_parity(out.float().cpu().numpy(), lse.cpu().numpy(), ro, rl, f"paged Hq={Hq} Hkv={Hkv}")
print("ok")
"""


@pytest.mark.parametrize("kernel", ["tc", "mma"])
def test_forced_prefill_kernel(kernel):
    env = dict(os.environ, SINKATTN_PREFILL_KERNEL=kernel)
    r = subprocess.run([sys.executable, "-c", CHILD, str(ROOT)], env=env, capture_output=True, text=True,
                       timeout=600)
    assert r.returncode == 0 and r.stdout.strip().endswith("ok"), r.stdout[-2000:] + r.stderr[-4000:]
