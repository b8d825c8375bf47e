"""Both tcgen05 prefill kernels, against the fp64 oracle.

The library runs the two-head kernel when the query-head group size is even
and the caller does not ask to share the SMs, and the one-head kernel when the
group size is odd or dims.share_sms = 1.  The default choice is covered by
test_prefill_gpu.py and test_paged_prefill_gpu.py; here share_sms = 1 sends
even groups through the one-head kernel too, causal and not, with ragged
lengths, contiguous and over pages.
"""
import pytest

import oracle
from gqa_attention_learned_head_gb300 import workloads as W
from parity_utils import assert_parity

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def S():
    from gqa_attention_learned_head_gb300 import sinkattn

    return sinkattn


@pytest.mark.parametrize("share_sms", [False, True])
@pytest.mark.parametrize("Hq,Hkv,lens,causal", [(8, 1, [1, 127, 300, 129], True), (16, 2, [200, 5, 1000], False),
                                                (6, 2, [64, 513], True), (64, 8, [777], True)])
def test_contiguous(S, share_sms, Hq, Hkv, lens, causal):
    inp = W.make_prefill(Hq, Hkv, lens, seed=Hq + len(lens), causal=causal)
    g = inp.to("cuda")
    out, lse = S.sinkattn_prefill(g.q, g.k, g.v, g.cu_seqlens, g.sinks, g.scale, g.causal, max_seqlen=inp.max_seqlen,
                                  share_sms=share_sms)
    assert S.sinkattn_get_error() == 0
    ro, rl = oracle.prefill(inp.q, inp.k, inp.v, inp.cu_seqlens, inp.sinks, inp.scale, inp.causal)
    assert_parity(out.float().cpu().numpy(), lse.cpu().numpy(), ro, rl,
                  f"Hq={Hq} Hkv={Hkv} lens={lens} causal={causal} share_sms={share_sms}")


@pytest.mark.parametrize("share_sms", [False, True])
@pytest.mark.parametrize("Hq,Hkv", [(64, 8), (6, 2)])
def test_paged(S, share_sms, Hq, Hkv):
    inp = W.make_paged_prefill(Hq, Hkv, [0, 300, 1000], [40, 129, 300], seed=Hq)
    g = inp.to("cuda")
    S.sinkattn_kv_append(g.k_new, g.v_new, g.cu_seqlens, g.start_pos, g.page_table, g.k_pages, g.v_pages)
    out, lse = S.sinkattn_prefill_paged(g.q, g.k_pages, g.v_pages, g.page_table, g.cu_seqlens, g.start_pos, g.sinks,
                                        g.scale, max_seqlen=inp.max_seqlen, share_sms=share_sms)
    assert S.sinkattn_get_error() == 0
    kb, vb = oracle.kv_append(inp.k_new, inp.v_new, inp.cu_seqlens, inp.start_pos, inp.page_table, inp.k_pages,
                              inp.v_pages)
    ro, rl = oracle.prefill_paged(inp.q, kb, vb, inp.page_table, inp.cu_seqlens, inp.start_pos, inp.sinks, inp.scale)
    assert_parity(out.float().cpu().numpy(), lse.cpu().numpy(), ro, rl, f"paged Hq={Hq} Hkv={Hkv} share_sms={share_sms}")


@pytest.mark.parametrize("share_sms", [False, True])
def test_growing_scores_rescale_o(S, share_sms):
    """Scores that rise along the keys by ~10 (log2 units) per 128-key tile: every row's running max
    passes the lazy-rescale threshold (8) tile after tile, so O is rescaled in tensor memory again and
    again, in both kernels.  q ~ 1 and k ~ r(pos) with r growing linearly to 5, so a row's scores
    span ~40 (natural units) and its lse stays well inside fp32's resolution."""
    import torch

    from gqa_attention_learned_head_gb300.workloads import PrefillInputs

    lens = [700, 300, 129]
    base = W.make_prefill(16, 2, lens, seed=77, causal=True)
    g = torch.Generator().manual_seed(78)
    T = base.q.shape[0]
    pos = torch.cat([torch.arange(L, dtype=torch.float32) for L in lens])
    q = (1.0 + 0.05 * torch.randn(T, 16, 64, generator=g)).to(torch.bfloat16)
    r = (5.0 / 700.0) * pos
    k = (r[:, None, None] + 0.05 * torch.randn(T, 2, 64, generator=g)).to(torch.bfloat16)
    inp = PrefillInputs(q, k, base.v, base.cu_seqlens, base.sinks, base.scale, True, lens)
    d = inp.to("cuda")
    out, lse = S.sinkattn_prefill(d.q, d.k, d.v, d.cu_seqlens, d.sinks, d.scale, True, max_seqlen=inp.max_seqlen,
                                  share_sms=share_sms)
    assert S.sinkattn_get_error() == 0
    ro, rl = oracle.prefill(inp.q, inp.k, inp.v, inp.cu_seqlens, inp.sinks, inp.scale, True)
    # the ramp really does climb past the threshold within a tile: the last row of sequence 0 sees
    # scores from ~0 to ~40 (natural units), ~10 log2 units per 128 keys
    assert float(rl[699].max()) > 35.0
    assert_parity(out.float().cpu().numpy(), lse.cpu().numpy(), ro, rl, f"growing scores share_sms={share_sms}")
