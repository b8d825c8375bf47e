"""GPU pre-attention prologue (QKV bias + YaRN rotary, k / v into pages) against the fp64 oracle."""
import numpy as np
import pytest
import torch

import oracle
from gqa_attention_learned_head_gb300 import workloads as W
from parity_utils import assert_parity

pytestmark = pytest.mark.gpu

YARN = dict(theta=150000.0, factor=32.0, original_max_position=4096, beta_fast=32.0, beta_slow=1.0)


@pytest.fixture(scope="module")
def S():
    from gqa_attention_learned_head_gb300 import sinkattn

    return sinkattn


def bf16_close(got, ref, what):
    """Rounded once to bf16 from fp32 arithmetic: within 2^-8 relative (+ a tiny absolute floor)."""
    got = np.asarray(got, dtype=np.float64)
    err = np.abs(got - ref)
    bound = np.abs(ref) * 2.0 ** -8 + 1e-6
    assert np.all(err <= bound), f"{what}: worst excess {float((err - bound).max()):.3e}"


def inputs(Hq, Hkv, prefix, new, seed):
    pp = W.make_paged_prefill(Hq, Hkv, prefix, new, seed=seed)
    g = torch.Generator().manual_seed(seed + 1000)
    qkv = torch.randn(pp.q.shape[0], (Hq + 2 * Hkv) * 64, generator=g).to(torch.bfloat16)
    bias = (0.5 * torch.randn((Hq + 2 * Hkv) * 64, generator=g)).to(torch.bfloat16)
    return pp, qkv, bias


def page_rows(pp, tensor_pages):
    """[T, Hkv, 64] read back from the pages at the new tokens' positions."""
    rows = []
    for n, (s0, L) in enumerate(zip(pp.start_pos.tolist(), pp.new_lens)):
        for i in range(L):
            pos = s0 + i
            rows.append(tensor_pages[int(pp.page_table[n, pos // 16]), :, pos % 16])
    return torch.stack(rows)


@pytest.mark.parametrize("interleaved", [False, True])
@pytest.mark.parametrize("Hq,Hkv", [(64, 8), (8, 2)])
def test_prologue_values(S, interleaved, Hq, Hkv):
    pp, qkv, bias = inputs(Hq, Hkv, [0, 130, 100000], [3, 40, 17], seed=Hq + int(interleaved))
    g = pp.to("cuda")
    q = S.sinkattn_qkv_prologue(qkv.cuda(), bias.cuda(), g.cu_seqlens, g.start_pos, g.page_table, g.k_pages,
                                g.v_pages, Hq, interleaved=interleaved, **YARN)
    assert S.sinkattn_get_error() == 0
    rq, rk, rv = oracle.qkv_prologue(qkv, bias, pp.cu_seqlens, pp.start_pos, Hq, Hkv, interleaved=interleaved, **YARN)
    bf16_close(q.float().cpu().numpy(), rq, "q")
    bf16_close(page_rows(pp, g.k_pages.cpu()).float().numpy(), rk, "k")
    bf16_close(page_rows(pp, g.v_pages.cpu()).float().numpy(), rv, "v")


def test_prologue_then_paged_prefill(S):
    """The serving step: prologue (bias, rotary, k/v into pages) then the paged prefill, against the
    oracle's prologue (rounded to bf16 like the device's) and its paged prefill."""
    Hq, Hkv = 64, 8
    pp, qkv, bias = inputs(Hq, Hkv, [300, 5000], [129, 64], seed=91)
    g = pp.to("cuda")
    q = S.sinkattn_qkv_prologue(qkv.cuda(), bias.cuda(), g.cu_seqlens, g.start_pos, g.page_table, g.k_pages,
                                g.v_pages, Hq, **YARN)
    out, lse = S.sinkattn_prefill_paged(q, g.k_pages, g.v_pages, g.page_table, g.cu_seqlens, g.start_pos, g.sinks,
                                        g.scale, max_seqlen=pp.max_seqlen)
    assert S.sinkattn_get_error() == 0
    rq, rk, rv = oracle.qkv_prologue(qkv, bias, pp.cu_seqlens, pp.start_pos, Hq, Hkv, **YARN)
    to_bf16 = lambda a: torch.from_numpy(a).float().to(torch.bfloat16)
    kb, vb = oracle.kv_append(to_bf16(rk), to_bf16(rv), pp.cu_seqlens, pp.start_pos, pp.page_table, pp.k_pages,
                              pp.v_pages)
    ro, rl = oracle.prefill_paged(to_bf16(rq), kb, vb, pp.page_table, pp.cu_seqlens, pp.start_pos, pp.sinks, pp.scale)
    assert_parity(out.float().cpu().numpy(), lse.cpu().numpy(), ro, rl, "prologue + paged prefill")


def test_plain_rope_without_bias(S):
    """factor 1, no bias: plain rotary embedding, attention temperature 1."""
    Hq, Hkv = 8, 2
    pp, qkv, _ = inputs(Hq, Hkv, [7], [50], seed=92)
    g = pp.to("cuda")
    cfg = dict(theta=10000.0, factor=1.0, original_max_position=2048, beta_fast=32.0, beta_slow=1.0)
    q = S.sinkattn_qkv_prologue(qkv.cuda(), None, g.cu_seqlens, g.start_pos, g.page_table, g.k_pages, g.v_pages, Hq,
                                **cfg)
    assert S.sinkattn_get_error() == 0
    rq, _, _ = oracle.qkv_prologue(qkv, torch.zeros(qkv.shape[1], dtype=torch.bfloat16), pp.cu_seqlens,
                                   pp.start_pos, Hq, Hkv, **cfg)
    bf16_close(q.float().cpu().numpy(), rq, "q")


def test_prologue_reports_bad_page_and_still_writes_q(S):
    Hq, Hkv = 8, 2
    pp, qkv, bias = inputs(Hq, Hkv, [16], [5], seed=93)
    g = pp.to("cuda")
    pt = g.page_table.clone()
    pt[0, 1] = pp.k_pages.shape[0] + 2
    before = g.k_pages.clone()
    q = S.sinkattn_qkv_prologue(qkv.cuda(), bias.cuda(), g.cu_seqlens, g.start_pos, pt, g.k_pages, g.v_pages, Hq,
                                **YARN)
    assert S.sinkattn_get_error() == S.ERR_BAD_PAGE
    assert torch.equal(g.k_pages, before)  # nothing written through the bad page id
    rq, _, _ = oracle.qkv_prologue(qkv, bias, pp.cu_seqlens, pp.start_pos, Hq, Hkv, **YARN)
    bf16_close(q.float().cpu().numpy(), rq, "q")
