"""A corrupted cu_seqlens through the C ABI: a decreasing entry, a last entry past the token count,
a negative entry.  Every call that takes cu_seqlens (the contiguous prefill, the append, the fused
prologue and the paged prefill) reports SINKATTN_ERR_BAD_LENGTH, reads and writes nothing outside
its buffers, and leaves the sequences the corruption does not reach with their correct results.
The corruption is made on the host; the kernels' own checks turn it into the error."""
import numpy as np
import pytest
import torch

import oracle
from gqa_attention_learned_head_gb300 import workloads as W
from parity_utils import assert_parity

pytestmark = pytest.mark.gpu

LENS = [100, 60, 140, 100]  # cu_seqlens = [0, 100, 160, 300, 400]
PREFIX = [30, 0, 200, 17]


def reported(S, kind):
    """The error word after a call with the corrupted packing.  Every kind sets the bad-length bit; in
    the negative one, tokens of sequence 0 land in sequence 1 past its pages, whose page-table
    entries are -1, so the bad-page bit is set too and is the one returned (the lowest code)."""
    err = S.sinkattn_get_error()
    return err == S.ERR_BAD_LENGTH or (kind == "negative" and err == S.ERR_BAD_PAGE), err


def corrupt(kind, cu):
    """The corrupted packing and the sequences it cannot reach."""
    cu = cu.clone()
    if kind == "decreasing":  # [0, 100, 90, 300, 400]: sequence 1 is negative, 2 overlaps 0 and 1
        cu[2] = 90
        return cu, [3]
    if kind == "past_end":  # [0, 100, 160, 300, 500]: sequence 3 runs past T
        cu[4] = 500
        return cu, [0, 1, 2]
    cu[1] = -5  # [0, -5, 160, 300, 400]: sequences 0 and 1 start or end outside [0, T)
    return cu, [2, 3]


KINDS = ["decreasing", "past_end", "negative"]


@pytest.fixture(scope="module")
def S():
    from gqa_attention_learned_head_gb300 import sinkattn

    return sinkattn


def seq_rows(cu, seqs):
    return np.concatenate([np.arange(int(cu[n]), int(cu[n + 1])) for n in seqs])


@pytest.mark.parametrize("kind", KINDS)
def test_prefill(S, kind):
    inp = W.make_prefill(8, 2, LENS, seed=90)
    g = inp.to("cuda")
    bad, untouched = corrupt(kind, inp.cu_seqlens)
    out, lse = S.sinkattn_prefill(g.q, g.k, g.v, bad.cuda(), g.sinks, g.scale, True, max_seqlen=256)
    assert S.sinkattn_get_error() == S.ERR_BAD_LENGTH
    ro, rl = oracle.prefill(inp.q, inp.k, inp.v, inp.cu_seqlens, inp.sinks, inp.scale, True)
    rows = seq_rows(inp.cu_seqlens, untouched)
    assert_parity(out.float().cpu().numpy()[rows], lse.cpu().numpy()[rows], ro[rows], rl[rows], kind)


def slots(pp, seqs):
    """(page, slot) of every new token of the given sequences."""
    out = []
    for n in seqs:
        for i in range(pp.new_lens[n]):
            pos = int(pp.start_pos[n]) + i
            out.append((int(pp.page_table[n, pos // 16]), pos % 16))
    return out


def bits(t):
    return t.detach().cpu().contiguous().view(torch.int16)


@pytest.mark.parametrize("kind", KINDS)
def test_kv_append_and_paged_prefill(S, kind):
    pp = W.make_paged_prefill(8, 2, PREFIX, LENS, seed=91)
    bad, untouched = corrupt(kind, pp.cu_seqlens)
    # the append with the corrupted packing: error, and the untouched sequences' slots as the oracle's
    g = pp.to("cuda")
    S.sinkattn_kv_append(g.k_new, g.v_new, bad.cuda(), g.start_pos, g.page_table, g.k_pages, g.v_pages)
    ok, err = reported(S, kind)
    assert ok, err
    kb, vb = oracle.kv_append(pp.k_new, pp.v_new, pp.cu_seqlens, pp.start_pos, pp.page_table, pp.k_pages,
                              pp.v_pages)
    kg, vg = bits(g.k_pages), bits(g.v_pages)
    kb, vb = torch.as_tensor(kb.view(np.int16)), torch.as_tensor(vb.view(np.int16))
    for page, slot in slots(pp, untouched):
        assert torch.equal(kg[page, :, slot], kb[page, :, slot]) and torch.equal(vg[page, :, slot], vb[page, :, slot])
    # the paged prefill with the corrupted packing over a correctly appended cache
    g = pp.to("cuda")
    S.sinkattn_kv_append(g.k_new, g.v_new, g.cu_seqlens, g.start_pos, g.page_table, g.k_pages, g.v_pages)
    assert S.sinkattn_get_error() == 0
    out, lse = S.sinkattn_prefill_paged(g.q, g.k_pages, g.v_pages, g.page_table, bad.cuda(), g.start_pos, g.sinks,
                                        g.scale, max_seqlen=256)
    ok, err = reported(S, kind)
    assert ok, err
    kf, vf = oracle.kv_append(pp.k_new, pp.v_new, pp.cu_seqlens, pp.start_pos, pp.page_table, pp.k_pages,
                              pp.v_pages)
    ro, rl = oracle.prefill_paged(pp.q, kf, vf, pp.page_table, pp.cu_seqlens, pp.start_pos, pp.sinks, pp.scale)
    rows = seq_rows(pp.cu_seqlens, untouched)
    assert_parity(out.float().cpu().numpy()[rows], lse.cpu().numpy()[rows], ro[rows], rl[rows], kind)


@pytest.mark.parametrize("kind", KINDS)
def test_qkv_prologue(S, kind):
    """The prologue with the corrupted packing against the same call with the correct one: error, and
    the untouched sequences' q rows and page slots bit for bit the same."""
    pp = W.make_paged_prefill(8, 2, PREFIX, LENS, seed=92)
    gen = torch.Generator().manual_seed(92)
    qkv = torch.randn(pp.q.shape[0], (8 + 2 * 2) * 64, generator=gen).to(torch.bfloat16).cuda()
    bias = (0.5 * torch.randn((8 + 2 * 2) * 64, generator=gen)).to(torch.bfloat16).cuda()
    bad, untouched = corrupt(kind, pp.cu_seqlens)
    yarn = dict(theta=150000.0, factor=32.0, original_max_position=4096, beta_fast=32.0, beta_slow=1.0)
    results = []
    for cu in (pp.cu_seqlens, bad):
        g = pp.to("cuda")
        q = torch.empty_like(g.q)
        S.sinkattn_qkv_prologue(qkv, bias, cu.cuda(), g.start_pos, g.page_table, g.k_pages, g.v_pages, 8, q_out=q,
                                **yarn)
        results.append((reported(S, kind), bits(q), bits(g.k_pages), bits(g.v_pages)))
    ((_, e0), q0, k0, v0), ((ok, e1), q1, k1, v1) = results
    assert e0 == 0 and ok, e1
    rows = torch.as_tensor(seq_rows(pp.cu_seqlens, untouched))
    assert torch.equal(q1[rows], q0[rows])
    for page, slot in slots(pp, untouched):
        assert torch.equal(k1[page, :, slot], k0[page, :, slot]) and torch.equal(v1[page, :, slot], v0[page, :, slot])
