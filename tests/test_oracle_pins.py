"""Pins of the fp64 oracle to facts that do not come from the oracle itself.

The blog posts that define the method ("GPT-OSS on day 0", section "Kernels
for GPT-OSS / Sink Attention") print no worked example: their equations were
lost.  What they fix in prose -- a per-head sink logit inside the softmax
normaliser with no value row, the online state seeded from the sink, and the
sink held by the first chunk only when the sequence is split -- is pinned
here through library routines, closed forms, invariants and special cases:

* sink = -inf reduces to ordinary attention: torch's fp64 SDPA;
* any sink equals SDPA over the keys plus one zero key whose logit is the
  sink (additive mask) and whose value row is zero;
* a single key has the closed form e^s / (e^s + e^sink) * v;
* a huge sink drives out to 0 and lse to the sink;
* constant V gives out = c * (1 - e^(sink - lse));
* one-hot V exposes the weights: ratios e^(s_j - s_k), mass 1 with the sink;
* split + merge equals unsplit for both sink routes, and the wrong rule
  (every chunk seeded) is caught;
* permuting the page pool with the page table changes nothing;
* prefill row i equals decode over keys 0..i; GQA equals explicit head repeat.
"""
import math

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle
from gqa_attention_learned_head_gb300 import workloads as W

TOL = 1e-12


def bf16(x):
    return torch.as_tensor(x, dtype=torch.float32).to(torch.bfloat16)


def gather_kv(inp, b, kvh):
    """Contiguous K, V rows [len, D] (float64) of request b, KV head kvh."""
    L = int(inp.kv_lens[b])
    t = torch.arange(L)
    pages = inp.page_table[b, t // W.PAGE_SIZE].long()
    k = inp.k_pages[pages, kvh, t % W.PAGE_SIZE].double()
    v = inp.v_pages[pages, kvh, t % W.PAGE_SIZE].double()
    return k, v


def sdpa_with_sink(q, k, v, sink, scale, causal=False):
    """torch SDPA (fp64) with the sink modelled as an extra zero key of logit `sink` and zero value.

    q [H, Lq, D], k/v [H, Lk, D]; sink [H].  causal aligns query i with key i.
    """
    H, Lq, D = q.shape
    Lk = k.shape[1]
    k1 = torch.cat([k, torch.zeros(H, 1, D, dtype=k.dtype)], 1)
    v1 = torch.cat([v, torch.zeros(H, 1, D, dtype=v.dtype)], 1)
    mask = torch.zeros(H, Lq, Lk + 1, dtype=torch.float64)
    if causal:
        mask[:, :, :Lk] = torch.triu(torch.full((Lq, Lk), float("-inf"), dtype=torch.float64), 1)
    mask[:, :, Lk] = torch.as_tensor(sink, dtype=torch.float64)[:, None]
    return F.scaled_dot_product_attention(q[None], k1[None], v1[None], attn_mask=mask[None],
                                          scale=scale)[0]


# ----------------------------------------------------------------------------------------
# decode against library SDPA


@pytest.mark.parametrize("Hq,Hkv", [(4, 1), (8, 2), (16, 2)])
def test_decode_minus_inf_sink_is_plain_attention(Hq, Hkv):
    inp = W.make_decode(3, Hq, Hkv, [1, 37, 64], seed=1)
    inp.sinks[:] = float("-inf")
    out, lse = oracle.decode(inp.q, inp.k_pages, inp.v_pages, inp.page_table, inp.kv_lens,
                             inp.sinks, inp.scale)
    G = Hq // Hkv
    for b in range(3):
        for kvh in range(Hkv):
            k, v = gather_kv(inp, b, kvh)
            q = inp.q[b, kvh * G:(kvh + 1) * G].double()[:, None]  # [G,1,D]
            ref = F.scaled_dot_product_attention(q, k.expand(G, -1, -1), v.expand(G, -1, -1),
                                                 scale=inp.scale)[:, 0]
            np.testing.assert_allclose(out[b, kvh * G:(kvh + 1) * G], ref.numpy(), rtol=0, atol=TOL)
            # lse of plain attention: log-sum-exp of the scaled scores (torch routine)
            s = inp.scale * (q[:, 0] @ k.T)
            np.testing.assert_allclose(lse[b, kvh * G:(kvh + 1) * G],
                                       torch.logsumexp(s, -1).numpy(), rtol=0, atol=TOL)


@pytest.mark.parametrize("sink_std", [0.5, 3.0])
def test_decode_sink_equals_sdpa_with_zero_value_key(sink_std):
    inp = W.make_decode(4, 8, 2, [5, 16, 17, 90], seed=2, sink_std=sink_std)
    out, _ = oracle.decode(inp.q, inp.k_pages, inp.v_pages, inp.page_table, inp.kv_lens,
                           inp.sinks, inp.scale)
    for b in range(4):
        for kvh in range(2):
            k, v = gather_kv(inp, b, kvh)
            q = inp.q[b, kvh * 4:(kvh + 1) * 4].double()[:, None]
            ref = sdpa_with_sink(q, k.expand(4, -1, -1), v.expand(4, -1, -1),
                                 inp.sinks[kvh * 4:(kvh + 1) * 4], inp.scale)[:, 0]
            np.testing.assert_allclose(out[b, kvh * 4:(kvh + 1) * 4], ref.numpy(), rtol=0, atol=TOL)


# ----------------------------------------------------------------------------------------
# closed forms and limits


def test_single_key_closed_form():
    inp = W.make_decode(1, 4, 1, [1], seed=3)
    out, lse = oracle.decode(inp.q, inp.k_pages, inp.v_pages, inp.page_table, inp.kv_lens,
                             inp.sinks, inp.scale)
    k, v = gather_kv(inp, 0, 0)
    for h in range(4):
        s = inp.scale * float(inp.q[0, h].double() @ k[0])
        sig = float(inp.sinks[h])
        w = math.exp(s) / (math.exp(s) + math.exp(sig))
        np.testing.assert_allclose(out[0, h], w * v[0].numpy(), rtol=0, atol=TOL)
        assert abs(lse[0, h] - math.log(math.exp(s) + math.exp(sig))) < TOL


def test_huge_sink_takes_all_mass():
    inp = W.make_decode(2, 4, 1, [3, 40], seed=4)
    inp.sinks[:] = 1.0e4
    out, lse = oracle.decode(inp.q, inp.k_pages, inp.v_pages, inp.page_table, inp.kv_lens,
                             inp.sinks, inp.scale)
    assert np.all(out == 0.0)
    assert np.all(lse == 1.0e4)


def test_growing_sink_shrinks_output():
    inp = W.make_decode(1, 4, 1, [50], seed=5)
    norms = []
    for sig in [-5.0, 0.0, 5.0, 10.0, 20.0, 40.0]:
        inp.sinks[:] = sig
        out, _ = oracle.decode(inp.q, inp.k_pages, inp.v_pages, inp.page_table, inp.kv_lens,
                               inp.sinks, inp.scale)
        norms.append(np.abs(out).max())
    assert all(a > b for a, b in zip(norms, norms[1:]))
    assert norms[-1] < 1e-12


def test_empty_cache_puts_all_mass_on_sink():
    inp = W.make_decode(2, 4, 1, [0, 0], seed=6)
    inp.sinks[2] = float("-inf")
    out, lse = oracle.decode(inp.q, inp.k_pages, inp.v_pages, inp.page_table, inp.kv_lens,
                             inp.sinks, inp.scale)
    assert np.all(out == 0.0)
    for h in range(4):
        assert lse[0, h] == float(inp.sinks[h])
    assert lse[1, 2] == float("-inf")


def test_constant_values():
    inp = W.make_decode(2, 8, 2, [7, 33], seed=7)
    c = 1.5
    inp.v_pages[:] = c
    out, lse = oracle.decode(inp.q, inp.k_pages, inp.v_pages, inp.page_table, inp.kv_lens,
                             inp.sinks, inp.scale)
    mass = 1.0 - np.exp(inp.sinks.double().numpy()[None, :] - lse)  # [B, Hq]
    np.testing.assert_allclose(out, c * mass[..., None] * np.ones(64), rtol=0, atol=TOL)


def test_one_hot_values_expose_weights():
    L = 48
    inp = W.make_decode(1, 4, 1, [L], seed=8, contiguous=True)
    pages = inp.page_table[0, :3].long()
    eye = torch.eye(64)[:L].reshape(3, W.PAGE_SIZE, 64)
    inp.v_pages[pages, 0] = eye.to(torch.bfloat16)
    out, lse = oracle.decode(inp.q, inp.k_pages, inp.v_pages, inp.page_table, inp.kv_lens,
                             inp.sinks, inp.scale)
    k, _ = gather_kv(inp, 0, 0)
    for h in range(4):
        s = inp.scale * (k @ inp.q[0, h].double()).numpy()
        w = out[0, h, :L]
        assert np.all(out[0, h, L:] == 0)
        # weights are the exponentials of the scores (ratio e^(s_j - s_0)) ...
        np.testing.assert_allclose(w / w[0], np.exp(s - s[0]), rtol=1e-12)
        # ... and, together with the sink's share, sum to one
        assert abs(w.sum() + math.exp(float(inp.sinks[h]) - lse[0, h]) - 1.0) < 1e-12


# ----------------------------------------------------------------------------------------
# split-KV + merge


@pytest.mark.parametrize("S", [1, 2, 7, 32])
def test_split_then_merge_equals_unsplit(S):
    lens = [0, 1, 15, 16, 17, 300, 511]
    inp = W.make_decode(len(lens), 8, 2, lens, seed=9)
    chunk = max(1, -(-max(lens) // S))
    ref_o, ref_l = oracle.decode(inp.q, inp.k_pages, inp.v_pages, inp.page_table, inp.kv_lens,
                                 inp.sinks, inp.scale)
    args = (inp.q, inp.k_pages, inp.v_pages, inp.page_table, inp.kv_lens, inp.sinks, inp.scale,
            S, chunk)
    # the page's rule: the first chunk holds the sink, the merge does not add it
    po, pl = oracle.decode_partials(*args, sink_mode=oracle.SINK_IN_FIRST_CHUNK)
    o, l = oracle.merge(po, pl)
    np.testing.assert_allclose(o, ref_o, rtol=0, atol=TOL)
    np.testing.assert_allclose(l, ref_l, rtol=0, atol=TOL)
    # the equivalent route: no chunk holds it, the merge adds it once
    po, pl = oracle.decode_partials(*args, sink_mode=oracle.SINK_IN_NO_CHUNK)
    o, l = oracle.merge(po, pl, inp.sinks)
    np.testing.assert_allclose(o, ref_o, rtol=0, atol=TOL)
    np.testing.assert_allclose(l, ref_l, rtol=0, atol=TOL)


def test_seeding_every_chunk_is_detected():
    """Planting the wrong rule (sink in every chunk) must break split == unsplit."""
    inp = W.make_decode(2, 4, 1, [100, 64], seed=10)
    ref_o, ref_l = oracle.decode(inp.q, inp.k_pages, inp.v_pages, inp.page_table, inp.kv_lens,
                                 inp.sinks, inp.scale)
    po, pl = oracle.decode_partials(inp.q, inp.k_pages, inp.v_pages, inp.page_table, inp.kv_lens,
                                    inp.sinks, inp.scale, 4, 25,
                                    sink_mode=oracle.SINK_IN_EVERY_CHUNK)
    o, l = oracle.merge(po, pl)
    assert np.abs(l - ref_l).max() > 1e-3
    assert np.abs(o - ref_o).max() > 1e-3


def test_merge_edge_rows():
    po = np.zeros((3, 2, 1, 4))
    pl = np.full((3, 2, 1), -np.inf)
    po[1, 1, 0] = [1, 2, 3, 4]
    pl[1, 1, 0] = 0.25
    o, l = oracle.merge(po, pl)
    assert np.all(o[0] == 0) and l[0, 0] == -np.inf          # nothing at all
    np.testing.assert_array_equal(o[1, 0], [1, 2, 3, 4])      # one live partial passes through
    assert l[1, 0] == 0.25
    o, l = oracle.merge(po, pl, np.array([0.25], np.float32))  # sink equal to the live lse
    np.testing.assert_allclose(o[1, 0], [0.5, 1, 1.5, 2], rtol=0, atol=TOL)
    assert abs(l[1, 0] - (0.25 + math.log(2))) < TOL
    assert np.all(o[0] == 0) and l[0, 0] == 0.25


# ----------------------------------------------------------------------------------------
# paging, GQA, prefill


def test_page_permutation_invariance():
    inp = W.make_decode(3, 8, 2, [40, 17, 64], seed=11)
    out, lse = oracle.decode(inp.q, inp.k_pages, inp.v_pages, inp.page_table, inp.kv_lens,
                             inp.sinks, inp.scale)
    P = inp.k_pages.shape[0]
    perm = torch.randperm(P, generator=torch.Generator().manual_seed(5))
    inv = torch.empty_like(perm)
    inv[perm] = torch.arange(P)
    pt = inp.page_table.clone()
    pt[pt >= 0] = inv[pt[pt >= 0].long()].int()
    out2, lse2 = oracle.decode(inp.q, inp.k_pages[perm], inp.v_pages[perm], pt, inp.kv_lens,
                               inp.sinks, inp.scale)
    np.testing.assert_array_equal(out, out2)
    np.testing.assert_array_equal(lse, lse2)


def test_bad_page_id_is_reported():
    inp = W.make_decode(1, 4, 1, [20], seed=12)
    inp.page_table[0, 1] = 99
    with pytest.raises(IndexError):
        oracle.decode(inp.q, inp.k_pages, inp.v_pages, inp.page_table, inp.kv_lens, inp.sinks,
                      inp.scale)


def test_gqa_equals_explicit_head_repeat():
    inp = W.make_decode(2, 8, 2, [30, 45], seed=13)
    out, lse = oracle.decode(inp.q, inp.k_pages, inp.v_pages, inp.page_table, inp.kv_lens,
                             inp.sinks, inp.scale)
    rep = W.DecodeInputs(inp.q, inp.k_pages.repeat_interleave(4, 1),
                         inp.v_pages.repeat_interleave(4, 1), inp.page_table, inp.kv_lens,
                         inp.sinks, inp.scale)
    out2, lse2 = oracle.decode(rep.q, rep.k_pages, rep.v_pages, rep.page_table, rep.kv_lens,
                               rep.sinks, rep.scale)
    np.testing.assert_array_equal(out, out2)
    np.testing.assert_array_equal(lse, lse2)


@pytest.mark.parametrize("causal", [True, False])
def test_prefill_against_sdpa(causal):
    inp = W.make_prefill(8, 2, [1, 37, 130], seed=14, causal=causal)
    out, lse = oracle.prefill(inp.q, inp.k, inp.v, inp.cu_seqlens, inp.sinks, inp.scale, causal)
    cu = inp.cu_seqlens.tolist()
    for n in range(3):
        a, b = cu[n], cu[n + 1]
        q = inp.q[a:b].double().transpose(0, 1)                       # [Hq, L, D]
        k = inp.k[a:b].double().transpose(0, 1).repeat_interleave(4, 0)
        v = inp.v[a:b].double().transpose(0, 1).repeat_interleave(4, 0)
        ref = sdpa_with_sink(q, k, v, inp.sinks, inp.scale, causal).transpose(0, 1)
        np.testing.assert_allclose(out[a:b], ref.numpy(), rtol=0, atol=TOL)


def test_prefill_rows_equal_decode_over_prefix():
    L = 70
    inp = W.make_prefill(4, 1, [L], seed=15)
    out, lse = oracle.prefill(inp.q, inp.k, inp.v, inp.cu_seqlens, inp.sinks, inp.scale, True)
    # the same keys as a contiguous paged cache
    npg = -(-L // W.PAGE_SIZE)
    kp = torch.zeros(npg * W.PAGE_SIZE, 1, 64, dtype=torch.bfloat16)
    vp = torch.zeros_like(kp)
    kp[:L], vp[:L] = inp.k, inp.v
    kp = kp.view(npg, W.PAGE_SIZE, 1, 64).transpose(1, 2).contiguous()
    vp = vp.view(npg, W.PAGE_SIZE, 1, 64).transpose(1, 2).contiguous()
    pt = torch.arange(npg, dtype=torch.int32)[None].repeat(L, 1)
    lens = torch.arange(1, L + 1, dtype=torch.int32)
    dout, dlse = oracle.decode(inp.q, kp, vp, pt, lens, inp.sinks, inp.scale)
    np.testing.assert_array_equal(out, dout)
    np.testing.assert_array_equal(lse, dlse)
    # row 0 of a sequence is the single-key closed form
    for h in range(4):
        s = inp.scale * float(inp.q[0, h].double() @ inp.k[0, 0].double())
        w = math.exp(s) / (math.exp(s) + math.exp(float(inp.sinks[h])))
        np.testing.assert_allclose(out[0, h], w * inp.v[0, 0].double().numpy(), rtol=0, atol=TOL)


def test_row_selection_matches_full_result():
    inp = W.make_decode(3, 8, 2, [10, 0, 33], seed=16)
    out, lse = oracle.decode(inp.q, inp.k_pages, inp.v_pages, inp.page_table, inp.kv_lens,
                             inp.sinks, inp.scale)
    rows = np.array([[2, 7], [0, 0], [1, 3]], np.int32)
    o, l = oracle.decode(inp.q, inp.k_pages, inp.v_pages, inp.page_table, inp.kv_lens,
                         inp.sinks, inp.scale, rows=rows)
    for i, (b, h) in enumerate(rows):
        np.testing.assert_array_equal(o[i], out[b, h])
        assert l[i] == lse[b, h]
    pin = W.make_prefill(4, 2, [9, 20], seed=17)
    out, lse = oracle.prefill(pin.q, pin.k, pin.v, pin.cu_seqlens, pin.sinks, pin.scale)
    rows = np.array([[28, 1], [0, 3], [9, 0]], np.int32)
    o, l = oracle.prefill(pin.q, pin.k, pin.v, pin.cu_seqlens, pin.sinks, pin.scale, rows=rows)
    for i, (t, h) in enumerate(rows):
        np.testing.assert_array_equal(o[i], out[t, h])
        assert l[i] == lse[t, h]


# ---- verification of drafted tokens (speculative decoding)

def test_verify_rows_equal_decode_over_their_prefix():
    """Token i of a q_len draft is a decode over cache tokens 0..kv_len-q_len+i."""
    QL = 3
    inp = W.make_decode(3, 8, 2, [5, 40, 33], seed=21, q_len=QL)
    out, lse = oracle.verify(inp.q, inp.k_pages, inp.v_pages, inp.page_table, inp.kv_lens, inp.sinks, inp.scale)
    for i in range(QL):
        lens = (inp.kv_lens - QL + i + 1).clamp(min=0)
        ro, rl = oracle.decode(inp.q[:, i].contiguous(), inp.k_pages, inp.v_pages, inp.page_table, lens, inp.sinks,
                               inp.scale)
        assert np.abs(out[:, i] - ro).max() <= TOL
        assert np.abs(lse[:, i] - rl).max() <= TOL


def test_verify_equals_causal_prefill_tail():
    """On a contiguous cache holding a whole sequence, the draft rows are the last rows of its causal prefill."""
    QL, L, Hq, Hkv = 4, 37, 8, 2
    pre = W.make_prefill(Hq, Hkv, [L], seed=22)
    po, pl = oracle.prefill(pre.q, pre.k, pre.v, pre.cu_seqlens, pre.sinks, pre.scale, True)
    npg = (L + W.PAGE_SIZE - 1) // W.PAGE_SIZE
    kp = torch.zeros(npg * W.PAGE_SIZE, Hkv, 64, dtype=torch.bfloat16)
    vp = torch.zeros_like(kp)
    kp[:L], vp[:L] = pre.k, pre.v
    kp = kp.view(npg, W.PAGE_SIZE, Hkv, 64).permute(0, 2, 1, 3).contiguous()
    vp = vp.view(npg, W.PAGE_SIZE, Hkv, 64).permute(0, 2, 1, 3).contiguous()
    pt = torch.arange(npg, dtype=torch.int32).view(1, npg)
    q = pre.q[L - QL:].unsqueeze(0).contiguous()  # [1, QL, Hq, D]
    out, lse = oracle.verify(q, kp, vp, pt, torch.tensor([L], dtype=torch.int32), pre.sinks, pre.scale)
    assert np.abs(out[0] - po[L - QL:]).max() <= TOL
    assert np.abs(lse[0] - pl[L - QL:]).max() <= TOL


def test_verify_brute_force_tiny():
    """Two drafted tokens over a 3-token cache, by explicit enumeration of each row's key set."""
    inp = W.make_decode(1, 2, 1, [3], seed=23, q_len=2)
    out, lse = oracle.verify(inp.q, inp.k_pages, inp.v_pages, inp.page_table, inp.kv_lens, inp.sinks, inp.scale)
    k, v = gather_kv(inp, 0, 0)
    for i, visible in ((0, 2), (1, 3)):  # token 0 sits at position 1, token 1 at position 2
        for h in range(2):
            qv = inp.q[0, i, h].double()
            logits = [inp.scale * float(qv @ k[j]) for j in range(visible)] + [float(inp.sinks[h])]
            m = max(logits)
            w = [math.exp(x - m) for x in logits]
            z = sum(w)
            ref = sum(w[j] / z * v[j].numpy() for j in range(visible))
            assert np.abs(out[0, i, h] - ref).max() <= TOL
            assert abs(lse[0, i, h] - (m + math.log(z))) <= TOL


def test_verify_short_cache_rows_fall_on_the_sink():
    """A cache shorter than the draft leaves the earliest rows without keys: out 0, lse = sink."""
    inp = W.make_decode(1, 4, 2, [2], seed=24, q_len=4)
    out, lse = oracle.verify(inp.q, inp.k_pages, inp.v_pages, inp.page_table, inp.kv_lens, inp.sinks, inp.scale)
    assert np.all(out[0, :2] == 0.0)
    assert np.abs(lse[0, :2] - inp.sinks.double().numpy()[None]).max() == 0.0
    assert np.all(np.abs(out[0, 2:]).max(axis=-1) > 0)


def test_verify_row_selection_matches_full_result():
    inp = W.make_decode(2, 8, 2, [20, 50], seed=25, q_len=3)
    out, lse = oracle.verify(inp.q, inp.k_pages, inp.v_pages, inp.page_table, inp.kv_lens, inp.sinks, inp.scale)
    rows = np.array([[1, 2, 7], [0, 0, 3], [1, 0, 0]], dtype=np.int32)
    so, sl = oracle.verify(inp.q, inp.k_pages, inp.v_pages, inp.page_table, inp.kv_lens, inp.sinks, inp.scale, rows=rows)
    for n, (b, i, h) in enumerate(rows):
        assert np.array_equal(so[n], out[b, i, h]) and sl[n] == lse[b, i, h]


# ---- chunked prefill over a paged cache, and writing new tokens into pages

def _pool_from_sequences(seqs, Hkv, extra_tokens, seed):
    """A permuted page pool holding each sequence's K/V [L, Hkv, 64] at positions 0..L-1, with room for
    `extra_tokens` more tokens per sequence; returns (k_pages, v_pages, page_table)."""
    g = torch.Generator().manual_seed(seed)
    npg = [(k.shape[0] + extra + 15) // 16 for (k, _), extra in zip(seqs, extra_tokens)]
    P = sum(npg)
    perm = torch.randperm(P, generator=g)
    pt = torch.full((len(seqs), max(npg)), -1, dtype=torch.int32)
    kp = torch.randn(P, Hkv, 16, 64, generator=g).to(torch.bfloat16)  # unused slots hold noise
    vp = torch.randn(P, Hkv, 16, 64, generator=g).to(torch.bfloat16)
    off = 0
    for n, ((k, v), m) in enumerate(zip(seqs, npg)):
        pt[n, :m] = perm[off:off + m].to(torch.int32)
        off += m
        for t in range(k.shape[0]):
            kp[pt[n, t // 16], :, t % 16] = k[t]
            vp[pt[n, t // 16], :, t % 16] = v[t]
    return kp, vp, pt


def test_append_then_paged_prefill_equals_causal_prefill():
    """Prefix in pages + new tokens appended into pages + paged prefill of the new tokens == the causal
    prefill of the whole sequences (an independent causal rule and contiguous K/V)."""
    Hq, Hkv = 8, 2
    full = W.make_prefill(Hq, Hkv, [40, 23, 70], seed=41)
    prefix = [17, 0, 64]  # cached tokens of each sequence; the rest is new
    cu = full.cu_seqlens.tolist()
    seqs = [(full.k[cu[n]:cu[n] + prefix[n]], full.v[cu[n]:cu[n] + prefix[n]]) for n in range(3)]
    new_len = [cu[n + 1] - cu[n] - prefix[n] for n in range(3)]
    kp, vp, pt = _pool_from_sequences(seqs, Hkv, new_len, seed=42)
    sel = torch.cat([torch.arange(cu[n] + prefix[n], cu[n + 1]) for n in range(3)])
    cu_new = torch.tensor([0] + list(np.cumsum(new_len)), dtype=torch.int32)
    sp = torch.tensor(prefix, dtype=torch.int32)
    kb, vb = oracle.kv_append(full.k[sel], full.v[sel], cu_new, sp, pt, kp, vp)
    out, lse = oracle.prefill_paged(full.q[sel], kb, vb, pt, cu_new, sp, full.sinks, full.scale)
    ro, rl = oracle.prefill(full.q, full.k, full.v, full.cu_seqlens, full.sinks, full.scale, True)
    assert np.abs(out - ro[sel.numpy()]).max() <= TOL
    assert np.abs(lse - rl[sel.numpy()]).max() <= TOL


def test_kv_append_writes_only_its_slots():
    inp = W.make_decode(2, 8, 2, [20, 5], seed=43, extra_pages=3, max_pages=4)
    k = bf16(torch.randn(7, 2, 64))
    v = bf16(torch.randn(7, 2, 64))
    cu, sp = torch.tensor([0, 4, 7], dtype=torch.int32), torch.tensor([20, 5], dtype=torch.int32)
    pt = inp.page_table.clone()
    used = set(int(x) for x in inp.page_table.flatten() if x >= 0)
    pt[0, 1] = min(set(range(inp.k_pages.shape[0])) - used)  # request 0's positions 16.. go to a spare page
    kb, vb = oracle.kv_append(k, v, cu, sp, pt, inp.k_pages, inp.v_pages)
    before = oracle._bf16_bits(inp.k_pages)
    changed = np.argwhere(np.any(kb != before, axis=-1))
    written = {(int(pt[n, (int(sp[n]) + i) // 16]), h, (int(sp[n]) + i) % 16)
               for n in range(2) for i in range(int(cu[n + 1] - cu[n])) for h in range(2)}
    assert {tuple(int(x) for x in c) for c in changed} <= written
    for n in range(2):
        for i in range(int(cu[n + 1] - cu[n])):
            pos = int(sp[n]) + i
            assert np.array_equal(kb[pt[n, pos // 16], :, pos % 16], oracle._bf16_bits(k)[cu[n] + i])
            assert np.array_equal(vb[pt[n, pos // 16], :, pos % 16], oracle._bf16_bits(v)[cu[n] + i])


def test_paged_prefill_with_uniform_chunks_is_verification():
    QL = 3
    inp = W.make_decode(3, 8, 2, [9, 40, 33], seed=44, q_len=QL)
    vo, vl = oracle.verify(inp.q, inp.k_pages, inp.v_pages, inp.page_table, inp.kv_lens, inp.sinks, inp.scale)
    cu = torch.arange(0, 3 * QL + 1, QL, dtype=torch.int32)
    po, pl = oracle.prefill_paged(inp.q.reshape(3 * QL, 8, 64), inp.k_pages, inp.v_pages, inp.page_table, cu,
                                  inp.kv_lens - QL, inp.sinks, inp.scale)
    assert np.abs(po - vo.reshape(3 * QL, 8, 64)).max() <= TOL
    assert np.abs(pl - vl.reshape(3 * QL, 8)).max() <= TOL


# ---- verification of a draft tree (EAGLE-style masks)

def test_tree_masks_from_parents():
    assert W.tree_masks([-1, 0, 0, 1]) == [0b1, 0b11, 0b101, 0b1011]
    assert W.tree_masks(W.DRAFT_TREE_PARENTS)[7] == (1 << 7) | (1 << 5) | (1 << 2) | 1


def test_chain_tree_is_linear_verification():
    QL = 4
    inp = W.make_decode(3, 8, 2, [9, 40, 33], seed=61, q_len=QL)
    chain = torch.tensor([W.tree_masks([-1, 0, 1, 2])] * 3, dtype=torch.int64)
    to, tl = oracle.verify_tree(inp.q, inp.k_pages, inp.v_pages, inp.page_table, inp.kv_lens, chain, inp.sinks,
                                inp.scale)
    vo, vl = oracle.verify(inp.q, inp.k_pages, inp.v_pages, inp.page_table, inp.kv_lens, inp.sinks, inp.scale)
    assert np.abs(to - vo).max() <= TOL and np.abs(tl - vl).max() <= TOL


def test_tree_brute_force_tiny():
    """A 4-token tree over a 6-token cache (2 tokens before the draft), by explicit key sets."""
    parents = [-1, 0, 0, 2]
    inp = W.make_decode(1, 2, 1, [6], seed=62, q_len=4)
    masks = W.tree_masks(parents)
    out, lse = oracle.verify_tree(inp.q, inp.k_pages, inp.v_pages, inp.page_table, inp.kv_lens,
                                  torch.tensor([masks], dtype=torch.int64), inp.sinks, inp.scale)
    k, v = gather_kv(inp, 0, 0)
    for i in range(4):
        keys = [0, 1] + [2 + j for j in range(4) if (masks[i] >> j) & 1]  # prefix + path to the root
        for h in range(2):
            qv = inp.q[0, i, h].double()
            logits = [inp.scale * float(qv @ k[j]) for j in keys] + [float(inp.sinks[h])]
            m = max(logits)
            w = [math.exp(x - m) for x in logits]
            z = sum(w)
            ref = sum(w[n] / z * v[j].numpy() for n, j in enumerate(keys))
            assert np.abs(out[0, i, h] - ref).max() <= TOL
            assert abs(lse[0, i, h] - (m + math.log(z))) <= TOL


def test_tree_siblings_do_not_see_each_other():
    """Two children of the same parent: each result is independent of the other's key and value."""
    parents = [-1, 0, 0]
    inp = W.make_decode(1, 4, 2, [30], seed=63, q_len=3)
    m = torch.tensor([W.tree_masks(parents)], dtype=torch.int64)
    base, _ = oracle.verify_tree(inp.q, inp.k_pages, inp.v_pages, inp.page_table, inp.kv_lens, m, inp.sinks, inp.scale)
    kp, vp = inp.k_pages.clone(), inp.v_pages.clone()
    sib = 30 - 3 + 2  # cache position of draft token 2
    kp[inp.page_table[0, sib // 16], :, sib % 16] = 7.0
    vp[inp.page_table[0, sib // 16], :, sib % 16] = -7.0
    moved, _ = oracle.verify_tree(inp.q, kp, vp, inp.page_table, inp.kv_lens, m, inp.sinks, inp.scale)
    assert np.array_equal(moved[0, :2], base[0, :2])  # tokens 0 and 1 never look at token 2
    assert not np.array_equal(moved[0, 2], base[0, 2])


def test_forest_brute_force():
    """Two roots: token 1's path does not contain token 0, token 3 hangs under token 1."""
    parents = [-1, -1, 0, 1]
    inp = W.make_decode(1, 2, 1, [7], seed=64, q_len=4)
    masks = W.tree_masks(parents)
    assert masks[1] == 0b10 and masks[3] == 0b1010
    out, lse = oracle.verify_tree(inp.q, inp.k_pages, inp.v_pages, inp.page_table, inp.kv_lens,
                                  torch.tensor([masks], dtype=torch.int64), inp.sinks, inp.scale)
    k, v = gather_kv(inp, 0, 0)
    for i in range(4):
        keys = [0, 1, 2] + [3 + j for j in range(4) if (masks[i] >> j) & 1]
        for h in range(2):
            qv = inp.q[0, i, h].double()
            logits = [inp.scale * float(qv @ k[j]) for j in keys] + [float(inp.sinks[h])]
            m = max(logits)
            w = [math.exp(x - m) for x in logits]
            z = sum(w)
            ref = sum(w[n] / z * v[j].numpy() for n, j in enumerate(keys))
            assert np.abs(out[0, i, h] - ref).max() <= TOL
            assert abs(lse[0, i, h] - (m + math.log(z))) <= TOL


# ---- pre-attention prologue: QKV bias + YaRN rotary embedding

YARN = dict(theta=150000.0, factor=32.0, original_max_position=4096, beta_fast=32.0, beta_slow=1.0)


def test_yarn_without_extension_is_plain_rope():
    inv = oracle.yarn_inv_freq(64, 10000.0, 1.0, 4096, 32.0, 1.0)
    assert np.allclose(inv, 10000.0 ** (-np.arange(32) / 32.0), rtol=1e-15, atol=0)
    assert oracle.yarn_mscale(1.0) == 1.0


def test_yarn_ramp_orientation():
    """Dimensions that turn many times within the original context keep their frequency; those that
    turn less than once are slowed down by the factor; the ramp between is monotone."""
    D, th, s, L = 64, 150000.0, 32.0, 4096
    base = th ** (-np.arange(32) / 32.0)
    turns = L * base / (2 * np.pi)  # full turns over the original context
    inv = oracle.yarn_inv_freq(D, th, s, L, 32.0, 1.0)
    fast, slow = turns > 32.0, turns < 1.0
    assert fast.any() and slow.any()
    assert np.allclose(inv[fast], base[fast], rtol=1e-15, atol=0)
    assert np.allclose(inv[slow], base[slow] / s, rtol=1e-15, atol=0)
    ratio = inv / base  # 1 for fast dims, 1/s for slow ones
    assert np.all(np.diff(ratio) <= 1e-15)
    assert abs(oracle.yarn_mscale(32.0) - (0.1 * math.log(32.0) + 1.0)) < 1e-15


def test_yarn_ramp_interior_value():
    """One dimension inside the ramp, worked by hand from the YaRN method's definition (the ramp is
    a linear function of r, the number of turns a pair makes over the original context).

    theta = 150000, s = 32, L = 4096, beta_fast = 32, beta_slow = 1, pair d = 16 of 32:
      theta_16 = 150000^(-32/64) = 1 / 387.2983...          = 2.5819888974716e-3
      r_16     = 4096 * theta_16 / (2 pi)                    = 1.6831950685839
      gamma    = (r_16 - 1) / (32 - 1)                       = 0.022038550599482
      angle    = ((1 - gamma) / 32 + gamma) * theta_16      = 1.3581221810508e-4 per position
    A ramp that is linear in the pair index between the (fractional) pairs where r = 32 and r = 1
    (8.0928 and 17.3980) would give gamma = 0.150240 and 4.5648e-4 instead."""
    inv = oracle.yarn_inv_freq(64, 150000.0, 32.0, 4096, 32.0, 1.0)
    assert abs(inv[16] - 1.3581221810508e-4) <= 1e-15
    assert abs(inv[16] - 4.5648e-4) > 1e-4  # the pair-index ramp is a different reading
    # the two ramp ends bracket it: pair 14 is inside too, pair 18 already fully slowed
    assert abs(inv[14] - 6.0249056412024e-4) <= 1e-15
    assert abs(inv[18] - 1.2258819959601083e-3 / 32.0) <= 1e-18


@pytest.mark.parametrize("interleaved", [False, True])
def test_rope_invariants(interleaved):
    rng = np.random.default_rng(81)
    inv = oracle.yarn_inv_freq(64, **YARN)
    ms = oracle.yarn_mscale(YARN["factor"])
    q, k = rng.standard_normal((1, 1, 64)), rng.standard_normal((1, 1, 64))
    rq = lambda p: oracle.rope(q, [p], inv, ms, interleaved)[0, 0]
    rk = lambda p: oracle.rope(k, [p], inv, ms, interleaved)[0, 0]
    assert np.allclose(rq(0), ms * q[0, 0], rtol=1e-15, atol=0)  # position 0: no turn
    for p in (1, 777, 131071):
        assert abs(np.linalg.norm(rq(p)) - ms * np.linalg.norm(q)) < 1e-12  # a rotation
    for m, n, delta in ((5, 2, 100), (4000, 17, 60000), (9, 9, 3)):  # only m - n matters
        assert abs(rq(m) @ rk(n) - rq(m + delta) @ rk(n + delta)) < 1e-9


def test_rope_pairs_by_hand():
    """One unit vector per convention, rotated by hand: (1, 0) -> (cos a, sin a) in its pair."""
    inv = oracle.yarn_inv_freq(64, **YARN)
    p, d = 1234, 5
    a = p * inv[d]
    x = np.zeros((1, 1, 64))
    x[0, 0, d] = 1.0
    y = oracle.rope(x, [p], inv, 1.0, False)[0, 0]
    assert abs(y[d] - math.cos(a)) < 1e-12 and abs(y[d + 32] - math.sin(a)) < 1e-12
    assert np.count_nonzero(np.abs(y) > 1e-15) == 2
    x = np.zeros((1, 1, 64))
    x[0, 0, 2 * d] = 1.0
    y = oracle.rope(x, [p], inv, 1.0, True)[0, 0]
    assert abs(y[2 * d] - math.cos(a)) < 1e-12 and abs(y[2 * d + 1] - math.sin(a)) < 1e-12


def test_conventions_are_a_permutation_apart():
    rng = np.random.default_rng(82)
    inv = oracle.yarn_inv_freq(64, **YARN)
    x = rng.standard_normal((3, 2, 64))
    perm = np.empty(64, dtype=int)
    perm[0::2], perm[1::2] = np.arange(32), np.arange(32, 64)  # interleaved slot -> halves slot
    a = oracle.rope(x[..., perm], [3, 50, 999], inv, 1.3, True)
    b = oracle.rope(x, [3, 50, 999], inv, 1.3, False)[..., perm]
    assert np.allclose(a, b, rtol=0, atol=1e-13)


def test_prologue_adds_bias_before_rotating_and_uses_cache_positions():
    Hq, Hkv = 4, 2
    g = torch.Generator().manual_seed(83)
    qkv = bf16(torch.randn(7, (Hq + 2 * Hkv) * 64, generator=g))
    bias = bf16(torch.randn((Hq + 2 * Hkv) * 64, generator=g))
    cu, sp = torch.tensor([0, 3, 7], dtype=torch.int32), torch.tensor([10, 0], dtype=torch.int32)
    q, k, v = oracle.qkv_prologue(qkv, bias, cu, sp, Hq, Hkv, **YARN)
    x = (qkv.double() + bias.double()).reshape(7, Hq + 2 * Hkv, 64).numpy()
    pos = [10, 11, 12, 0, 1, 2, 3]
    inv, ms = oracle.yarn_inv_freq(64, **YARN), oracle.yarn_mscale(32.0)
    assert np.allclose(q, oracle.rope(x[:, :Hq], pos, inv, ms), rtol=0, atol=1e-12)
    assert np.allclose(k, oracle.rope(x[:, Hq:Hq + Hkv], pos, inv, ms), rtol=0, atol=1e-12)
    assert np.array_equal(v, x[:, Hq + Hkv:])
