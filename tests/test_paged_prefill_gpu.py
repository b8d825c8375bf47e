"""GPU writing of new tokens into pages and chunked prefill over the paged cache, against the
fp64 oracle, through the C ABI."""
import numpy as np
import pytest
import torch

import oracle
from gqa_attention_learned_head_gb300 import workloads as W
from parity_utils import assert_parity

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def S():
    from gqa_attention_learned_head_gb300 import sinkattn

    return sinkattn


def bits(t):
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def append_and_prefill(S, inp, rows=None):
    """GPU: append the new tokens, then the paged prefill; oracle: its own append, then its prefill."""
    g = inp.to("cuda")
    S.sinkattn_kv_append(g.k_new, g.v_new, g.cu_seqlens, g.start_pos, g.page_table, g.k_pages, g.v_pages)
    out, lse = S.sinkattn_prefill_paged(g.q, g.k_pages, g.v_pages, g.page_table, g.cu_seqlens, g.start_pos, g.sinks,
                                        g.scale, max_seqlen=inp.max_seqlen)
    err = S.sinkattn_get_error()
    kb, vb = oracle.kv_append(inp.k_new, inp.v_new, inp.cu_seqlens, inp.start_pos, inp.page_table, inp.k_pages,
                              inp.v_pages)
    return g, out.float().cpu().numpy(), lse.cpu().numpy(), err, kb, vb


@pytest.mark.parametrize("Hq,Hkv", [(8, 2), (8, 8), (64, 8), (6, 2)])
@pytest.mark.parametrize("prefix,new", [([0, 17, 64, 130], [1, 127, 128, 129]), ([300, 5, 1000], [40, 300, 17])])
def test_small_shapes(S, Hq, Hkv, prefix, new):
    inp = W.make_paged_prefill(Hq, Hkv, prefix, new, seed=Hq + len(prefix))
    g, out, lse, err, kb, vb = append_and_prefill(S, inp)
    assert err == 0
    assert np.array_equal(bits(g.k_pages), kb) and np.array_equal(bits(g.v_pages), vb)  # append is bit-exact
    ro, rl = oracle.prefill_paged(inp.q, kb, vb, inp.page_table, inp.cu_seqlens, inp.start_pos, inp.sinks, inp.scale)
    assert_parity(out, lse, ro, rl, f"Hq={Hq} Hkv={Hkv} prefix={prefix} new={new}")


@pytest.mark.parametrize("N", [40, 140])
@pytest.mark.parametrize("Hq,Hkv", [(8, 2), (6, 2)])
def test_many_sequences(S, N, Hq, Hkv):
    """Batches ranked by cached prefix + new tokens (40 sequences) and past the ranked limit (140,
    index order); prefixes and new lengths repeat, so equal weights occur."""
    rng = np.random.default_rng(N + Hq)
    prefix = rng.choice([0, 5, 16, 200, 700], size=N).tolist()
    new = rng.choice([1, 30, 128, 129], size=N).tolist()
    inp = W.make_paged_prefill(Hq, Hkv, prefix, new, seed=N + Hq)
    g, out, lse, err, kb, vb = append_and_prefill(S, inp)
    assert err == 0
    ro, rl = oracle.prefill_paged(inp.q, kb, vb, inp.page_table, inp.cu_seqlens, inp.start_pos, inp.sinks, inp.scale)
    assert_parity(out, lse, ro, rl, f"N={N} Hq={Hq} Hkv={Hkv}")


def test_maximum_sequence_count(S):
    """16384 sequences (the most a paged prefill call takes), 0..20 cached and 1..3 new tokens each."""
    rng = np.random.default_rng(16383)
    prefix = rng.integers(0, 21, 16384).tolist()
    new = rng.integers(1, 4, 16384).tolist()
    inp = W.make_paged_prefill(8, 2, prefix, new, seed=12)
    g, out, lse, err, kb, vb = append_and_prefill(S, inp)
    assert err == 0
    ro, rl = oracle.prefill_paged(inp.q, kb, vb, inp.page_table, inp.cu_seqlens, inp.start_pos, inp.sinks, inp.scale)
    assert_parity(out, lse, ro, rl, "16384 sequences")


def test_share_sms_matches_oracle(S):
    """The paged prefill's kernel that leaves room on every SM computes the same attention."""
    inp = W.make_paged_prefill(64, 8, [300, 5, 1000], [40, 300, 17], seed=35)
    g = inp.to("cuda")
    S.sinkattn_kv_append(g.k_new, g.v_new, g.cu_seqlens, g.start_pos, g.page_table, g.k_pages, g.v_pages)
    out, lse = S.sinkattn_prefill_paged(g.q, g.k_pages, g.v_pages, g.page_table, g.cu_seqlens, g.start_pos, g.sinks,
                                        g.scale, max_seqlen=inp.max_seqlen, share_sms=True)
    assert S.sinkattn_get_error() == 0
    kb, vb = oracle.kv_append(inp.k_new, inp.v_new, inp.cu_seqlens, inp.start_pos, inp.page_table, inp.k_pages,
                              inp.v_pages)
    ro, rl = oracle.prefill_paged(inp.q, kb, vb, inp.page_table, inp.cu_seqlens, inp.start_pos, inp.sinks, inp.scale)
    assert_parity(out.float().cpu().numpy(), lse.cpu().numpy(), ro, rl, "paged share_sms")


def test_no_prefix_equals_plain_prefill(S):
    """start_pos = 0: the paged prefill is the causal prefill of the new tokens."""
    inp = W.make_paged_prefill(16, 2, [0, 0, 0], [200, 1, 129], seed=51)
    g, out, lse, err, kb, vb = append_and_prefill(S, inp)
    assert err == 0
    ro, rl = oracle.prefill(inp.q, inp.k_new, inp.v_new, inp.cu_seqlens, inp.sinks, inp.scale, True)
    assert_parity(out, lse, ro, rl, "no prefix")


def test_nan_in_unused_slots_is_ignored(S):
    """Pool slots past each sequence's end hold NaN: no output may see them."""
    inp = W.make_paged_prefill(8, 2, [21, 70], [10, 35], seed=52)
    kb, vb = oracle.kv_append(inp.k_new, inp.v_new, inp.cu_seqlens, inp.start_pos, inp.page_table, inp.k_pages,
                              inp.v_pages)
    ro, rl = oracle.prefill_paged(inp.q, kb, vb, inp.page_table, inp.cu_seqlens, inp.start_pos, inp.sinks, inp.scale)
    for n, (s0, L) in enumerate(zip(inp.start_pos.tolist(), inp.new_lens)):
        end = s0 + L
        last = int(inp.page_table[n, (end - 1) // 16])
        inp.k_pages[last, :, end % 16 or 16:] = float("nan")
        inp.v_pages[last, :, end % 16 or 16:] = float("nan")
    g, out, lse, err, _, _ = append_and_prefill(S, inp)
    assert err == 0
    assert_parity(out, lse, ro, rl, "NaN past the end")


def test_bad_page_is_reported(S):
    inp = W.make_paged_prefill(8, 2, [40, 40], [20, 20], seed=53)
    inp.page_table[1, 0] = inp.k_pages.shape[0] + 3
    g = inp.to("cuda")
    out, lse = S.sinkattn_prefill_paged(g.q, g.k_pages, g.v_pages, g.page_table, g.cu_seqlens, g.start_pos, g.sinks,
                                        g.scale, max_seqlen=inp.max_seqlen)
    assert S.sinkattn_get_error() == S.ERR_BAD_PAGE
    assert torch.isfinite(out.float()).all() and torch.isfinite(lse).all()


def test_chunked_prefill_full_size_sampled(S):
    """Full-size workload in the launch configuration the benchmark times; 96 sampled rows."""
    inp = W.chunked_prefill()
    g, out, lse, err, kb, vb = append_and_prefill(S, inp)
    assert err == 0
    rng = np.random.default_rng(2)
    rows = np.stack([rng.integers(0, inp.q.shape[0], 96), rng.integers(0, 64, 96)], 1).astype(np.int32)
    ro, rl = oracle.prefill_paged(inp.q, kb, vb, inp.page_table, inp.cu_seqlens, inp.start_pos, inp.sinks, inp.scale,
                                  rows=rows)
    assert_parity(out[rows[:, 0], rows[:, 1]], lse[rows[:, 0], rows[:, 1]], ro, rl, "chunked prefill")
    assert np.all(np.isfinite(out)) and np.all(np.isfinite(lse))


def test_append_reports_bad_pages_and_positions(S):
    inp = W.make_paged_prefill(8, 2, [16, 16], [4, 4], seed=54)
    g = inp.to("cuda")
    before_k = g.k_pages.clone()
    pt = g.page_table.clone()
    pt[1, 1] = -7  # sequence 1's new tokens (positions 16..19) land in page index 1
    S.sinkattn_kv_append(g.k_new, g.v_new, g.cu_seqlens, g.start_pos, pt, g.k_pages, g.v_pages)
    assert S.sinkattn_get_error() == S.ERR_BAD_PAGE
    # sequence 0's tokens were written, sequence 1's skipped: only sequence 0's slots changed
    changed = (g.k_pages != before_k).any(dim=-1).nonzero().tolist()
    assert changed and all(p == int(inp.page_table[0, 1]) for p, _, _ in changed)
    far = torch.tensor([10 ** 6, 0], dtype=torch.int32, device="cuda")  # past max_pages * 16
    S.sinkattn_kv_append(g.k_new, g.v_new, g.cu_seqlens, far, g.page_table, g.k_pages, g.v_pages)
    assert S.sinkattn_get_error() == S.ERR_BAD_LENGTH


def test_paged_prefill_reports_bad_length(S):
    inp = W.make_paged_prefill(8, 2, [16, 16], [4, 4], seed=55)
    g = inp.to("cuda")
    far = torch.tensor([10 ** 6, 16], dtype=torch.int32, device="cuda")
    out, lse = S.sinkattn_prefill_paged(g.q, g.k_pages, g.v_pages, g.page_table, g.cu_seqlens, far, g.sinks, g.scale,
                                        max_seqlen=inp.max_seqlen)
    assert S.sinkattn_get_error() == S.ERR_BAD_LENGTH
    assert torch.isfinite(out.float()).all() and torch.isfinite(lse).all()


def test_graph_replay_append_and_prefill(S):
    """The chunked step (append, then the paged prefill, a programmatic dependent of the append) captured
    once in a CUDA graph and replayed after the inputs in the same buffers changed (other tokens, pool
    contents and page layout): every replay matches the oracle on its inputs."""
    prefix, new = [0, 300, 1000, 17], [129, 40, 300, 1]
    srcs = [W.make_paged_prefill(8, 2, prefix, new, seed=s) for s in (61, 62, 63)]
    for s in srcs[1:]:
        assert s.k_pages.shape == srcs[0].k_pages.shape and s.page_table.shape == srcs[0].page_table.shape
    g = srcs[0].to("cuda")
    out = torch.empty_like(g.q)
    lse = torch.empty(g.q.shape[:2], dtype=torch.float32, device="cuda")
    stream = torch.cuda.Stream()

    def step():
        S.sinkattn_kv_append(g.k_new, g.v_new, g.cu_seqlens, g.start_pos, g.page_table, g.k_pages, g.v_pages,
                             stream=stream)
        S.sinkattn_prefill_paged(g.q, g.k_pages, g.v_pages, g.page_table, g.cu_seqlens, g.start_pos, g.sinks,
                                 g.scale, max_seqlen=srcs[0].max_seqlen, out=out, lse=lse, stream=stream)

    with torch.cuda.stream(stream):
        step()  # warm-up outside the capture
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        step()
    for src in srcs + srcs[:1]:
        for name in ("q", "k_new", "v_new", "k_pages", "v_pages", "page_table", "sinks"):
            getattr(g, name).copy_(getattr(src, name))
        torch.cuda.synchronize()
        graph.replay()
        torch.cuda.synchronize()
        assert S.sinkattn_get_error() == 0
        kb, vb = oracle.kv_append(src.k_new, src.v_new, src.cu_seqlens, src.start_pos, src.page_table, src.k_pages,
                                  src.v_pages)
        ro, rl = oracle.prefill_paged(src.q, kb, vb, src.page_table, src.cu_seqlens, src.start_pos, src.sinks,
                                      src.scale)
        assert_parity(out.float().cpu().numpy(), lse.cpu().numpy(), ro, rl, "graph replay")
