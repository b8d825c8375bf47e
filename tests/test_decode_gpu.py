"""GPU decode (split-KV + merge) against the fp64 oracle, through the C ABI."""
import math

import numpy as np
import pytest
import torch

import oracle
from gqa_attention_learned_head_gb300 import workloads as W
from parity_utils import assert_parity, growing_scores

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def S():
    from gqa_attention_learned_head_gb300 import sinkattn

    return sinkattn


def run(S, inp, **kw):
    g = inp.to("cuda")
    out, lse = S.sinkattn_decode(g.q, g.k_pages, g.v_pages, g.page_table, g.kv_lens, g.sinks, g.scale, **kw)
    err = S.sinkattn_get_error()
    return out.float().cpu().numpy(), lse.cpu().numpy(), err


def ref(inp, rows=None):
    return oracle.decode(inp.q, inp.k_pages, inp.v_pages, inp.page_table, inp.kv_lens, inp.sinks, inp.scale,
                         rows=rows)


def test_tiny_decode(S):
    inp = W.tiny_decode()
    out, lse, err = run(S, inp)
    assert err == 0
    assert_parity(out, lse, *ref(inp), "tiny decode")


def test_batched_paged_decode(S):
    inp = W.batched_paged_decode()
    out, lse, err = run(S, inp)
    assert err == 0
    assert_parity(out, lse, *ref(inp), "batched paged decode")


@pytest.mark.parametrize("workers", [0, 4 * 8 * 32])
def test_long_context_every_row(S, workers):
    """Full-size long-context workload, every (request, head) row against the oracle.

    workers = B * Hkv * 32 cuts every request into exactly 32 chunks of 4096 tokens."""
    inp = W.long_context_decode()
    out, lse, err = run(S, inp, num_workers=workers)
    assert err == 0
    assert_parity(out, lse, *ref(inp), "long context")


def test_mixed_serving_decode_every_row(S):
    """The decode half of the mixed serving batch (256 requests, kv_len U[1024, 32768]) in full."""
    inp = W.mixed_serving_decode()
    out, lse, err = run(S, inp)
    assert err == 0
    assert_parity(out, lse, *ref(inp), "mixed decode")


@pytest.mark.parametrize("lens", [[0, 1, 15, 16, 17], [255, 256, 257, 4097], [0, 0, 0], [33]])
@pytest.mark.parametrize("Hq,Hkv", [(4, 1), (64, 8), (16, 1), (6, 2)])
def test_lengths_and_groups(S, lens, Hq, Hkv):
    inp = W.make_decode(len(lens), Hq, Hkv, lens, seed=sum(lens) + Hq)
    out, lse, err = run(S, inp)
    assert err == 0
    assert_parity(out, lse, *ref(inp), f"lens={lens} Hq={Hq} Hkv={Hkv}")


@pytest.mark.parametrize("sink", [float("-inf"), -30.0, 0.0, 30.0])
def test_sink_values(S, sink):
    inp = W.make_decode(3, 16, 2, [0, 40, 700], seed=3)
    inp.sinks[:] = sink
    out, lse, err = run(S, inp)
    assert err == 0
    assert_parity(out, lse, *ref(inp), f"sink={sink}")


@pytest.mark.parametrize("workers", [1, 2, 3, 7, 64, 1000, 5000])
def test_split_count_does_not_change_result(S, workers):
    inp = W.make_decode(5, 32, 4, [1, 100, 1000, 3000, 17], seed=4)
    out, lse, err = run(S, inp, num_workers=workers)
    assert err == 0
    assert_parity(out, lse, *ref(inp), f"workers={workers}")


def test_partial_last_page_garbage_is_ignored(S):
    inp = W.make_decode(2, 8, 1, [17, 30], seed=5)
    # slots past kv_len in each last page: fill with NaN and huge values
    for b, L in enumerate([17, 30]):
        last = int(inp.page_table[b, (L - 1) // 16])
        inp.k_pages[last, :, L % 16:] = float("nan")
        inp.v_pages[last, :, L % 16:] = float("inf")
    out, lse, err = run(S, inp)
    assert err == 0
    assert_parity(out, lse, *ref(inp), "garbage tail")


def test_bad_page_is_reported_and_skipped(S):
    inp = W.make_decode(2, 8, 2, [40, 40], seed=6)
    good = ref(inp)
    inp.page_table[1, 1] = inp.k_pages.shape[0] + 5  # request 1 points outside the pool
    out, lse, err = run(S, inp)
    assert err == S.ERR_BAD_PAGE
    assert_parity(out[0], lse[0], good[0][0], good[1][0], "untouched request")
    assert np.all(np.isfinite(out[1]))


def test_bad_length_is_reported(S):
    inp = W.make_decode(2, 8, 2, [48, 48], seed=7)  # full page-table rows: 3 pages each
    g = inp.to("cuda")
    g.kv_lens[1] = 10_000  # beyond max_pages * 16 = 48: clamped to 48
    S.sinkattn_decode(g.q, g.k_pages, g.v_pages, g.page_table, g.kv_lens, g.sinks, g.scale)
    assert S.sinkattn_get_error() == S.ERR_BAD_LENGTH
    assert S.sinkattn_get_error() == 0  # cleared by the read


def test_workspace_too_small(S):
    inp = W.make_decode(2, 8, 2, [40, 20], seed=8).to("cuda")
    ws = torch.empty(16, dtype=torch.uint8, device="cuda")
    with pytest.raises(S.SinkAttnError) as e:
        S.sinkattn_decode(inp.q, inp.k_pages, inp.v_pages, inp.page_table, inp.kv_lens, inp.sinks, inp.scale,
                          workspace=ws)
    assert e.value.status == S.ERR_WORKSPACE


def test_lse_optional_and_repeatable(S):
    inp = W.make_decode(4, 64, 8, (100, 2000), seed=9).to("cuda")
    o1, _ = S.sinkattn_decode(inp.q, inp.k_pages, inp.v_pages, inp.page_table, inp.kv_lens, inp.sinks, inp.scale,
                              return_lse=False)
    o2, _ = S.sinkattn_decode(inp.q, inp.k_pages, inp.v_pages, inp.page_table, inp.kv_lens, inp.sinks, inp.scale)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2)  # deterministic


def test_empty_batch(S):
    inp = W.make_decode(1, 8, 2, [5], seed=10).to("cuda")
    q = inp.q[:0]
    out, lse = S.sinkattn_decode(q, inp.k_pages, inp.v_pages, inp.page_table[:0], inp.kv_lens[:0], inp.sinks,
                                 inp.scale)
    assert out.shape == (0, 8, 64) and S.sinkattn_get_error() == 0


def test_maximum_batch(S):
    """32768 requests, the most a decode call takes (the per-CTA page prefix fills 128 KB of shared
    memory); cache lengths 0..40, so empty requests and partial pages occur throughout."""
    lens = np.random.default_rng(32768).integers(0, 41, 32768).tolist()
    inp = W.make_decode(32768, 8, 2, lens, seed=9)
    out, lse, err = run(S, inp)
    assert err == 0
    assert_parity(out, lse, *ref(inp), "32768 requests")


def test_one_million_token_request(S):
    """Maximum-size case: a 2^20-token request (65536 pages, 2 GiB of K/V) beside a 5-token one; every
    head of both requests against the oracle (inputs drawn on the device, copied to the host)."""
    g = W.make_decode(2, 64, 8, [1 << 20, 5], seed=77, device="cuda")
    out, lse = S.sinkattn_decode(g.q, g.k_pages, g.v_pages, g.page_table, g.kv_lens, g.sinks, g.scale)
    assert S.sinkattn_get_error() == 0
    out, lse = out.float().cpu().numpy(), lse.cpu().numpy()
    c = g.to("cpu")
    del g
    ro, rl = ref(c)
    assert_parity(out, lse, ro, rl, "2^20-token request")


def test_workspace_needs_no_initialisation(S):
    """The caller's workspace may hold anything: random bytes give the same result as a fresh one."""
    inp = W.make_decode(6, 64, 8, [300, 5000, 17, 0, 2048, 777], seed=11)
    g = inp.to("cuda")
    n = S.sinkattn_decode_workspace_size(g.q, g.k_pages, g.page_table, 40)
    ws = torch.randint(0, 256, (n,), dtype=torch.uint8, device="cuda")
    out, lse = S.sinkattn_decode(g.q, g.k_pages, g.v_pages, g.page_table, g.kv_lens, g.sinks, g.scale,
                                 workspace=ws, num_workers=40)
    assert S.sinkattn_get_error() == 0
    assert_parity(out.float().cpu().numpy(), lse.cpu().numpy(), *ref(inp), "random workspace")


def test_graph_replay_with_new_inputs(S):
    """The decode (split kernel and its dependent merge) captured once in a CUDA graph and replayed
    after the inputs in the same buffers changed: every replay matches the oracle on its inputs."""
    a = W.make_decode(8, 64, 8, (512, 4096), seed=12)
    b = W.make_decode(8, 64, 8, a.kv_lens.tolist(), seed=13)
    b.page_table = a.page_table.clone()  # same lengths and pool size, other contents and layout
    c = W.make_decode(8, 64, 8, a.kv_lens.tolist(), seed=14)
    c.page_table = a.page_table.clone()
    c.kv_lens = a.kv_lens // 3 + 1  # shorter caches: the split of the work moves
    g = a.to("cuda")
    out = torch.empty_like(g.q)
    lse = torch.empty(g.q.shape[:2], dtype=torch.float32, device="cuda")
    ws = torch.empty(S.sinkattn_decode_workspace_size(g.q, g.k_pages, g.page_table), dtype=torch.uint8,
                     device="cuda")
    stream = torch.cuda.Stream()
    S.sinkattn_decode(g.q, g.k_pages, g.v_pages, g.page_table, g.kv_lens, g.sinks, g.scale, out=out, lse=lse,
                      workspace=ws, stream=stream)  # warm-up outside the capture
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        S.sinkattn_decode(g.q, g.k_pages, g.v_pages, g.page_table, g.kv_lens, g.sinks, g.scale, out=out, lse=lse,
                          workspace=ws, stream=stream)
    for src in (a, b, c, a):
        for name in ("q", "k_pages", "v_pages", "kv_lens", "sinks"):
            getattr(g, name).copy_(getattr(src, name))
        torch.cuda.synchronize()
        graph.replay()
        torch.cuda.synchronize()
        assert S.sinkattn_get_error() == 0
        assert_parity(out.float().cpu().numpy(), lse.cpu().numpy(), *ref(src), "graph replay")


def test_benchmark_draw_of_the_batched_workload(S):
    """The exact bytes the benchmark times: the batched paged decode drawn on the device (seed 0,
    the draw of rank 0), checked against the oracle on a host copy of the same inputs."""
    g = W.batched_paged_decode(device="cuda", seed=0)
    out, lse = S.sinkattn_decode(g.q, g.k_pages, g.v_pages, g.page_table, g.kv_lens, g.sinks, g.scale)
    assert S.sinkattn_get_error() == 0
    c = g.to("cpu")
    assert_parity(out.float().cpu().numpy(), lse.cpu().numpy(), *ref(c), "benchmark draw")


@pytest.mark.parametrize("workers", [0, 13])
def test_growing_scores(S, workers):
    """Scores that rise along the cache (the running max moves on every page), whole and split."""
    inp = growing_scores(W.make_decode(4, 64, 8, [700, 300, 2000, 129], seed=83), seed=84)
    out, lse, err = run(S, inp, num_workers=workers)
    assert err == 0
    assert_parity(out, lse, *ref(inp), f"workers={workers}")
