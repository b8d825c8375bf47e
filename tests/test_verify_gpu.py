"""GPU verification of drafted tokens (q_len query tokens per request over the paged cache)
against the fp64 oracle, through the C ABI."""
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
    out, lse = S.sinkattn_verify(g.q, g.k_pages, g.v_pages, g.page_table, g.kv_lens, g.sinks, g.scale, **kw)
    err = S.sinkattn_get_error()
    return out.float().cpu().numpy(), lse.cpu().numpy(), err


def ref(inp, rows=None):
    return oracle.verify(inp.q, inp.k_pages, inp.v_pages, inp.page_table, inp.kv_lens, inp.sinks, inp.scale,
                         rows=rows)


# (Hq, Hkv, q_len): rows q_len * Hq/Hkv of 2, 8, 12, 16, 24, 32, 64 -> 1, 2, 4 and 8 warps
SHAPES = [(2, 1, 1), (8, 1, 1), (8, 2, 3), (8, 8, 16), (16, 2, 3), (64, 8, 4), (64, 8, 8), (32, 2, 4), (4, 2, 1)]


@pytest.mark.parametrize("Hq,Hkv,QL", SHAPES)
@pytest.mark.parametrize("lens", [[1, 16, 17], [300, 2, 64, 1000, 0, 33]])
def test_small_shapes(S, Hq, Hkv, QL, lens):
    inp = W.make_decode(len(lens), Hq, Hkv, lens, seed=Hq + QL + len(lens), q_len=QL)
    out, lse, err = run(S, inp)
    assert err == 0
    assert_parity(out, lse, *ref(inp), f"Hq={Hq} Hkv={Hkv} q_len={QL} lens={lens}")


@pytest.mark.parametrize("workers", [1, 7, 50, 300])
def test_forced_splits(S, workers):
    """Equal shares cut segments anywhere: pieces of every size, merged by log-sum-exp."""
    inp = W.make_decode(6, 64, 8, (20, 700), seed=31, q_len=4)
    out, lse, err = run(S, inp, num_workers=workers)
    assert err == 0
    assert_parity(out, lse, *ref(inp), f"workers={workers}")


@pytest.mark.parametrize("sink", [float("-inf"), -30.0, 30.0])
def test_sink_values(S, sink):
    inp = W.make_decode(3, 16, 2, [40, 3, 129], seed=32, q_len=5)
    inp.sinks[:] = sink
    out, lse, err = run(S, inp)
    assert err == 0
    assert_parity(out, lse, *ref(inp), f"sink={sink}")


def test_short_caches_put_early_tokens_on_the_sink(S):
    """kv_len < q_len: the earliest drafted tokens see no key at all."""
    inp = W.make_decode(3, 8, 2, [1, 2, 5], seed=33, q_len=6)
    out, lse, err = run(S, inp)
    assert err == 0
    ro, rl = ref(inp)
    assert_parity(out, lse, ro, rl, "short caches")
    assert np.all(out[0, :5] == 0)  # exactly: no key, the sink carries no value row
    assert np.abs(lse[0, :5] - inp.sinks.numpy()[None]).max() <= 1e-5  # sink, up to the log2 / ln round trip


def test_q_len_one_matches_decode(S):
    """q_len = 1 is decode: both calls against the same oracle rows."""
    inp = W.make_decode(5, 64, 8, (1, 900), seed=34, q_len=1)
    out, lse, err = run(S, inp)
    assert err == 0
    g = inp.to("cuda")
    dout, dlse = S.sinkattn_decode(g.q[:, 0].contiguous(), g.k_pages, g.v_pages, g.page_table, g.kv_lens, g.sinks,
                                   g.scale)
    ro, rl = oracle.decode(inp.q[:, 0].contiguous(), inp.k_pages, inp.v_pages, inp.page_table, inp.kv_lens,
                           inp.sinks, inp.scale)
    assert_parity(out[:, 0], lse[:, 0], ro, rl, "verify q_len 1")
    assert_parity(dout.float().cpu().numpy(), dlse.cpu().numpy(), ro, rl, "decode")


def test_bad_page_is_skipped_and_reported(S):
    inp = W.make_decode(2, 8, 2, [40, 40], seed=35, q_len=2)
    P = inp.k_pages.shape[0]
    inp.page_table[1, 1] = P + 5  # out of range: its tokens count as absent
    out, lse, err = run(S, inp)
    assert err == S.ERR_BAD_PAGE
    ro, rl = ref(W.make_decode(2, 8, 2, [40, 40], seed=35, q_len=2), rows=np.array([[0, i, h] for i in range(2) for h in range(8)], dtype=np.int32))
    assert_parity(out[0].reshape(-1, 64), lse[0].reshape(-1), ro, rl, "unaffected request")
    assert np.all(np.isfinite(out)) and np.all(np.isfinite(lse))


def test_maximum_batch(S):
    """32768 requests of 2 drafted tokens (the most a verification call takes): the share search
    walks the requests in many passes; cache lengths 2..40."""
    lens = np.random.default_rng(32767).integers(2, 41, 32768).tolist()
    inp = W.make_decode(32768, 8, 2, lens, seed=10, q_len=2)
    out, lse, err = run(S, inp)
    assert err == 0
    assert_parity(out, lse, *ref(inp), "32768 requests")


def test_speculative_verify_full_size_sampled(S):
    """Full-size workload in the launch configuration the benchmark times; 96 sampled rows."""
    inp = W.speculative_verify()
    out, lse, err = run(S, inp)
    assert err == 0
    rng = np.random.default_rng(1)
    rows = np.stack([rng.integers(0, 32, 96), rng.integers(0, 4, 96), rng.integers(0, 64, 96)], 1).astype(np.int32)
    ro, rl = ref(inp, rows)
    assert_parity(out[rows[:, 0], rows[:, 1], rows[:, 2]], lse[rows[:, 0], rows[:, 1], rows[:, 2]], ro, rl,
                  "speculative verify")
    assert np.all(np.isfinite(out)) and np.all(np.isfinite(lse))


def test_garbage_past_the_cache_end_is_ignored(S):
    """Slots past kv_len in the last page hold NaN: no output may see them."""
    inp = W.make_decode(2, 16, 2, [21, 37], seed=36, q_len=3)
    ro, rl = ref(inp)
    kp, vp = inp.k_pages.clone(), inp.v_pages.clone()
    for b, L in enumerate(inp.kv_lens.tolist()):
        last = int(inp.page_table[b, (L - 1) // 16])
        kp[last, :, L % 16:] = float("nan")
        vp[last, :, L % 16:] = float("nan")
    inp.k_pages, inp.v_pages = kp, vp
    out, lse, err = run(S, inp)
    assert err == 0
    assert_parity(out, lse, ro, rl, "NaN past the end")


# ---- draft trees (EAGLE-style masks)

def run_tree(S, inp, masks, **kw):
    g = inp.to("cuda")
    m = torch.as_tensor(masks, dtype=torch.int64).cuda()
    out, lse = S.sinkattn_verify_tree(g.q, g.k_pages, g.v_pages, g.page_table, g.kv_lens, m, g.sinks, g.scale, **kw)
    err = S.sinkattn_get_error()
    return out.float().cpu().numpy(), lse.cpu().numpy(), err


def ref_tree(inp, masks, rows=None):
    return oracle.verify_tree(inp.q, inp.k_pages, inp.v_pages, inp.page_table, inp.kv_lens,
                              torch.as_tensor(masks, dtype=torch.int64), inp.sinks, inp.scale, rows=rows)


@pytest.mark.parametrize("parents", [W.DRAFT_TREE_PARENTS, [-1, -1, 0, 1], [-1, 0, 1, 2, 3], [-1, 0, 0, 0, 0, 0]])
@pytest.mark.parametrize("Hq,Hkv", [(64, 8), (8, 2), (4, 4)])
def test_tree_shapes(S, parents, Hq, Hkv):
    QL = len(parents)
    if QL * Hq // Hkv > 64:
        pytest.skip("more than 64 query rows per (request, KV head)")
    lens = [QL, 17, 300, 1000, QL + 16]
    inp = W.make_decode(len(lens), Hq, Hkv, lens, seed=QL + Hq, q_len=QL)
    masks = [W.tree_masks(parents)] * len(lens)
    out, lse, err = run_tree(S, inp, masks)
    assert err == 0
    assert_parity(out, lse, *ref_tree(inp, masks), f"parents={parents} Hq={Hq} Hkv={Hkv}")


def test_tree_per_request_masks_and_splits(S):
    """Different trees per request, forced splits so that drafts land in merged pieces."""
    rng = np.random.default_rng(5)
    QL, B = 6, 5
    masks = []
    for _ in range(B):
        parents = [-1] + [int(rng.integers(-1, i)) for i in range(1, QL)]
        masks.append(W.tree_masks(parents))
    inp = W.make_decode(B, 16, 2, (20, 400), seed=71, q_len=QL)
    for workers in (0, 7, 40):
        out, lse, err = run_tree(S, inp, masks, num_workers=workers)
        assert err == 0
        assert_parity(out, lse, *ref_tree(inp, masks), f"workers={workers}")


def test_chain_tree_matches_linear_kernel(S):
    inp = W.make_decode(4, 64, 8, (100, 900), seed=72, q_len=4)
    masks = [W.tree_masks([-1, 0, 1, 2])] * 4
    out, lse, err = run_tree(S, inp, masks)
    lo, ll, lerr = run(S, inp)
    assert err == 0 and lerr == 0
    ro, rl = ref(inp)
    assert_parity(out, lse, ro, rl, "chain tree")
    assert_parity(lo, ll, ro, rl, "linear")


def test_tree_verify_full_size_sampled(S):
    inp, masks = W.tree_verify()
    out, lse, err = run_tree(S, inp, masks)
    assert err == 0
    rng = np.random.default_rng(3)
    rows = np.stack([rng.integers(0, 32, 96), rng.integers(0, 8, 96), rng.integers(0, 64, 96)], 1).astype(np.int32)
    ro, rl = ref_tree(inp, masks, rows)
    assert_parity(out[rows[:, 0], rows[:, 1], rows[:, 2]], lse[rows[:, 0], rows[:, 1], rows[:, 2]], ro, rl, "tree")
    assert np.all(np.isfinite(out)) and np.all(np.isfinite(lse))


def test_bad_page_tokens_count_as_absent(S):
    """A page id outside the pool: its tokens count as absent -- the request's rows equal
    the oracle's on the same cache with that page's 16 tokens left out (the page lies before the draft,
    and visibility depends only on positions relative to the draft)."""
    inp = W.make_decode(2, 8, 2, [40, 40], seed=37, q_len=2)
    ok = W.make_decode(2, 8, 2, [40, 40], seed=37, q_len=2)
    P = inp.k_pages.shape[0]
    pt = inp.page_table.clone()
    inp.page_table[1, 0] = P + 5
    out, lse, err = run(S, inp)
    assert err == S.ERR_BAD_PAGE
    ok.page_table[1, 0], ok.page_table[1, 1] = pt[1, 1], pt[1, 2]  # the cache without its first page
    ok.kv_lens[1] = 24
    rows = np.array([[1, i, h] for i in range(2) for h in range(8)], dtype=np.int32)
    ro, rl = ref(ok, rows)
    assert_parity(out[1].reshape(-1, 64), lse[1].reshape(-1), ro, rl, "request with an absent page")


def test_empty_pool(S):
    """No page in the pool: every cached token is absent, so each row is the sink's alone (out = 0,
    lse = sink); a request that claims cached tokens is reported as pointing outside the pool."""
    Hq, Hkv, QL = 16, 2, 3
    q = torch.randn(3, QL, Hq, 64, device="cuda").to(torch.bfloat16)
    pages = torch.empty(0, Hkv, 16, 64, dtype=torch.bfloat16, device="cuda")
    pt = torch.full((3, 2), -1, dtype=torch.int32, device="cuda")
    sinks = torch.randn(Hq, device="cuda")
    lens = torch.zeros(3, dtype=torch.int32, device="cuda")
    out, lse = S.sinkattn_verify(q, pages, pages, pt, lens, sinks, 0.125)
    assert S.sinkattn_get_error() == 0
    assert bool((out == 0).all())
    assert torch.equal(lse, sinks.expand(3, QL, Hq))
    lens[1] = 20  # two pages' worth of tokens, none of them in the pool
    out, lse = S.sinkattn_verify(q, pages, pages, pt, lens, sinks, 0.125)
    assert S.sinkattn_get_error() == S.ERR_BAD_PAGE
    assert bool((out == 0).all()) and torch.equal(lse, sinks.expand(3, QL, Hq))


def test_growing_scores_rescale_o(S):
    """Scores that rise along the cache by ~10 (log2 units) per 128-key tile at kv_len 700: each row's
    running max passes the lazy-rescale threshold tile after tile, so O is rescaled in tensor memory
    again and again; linear drafts and a tree, with and without split segments."""
    inp = growing_scores(W.make_decode(4, 64, 8, [700, 300, 2000, 129], seed=81, q_len=4), seed=82)
    _, rl = ref(inp)
    assert float(rl[0].max()) > 35.0  # the first request's last row sees scores from ~0 to ~40
    masks = [W.tree_masks([-1, 0, 0, 1])] * 4
    for workers in (0, 9):
        out, lse, err = run(S, inp, num_workers=workers)
        assert err == 0
        assert_parity(out, lse, *ref(inp), f"linear workers={workers}")
        out, lse, err = run_tree(S, inp, masks, num_workers=workers)
        assert err == 0
        assert_parity(out, lse, *ref_tree(inp, masks), f"tree workers={workers}")
