"""The seeded generators: deterministic, and shaped like the named workloads."""
import torch

from gqa_attention_learned_head_gb300 import workloads as W


def test_same_seed_same_bytes():
    a = W.make_decode(4, 8, 2, (10, 100), seed=3)
    b = W.make_decode(4, 8, 2, (10, 100), seed=3)
    for x, y in zip((a.q, a.k_pages, a.v_pages, a.page_table, a.kv_lens, a.sinks),
                    (b.q, b.k_pages, b.v_pages, b.page_table, b.kv_lens, b.sinks)):
        assert torch.equal(x, y)
    c = W.make_decode(4, 8, 2, (10, 100), seed=4)
    assert not torch.equal(a.q, c.q)


def test_tiny_decode_shape():
    t = W.tiny_decode()
    assert t.q.shape == (1, 4, 64) and t.k_pages.shape == (8, 1, 16, 64)
    assert t.page_table.tolist() == [list(range(8))]
    assert t.kv_lens.tolist() == [128]
    assert abs(t.scale - 0.125) < 1e-12


def test_batched_paged_decode_shape():
    d = W.batched_paged_decode()
    lens = d.kv_lens.tolist()
    assert len(lens) == 32 and all(512 <= L <= 4096 for L in lens)
    npg = [(L + 15) // 16 for L in lens]
    assert d.k_pages.shape == (sum(npg), 8, 16, 64) and d.q.shape == (32, 64, 64)
    used = torch.cat([d.page_table[b, :n] for b, n in enumerate(npg)])
    assert sorted(used.tolist()) == list(range(sum(npg)))  # every pool page used exactly once
    assert all((d.page_table[b, n:] == -1).all() for b, n in enumerate(npg))


def test_prefill_shape():
    p = W.make_prefill(8, 2, (5, 3, 40), seed=1)
    cu = p.cu_seqlens.tolist()
    assert cu[0] == 0 and len(cu) == 6 and cu[-1] == p.q.shape[0]
    assert all(3 <= L <= 40 for L in p.seqlens)
    assert p.visible_pairs() == sum(L * (L + 1) // 2 for L in p.seqlens)


def test_speculative_verify_shape():
    d = W.speculative_verify()
    lens = d.kv_lens.tolist()
    assert d.q.shape == (32, 4, 64, 64) and len(lens) == 32 and all(512 <= L <= 4096 for L in lens)
    npg = [(L + 15) // 16 for L in lens]
    assert d.k_pages.shape == (sum(npg), 8, 16, 64)
    # the same lengths and pool as the one-token workload: only q differs in size
    b = W.batched_paged_decode()
    assert lens == b.kv_lens.tolist() and torch.equal(d.page_table, b.page_table)
