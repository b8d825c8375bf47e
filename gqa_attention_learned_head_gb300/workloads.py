"""Seeded synthetic inputs for sink attention.

This module draws random inputs and nothing else: it holds none of the
method's arithmetic.  Both the CUDA path and the CPU oracle are fed from it.

Draw order, for every workload: lengths -> page permutation -> q -> k -> v
-> sinks, from one ``torch.Generator`` seeded with ``seed``.  Normals are
drawn in fp32 and rounded to bf16 (round-to-nearest-even); sinks stay fp32.
Lengths are inclusive-uniform.  A normal written N(0, v) has variance v.

The five named workloads reproduce the sizes and distributions of the
benchmark set used for this library (decode over a paged KV cache, long
context split-KV decode, causal varlen prefill and a mixed serving batch);
the blog posts that describe the method publish no inputs, so all of them
are synthetic.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import torch

HEAD_DIM = 64
PAGE_SIZE = 16


@dataclass
class DecodeInputs:
    q: torch.Tensor           # [B, Hq, D] bf16
    k_pages: torch.Tensor     # [P, Hkv, PS, D] bf16
    v_pages: torch.Tensor     # [P, Hkv, PS, D] bf16
    page_table: torch.Tensor  # [B, max_pages] int32, unused entries -1
    kv_lens: torch.Tensor     # [B] int32
    sinks: torch.Tensor       # [Hq] f32
    scale: float

    @property
    def shape(self):
        B, Hq, D = self.q.shape
        return dict(B=B, Hq=Hq, Hkv=self.k_pages.shape[1], D=D,
                    num_pages=self.k_pages.shape[0], max_pages=self.page_table.shape[1])

    def to(self, device):
        return DecodeInputs(*(t.to(device) for t in (self.q, self.k_pages, self.v_pages,
                                                     self.page_table, self.kv_lens, self.sinks)),
                            self.scale)

    def kv_tokens(self) -> int:
        return int(self.kv_lens.to(torch.int64).sum())


@dataclass
class PrefillInputs:
    q: torch.Tensor           # [T, Hq, D] bf16
    k: torch.Tensor           # [T, Hkv, D] bf16
    v: torch.Tensor           # [T, Hkv, D] bf16
    cu_seqlens: torch.Tensor  # [N+1] int32
    sinks: torch.Tensor       # [Hq] f32
    scale: float
    causal: bool = True
    seqlens: list = field(default_factory=list)

    def to(self, device):
        return PrefillInputs(self.q.to(device), self.k.to(device), self.v.to(device),
                             self.cu_seqlens.to(device), self.sinks.to(device), self.scale,
                             self.causal, list(self.seqlens))

    @property
    def max_seqlen(self) -> int:
        return max(self.seqlens) if self.seqlens else 0

    def visible_pairs(self) -> int:
        """Number of (query row, visible key) pairs per head."""
        if self.causal:
            return sum(L * (L + 1) // 2 for L in self.seqlens)
        return sum(L * L for L in self.seqlens)


def _normal_bf16(gen, shape, device, std=1.0, chunk=1 << 26):
    """N(0, std^2) in fp32, rounded to bf16, drawn in fixed-size chunks."""
    n = math.prod(shape)
    out = torch.empty(n, dtype=torch.bfloat16, device=device)
    for lo in range(0, n, chunk):
        hi = min(n, lo + chunk)
        x = torch.randn(hi - lo, generator=gen, device=device, dtype=torch.float32)
        if std != 1.0:
            x.mul_(std)
        out[lo:hi] = x.to(torch.bfloat16)
    return out.view(shape)


def _generator(seed, device):
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def make_decode(B, Hq, Hkv, kv_lens, seed=0, sink_std=1.0, contiguous=False,
                device="cpu", D=HEAD_DIM, PS=PAGE_SIZE, extra_pages=0,
                max_pages=None, q_len=None) -> DecodeInputs:
    """Paged decode inputs.

    kv_lens: a list of B ints, or a (lo, hi) tuple for inclusive-uniform
    lengths.  The pool holds exactly the pages the requests need (plus
    ``extra_pages`` unused ones), in a random order unless ``contiguous``.
    q_len: None for one query token per request (q [B, Hq, D]); an int for
    verification inputs, q [B, q_len, Hq, D] -- the last q_len cached tokens
    of every request (kv_lens counts them).
    """
    g = _generator(seed, device)
    if isinstance(kv_lens, tuple):
        lo, hi = kv_lens
        lens = torch.randint(lo, hi + 1, (B,), generator=g, device=device).cpu().tolist()
    else:
        lens = [int(x) for x in kv_lens]
        assert len(lens) == B
    npages = [(L + PS - 1) // PS for L in lens]
    P = sum(npages) + extra_pages
    if contiguous:
        perm = torch.arange(P)
    else:
        perm = torch.randperm(P, generator=g, device=device).cpu()
    mp = max(max(npages, default=0), 1) if max_pages is None else max_pages
    pt = torch.full((B, mp), -1, dtype=torch.int32)
    off = 0
    for b, n in enumerate(npages):
        pt[b, :n] = perm[off:off + n].to(torch.int32)
        off += n
    q = _normal_bf16(g, (B, Hq, D) if q_len is None else (B, q_len, Hq, D), device)
    kp = _normal_bf16(g, (P, Hkv, PS, D), device)
    vp = _normal_bf16(g, (P, Hkv, PS, D), device)
    sinks = torch.randn(Hq, generator=g, device=device, dtype=torch.float32) * sink_std
    return DecodeInputs(q, kp, vp, pt.to(device), torch.tensor(lens, dtype=torch.int32, device=device),
                        sinks, 1.0 / math.sqrt(D))


@dataclass
class PagedPrefillInputs:
    q: torch.Tensor           # [T, Hq, D] bf16   new tokens packed by cu_seqlens
    k_new: torch.Tensor       # [T, Hkv, D] bf16  their keys, to be appended to the pages
    v_new: torch.Tensor       # [T, Hkv, D] bf16
    k_pages: torch.Tensor     # [P, Hkv, PS, D] bf16  holds the cached prefixes
    v_pages: torch.Tensor
    page_table: torch.Tensor  # [N, max_pages] int32, room for prefix + new tokens
    cu_seqlens: torch.Tensor  # [N+1] int32 over the new tokens
    start_pos: torch.Tensor   # [N] int32 cached tokens of each sequence
    sinks: torch.Tensor       # [Hq] f32
    scale: float
    new_lens: list = field(default_factory=list)

    def to(self, device):
        return PagedPrefillInputs(*(t.to(device) for t in (self.q, self.k_new, self.v_new, self.k_pages,
                                                           self.v_pages, self.page_table, self.cu_seqlens,
                                                           self.start_pos, self.sinks)),
                                  self.scale, list(self.new_lens))

    @property
    def max_seqlen(self) -> int:
        return max(self.new_lens) if self.new_lens else 0

    def visible_pairs(self) -> int:
        """(new token, visible cached token) pairs per head."""
        return sum(L * s + L * (L + 1) // 2 for L, s in zip(self.new_lens, self.start_pos.tolist()))


def make_paged_prefill(Hq, Hkv, prefix_lens, new_lens, seed=0, device="cpu", D=HEAD_DIM, PS=PAGE_SIZE):
    """Chunked prefill inputs over a paged cache.

    prefix_lens / new_lens: lists of N ints, or (lo, hi) tuples for inclusive-uniform lengths (N from
    the other argument, or 8).  Each sequence gets the pages for prefix + new tokens, randomly
    permuted in the pool; the pool is drawn whole (the prefix slots hold the cached K/V, the others
    noise that the appended tokens overwrite).  Draw order: lengths -> page permutation -> q ->
    k_pages -> v_pages -> k_new -> v_new -> sinks.
    """
    g = _generator(seed, device)
    N = len(prefix_lens) if isinstance(prefix_lens, list) else (len(new_lens) if isinstance(new_lens, list) else 8)

    def draw(spec):
        if isinstance(spec, tuple):
            return torch.randint(spec[0], spec[1] + 1, (N,), generator=g, device=device).cpu().tolist()
        return [int(x) for x in spec]

    pre, new = draw(prefix_lens), draw(new_lens)
    npages = [(p + n + PS - 1) // PS for p, n in zip(pre, new)]
    P = max(sum(npages), 1)
    perm = torch.randperm(P, generator=g, device=device).cpu()
    pt = torch.full((N, max(max(npages, default=0), 1)), -1, dtype=torch.int32)
    off = 0
    for b, n in enumerate(npages):
        pt[b, :n] = perm[off:off + n].to(torch.int32)
        off += n
    T = sum(new)
    q = _normal_bf16(g, (T, Hq, D), device)
    kp = _normal_bf16(g, (P, Hkv, PS, D), device)
    vp = _normal_bf16(g, (P, Hkv, PS, D), device)
    kn = _normal_bf16(g, (T, Hkv, D), device)
    vn = _normal_bf16(g, (T, Hkv, D), device)
    sinks = torch.randn(Hq, generator=g, device=device, dtype=torch.float32)
    cu = torch.tensor([0] + list(torch.tensor(new).cumsum(0).tolist()), dtype=torch.int32, device=device)
    return PagedPrefillInputs(q, kn, vn, kp, vp, pt.to(device), cu, torch.tensor(pre, dtype=torch.int32, device=device),
                              sinks, 1.0 / math.sqrt(D), new)


def make_prefill(Hq, Hkv, seqlens, seed=0, causal=True, device="cpu", D=HEAD_DIM,
                 sink_std=1.0) -> PrefillInputs:
    """Packed varlen prefill inputs; seqlens: list, or (N, lo, hi) for inclusive-uniform."""
    g = _generator(seed, device)
    if isinstance(seqlens, tuple):
        N, lo, hi = seqlens
        lens = torch.randint(lo, hi + 1, (N,), generator=g, device=device).cpu().tolist()
    else:
        lens = [int(x) for x in seqlens]
    cu = [0]
    for L in lens:
        cu.append(cu[-1] + L)
    T = cu[-1]
    q = _normal_bf16(g, (T, Hq, D), device)
    k = _normal_bf16(g, (T, Hkv, D), device)
    v = _normal_bf16(g, (T, Hkv, D), device)
    sinks = torch.randn(Hq, generator=g, device=device, dtype=torch.float32) * sink_std
    return PrefillInputs(q, k, v, torch.tensor(cu, dtype=torch.int32, device=device), sinks,
                         1.0 / math.sqrt(D), causal, lens)


# ---- the named benchmark workloads -------------------------------------------------

def tiny_decode(device="cpu", seed=0):
    """Batch 1, 4 query heads on 1 KV head, kv_len 128, contiguous pages, seed 0."""
    return make_decode(1, 4, 1, [128], seed=seed, contiguous=True, device=device)


def batched_paged_decode(device="cpu", seed=0):
    """Batch 32, 64 q / 8 KV heads, kv_len uniform in [512, 4096], permuted pages."""
    return make_decode(32, 64, 8, (512, 4096), seed=seed, device=device)


def tree_masks(parents) -> list:
    """Attention masks of a draft tree (or forest) given by parent indices (-1 for a root, parents
    before children): bit j of mask i is set iff draft token j is token i or one of its ancestors."""
    masks = []
    for i, p in enumerate(parents):
        assert p < i, "parents must come before their children"
        masks.append((masks[p] if p >= 0 else 0) | (1 << i))
    return masks


# An EAGLE-style draft tree of 8 tokens, depth 4: the last accepted token (0) with two candidate
# continuations, the first of them expanded twice, then one more level on two branches.
DRAFT_TREE_PARENTS = [-1, 0, 0, 1, 1, 2, 3, 5]


def tree_verify(device="cpu", seed=0):
    """Verification of a draft tree: the batched paged decode's lengths and pool with 8 drafted
    tokens per request (the tree DRAFT_TREE_PARENTS, same for every request), 64 q / 8 KV heads.
    Returns (inputs, tree_mask [B, 8] int64)."""
    inp = make_decode(32, 64, 8, (512, 4096), seed=seed, device=device, q_len=len(DRAFT_TREE_PARENTS))
    m = torch.tensor(tree_masks(DRAFT_TREE_PARENTS), dtype=torch.int64, device=device)
    return inp, m.expand(32, -1).contiguous()


def speculative_verify(device="cpu", seed=0):
    """Verification of drafts: batch 32, 4 query tokens per request (3 drafted + the last
    accepted one), 64 q / 8 KV heads, kv_len U[512, 4096] including the 4, permuted pages."""
    return make_decode(32, 64, 8, (512, 4096), seed=seed, device=device, q_len=4)


def long_context_decode(device="cpu", seed=0):
    """Batch 4, 64 q / 8 KV heads, kv_len 131072 each (8192 pages), sinks N(0, 2)."""
    return make_decode(4, 64, 8, [131072] * 4, seed=seed, sink_std=math.sqrt(2.0), device=device)


LONG_CONTEXT_CHUNKS = 32  # the long-context workload splits each request into 32 chunks


def causal_prefill(device="cpu", seed=0):
    """Two sequences of 8192 tokens, 64 q / 8 KV heads, causal."""
    return make_prefill(64, 8, [8192, 8192], seed=seed, device=device)


def chunked_prefill(device="cpu", seed=0):
    """Chunked prefill over the paged cache: 8 sequences with U[1024, 8192] cached tokens each taking
    U[256, 2048] new tokens, 64 q / 8 KV heads."""
    return make_paged_prefill(64, 8, (1024, 8192), (256, 2048), seed=seed, device=device)


def mixed_serving_prefill(device="cpu", seed=0):
    """The prefill half of the mixed serving batch: 8 causal sequences, lengths in [256, 4096]."""
    return make_prefill(64, 8, (8, 256, 4096), seed=seed, device=device)


def mixed_serving_decode(device="cpu", seed=0):
    """The decode half of the mixed serving batch: 256 paged requests, kv_len in [1024, 32768]."""
    return make_decode(256, 64, 8, (1024, 32768), seed=seed + 1, device=device)


def mixed_serving(device="cpu", seed=0):
    """8 causal prefills with lengths in [256, 4096] plus 256 paged decodes with kv_len in [1024, 32768].

    The prefill part is drawn from ``seed`` and the decode part from ``seed + 1``.
    """
    return mixed_serving_prefill(device, seed), mixed_serving_decode(device, seed)


WORKLOADS = {
    "tiny_decode": tiny_decode,
    "batched_paged_decode": batched_paged_decode,
    "long_context_decode": long_context_decode,
    "causal_prefill": causal_prefill,
    "mixed_serving": mixed_serving,
}
