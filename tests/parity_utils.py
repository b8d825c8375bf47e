"""Shared helpers for GPU-vs-oracle parity tests.

Tolerances are the ones the method's benchmark set states for bf16 outputs:
max |out - ref| <= 2e-2, mean |out - ref| <= 2e-3, and |lse - ref| <= 1e-3
(natural log).  An lse of -inf must match -inf exactly.
"""
import numpy as np

MAX_ABS = 2e-2
MEAN_ABS = 2e-3
LSE_TOL = 1e-3


def assert_parity(out, lse, ref_out, ref_lse, what=""):
    out = np.asarray(out, dtype=np.float64)
    ref_out = np.asarray(ref_out, dtype=np.float64)
    assert out.shape == ref_out.shape, (what, out.shape, ref_out.shape)
    assert np.all(np.isfinite(out)), f"{what}: non-finite output"
    diff = np.abs(out - ref_out)
    assert diff.max() <= MAX_ABS, f"{what}: max abs error {diff.max():.3e}"
    assert diff.mean() <= MEAN_ABS, f"{what}: mean abs error {diff.mean():.3e}"
    if lse is not None:
        lse = np.asarray(lse, dtype=np.float64)
        ref_lse = np.asarray(ref_lse, dtype=np.float64)
        assert lse.shape == ref_lse.shape
        inf_g, inf_r = np.isneginf(lse), np.isneginf(ref_lse)
        assert np.array_equal(inf_g, inf_r), f"{what}: -inf pattern of lse differs"
        assert not np.any(np.isnan(lse)), f"{what}: NaN lse"
        if (~inf_r).any():
            dl = np.abs(lse[~inf_r] - ref_lse[~inf_r]).max()
            assert dl <= LSE_TOL, f"{what}: lse error {dl:.3e}"
    return float(np.abs(out - ref_out).max())


def growing_scores(inp, top=5.0, seed=0):
    """The same request set with scores that rise along the cache: q ~ 1 and the key of cache position
    pos ~ top * pos / kv_len (plus a little noise), so at the 1/8 scale of head_dim 64 a request's last
    query sees scores from ~0 to ~8 * top (natural units).  The running max of an online softmax then
    grows steadily, past any lazy-rescale threshold, instead of settling early."""
    import torch

    from gqa_attention_learned_head_gb300.workloads import DecodeInputs

    g = torch.Generator().manual_seed(seed)
    q = (1.0 + 0.05 * torch.randn(inp.q.shape, generator=g)).to(torch.bfloat16)
    k = inp.k_pages.float().clone()
    _, Hkv, PS, D = k.shape
    for b in range(inp.kv_lens.shape[0]):
        L = int(inp.kv_lens[b])
        for j in range((L + PS - 1) // PS):
            p = int(inp.page_table[b, j])
            pos = torch.arange(j * PS, (j + 1) * PS, dtype=torch.float32)
            k[p] = (top * pos / L)[None, :, None] + 0.05 * torch.randn(Hkv, PS, D, generator=g)
    return DecodeInputs(q, k.to(torch.bfloat16), inp.v_pages, inp.page_table, inp.kv_lens, inp.sinks, inp.scale)
