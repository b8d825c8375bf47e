"""GPU causal varlen prefill against the fp64 oracle, through the C ABI."""
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


def run(S, inp, max_seqlen=None):
    g = inp.to("cuda")
    out, lse = S.sinkattn_prefill(g.q, g.k, g.v, g.cu_seqlens, g.sinks, g.scale, g.causal,
                                  max_seqlen=inp.max_seqlen if max_seqlen is None else max_seqlen)
    err = S.sinkattn_get_error()
    return out.float().cpu().numpy(), lse.cpu().numpy(), err


def ref(inp, rows=None):
    return oracle.prefill(inp.q, inp.k, inp.v, inp.cu_seqlens, inp.sinks, inp.scale, inp.causal, rows=rows)


@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("lens", [[1], [127, 128, 129], [300, 5, 64, 1000]])
@pytest.mark.parametrize("Hq,Hkv", [(8, 2), (16, 2), (4, 4)])
def test_small_varlen(S, causal, lens, Hq, Hkv):
    inp = W.make_prefill(Hq, Hkv, lens, seed=len(lens) + Hq, causal=causal)
    out, lse, err = run(S, inp)
    assert err == 0
    assert_parity(out, lse, *ref(inp), f"lens={lens} causal={causal} Hq={Hq} Hkv={Hkv}")


@pytest.mark.parametrize("sink", [float("-inf"), -30.0, 30.0])
def test_sink_values(S, sink):
    inp = W.make_prefill(8, 1, [200, 77], seed=2)
    inp.sinks[:] = sink
    out, lse, err = run(S, inp)
    assert err == 0
    assert_parity(out, lse, *ref(inp), f"sink={sink}")


def test_empty_sequences_in_batch(S):
    inp = W.make_prefill(8, 2, [0, 50, 0, 130, 0], seed=3)
    out, lse, err = run(S, inp)
    assert err == 0
    assert_parity(out, lse, *ref(inp), "empty sequences")


@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("N", [33, 128, 129, 300])
@pytest.mark.parametrize("Hq,Hkv", [(8, 2), (6, 2)])
def test_many_sequences(S, causal, N, Hq, Hkv):
    """Batches ranked four keys per lane (33..128 sequences) and past the ranked limit (index order);
    lengths repeat and include 0, so ties and empty sequences occur in the order."""
    lens = np.random.default_rng(N).choice([0, 1, 17, 64, 129, 200], size=N).tolist()
    inp = W.make_prefill(Hq, Hkv, lens, seed=N + Hq, causal=causal)
    out, lse, err = run(S, inp)
    assert err == 0
    assert_parity(out, lse, *ref(inp), f"N={N} causal={causal} Hq={Hq} Hkv={Hkv}")


def test_maximum_sequence_count(S):
    """16384 sequences, the most a prefill call takes: the tile order runs in index order from its
    largest table.  Lengths 0..3 with 40 sequences of 130 (two tiles, the second ragged)."""
    rng = np.random.default_rng(16384)
    lens = rng.choice([0, 1, 2, 3], size=16384)
    lens[rng.choice(16384, 40, replace=False)] = 130
    inp = W.make_prefill(8, 2, lens.tolist(), seed=5)
    out, lse, err = run(S, inp)
    assert err == 0
    assert_parity(out, lse, *ref(inp), "16384 sequences")


@pytest.mark.parametrize("causal", [True, False])
def test_share_sms_matches_oracle(S, causal):
    """The kernel that leaves room on every SM (share_sms) computes the same attention."""
    inp = W.make_prefill(64, 8, [300, 5, 64, 1000, 129], seed=31, causal=causal)
    g = inp.to("cuda")
    out, lse = S.sinkattn_prefill(g.q, g.k, g.v, g.cu_seqlens, g.sinks, g.scale, causal, max_seqlen=inp.max_seqlen,
                                  share_sms=True)
    assert S.sinkattn_get_error() == 0
    assert_parity(out.float().cpu().numpy(), lse.cpu().numpy(), *ref(inp), f"share_sms causal={causal}")


def test_decode_and_prefill_side_by_side(S):
    """A decode with two shares per SM and a prefill that shares the SMs, launched on two streams
    at once (the mixed-batch schedule): both match the oracle."""
    dec = W.make_decode(64, 64, 8, (256, 2048), seed=33)
    pre = W.make_prefill(64, 8, [700, 1300, 90, 2048], seed=34)
    gd, gp = dec.to("cuda"), pre.to("cuda")
    workers = 2 * torch.cuda.get_device_properties(0).multi_processor_count
    ws = torch.empty(S.sinkattn_decode_workspace_size(gd.q, gd.k_pages, gd.page_table, workers), dtype=torch.uint8,
                     device="cuda")
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    main = torch.cuda.current_stream()
    s1.wait_stream(main)
    s2.wait_stream(main)
    dout, dlse = S.sinkattn_decode(gd.q, gd.k_pages, gd.v_pages, gd.page_table, gd.kv_lens, gd.sinks, gd.scale,
                                   workspace=ws, num_workers=workers, stream=s2)
    pout, plse = S.sinkattn_prefill(gp.q, gp.k, gp.v, gp.cu_seqlens, gp.sinks, gp.scale, True,
                                    max_seqlen=pre.max_seqlen, share_sms=True, stream=s1)
    main.wait_stream(s1)
    main.wait_stream(s2)
    torch.cuda.synchronize()
    assert S.sinkattn_get_error() == 0
    ro, rl = oracle.decode(dec.q, dec.k_pages, dec.v_pages, dec.page_table, dec.kv_lens, dec.sinks, dec.scale)
    assert_parity(dout.float().cpu().numpy(), dlse.cpu().numpy(), ro, rl, "decode beside the prefill")
    assert_parity(pout.float().cpu().numpy(), plse.cpu().numpy(), *ref(pre), "prefill beside the decode")


def sampled_rows(inp, n, seed):
    rng = np.random.default_rng(seed)
    cu = inp.cu_seqlens.tolist()
    T, Hq = inp.q.shape[0], inp.q.shape[1]
    toks = list(rng.integers(0, T, n))
    # always include every sequence's first and last row and a tile boundary
    for s in range(len(cu) - 1):
        if cu[s + 1] > cu[s]:
            toks += [cu[s], cu[s + 1] - 1, min(cu[s] + 128, cu[s + 1] - 1)]
    hs = rng.integers(0, Hq, len(toks))
    return np.stack([np.array(toks), hs], 1).astype(np.int32)


def test_causal_prefill_full_size_sampled(S):
    inp = W.causal_prefill()
    out, lse, err = run(S, inp)
    assert err == 0
    assert np.all(np.isfinite(out)) and np.all(np.isfinite(lse))
    rows = sampled_rows(inp, 96, 0)
    ro, rl = ref(inp, rows)
    assert_parity(out[rows[:, 0], rows[:, 1]], lse[rows[:, 0], rows[:, 1]], ro, rl, "causal prefill 2x8192")


def test_mixed_serving_prefill_sampled(S):
    inp = W.mixed_serving_prefill()
    out, lse, err = run(S, inp)
    assert err == 0
    rows = sampled_rows(inp, 96, 1)
    ro, rl = ref(inp, rows)
    assert_parity(out[rows[:, 0], rows[:, 1]], lse[rows[:, 0], rows[:, 1]], ro, rl, "mixed prefill")


def test_causal_prefill_every_row(S):
    """The full-size causal prefill (2 x 8192 tokens, 64 q / 8 KV heads), every one of its 1 048 576
    rows against the oracle (a minute or two of the oracle on the host cores)."""
    inp = W.causal_prefill()
    out, lse, err = run(S, inp)
    assert err == 0
    assert_parity(out, lse, *ref(inp), "causal prefill 2x8192, every row")


def test_mixed_serving_prefill_every_row(S):
    inp = W.mixed_serving_prefill()
    out, lse, err = run(S, inp)
    assert err == 0
    assert_parity(out, lse, *ref(inp), "mixed prefill, every row")


def test_too_long_sequence_is_reported(S):
    inp = W.make_prefill(4, 1, [100, 40], seed=4)
    out, lse, err = run(S, inp, max_seqlen=64)
    assert err == S.ERR_BAD_LENGTH


def test_long_single_sequence_sampled(S):
    """A 65536-token causal sequence (512 query tiles) next to a 3-token one; sampled rows include the
    last rows, which see every key."""
    inp = W.make_prefill(16, 2, [65536, 3], seed=21)
    out, lse, err = run(S, inp)
    assert err == 0
    rows = sampled_rows(inp, 64, 2)
    rows = np.concatenate([rows, np.array([[65535, h] for h in range(16)], dtype=np.int32)])
    ro, rl = ref(inp, rows)
    assert_parity(out[rows[:, 0], rows[:, 1]], lse[rows[:, 0], rows[:, 1]], ro, rl, "65536-token sequence")
