"""GPU LSE merge against the fp64 oracle merge, through the C ABI."""
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


def gpu_merge(S, po, pl, sinks=None):
    t = lambda x: torch.as_tensor(np.ascontiguousarray(x), dtype=torch.float32, device="cuda")
    out, lse = S.sinkattn_merge(t(po), t(pl), None if sinks is None else t(sinks))
    assert S.sinkattn_get_error() == 0
    return out.float().cpu().numpy(), lse.cpu().numpy()


@pytest.mark.parametrize("S_", [1, 2, 7, 32])
@pytest.mark.parametrize("route", ["first_chunk", "merge_adds"])
def test_merge_of_decode_partials(S, S_, route):
    lens = [0, 1, 15, 16, 17, 300, 511, 2048]
    inp = W.make_decode(len(lens), 16, 2, lens, seed=S_)
    chunk = max(1, -(-max(lens) // S_))
    mode = oracle.SINK_IN_FIRST_CHUNK if route == "first_chunk" else oracle.SINK_IN_NO_CHUNK
    po, pl = oracle.decode_partials(inp.q, inp.k_pages, inp.v_pages, inp.page_table, inp.kv_lens, inp.sinks,
                                    inp.scale, S_, chunk, sink_mode=mode)
    sinks = None if route == "first_chunk" else inp.sinks.numpy()
    # the GPU merges the fp32-rounded partials; the oracle merges the same fp32 values
    po32, pl32 = po.astype(np.float32), pl.astype(np.float32)
    ro, rl = oracle.merge(po32.astype(np.float64), pl32.astype(np.float64), sinks)
    go, gl = gpu_merge(S, po32, pl32, sinks)
    assert_parity(go, gl, ro, rl, f"S={S_} {route}")
    # and split + merge equals the unsplit decode
    uo, ul = oracle.decode(inp.q, inp.k_pages, inp.v_pages, inp.page_table, inp.kv_lens, inp.sinks, inp.scale)
    assert_parity(go, gl, uo, ul, "vs unsplit")


def test_merge_edge_rows(S):
    po = np.random.default_rng(0).standard_normal((3, 4, 2, 64)).astype(np.float32)
    pl = np.full((3, 4, 2), -np.inf, np.float32)
    pl[1, 1, 0] = 0.5                     # one live split
    pl[:, 2, 1] = [1.0, 2.0, -np.inf]     # two live + one empty (its o is ignored)
    po[2, 2, 1] = np.nan
    for sinks in (None, np.array([0.25, -np.inf], np.float32)):
        ro, rl = oracle.merge(po.astype(np.float64), pl.astype(np.float64), sinks)
        go, gl = gpu_merge(S, po, pl, sinks)
        assert_parity(go, gl, ro, rl, f"edge rows sinks={sinks}")


def test_merge_zero_splits_with_sink(S):
    po = np.zeros((0, 3, 2, 64), np.float32)
    pl = np.zeros((0, 3, 2), np.float32)
    go, gl = gpu_merge(S, po, pl, np.array([0.5, -1.0], np.float32))
    assert np.all(go == 0)
    np.testing.assert_allclose(gl, np.tile([0.5, -1.0], (3, 1)), rtol=0, atol=1e-6)
