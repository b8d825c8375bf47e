"""The cubic for 2^f used by the prefill kernel's FMA-pipe exp2 path: the constants in the kernel
source are the ones the derivation script produces, and its relative error on [-1/2, 1/2] is
below 1e-4 (bf16 probabilities are rounded at 2^-9, so the approximation is invisible)."""
import importlib.util
import re
from pathlib import Path

import numpy as np

CSRC = Path(__file__).resolve().parents[1] / "gqa_attention_learned_head_gb300" / "csrc"


def _script():
    spec = importlib.util.spec_from_file_location("exp2_poly", CSRC / "exp2_poly.py")
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def kernel_constants():
    src = (CSRC / "tc_tile.cuh").read_text()
    return np.array([float(re.search(rf"kExp2C{i} = ([0-9.e+-]+)f;", src).group(1)) for i in range(4)],
                    dtype=np.float32)


def test_kernel_constants_match_derivation():
    np.testing.assert_array_equal(kernel_constants(), _script().fit())


def test_relative_error_bound():
    c = kernel_constants().astype(np.float64)
    f = np.linspace(-0.5, 0.5, 100001)
    p = ((c[3] * f + c[2]) * f + c[1]) * f + c[0]
    assert np.max(np.abs(p / 2.0 ** f - 1.0)) < 1e-4


def test_full_range_reconstruction_in_float32():
    """2^x = 2^round(x) * p(x - round(x)) rebuilt with float32 bit arithmetic, as the kernel does."""
    c = kernel_constants()
    x = np.linspace(-125.0, 15.0, 200001).astype(np.float32)  # the kernel clamps at -125
    t = x + np.float32(12582912.0)
    r = t - np.float32(12582912.0)
    f = x - r
    p = ((c[3] * f + c[2]) * f + c[1]) * f + c[0]
    bits = p.view(np.int32) + (t.view(np.int32) << 23)
    y = bits.view(np.float32).astype(np.float64)
    np.testing.assert_allclose(y, 2.0 ** x.astype(np.float64), rtol=1e-4, atol=0)
