"""libsinkattn loads, exports every entry point its header declares, and
rejects bad arguments on the host before touching a device (no GPU needed)."""
import ctypes
import re
from pathlib import Path

import pytest

ROOT = Path(__file__).resolve().parents[1]


@pytest.fixture(scope="module")
def S():
    from gqa_attention_learned_head_gb300 import build

    build.build()
    from gqa_attention_learned_head_gb300 import sinkattn

    return sinkattn


def declared_functions():
    text = (ROOT / "include" / "sinkattn.h").read_text()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(sinkattn_\w+)\s*\(", text)))


def test_header_declares_the_three_calls():
    names = declared_functions()
    for fn in ("sinkattn_decode", "sinkattn_prefill", "sinkattn_merge"):
        assert fn in names


def documented_functions():
    """Entry points listed in the design document's boundary section (the paragraph that opens with
    "Exported entry points")."""
    text = (ROOT / "DESIGN.md").read_text()
    para = text[text.index("Exported entry points"):]
    para = para[:para.index("\n\n")]
    para = para[para.index(":\n") + 2:]
    return sorted(set(re.findall(r"`(sinkattn_\w+)`", para)))


def test_documented_entry_points_match_the_header():
    assert documented_functions() == declared_functions()


def test_library_exports_every_declared_symbol(S):
    lib = ctypes.CDLL(S.library_path)
    for fn in declared_functions():
        assert hasattr(lib, fn), f"{fn} not exported"
    assert set(S.EXPORTS) <= set(declared_functions())


def test_status_strings(S):
    assert S.status_string(0) == "ok"
    assert "page" in S.status_string(S.ERR_BAD_PAGE)
    assert S.status_string(99) == "unknown status"
    assert S.version() >= 10000


def test_host_validation_without_device(S):
    lib = S._lib
    d = S.DecodeDims(2, 8, 2, 32, 16, 10, 4, 0)  # head_dim 32
    st = lib.sinkattn_decode(None, None, None, None, None, None, 0.125, None, None, ctypes.byref(d), None, 0, None)
    assert st == S.ERR_UNSUPPORTED
    d = S.DecodeDims(2, 8, 3, 64, 16, 10, 4, 0)  # Hq % Hkv != 0
    assert lib.sinkattn_decode(None, None, None, None, None, None, 0.125, None, None, ctypes.byref(d), None, 0,
                               None) == S.ERR_INVALID_ARG
    d = S.DecodeDims(2, 64, 2, 64, 16, 10, 4, 0)  # group of 32 heads
    assert lib.sinkattn_decode(None, None, None, None, None, None, 0.125, None, None, ctypes.byref(d), None, 0,
                               None) == S.ERR_UNSUPPORTED
    d = S.DecodeDims(2, 8, 2, 64, 8, 10, 4, 0)  # page size 8
    assert lib.sinkattn_decode(None, None, None, None, None, None, 0.125, None, None, ctypes.byref(d), None, 0,
                               None) == S.ERR_UNSUPPORTED
    assert lib.sinkattn_decode_workspace_size(ctypes.byref(d)) == 0
    p = S.PrefillDims(1, 10, 10, 8, 2, 128)
    assert lib.sinkattn_prefill(None, None, None, None, None, 0.1, 1, None, None, ctypes.byref(p), None) == \
        S.ERR_UNSUPPORTED
    p = S.PrefillDims(-1, 10, 10, 8, 2, 64)
    assert lib.sinkattn_prefill(None, None, None, None, None, 0.1, 1, None, None, ctypes.byref(p), None) == \
        S.ERR_INVALID_ARG
    p = S.PrefillDims(1, 10, 10, 8, 2, 64, 2)  # share_sms is 0 or 1
    assert lib.sinkattn_prefill(None, None, None, None, None, 0.1, 1, None, None, ctypes.byref(p), None) == \
        S.ERR_INVALID_ARG
    m = S.MergeDims(2, 4, 0, 64)
    assert lib.sinkattn_merge(None, None, None, None, None, ctypes.byref(m), None) == S.ERR_INVALID_ARG
    assert lib.sinkattn_merge(None, None, None, None, None, None, None) == S.ERR_INVALID_ARG


def test_verify_host_validation_without_device(S):
    lib = S._lib
    nul = [None] * 6

    def call(d):
        return lib.sinkattn_verify(*nul, 0.125, None, None, ctypes.byref(d), None, 0, None)

    assert call(S.VerifyDims(2, 0, 8, 2, 64, 16, 10, 4, 0)) == S.ERR_INVALID_ARG       # q_len 0
    assert call(S.VerifyDims(2, 17, 8, 8, 64, 16, 10, 4, 0)) == S.ERR_UNSUPPORTED      # q_len 17
    assert call(S.VerifyDims(2, 9, 64, 8, 64, 16, 10, 4, 0)) == S.ERR_UNSUPPORTED      # 9 x 8 = 72 rows
    assert call(S.VerifyDims(2, 4, 8, 3, 64, 16, 10, 4, 0)) == S.ERR_INVALID_ARG       # Hq % Hkv != 0
    assert call(S.VerifyDims(2, 4, 8, 2, 32, 16, 10, 4, 0)) == S.ERR_UNSUPPORTED       # head_dim 32
    assert lib.sinkattn_verify_workspace_size(ctypes.byref(S.VerifyDims(2, 9, 64, 8, 64, 16, 10, 4, 0))) == 0
    assert call(S.VerifyDims(0, 4, 8, 2, 64, 16, 10, 4, 0)) == 0                       # empty batch: nothing to do


def test_paged_host_validation_without_device(S):
    lib = S._lib
    d = S.PagedDims(2, 10, 8, 8, 2, 32, 16, 10, 4)  # head_dim 32
    assert lib.sinkattn_kv_append(*([None] * 7), ctypes.byref(d), None) == S.ERR_UNSUPPORTED
    assert lib.sinkattn_prefill_paged(*([None] * 7), 0.125, None, None, ctypes.byref(d), None) == S.ERR_UNSUPPORTED
    d = S.PagedDims(2, 10, 8, 8, 3, 64, 16, 10, 4)  # Hq % Hkv != 0
    assert lib.sinkattn_prefill_paged(*([None] * 7), 0.125, None, None, ctypes.byref(d), None) == S.ERR_INVALID_ARG
    d = S.PagedDims(2, 10, 8, 8, 2, 64, 16, 10, 0)  # max_pages 0
    assert lib.sinkattn_kv_append(*([None] * 7), ctypes.byref(d), None) == S.ERR_INVALID_ARG
    d = S.PagedDims(2, 10, 8, 8, 2, 64, 16, 10, 4, 3)  # share_sms is 0 or 1
    assert lib.sinkattn_prefill_paged(*([None] * 7), 0.125, None, None, ctypes.byref(d), None) == S.ERR_INVALID_ARG
    d = S.PagedDims(0, 0, 0, 8, 2, 64, 16, 10, 4)  # nothing to do
    assert lib.sinkattn_kv_append(*([None] * 7), ctypes.byref(d), None) == 0
    assert lib.sinkattn_prefill_paged(*([None] * 7), 0.125, None, None, ctypes.byref(d), None) == 0


def test_prologue_host_validation_without_device(S):
    lib = S._lib
    d = S.PagedDims(1, 4, 4, 8, 2, 64, 16, 10, 4)
    ok = S.RopeParams(150000.0, 32.0, 4096, 32.0, 1.0, 0.0, 0)
    call = lambda r, dd=d: lib.sinkattn_qkv_prologue(*([None] * 5), ctypes.byref(r) if r else None, None, None, None,
                                                      ctypes.byref(dd), None)
    assert call(None) == S.ERR_INVALID_ARG
    assert call(S.RopeParams(150000.0, 0.5, 4096, 32.0, 1.0, 0.0, 0)) == S.ERR_INVALID_ARG   # factor < 1
    assert call(S.RopeParams(150000.0, 32.0, 4096, 1.0, 32.0, 0.0, 0)) == S.ERR_INVALID_ARG  # beta_fast <= beta_slow
    assert call(ok) == S.ERR_INVALID_ARG  # null buffers
    assert call(ok, S.PagedDims(0, 0, 0, 8, 2, 64, 16, 10, 4)) == 0  # nothing to do


SANITIZED_CHILD = r"""
import ctypes, sys
sys.path.insert(0, sys.argv[1])
from gqa_attention_learned_head_gb300 import abi
lib = abi.declare(ctypes.CDLL(sys.argv[2]))
nul = [None] * 7
codes = []
for d in (abi.DecodeDims(2, 8, 2, 32, 16, 10, 4, 0), abi.DecodeDims(2, 8, 3, 64, 16, 10, 4, 0),
          abi.DecodeDims(2, 64, 2, 64, 16, 10, 4, 0), abi.DecodeDims(-1, 8, 2, 64, 16, 10, 4, 0),
          abi.DecodeDims(2, 8, 2, 64, 16, 10, 0, 0)):
    codes.append(lib.sinkattn_decode(*nul[:6], 0.125, None, None, ctypes.byref(d), None, 0, None))
    codes.append(lib.sinkattn_decode_noalloc(*nul[:6], 0.125, None, None, ctypes.byref(d), None))
    codes.append(int(lib.sinkattn_decode_workspace_size(ctypes.byref(d)) == 0))
codes.append(lib.sinkattn_decode(*nul[:6], 0.125, None, None, None, None, 0, None))
for d in (abi.VerifyDims(2, 0, 8, 2, 64, 16, 10, 4, 0), abi.VerifyDims(2, 17, 8, 8, 64, 16, 10, 4, 0),
          abi.VerifyDims(2, 9, 64, 8, 64, 16, 10, 4, 0), abi.VerifyDims(2, 4, 8, 3, 64, 16, 10, 4, 0)):
    codes.append(lib.sinkattn_verify(*nul[:6], 0.125, None, None, ctypes.byref(d), None, 0, None))
    codes.append(lib.sinkattn_verify_tree(*nul[:7], 0.125, None, None, ctypes.byref(d), None, 0, None))
for d in (abi.PrefillDims(1, 10, 10, 8, 2, 128), abi.PrefillDims(-1, 10, 10, 8, 2, 64),
          abi.PrefillDims(1, 10, 10, 8, 2, 64, 2), abi.PrefillDims(1, 10, 10, 8, 3, 64)):
    codes.append(lib.sinkattn_prefill(*nul[:5], 0.1, 1, None, None, ctypes.byref(d), None))
for d in (abi.PagedDims(2, 10, 8, 8, 2, 32, 16, 10, 4), abi.PagedDims(2, 10, 8, 8, 3, 64, 16, 10, 4),
          abi.PagedDims(2, 10, 8, 8, 2, 64, 16, 10, 0), abi.PagedDims(2, 10, 8, 8, 2, 64, 16, 10, 4, 3),
          abi.PagedDims(20000, 10, 8, 8, 2, 64, 16, 10, 4)):
    codes.append(lib.sinkattn_kv_append(*nul[:7], ctypes.byref(d), None))
    codes.append(lib.sinkattn_prefill_paged(*nul[:7], 0.125, None, None, ctypes.byref(d), None))
    r = abi.RopeParams(150000.0, 0.5, 4096, 32.0, 1.0, 0.0, 0)
    codes.append(lib.sinkattn_qkv_prologue(*nul[:5], ctypes.byref(r), None, None, None, ctypes.byref(d), None))
for d in (abi.MergeDims(2, 4, 0, 64), abi.MergeDims(2, 4, 8, 32), abi.MergeDims(-1, 4, 8, 64)):
    codes.append(lib.sinkattn_merge(*nul[:5], ctypes.byref(d), None))
codes.append(lib.sinkattn_merge(*nul[:5], None, None))
for st in list(range(-3, 12)) + [1 << 30]:
    lib.sinkattn_status_string(st)
assert all(c != 0 for c in codes), codes
print("ok", len(codes))
"""


def test_host_validation_under_sanitizers():
    """The host code of the C ABI layer and the no-allocation entry point, built with AddressSanitizer
    and UndefinedBehaviorSanitizer, rejects every malformed call of the validation tests (and status
    strings out of range) without a sanitizer report."""
    import os
    import subprocess
    import sys

    from gqa_attention_learned_head_gb300 import build

    asan = subprocess.run(["gcc", "-print-file-name=libasan.so"], capture_output=True, text=True).stdout.strip()
    if not asan or not os.path.isabs(asan) or not os.path.exists(asan):
        pytest.skip("the AddressSanitizer runtime is not installed")
    lib = build.build_sanitized()
    env = dict(os.environ, LD_PRELOAD=asan, ASAN_OPTIONS="detect_leaks=0:abort_on_error=1",
               UBSAN_OPTIONS="halt_on_error=1:print_stacktrace=1")
    r = subprocess.run([sys.executable, "-c", SANITIZED_CHILD, str(ROOT), str(lib)], env=env, capture_output=True,
                       text=True, timeout=600)
    assert r.returncode == 0 and r.stdout.startswith("ok"), r.stdout[-2000:] + r.stderr[-4000:]
    assert "AddressSanitizer" not in r.stderr and "runtime error" not in r.stderr, r.stderr[-4000:]
