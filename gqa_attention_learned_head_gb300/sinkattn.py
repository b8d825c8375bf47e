"""Python binding of libsinkattn: argument marshalling only.

Each function takes torch tensors already on the GPU, checks dtypes and
shapes, allocates missing outputs with ``torch.empty`` and calls the C ABI
(``include/sinkattn.h``) with raw device pointers and the current CUDA stream.
Every arithmetic step runs in the library's kernels; there is no fallback:
if ``libsinkattn.so`` is absent, importing this module raises.
"""
from __future__ import annotations

import ctypes
from pathlib import Path

import torch

from .abi import (EXPORTS, ERR_BAD_LENGTH, ERR_BAD_PAGE, ERR_CUDA, ERR_INVALID_ARG, ERR_TIMEOUT,  # noqa: F401
                  ERR_UNSUPPORTED, ERR_WORKSPACE, OK, DecodeDims, MergeDims, PagedDims, PrefillDims, RopeParams,
                  VerifyDims, declare)

_LIB_PATH = Path(__file__).resolve().parent / "_build" / "libsinkattn.so"


class SinkAttnError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {status_string(status)} (status {status})")


def _load():
    if not _LIB_PATH.exists():
        raise ImportError(f"libsinkattn is not built ({_LIB_PATH} missing); run "
                          "`python -m gqa_attention_learned_head_gb300.build` (needs nvcc)")
    return declare(ctypes.CDLL(str(_LIB_PATH)))


_lib = _load()
library_path = str(_LIB_PATH)


def status_string(status: int) -> str:
    return _lib.sinkattn_status_string(int(status)).decode()


def version() -> int:
    return int(_lib.sinkattn_version())


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _need(t, name, dtype, ndim):
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if t.dim() != ndim or not t.is_contiguous():
        raise ValueError(f"{name} must be a contiguous {ndim}-d tensor, got shape {tuple(t.shape)}")


def _check(status, what):
    if status != OK:
        raise SinkAttnError(status, what)


def decode_dims(q, k_pages, page_table, num_workers=0) -> DecodeDims:
    B, Hq, D = q.shape
    P, Hkv, PS, _ = k_pages.shape
    return DecodeDims(B, Hq, Hkv, D, PS, P, page_table.shape[1], num_workers)


def sinkattn_decode_workspace_size(q, k_pages, page_table, num_workers=0) -> int:
    return int(_lib.sinkattn_decode_workspace_size(ctypes.byref(decode_dims(q, k_pages, page_table, num_workers))))


def sinkattn_decode(q, k_pages, v_pages, page_table, kv_lens, sinks, scale, out=None, lse=None, workspace=None,
                    num_workers=0, return_lse=True, stream=None):
    """Paged split-KV decode.  Shapes: see ``include/sinkattn.h``.  Returns (out, lse)."""
    _need(q, "q", torch.bfloat16, 3)
    _need(k_pages, "k_pages", torch.bfloat16, 4)
    _need(v_pages, "v_pages", torch.bfloat16, 4)
    _need(page_table, "page_table", torch.int32, 2)
    _need(kv_lens, "kv_lens", torch.int32, 1)
    _need(sinks, "sinks", torch.float32, 1)
    if v_pages.shape != k_pages.shape:
        raise ValueError("k_pages and v_pages must have the same shape")
    B, Hq, D = q.shape
    if page_table.shape[0] != B or kv_lens.shape[0] != B or sinks.shape[0] != Hq or k_pages.shape[1] == 0:
        raise ValueError("inconsistent decode shapes")
    dims = decode_dims(q, k_pages, page_table, num_workers)
    if out is None:
        out = torch.empty_like(q)
    if lse is None and return_lse:
        lse = torch.empty(B, Hq, device=q.device, dtype=torch.float32)
    if workspace is None:
        nbytes = int(_lib.sinkattn_decode_workspace_size(ctypes.byref(dims)))
        if nbytes == 0:
            raise SinkAttnError(ERR_INVALID_ARG, "sinkattn_decode_workspace_size")
        workspace = torch.empty(nbytes, device=q.device, dtype=torch.uint8)
    st = _lib.sinkattn_decode(_ptr(q), _ptr(k_pages), _ptr(v_pages), _ptr(page_table), _ptr(kv_lens), _ptr(sinks),
                              float(scale), _ptr(out), _ptr(lse), ctypes.byref(dims), _ptr(workspace),
                              workspace.numel() * workspace.element_size(), _stream(stream))
    _check(st, "sinkattn_decode")
    return out, lse


def verify_dims(q, k_pages, page_table, num_workers=0) -> VerifyDims:
    B, QL, Hq, D = q.shape
    P, Hkv, PS, _ = k_pages.shape
    return VerifyDims(B, QL, Hq, Hkv, D, PS, P, page_table.shape[1], num_workers)


def sinkattn_verify_workspace_size(q, k_pages, page_table, num_workers=0) -> int:
    return int(_lib.sinkattn_verify_workspace_size(ctypes.byref(verify_dims(q, k_pages, page_table, num_workers))))


def sinkattn_verify(q, k_pages, v_pages, page_table, kv_lens, sinks, scale, out=None, lse=None, workspace=None,
                    num_workers=0, return_lse=True, stream=None):
    """Attention of q_len drafted tokens per request over the paged cache (their K/V already in it).

    q [B, q_len, Hq, 64]; kv_lens counts the drafted tokens.  Shapes: see ``include/sinkattn.h``.
    Returns (out [B, q_len, Hq, 64], lse [B, q_len, Hq]).
    """
    _need(q, "q", torch.bfloat16, 4)
    _need(k_pages, "k_pages", torch.bfloat16, 4)
    _need(v_pages, "v_pages", torch.bfloat16, 4)
    _need(page_table, "page_table", torch.int32, 2)
    _need(kv_lens, "kv_lens", torch.int32, 1)
    _need(sinks, "sinks", torch.float32, 1)
    if v_pages.shape != k_pages.shape:
        raise ValueError("k_pages and v_pages must have the same shape")
    B, QL, Hq, D = q.shape
    if page_table.shape[0] != B or kv_lens.shape[0] != B or sinks.shape[0] != Hq or k_pages.shape[1] == 0:
        raise ValueError("inconsistent verify shapes")
    dims = verify_dims(q, k_pages, page_table, num_workers)
    if out is None:
        out = torch.empty_like(q)
    if lse is None and return_lse:
        lse = torch.empty(B, QL, Hq, device=q.device, dtype=torch.float32)
    if workspace is None:
        nbytes = int(_lib.sinkattn_verify_workspace_size(ctypes.byref(dims)))
        if nbytes == 0:
            raise SinkAttnError(ERR_INVALID_ARG, "sinkattn_verify_workspace_size")
        workspace = torch.empty(nbytes, device=q.device, dtype=torch.uint8)
    st = _lib.sinkattn_verify(_ptr(q), _ptr(k_pages), _ptr(v_pages), _ptr(page_table), _ptr(kv_lens), _ptr(sinks),
                              float(scale), _ptr(out), _ptr(lse), ctypes.byref(dims), _ptr(workspace),
                              workspace.numel() * workspace.element_size(), _stream(stream))
    _check(st, "sinkattn_verify")
    return out, lse


def sinkattn_verify_tree(q, k_pages, v_pages, page_table, kv_lens, tree_mask, sinks, scale, out=None, lse=None,
                         workspace=None, num_workers=0, return_lse=True, stream=None):
    """sinkattn_verify for a draft tree: tree_mask [B, q_len] int64 on the device, bit j of mask i = drafted
    token i sees drafted token j (its ancestors and itself).  Returns (out, lse)."""
    _need(tree_mask, "tree_mask", torch.int64, 2)
    B, QL = q.shape[0], q.shape[1]
    if tuple(tree_mask.shape) != (B, QL):
        raise ValueError("tree_mask must be [batch, q_len]")
    _need(q, "q", torch.bfloat16, 4)
    _need(k_pages, "k_pages", torch.bfloat16, 4)
    _need(v_pages, "v_pages", torch.bfloat16, 4)
    _need(page_table, "page_table", torch.int32, 2)
    _need(kv_lens, "kv_lens", torch.int32, 1)
    _need(sinks, "sinks", torch.float32, 1)
    Hq = q.shape[2]
    dims = verify_dims(q, k_pages, page_table, num_workers)
    if out is None:
        out = torch.empty_like(q)
    if lse is None and return_lse:
        lse = torch.empty(B, QL, Hq, device=q.device, dtype=torch.float32)
    if workspace is None:
        nbytes = int(_lib.sinkattn_verify_workspace_size(ctypes.byref(dims)))
        if nbytes == 0:
            raise SinkAttnError(ERR_INVALID_ARG, "sinkattn_verify_workspace_size")
        workspace = torch.empty(nbytes, device=q.device, dtype=torch.uint8)
    st = _lib.sinkattn_verify_tree(_ptr(q), _ptr(k_pages), _ptr(v_pages), _ptr(page_table), _ptr(kv_lens),
                                   _ptr(tree_mask), _ptr(sinks), float(scale), _ptr(out), _ptr(lse), ctypes.byref(dims),
                                   _ptr(workspace), workspace.numel() * workspace.element_size(), _stream(stream))
    _check(st, "sinkattn_verify_tree")
    return out, lse


def paged_dims(k_pages, page_table, cu_seqlens, total_tokens, max_seqlen, num_q_heads=0, share_sms=False) -> PagedDims:
    P, Hkv, PS, D = k_pages.shape
    return PagedDims(cu_seqlens.shape[0] - 1, total_tokens, max_seqlen, num_q_heads, Hkv, D, PS, P,
                     page_table.shape[1], int(bool(share_sms)))


def sinkattn_kv_append(k, v, cu_seqlens, start_pos, page_table, k_pages, v_pages, max_seqlen=0, stream=None):
    """Writes new tokens' k / v [T, Hkv, 64] into the pages, in place, at cache positions start_pos[n] + i."""
    _need(k, "k", torch.bfloat16, 3)
    _need(v, "v", torch.bfloat16, 3)
    _need(cu_seqlens, "cu_seqlens", torch.int32, 1)
    _need(start_pos, "start_pos", torch.int32, 1)
    _need(page_table, "page_table", torch.int32, 2)
    _need(k_pages, "k_pages", torch.bfloat16, 4)
    _need(v_pages, "v_pages", torch.bfloat16, 4)
    if v.shape != k.shape or v_pages.shape != k_pages.shape or k.shape[1] != k_pages.shape[1]:
        raise ValueError("inconsistent append shapes")
    dims = paged_dims(k_pages, page_table, cu_seqlens, k.shape[0], max_seqlen)
    st = _lib.sinkattn_kv_append(_ptr(k), _ptr(v), _ptr(cu_seqlens), _ptr(start_pos), _ptr(page_table),
                                 _ptr(k_pages), _ptr(v_pages), ctypes.byref(dims), _stream(stream))
    _check(st, "sinkattn_kv_append")


def sinkattn_qkv_prologue(qkv, bias, cu_seqlens, start_pos, page_table, k_pages, v_pages, num_q_heads, theta,
                          factor, original_max_position, beta_fast, beta_slow, attn_factor=0.0, interleaved=False,
                          q_out=None, stream=None):
    """QKV bias + YaRN rotary embedding of new tokens qkv [T, (Hq + 2 Hkv) * 64]; returns q [T, Hq, 64] and
    writes the rotated k and the v into the pages at positions start_pos[n] + i (in place)."""
    _need(qkv, "qkv", torch.bfloat16, 2)
    if bias is not None:
        _need(bias, "bias", torch.bfloat16, 1)
    _need(cu_seqlens, "cu_seqlens", torch.int32, 1)
    _need(start_pos, "start_pos", torch.int32, 1)
    _need(page_table, "page_table", torch.int32, 2)
    _need(k_pages, "k_pages", torch.bfloat16, 4)
    _need(v_pages, "v_pages", torch.bfloat16, 4)
    T = qkv.shape[0]
    Hkv = k_pages.shape[1]
    if qkv.shape[1] != (num_q_heads + 2 * Hkv) * 64 or (bias is not None and bias.shape[0] != qkv.shape[1]):
        raise ValueError("qkv must be [T, (Hq + 2 Hkv) * 64] and bias [(Hq + 2 Hkv) * 64]")
    if q_out is None:
        q_out = torch.empty(T, num_q_heads, 64, device=qkv.device, dtype=torch.bfloat16)
    dims = paged_dims(k_pages, page_table, cu_seqlens, T, 0, num_q_heads)
    rope = RopeParams(theta, factor, original_max_position, beta_fast, beta_slow, attn_factor, int(bool(interleaved)))
    st = _lib.sinkattn_qkv_prologue(_ptr(qkv), _ptr(bias), _ptr(cu_seqlens), _ptr(start_pos), _ptr(page_table),
                                    ctypes.byref(rope), _ptr(q_out), _ptr(k_pages), _ptr(v_pages), ctypes.byref(dims),
                                    _stream(stream))
    _check(st, "sinkattn_qkv_prologue")
    return q_out


def sinkattn_prefill_paged(q, k_pages, v_pages, page_table, cu_seqlens, start_pos, sinks, scale, max_seqlen=None,
                           out=None, lse=None, return_lse=True, stream=None, share_sms=False):
    """Chunked prefill of new tokens q [T, Hq, 64] over the paged cache (their K/V already appended):
    new token i of sequence n sees cache tokens 0 .. start_pos[n] + i.  Returns (out, lse).
    ``share_sms`` as in sinkattn_prefill."""
    _need(q, "q", torch.bfloat16, 3)
    _need(k_pages, "k_pages", torch.bfloat16, 4)
    _need(v_pages, "v_pages", torch.bfloat16, 4)
    _need(page_table, "page_table", torch.int32, 2)
    _need(cu_seqlens, "cu_seqlens", torch.int32, 1)
    _need(start_pos, "start_pos", torch.int32, 1)
    _need(sinks, "sinks", torch.float32, 1)
    if max_seqlen is None:
        raise ValueError("max_seqlen is required (an upper bound of the new tokens per sequence)")
    T, Hq, D = q.shape
    dims = paged_dims(k_pages, page_table, cu_seqlens, T, max_seqlen, Hq, share_sms)
    if out is None:
        out = torch.empty_like(q)
    if lse is None and return_lse:
        lse = torch.empty(T, Hq, device=q.device, dtype=torch.float32)
    st = _lib.sinkattn_prefill_paged(_ptr(q), _ptr(k_pages), _ptr(v_pages), _ptr(page_table), _ptr(cu_seqlens),
                                     _ptr(start_pos), _ptr(sinks), float(scale), _ptr(out), _ptr(lse),
                                     ctypes.byref(dims), _stream(stream))
    _check(st, "sinkattn_prefill_paged")
    return out, lse


def sinkattn_prefill(q, k, v, cu_seqlens, sinks, scale, causal=True, max_seqlen=None, out=None, lse=None,
                     return_lse=True, stream=None, share_sms=False):
    """Packed varlen prefill.  ``max_seqlen`` (an upper bound of the lengths) is required.  ``share_sms``
    picks the kernel that leaves room on every SM for a decode launched just before it on another
    stream with two shares per SM."""
    _need(q, "q", torch.bfloat16, 3)
    _need(k, "k", torch.bfloat16, 3)
    _need(v, "v", torch.bfloat16, 3)
    _need(cu_seqlens, "cu_seqlens", torch.int32, 1)
    _need(sinks, "sinks", torch.float32, 1)
    if max_seqlen is None:
        raise ValueError("max_seqlen is required (an upper bound of the sequence lengths)")
    T, Hq, D = q.shape
    if k.shape != v.shape or k.shape[0] != T or sinks.shape[0] != Hq:
        raise ValueError("inconsistent prefill shapes")
    dims = PrefillDims(cu_seqlens.shape[0] - 1, T, int(max_seqlen), Hq, k.shape[1], D, int(bool(share_sms)))
    if out is None:
        out = torch.empty_like(q)
    if lse is None and return_lse:
        lse = torch.empty(T, Hq, device=q.device, dtype=torch.float32)
    st = _lib.sinkattn_prefill(_ptr(q), _ptr(k), _ptr(v), _ptr(cu_seqlens), _ptr(sinks), float(scale),
                               int(bool(causal)), _ptr(out), _ptr(lse), ctypes.byref(dims), _stream(stream))
    _check(st, "sinkattn_prefill")
    return out, lse


def sinkattn_merge(partial_o, partial_lse, sinks=None, out=None, lse=None, return_lse=True, stream=None):
    """LSE merge of partials [S,R,H,64] / [S,R,H]; ``sinks`` adds the sink once."""
    _need(partial_o, "partial_o", torch.float32, 4)
    _need(partial_lse, "partial_lse", torch.float32, 3)
    if sinks is not None:
        _need(sinks, "sinks", torch.float32, 1)
    S, R, H, D = partial_o.shape
    if partial_lse.shape != (S, R, H):
        raise ValueError("partial_lse must be [S, R, H]")
    dims = MergeDims(S, R, H, D)
    if out is None:
        out = torch.empty(R, H, D, device=partial_o.device, dtype=torch.bfloat16)
    if lse is None and return_lse:
        lse = torch.empty(R, H, device=partial_o.device, dtype=torch.float32)
    st = _lib.sinkattn_merge(_ptr(partial_o), _ptr(partial_lse), _ptr(sinks), _ptr(out), _ptr(lse),
                             ctypes.byref(dims), _stream(stream))
    _check(st, "sinkattn_merge")
    return out, lse


NOALLOC_SCRATCH_BYTES = 16 << 20  # SINKATTN_DECODE_NOALLOC_SCRATCH_BYTES


def sinkattn_decode_noalloc(q, k_pages, v_pages, page_table, kv_lens, sinks, scale, out, lse=None, stream=None):
    """Decode with the library's built-in scratch instead of a workspace.

    For callers that cannot allocate device memory on this path (a framework
    owning the whole device through its own pool, a plugin interface that
    passes only inputs and outputs, a loop that must avoid cudaMalloc's
    device synchronisation).  ``out`` (and ``lse`` if wanted) must be given:
    this function allocates nothing.  Problems needing more than 16 MiB of
    scratch raise SinkAttnError(ERR_WORKSPACE); calls must not overlap on the GPU.
    """
    for t, name, dt, nd in ((q, "q", torch.bfloat16, 3), (k_pages, "k_pages", torch.bfloat16, 4),
                            (v_pages, "v_pages", torch.bfloat16, 4), (page_table, "page_table", torch.int32, 2),
                            (kv_lens, "kv_lens", torch.int32, 1), (sinks, "sinks", torch.float32, 1),
                            (out, "out", torch.bfloat16, 3)):
        _need(t, name, dt, nd)
    if lse is not None:
        _need(lse, "lse", torch.float32, 2)
    dims = decode_dims(q, k_pages, page_table)
    st = _lib.sinkattn_decode_noalloc(_ptr(q), _ptr(k_pages), _ptr(v_pages), _ptr(page_table), _ptr(kv_lens),
                                      _ptr(sinks), float(scale), _ptr(out), _ptr(lse), ctypes.byref(dims),
                                      _stream(stream))
    _check(st, "sinkattn_decode_noalloc")
    return out, lse


def sinkattn_selftest_wait_timeout(stream=None) -> None:
    """Enqueues the bounded-wait failure path (one thread waiting on an mbarrier nothing completes);
    the device error word then holds ERR_TIMEOUT (see include/sinkattn.h)."""
    _check(_lib.sinkattn_selftest_wait_timeout(_stream(stream)), "sinkattn_selftest_wait_timeout")


def sinkattn_get_error(stream=None) -> int:
    """Synchronises the stream; returns and clears the device error word (0 = no problem)."""
    return int(_lib.sinkattn_get_error(_stream(stream)))
