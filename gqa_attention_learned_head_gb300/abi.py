"""The C ABI of libsinkattn as ctypes declarations: status codes, the dims structs of
include/sinkattn.h and the prototypes of its entry points.  Plain ctypes, no torch: the torch
binding (sinkattn.py) and tools that load another build of the library share these."""
from __future__ import annotations

import ctypes

OK = 0
ERR_INVALID_ARG = 1
ERR_UNSUPPORTED = 2
ERR_WORKSPACE = 3
ERR_BAD_PAGE = 4
ERR_TIMEOUT = 5
ERR_CUDA = 6
ERR_BAD_LENGTH = 7


class DecodeDims(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in ("batch", "num_q_heads", "num_kv_heads", "head_dim", "page_size",
                                              "num_pages", "max_pages", "num_workers")]


class VerifyDims(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in ("batch", "q_len", "num_q_heads", "num_kv_heads", "head_dim",
                                              "page_size", "num_pages", "max_pages", "num_workers")]


class PagedDims(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in ("num_seqs", "total_tokens", "max_seqlen", "num_q_heads", "num_kv_heads",
                                              "head_dim", "page_size", "num_pages", "max_pages", "share_sms")]


class RopeParams(ctypes.Structure):
    _fields_ = [("theta", ctypes.c_float), ("factor", ctypes.c_float), ("original_max_position", ctypes.c_int32),
                ("beta_fast", ctypes.c_float), ("beta_slow", ctypes.c_float), ("attn_factor", ctypes.c_float),
                ("interleaved", ctypes.c_int32)]


class PrefillDims(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in ("num_seqs", "total_tokens", "max_seqlen", "num_q_heads",
                                              "num_kv_heads", "head_dim", "share_sms")]


class MergeDims(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in ("num_splits", "num_rows", "num_heads", "head_dim")]


EXPORTS = ("sinkattn_decode", "sinkattn_prefill", "sinkattn_merge", "sinkattn_decode_workspace_size", "sinkattn_verify",
           "sinkattn_verify_workspace_size", "sinkattn_kv_append", "sinkattn_prefill_paged", "sinkattn_verify_tree", "sinkattn_qkv_prologue",
           "sinkattn_get_error", "sinkattn_status_string", "sinkattn_version", "sinkattn_selftest_wait_timeout")


def declare(lib):
    """Sets the argument and result types of every entry point on a loaded library; returns it."""
    P, i32, f32, sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_float, ctypes.c_size_t
    lib.sinkattn_decode.argtypes = [P, P, P, P, P, P, f32, P, P, ctypes.POINTER(DecodeDims), P, sz, P]
    lib.sinkattn_prefill.argtypes = [P, P, P, P, P, f32, i32, P, P, ctypes.POINTER(PrefillDims), P]
    lib.sinkattn_merge.argtypes = [P, P, P, P, P, ctypes.POINTER(MergeDims), P]
    lib.sinkattn_decode_noalloc.argtypes = [P, P, P, P, P, P, f32, P, P, ctypes.POINTER(DecodeDims), P]
    lib.sinkattn_decode_noalloc.restype = ctypes.c_int
    lib.sinkattn_decode_workspace_size.argtypes = [ctypes.POINTER(DecodeDims)]
    lib.sinkattn_decode_workspace_size.restype = sz
    lib.sinkattn_verify.argtypes = [P, P, P, P, P, P, f32, P, P, ctypes.POINTER(VerifyDims), P, sz, P]
    lib.sinkattn_verify_workspace_size.argtypes = [ctypes.POINTER(VerifyDims)]
    lib.sinkattn_verify_workspace_size.restype = sz
    lib.sinkattn_verify_tree.argtypes = [P, P, P, P, P, P, P, f32, P, P, ctypes.POINTER(VerifyDims), P, sz, P]
    lib.sinkattn_kv_append.argtypes = [P, P, P, P, P, P, P, ctypes.POINTER(PagedDims), P]
    lib.sinkattn_qkv_prologue.argtypes = [P, P, P, P, P, ctypes.POINTER(RopeParams), P, P, P,
                                          ctypes.POINTER(PagedDims), P]
    lib.sinkattn_prefill_paged.argtypes = [P, P, P, P, P, P, P, f32, P, P, ctypes.POINTER(PagedDims), P]
    lib.sinkattn_get_error.argtypes = [P]
    lib.sinkattn_selftest_wait_timeout.argtypes = [P]
    lib.sinkattn_selftest_wait_timeout.restype = ctypes.c_int
    lib.sinkattn_status_string.argtypes = [ctypes.c_int]
    lib.sinkattn_status_string.restype = ctypes.c_char_p
    lib.sinkattn_version.restype = i32
    for fn in ("sinkattn_decode", "sinkattn_prefill", "sinkattn_merge", "sinkattn_get_error", "sinkattn_verify",
               "sinkattn_kv_append", "sinkattn_prefill_paged", "sinkattn_verify_tree", "sinkattn_qkv_prologue"):
        getattr(lib, fn).restype = ctypes.c_int
    return lib


