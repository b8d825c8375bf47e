"""fp64 CPU oracle for sink attention -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product (the CUDA library and its
Python binding) never imports it and has no CPU fallback.

The arithmetic lives in ``sinkattn_oracle.c`` (plain C, double precision);
this module compiles it with gcc into ``oracle/_build/`` and wraps it for
numpy arrays.  The method it states is the one described in the "GPT-OSS on
day 0" blog post, section "Kernels for GPT-OSS / Sink Attention": a per-head
learned sink logit that enters the softmax normaliser and has no value row.
"""
from __future__ import annotations

import ctypes
import math
import os
import subprocess
from pathlib import Path

import numpy as np

_HERE = Path(__file__).resolve().parent
_SRC = _HERE / "sinkattn_oracle.c"
_BUILD = _HERE / "_build"
_LIB_PATH = _BUILD / "libsinkattn_oracle.so"
_lib = None


def build(force: bool = False) -> Path:
    """Compile the oracle shared library (gcc, OpenMP when available)."""
    if _LIB_PATH.exists() and not force and _LIB_PATH.stat().st_mtime >= _SRC.stat().st_mtime:
        return _LIB_PATH
    _BUILD.mkdir(exist_ok=True)
    tmp = _LIB_PATH.with_suffix(f".{os.getpid()}.tmp")
    base = ["gcc", "-O2", "-std=c11", "-shared", "-fPIC", str(_SRC), "-o", str(tmp), "-lm"]
    try:
        subprocess.run(base[:1] + ["-fopenmp"] + base[1:], check=True, capture_output=True)
    except subprocess.CalledProcessError:
        subprocess.run(base, check=True, capture_output=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    if _lib is None:
        _lib = ctypes.CDLL(str(build()))
        P = ctypes.c_void_p
        i = ctypes.c_int
        f = ctypes.c_float
        _lib.oracle_decode.argtypes = [i, i, i, i, i, i, i, P, P, P, P, P, P, f, i, P, P, P]
        _lib.oracle_prefill.argtypes = [i, P, i, i, i, i, P, P, P, P, f, i, i, P, P, P]
        _lib.oracle_decode_partials.argtypes = [i, i, i, i, i, i, i, P, P, P, P, P, P, f, i, i, i, P, P]
        _lib.oracle_merge.argtypes = [i, i, i, i, P, P, P, P, P]
        _lib.oracle_verify.argtypes = [i, i, i, i, i, i, i, i, P, P, P, P, P, P, f, i, P, P, P]
        _lib.oracle_prefill_paged.argtypes = [i, P, P, i, i, i, i, i, i, i, P, P, P, P, P, f, i, P, P, P]
        _lib.oracle_verify_tree.argtypes = [i, i, i, i, i, i, i, i, P, P, P, P, P, P, P, f, i, P, P, P]
        for fn in ("oracle_decode", "oracle_prefill", "oracle_decode_partials", "oracle_merge", "oracle_verify", "oracle_prefill_paged", "oracle_verify_tree",
                   "oracle_num_threads"):
            getattr(_lib, fn).restype = ctypes.c_int
        _lib.oracle_set_num_threads.argtypes = [i]
        _lib.oracle_set_num_threads.restype = None
    return _lib


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _bf16_bits(a) -> np.ndarray:
    """Accept a uint16 array of bf16 bit patterns or a torch bf16 tensor."""
    if hasattr(a, "dtype") and str(a.dtype) == "torch.bfloat16":
        import torch

        a = a.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)
    a = np.ascontiguousarray(a)
    if a.dtype != np.uint16:
        raise TypeError("bf16 inputs must be uint16 bit patterns or torch.bfloat16")
    return a


def _np(a, dtype):
    if hasattr(a, "detach"):
        a = a.detach().cpu().numpy()
    return np.ascontiguousarray(a, dtype=dtype)


def _check(rc: int, what: str):
    if rc == -2:
        raise IndexError(f"{what}: page id out of range")
    if rc != 0:
        raise ValueError(f"{what}: bad arguments (code {rc})")


def num_threads() -> int:
    return int(_load().oracle_num_threads())


def set_num_threads(n: int) -> None:
    """Threads the oracle's later calls use (OpenMP); returns with the count changed for the process."""
    _load().oracle_set_num_threads(int(n))


def decode(q, k_pages, v_pages, page_table, kv_lens, sinks, scale, rows=None):
    """Sink-attention decode by definition.

    q [B,Hq,D] bf16; k_pages/v_pages [P,Hkv,PS,D] bf16; page_table [B,maxpg]
    int32; kv_lens [B] int32; sinks [Hq] f32.  rows: optional int array of
    (b, h) pairs.  Returns (out float64 [B,Hq,D] or [n,D], lse float64).
    """
    q, kp, vp = _bf16_bits(q), _bf16_bits(k_pages), _bf16_bits(v_pages)
    pt, kl, sk = _np(page_table, np.int32), _np(kv_lens, np.int32), _np(sinks, np.float32)
    B, Hq, D = q.shape
    P, Hkv, PS, _ = kp.shape
    if rows is not None:
        rows = _np(rows, np.int32).reshape(-1, 2)
        n = rows.shape[0]
        out, lse = np.empty((n, D)), np.empty(n)
    else:
        n = B * Hq
        out, lse = np.empty((B, Hq, D)), np.empty((B, Hq))
    rc = _load().oracle_decode(B, Hq, Hkv, D, PS, pt.shape[1], P, _ptr(q), _ptr(kp), _ptr(vp),
                               _ptr(pt), _ptr(kl), _ptr(sk), float(scale), n, _ptr(rows),
                               _ptr(out), _ptr(lse))
    _check(rc, "oracle.decode")
    return out, lse


def verify(q, k_pages, v_pages, page_table, kv_lens, sinks, scale, rows=None):
    """Verification attention over drafted tokens by definition.

    q [B,q_len,Hq,D] bf16: the last q_len cached tokens of each request; token
    i sees cache tokens 0..kv_lens[b]-q_len+i.  Other arguments as decode.
    rows: optional (b, i, h) triples.  Returns (out float64 [B,q_len,Hq,D] or
    [n,D], lse float64).
    """
    q, kp, vp = _bf16_bits(q), _bf16_bits(k_pages), _bf16_bits(v_pages)
    pt, kl, sk = _np(page_table, np.int32), _np(kv_lens, np.int32), _np(sinks, np.float32)
    B, QL, Hq, D = q.shape
    P, Hkv, PS, _ = kp.shape
    if rows is not None:
        rows = _np(rows, np.int32).reshape(-1, 3)
        n = rows.shape[0]
        out, lse = np.empty((n, D)), np.empty(n)
    else:
        n = B * QL * Hq
        out, lse = np.empty((B, QL, Hq, D)), np.empty((B, QL, Hq))
    rc = _load().oracle_verify(B, QL, Hq, Hkv, D, PS, pt.shape[1], P, _ptr(q), _ptr(kp), _ptr(vp),
                               _ptr(pt), _ptr(kl), _ptr(sk), float(scale), n, _ptr(rows),
                               _ptr(out), _ptr(lse))
    _check(rc, "oracle.verify")
    return out, lse


def verify_tree(q, k_pages, v_pages, page_table, kv_lens, tree_mask, sinks, scale, rows=None):
    """Verification of a tree of drafted tokens by definition.

    As verify, but drafted token i sees drafted token j iff bit j of tree_mask[b, i] is set
    (tree_mask [B, q_len] integers, q_len <= 64); every cache token before the draft is seen.
    """
    q, kp, vp = _bf16_bits(q), _bf16_bits(k_pages), _bf16_bits(v_pages)
    pt, kl, sk = _np(page_table, np.int32), _np(kv_lens, np.int32), _np(sinks, np.float32)
    tm = np.ascontiguousarray(np.asarray(tree_mask.cpu() if hasattr(tree_mask, "cpu") else tree_mask,
                                         dtype=np.int64).view(np.uint64))
    B, QL, Hq, D = q.shape
    P, Hkv, PS, _ = kp.shape
    if rows is not None:
        rows = _np(rows, np.int32).reshape(-1, 3)
        n = rows.shape[0]
        out, lse = np.empty((n, D)), np.empty(n)
    else:
        n = B * QL * Hq
        out, lse = np.empty((B, QL, Hq, D)), np.empty((B, QL, Hq))
    rc = _load().oracle_verify_tree(B, QL, Hq, Hkv, D, PS, pt.shape[1], P, _ptr(q), _ptr(kp), _ptr(vp), _ptr(pt),
                                    _ptr(kl), _ptr(tm), _ptr(sk), float(scale), n, _ptr(rows), _ptr(out), _ptr(lse))
    _check(rc, "oracle.verify_tree")
    return out, lse


def prefill(q, k, v, cu_seqlens, sinks, scale, causal=True, rows=None):
    """Sink-attention prefill by definition over packed varlen sequences.

    q [T,Hq,D], k/v [T,Hkv,D] bf16; cu_seqlens [N+1] int32.  rows: optional
    (t, h) pairs.  Returns (out float64, lse float64).
    """
    q, k, v = _bf16_bits(q), _bf16_bits(k), _bf16_bits(v)
    cu, sk = _np(cu_seqlens, np.int32), _np(sinks, np.float32)
    T, Hq, D = q.shape
    Hkv = k.shape[1]
    if rows is not None:
        rows = _np(rows, np.int32).reshape(-1, 2)
        n = rows.shape[0]
        out, lse = np.empty((n, D)), np.empty(n)
    else:
        n = T * Hq
        out, lse = np.empty((T, Hq, D)), np.empty((T, Hq))
    rc = _load().oracle_prefill(len(cu) - 1, _ptr(cu), T, Hq, Hkv, D, _ptr(q), _ptr(k), _ptr(v),
                                _ptr(sk), float(scale), int(bool(causal)), n, _ptr(rows),
                                _ptr(out), _ptr(lse))
    _check(rc, "oracle.prefill")
    return out, lse


def kv_append(k, v, cu_seqlens, start_pos, page_table, k_pages, v_pages):
    """Writing new tokens into their requests' pages, by definition (returns new pool arrays).

    k/v [T,Hkv,D] bf16: the new tokens of N sequences packed by cu_seqlens [N+1]; new token i of
    sequence n goes to cache position start_pos[n] + i, i.e. page page_table[n][pos // PS], slot
    pos % PS.  k_pages/v_pages [P,Hkv,PS,D] bf16 are not modified.  Returns (k_pages, v_pages) as
    bf16 bit patterns (uint16), every other slot unchanged.
    """
    kb, vb = _bf16_bits(k), _bf16_bits(v)
    kp, vp = _bf16_bits(k_pages).copy(), _bf16_bits(v_pages).copy()
    cu, sp, pt = _np(cu_seqlens, np.int32), _np(start_pos, np.int32), _np(page_table, np.int32)
    PS = kp.shape[2]
    for n in range(len(cu) - 1):
        for i in range(int(cu[n + 1] - cu[n])):
            pos = int(sp[n]) + i
            page = int(pt[n, pos // PS])
            if not 0 <= page < kp.shape[0]:
                raise IndexError("oracle.kv_append: page id out of range")
            kp[page, :, pos % PS] = kb[cu[n] + i]
            vp[page, :, pos % PS] = vb[cu[n] + i]
    return kp, vp


def prefill_paged(q, k_pages, v_pages, page_table, cu_seqlens, start_pos, sinks, scale, rows=None):
    """Chunked prefill over a paged cache by definition.

    q [T,Hq,D] bf16: the new tokens of N sequences packed by cu_seqlens [N+1]; new token i of
    sequence n sits at cache position start_pos[n] + i (its K/V already in the pages) and sees
    cache tokens 0..that position.  k_pages/v_pages [P,Hkv,PS,D] (bf16 tensors or uint16 bit
    arrays), page_table [N,max_pages].  rows: optional (t, h) pairs.  Returns (out, lse) float64.
    """
    q, kp, vp = _bf16_bits(q), _bf16_bits(k_pages), _bf16_bits(v_pages)
    pt, cu, sp, sk = (_np(page_table, np.int32), _np(cu_seqlens, np.int32), _np(start_pos, np.int32),
                      _np(sinks, np.float32))
    T, Hq, D = q.shape
    P, Hkv, PS, _ = kp.shape
    if rows is not None:
        rows = _np(rows, np.int32).reshape(-1, 2)
        n = rows.shape[0]
        out, lse = np.empty((n, D)), np.empty(n)
    else:
        n = T * Hq
        out, lse = np.empty((T, Hq, D)), np.empty((T, Hq))
    rc = _load().oracle_prefill_paged(len(cu) - 1, _ptr(cu), _ptr(sp), T, Hq, Hkv, D, PS, pt.shape[1], P, _ptr(q),
                                      _ptr(kp), _ptr(vp), _ptr(pt), _ptr(sk), float(scale), n, _ptr(rows),
                                      _ptr(out), _ptr(lse))
    _check(rc, "oracle.prefill_paged")
    return out, lse


# ---------------------------------------------------------------------------- pre-attention prologue
# "GPT-OSS on day 0", section "Attention: GQA with attention sinks": the QKV projections carry a bias
# and positions are encoded with YaRN rotary embeddings (as in DeepSeek-V3).  The page gives no
# formulas; these follow the YaRN method as published ("YaRN: Efficient Context Window Extension of
# Large Language Models"): rotary frequency theta_d = theta^(-2d/D); wavelength lambda_d = 2 pi /
# theta_d; ratio r_d = L / lambda_d for the original context L; ramp gamma(r) = 0 for r < beta_slow,
# 1 for r > beta_fast, linear between; new frequency (1 - gamma) theta_d / s + gamma theta_d; and the
# attention temperature 1/t with sqrt(1/t) = 0.1 ln s + 1, applied by scaling q and k.

def yarn_inv_freq(D, theta, factor, original_max_position, beta_fast, beta_slow) -> np.ndarray:
    """Rotary angle per position of each of the D/2 dimension pairs, float64."""
    d = np.arange(D // 2, dtype=np.float64)
    theta_d = np.power(float(theta), -2.0 * d / D)
    r = float(original_max_position) * theta_d / (2.0 * np.pi)  # L / wavelength
    gamma = np.clip((r - beta_slow) / (beta_fast - beta_slow), 0.0, 1.0)
    return (1.0 - gamma) * theta_d / float(factor) + gamma * theta_d


def yarn_mscale(factor, attn_factor=0.0) -> float:
    """Multiplier of q and k after the rotation: the given one, else 0.1 ln(s) + 1 (1 for s <= 1)."""
    if attn_factor:
        return float(attn_factor)
    return 0.1 * math.log(factor) + 1.0 if factor > 1.0 else 1.0


def rope(x, positions, inv_freq, mscale, interleaved=False):
    """Rotates the last axis (D) of x [..., T, H, D] (float64) by positions [T] x inv_freq [D/2].

    Pairs are (d, d + D/2) (interleaved=False) or (2d, 2d + 1); the result is scaled by mscale."""
    x = np.asarray(x, dtype=np.float64)
    D = x.shape[-1]
    ang = np.asarray(positions, dtype=np.float64)[:, None] * inv_freq[None, :]  # [T, D/2]
    c, s = np.cos(ang)[:, None, :], np.sin(ang)[:, None, :]
    if interleaved:
        a, b = x[..., 0::2], x[..., 1::2]
    else:
        a, b = x[..., : D // 2], x[..., D // 2:]
    ra, rb = a * c - b * s, b * c + a * s
    out = np.empty_like(x)
    if interleaved:
        out[..., 0::2], out[..., 1::2] = ra, rb
    else:
        out[..., : D // 2], out[..., D // 2:] = ra, rb
    return out * mscale


def qkv_prologue(qkv, bias, cu_seqlens, start_pos, Hq, Hkv, theta, factor, original_max_position, beta_fast,
                 beta_slow, attn_factor=0.0, interleaved=False):
    """Bias + YaRN rotary embedding of new tokens, by definition.

    qkv [T, (Hq + 2 Hkv) * D] bf16 (q heads, then k heads, then v heads), bias [(Hq + 2 Hkv) * D]
    bf16; new token i of sequence n is at position start_pos[n] + i.  Returns float64 q [T, Hq, D],
    k [T, Hkv, D] (both rotated and scaled) and v [T, Hkv, D] (bias only)."""
    x = _bf16_bits(qkv)
    T = x.shape[0]
    D = x.shape[1] // (Hq + 2 * Hkv)
    xf = _bits_to_f64(x).reshape(T, Hq + 2 * Hkv, D) + _bits_to_f64(_bf16_bits(bias)).reshape(1, Hq + 2 * Hkv, D)
    cu, sp = _np(cu_seqlens, np.int32), _np(start_pos, np.int32)
    pos = np.concatenate([sp[n] + np.arange(cu[n + 1] - cu[n]) for n in range(len(cu) - 1)]).astype(np.float64)
    inv = yarn_inv_freq(D, theta, factor, original_max_position, beta_fast, beta_slow)
    ms = yarn_mscale(factor, attn_factor)
    q = rope(xf[:, :Hq], pos, inv, ms, interleaved)
    k = rope(xf[:, Hq:Hq + Hkv], pos, inv, ms, interleaved)
    return q, k, xf[:, Hq + Hkv:]


def _bits_to_f64(bits) -> np.ndarray:
    return (np.asarray(bits, dtype=np.uint32) << 16).view(np.float32).astype(np.float64)


SINK_IN_FIRST_CHUNK = 0
SINK_IN_NO_CHUNK = 1
SINK_IN_EVERY_CHUNK = 2  # the wrong rule; exists only for a negative test


def decode_partials(q, k_pages, v_pages, page_table, kv_lens, sinks, scale, num_chunks,
                    chunk_tokens, sink_mode=SINK_IN_FIRST_CHUNK):
    """Per-chunk partial results (o_c, lse_c) of decode, by definition."""
    q, kp, vp = _bf16_bits(q), _bf16_bits(k_pages), _bf16_bits(v_pages)
    pt, kl, sk = _np(page_table, np.int32), _np(kv_lens, np.int32), _np(sinks, np.float32)
    B, Hq, D = q.shape
    P, Hkv, PS, _ = kp.shape
    po = np.empty((num_chunks, B, Hq, D))
    pl = np.empty((num_chunks, B, Hq))
    rc = _load().oracle_decode_partials(B, Hq, Hkv, D, PS, pt.shape[1], P, _ptr(q), _ptr(kp),
                                        _ptr(vp), _ptr(pt), _ptr(kl), _ptr(sk), float(scale),
                                        num_chunks, chunk_tokens, sink_mode, _ptr(po), _ptr(pl))
    _check(rc, "oracle.decode_partials")
    return po, pl


def merge(partial_o, partial_lse, sinks=None):
    """Log-sum-exp merge of partials [S,R,H,D] / [S,R,H]; sinks [H] adds the sink once."""
    po = _np(partial_o, np.float64)
    pl = _np(partial_lse, np.float64)
    S, R, H, D = po.shape
    sk = None if sinks is None else _np(sinks, np.float32)
    out, lse = np.empty((R, H, D)), np.empty((R, H))
    rc = _load().oracle_merge(S, R, H, D, _ptr(po), _ptr(pl), _ptr(sk), _ptr(out), _ptr(lse))
    _check(rc, "oracle.merge")
    return out, lse
