#!/usr/bin/env python3
"""Benchmark of libsinkattn (sink attention, GQA, paged split-KV decode + causal prefill).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload batched_paged_decode|long_context_decode|speculative_verify|tree_verify|
                                causal_prefill|chunked_prefill|serving_step]

Headline: decode KV GB/s on the batched paged decode workload (batch 32,
64 q / 8 KV heads, head_dim 64, kv_len uniform in [512, 4096], 16-token pages
randomly permuted in the pool).  One step = one sinkattn_decode call (split
pass + merge), i.e. the whole decode hot path, on inputs resident in HBM.
The decode and verification workloads are timed in the steady state: K calls
back to back, captured in one CUDA graph and timed as one replay, cycling over
4 independent input sets that together outgrow L2 (each call reads its K/V
from DRAM); the same call
timed alone after an L2 flush (256 MiB write, then a 512 MiB read) is
reported beside it.  The prefill workloads flush L2 before every step.  Secondary lines
for the long-context split-KV decode, the verification of drafted tokens (4 per request, and a
draft tree of 8), the causal prefill, the chunked prefill over the paged cache and the mixed serving batch ride in the
same JSON object under "secondary".

Prints ONE JSON line on rank 0.  Under torchrun every rank runs its own
independent batch (weak scaling, no collective on the data path); the
barrier / max-over-ranks reduction only brackets the timing.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time
from pathlib import Path

import torch

ROOT = Path(__file__).resolve().parent
sys.path.insert(0, str(ROOT))

METRIC = "decode KV GB/s (% of HBM peak); prefill TFLOP/s (% of bf16 TC peak)"
HBM_FALLBACK_GBS = 6800.0
BF16_FALLBACK_TFLOPS = 1900.0
L2_FLUSH_BYTES = 256 << 20  # twice the 126.5 MiB L2

WORKLOAD_TEXT = {
    "tiny_decode": "tiny decode: batch 1, 4 q / 1 KV head, head_dim 64, kv_len 128, contiguous pages",
    "batched_paged_decode": "batched paged decode: batch 32, 64 q / 8 KV heads, head_dim 64, kv_len U[512,4096], "
                            "16-token pages randomly permuted in the pool",
    "long_context_decode": "long-context split-KV decode: batch 4, 64 q / 8 KV heads, head_dim 64, kv_len 131072, "
                           "split into chunks merged by LSE (the sink counted once)",
    "causal_prefill": "causal prefill: 2 x 8192 tokens (varlen), 64 q / 8 KV heads, head_dim 64",
    "chunked_prefill": "chunked prefill over the paged cache: 8 sequences, U[1024,8192] cached + U[256,2048] new "
                       "tokens each, 64 q / 8 KV heads, head_dim 64; one step = append the new K/V into the pages "
                       "+ paged prefill",
    "tree_verify": "verification of a draft tree: batch 32, an EAGLE-style tree of 8 drafted tokens per request "
                   "(depth 4) over the paged cache, 64 q / 8 KV heads, kv_len U[512,4096] (drafts included)",
    "serving_step": "serving step of the chunked prefill: fused prologue (QKV bias + YaRN rotary of the new tokens, "
                    "q out, k/v into the pages) + paged prefill; 8 sequences, U[1024,8192] cached + U[256,2048] new "
                    "tokens each, 64 q / 8 KV heads, head_dim 64",
    "speculative_verify": "verification of drafts: batch 32, 4 query tokens per request over the paged cache, "
                          "64 q / 8 KV heads, head_dim 64, kv_len U[512,4096] (drafts included), permuted pages",
    "mixed_serving": "mixed serving batch: 8 causal prefills L~U[256,4096] + 256 paged decodes kv_len~U[1024,32768], "
                     "64 q / 8 KV heads, two streams",
}


# ----------------------------------------------------------------------------- helpers

def peaks():
    p = ROOT / "MEASURED_PEAKS.json"
    if p.exists():
        try:
            d = json.loads(p.read_text())
            return float(d["hbm_gbs"]), float(d["bf16_tflops"]), float(d.get("bf16_tflops_sustained", d["bf16_tflops"])), "measured"
        except Exception:
            pass
    return HBM_FALLBACK_GBS, BF16_FALLBACK_TFLOPS, 1700.0, "fallback"


# Sources each profiled kernel is compiled from (its own file, the headers it includes).
KERNEL_SOURCES = {
    "decode_split_kernel": ["decode.cu", "ptx.cuh", "split_kv.cuh", "args_decode.h", "args_merge.h", "args_common.h"],
    "verify_tc_kernel": ["verify_tc.cu", "ptx.cuh", "split_kv.cuh", "tc_tile.cuh", "args_verify.h", "args_merge.h",
                         "args_common.h"],
    "prefill_pp_kernel": ["prefill_pp.cu", "ptx.cuh", "tc_tile.cuh", "tile_order.cuh", "args_prefill.h",
                          "args_common.h"],
    "prefill_tc_kernel": ["prefill_tc.cu", "ptx.cuh", "tc_tile.cuh", "tile_order.cuh", "args_prefill.h",
                          "args_common.h"],
    "prefill_pp_kernel_paged": ["prefill_pp.cu", "ptx.cuh", "tc_tile.cuh", "tile_order.cuh", "args_prefill.h",
                                "args_common.h"],
    "qkv_prologue_kernel": ["prologue.cu", "ptx.cuh", "args_paged.h", "args_common.h"],
}


def kernel_source_hash(names):
    h = hashlib.sha256()
    for n in names:
        h.update((ROOT / "gqa_attention_learned_head_gb300" / "csrc" / n).read_bytes())
    return h.hexdigest()[:16]


def profiled_traffic(kernel, workload, sources):
    """DRAM bytes per launch from a committed ncu summary, if taken on the current kernel source."""
    p = ROOT / "profiles" / f"{kernel}.{workload}.txt"
    if not p.exists():
        return None
    kv = {}
    for line in p.read_text().splitlines():
        if "=" in line and not line.startswith("#"):
            k, v = line.split("=", 1)
            kv[k.strip()] = v.strip()
    if kv.get("source_hash") != kernel_source_hash(sources):
        return None
    try:
        return float(kv["dram_bytes_per_launch_full"])
    except (KeyError, ValueError):
        return None


class ClockSampler:
    """nvidia-smi clock / throttle sampling in the background."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.lines = []
        self.t = None

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
            return
        self.t = threading.Thread(target=self._read, daemon=True)
        self.t.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line.strip()))

    def stop(self):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
        if self.t:
            self.t.join(timeout=2)

    def summary(self, t0, t1):
        sm, smax, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ts, line in self.lines:
            if not (t0 <= ts <= t1):
                continue
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                smax = float(f[2])
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": smax, "reasons": sorted(reasons), "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": smax, "reasons": sorted(reasons),
                "samples": len(sm)}


def dist_setup(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist

        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    elif torch.cuda.is_available():
        torch.cuda.set_device(0)
    return rank, world, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist

        dist.barrier()


def _reduce(x, world, op):
    """All-reduce one float over the ranks (NCCL: on the GPU; gloo: on the CPU)."""
    if world == 1:
        return x
    import torch.distributed as dist

    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=op)
    return float(t.item())


def max_over_ranks(x, world):
    import torch.distributed as dist

    return _reduce(x, world, dist.ReduceOp.MAX)


def sum_over_ranks(x, world):
    import torch.distributed as dist

    return _reduce(x, world, dist.ReduceOp.SUM)


def weak_scaling_value(units_this_rank, ms_this_rank, world):
    """Whole-job throughput: units all ranks processed / the slowest rank's time (units per second)."""
    total = sum_over_ranks(float(units_this_rank), world)
    slowest = max_over_ranks(float(ms_this_rank), world)
    return total / (slowest * 1e-3), slowest


def timed_steps(step, K, warmup, flush, stream):
    """W warm-up steps, then K steps each preceded by an L2 flush; device ms per step (events on `stream`)."""
    for _ in range(warmup):
        flush()
        step()
    torch.cuda.synchronize()
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    for i in range(K):
        flush()
        starts[i].record(stream)
        step()
        ends[i].record(stream)
    torch.cuda.synchronize()
    return [s.elapsed_time(e) for s, e in zip(starts, ends)]


STEADY_SETS = 4  # independent input sets the steady-state decode / verification steps cycle over
SEEDS_PER_RANK = 16


def steady_ms(steps, K, warmup, stream):
    """Mean ms per step of K steps run back to back, cycling over `steps` (one per independent input
    set): each step's inputs were last touched len(steps) - 1 steps earlier, and the sets together are
    larger than L2, so every step reads its K/V from DRAM.  The K steps are captured in one CUDA graph
    (as a serving loop replays its decode graph) and timed as one replay between an event pair on
    `stream`, after an untimed replay: no per-step event, flush or host launch sits between the
    kernels, and each launch overlaps the previous kernel's tail."""
    n = len(steps)
    with torch.cuda.stream(stream):
        for i in range(max(warmup, n)):
            steps[i % n]()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        for i in range(K):
            steps[i % n]()
    torch.cuda.synchronize()
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        g.replay()
        torch.cuda.synchronize()
        t0.record(stream)
        g.replay()
        t1.record(stream)
    torch.cuda.synchronize()
    return t0.elapsed_time(t1) / K


def graph_ms(step, n, reps, stream, flush=None):
    """Per-call ms of n calls captured back to back in one CUDA graph and replayed `reps` times (the
    host's launch overhead stripped).  With `flush`, every call is preceded by the L2 flush inside the
    graph, and the time of a graph of n flushes alone is subtracted."""
    def capture(body):
        g = torch.cuda.CUDAGraph()
        torch.cuda.synchronize()
        with torch.cuda.graph(g, stream=stream):
            for _ in range(n):
                body()
        torch.cuda.synchronize()
        return g

    def per_call(g):
        t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            g.replay()
            torch.cuda.synchronize()
            t0.record(stream)
            for _ in range(reps):
                g.replay()
            t1.record(stream)
        torch.cuda.synchronize()
        return t0.elapsed_time(t1) / (reps * n)

    if flush is None:
        return per_call(capture(step))

    def both():
        flush()
        step()

    return per_call(capture(both)) - per_call(capture(flush))


class Staging:
    """Tensors packed back to back (each at a 256-byte offset) in one pinned host buffer and one
    device buffer, so that a step's inputs (or results) cross to the other side in one copy."""

    def __init__(self, specs):
        offs, off = [], 0
        for shape, dtype in specs:
            off = (off + 255) & ~255
            offs.append(off)
            off += math.prod(shape) * torch.empty(0, dtype=dtype).element_size()
        self.nbytes = off
        self.host = torch.empty(off, dtype=torch.uint8).pin_memory()
        self.dev = torch.empty(off, dtype=torch.uint8, device="cuda")

        def views(buf):
            return [buf[o:o + math.prod(sh) * torch.empty(0, dtype=dt).element_size()].view(dt).view(sh)
                    for o, (sh, dt) in zip(offs, specs)]

        self.h, self.d = views(self.host), views(self.dev)

    def to_device(self):
        self.dev.copy_(self.host, non_blocking=True)

    def to_host(self):
        self.host.copy_(self.dev, non_blocking=True)


def pipelined_ms(api, ins, outs, K, warmup, stream):
    """Mean ms per step of a double-buffered loop through the public API: the inputs of step i go up
    on one copy stream, step i runs on `stream`, its results come back on another copy stream; slot
    i % 2 is reused only after step i - 2 has released it.  The K steps are captured in one CUDA
    graph (the three streams fork from and join `stream`) and timed as one replay, from the first
    upload to the last download, so the host's enqueue cost is not in the figure."""
    up, down = torch.cuda.Stream(), torch.cuda.Stream()

    def loop(n):
        up.wait_stream(stream)
        down.wait_stream(stream)
        ev_in = [torch.cuda.Event() for _ in range(n)]
        ev_run = [torch.cuda.Event() for _ in range(n)]
        ev_out = [torch.cuda.Event() for _ in range(n)]
        for i in range(n):
            slot = i % 2
            with torch.cuda.stream(up):
                if i >= 2:
                    up.wait_event(ev_run[i - 2])  # step i - 2 has read this slot's inputs
                ins[slot].to_device()
                ev_in[i].record(up)
            with torch.cuda.stream(stream):
                stream.wait_event(ev_in[i])
                if i >= 2:
                    stream.wait_event(ev_out[i - 2])  # this slot's previous results are on the host
                api(ins[slot].d, outs[slot].d)
                ev_run[i].record(stream)
            with torch.cuda.stream(down):
                down.wait_event(ev_run[i])
                outs[slot].to_host()
                ev_out[i].record(down)
        stream.wait_stream(up)
        stream.wait_stream(down)

    with torch.cuda.stream(stream):
        loop(warmup)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        loop(K)
    torch.cuda.synchronize()
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        g.replay()  # warm
        torch.cuda.synchronize()
        t0.record(stream)
        g.replay()
        t1.record(stream)
    torch.cuda.synchronize()
    return t0.elapsed_time(t1) / K


# ----------------------------------------------------------------------------- workloads

def decode_bytes(kv_lens, Hkv, D=64):
    return int(kv_lens.to(torch.int64).sum()) * Hkv * D * 2 * 2


def decode_launches_per_call(B, Hkv, max_pages, workers):
    """Kernels one decode call launches: the split pass, plus the split merge unless a single share
    covers the whole call (the rule the library applies on the host)."""
    n_sms = torch.cuda.get_device_properties(torch.cuda.current_device()).multi_processor_count
    may_split = (workers or n_sms) > 1 and (workers > 0 or B * Hkv * max_pages > 32)
    return 2 if may_split else 1


def bench_decode(S, W, name, rank, K, warmup, flush, stream, num_workers=0, sets=1):
    """Per-call times (L2 flushed before each) on input set 0, and, with sets > 1, the steady-state
    ms per step over `sets` independent input sets.  Returns (inputs of set 0, its step, per-call
    times, its bytes, steady (ms, mean bytes per step) or None)."""
    gen = getattr(W, name)
    steps, nbytes = [], []
    inps = []
    for j in range(sets):
        inp = gen(device="cuda", seed=SEEDS_PER_RANK * rank + j)
        B, Hq, D = inp.q.shape
        Hkv = inp.k_pages.shape[1]
        ws = torch.empty(S.sinkattn_decode_workspace_size(inp.q, inp.k_pages, inp.page_table, num_workers),
                         dtype=torch.uint8, device="cuda")
        out = torch.empty_like(inp.q)
        lse = torch.empty(B, Hq, dtype=torch.float32, device="cuda")

        def step(inp=inp, ws=ws, out=out, lse=lse):
            S.sinkattn_decode(inp.q, inp.k_pages, inp.v_pages, inp.page_table, inp.kv_lens, inp.sinks, inp.scale,
                              out=out, lse=lse, workspace=ws, num_workers=num_workers, stream=stream)

        steps.append(step)
        nbytes.append(decode_bytes(inp.kv_lens, Hkv, D))
        inps.append(inp)
    with torch.cuda.stream(stream):
        times = timed_steps(steps[0], K, warmup, flush, stream)
        steady = None
        if sets > 1:
            ms = steady_ms(steps, K, warmup, stream)
            steady = (ms, sum(nbytes[i % sets] for i in range(K)) / K)
    err = S.sinkattn_get_error(stream)
    if err:
        raise RuntimeError(f"device error {S.status_string(err)}")
    return inps[0], steps[0], times, nbytes[0], steady


def bench_verify(S, W, rank, K, warmup, flush, stream, sets=1, tree=False):
    """As bench_decode, for the verification of drafted tokens (linear, or the draft tree)."""
    steps, nbytes, inps, all_masks = [], [], [], []
    for j in range(sets):
        seed = SEEDS_PER_RANK * rank + j
        if tree:
            inp, masks = W.tree_verify(device="cuda", seed=seed)
            mt = torch.as_tensor(masks, dtype=torch.int64, device="cuda")
        else:
            inp, masks, mt = W.speculative_verify(device="cuda", seed=seed), None, None
        B, QL, Hq, D = inp.q.shape
        Hkv = inp.k_pages.shape[1]
        ws = torch.empty(S.sinkattn_verify_workspace_size(inp.q, inp.k_pages, inp.page_table), dtype=torch.uint8,
                         device="cuda")
        out = torch.empty_like(inp.q)
        lse = torch.empty(B, QL, Hq, dtype=torch.float32, device="cuda")

        def step(inp=inp, ws=ws, out=out, lse=lse, mt=mt):
            kw = dict(out=out, lse=lse, workspace=ws, stream=stream)
            if mt is not None:
                S.sinkattn_verify_tree(inp.q, inp.k_pages, inp.v_pages, inp.page_table, inp.kv_lens, mt, inp.sinks,
                                       inp.scale, **kw)
            else:
                S.sinkattn_verify(inp.q, inp.k_pages, inp.v_pages, inp.page_table, inp.kv_lens, inp.sinks,
                                  inp.scale, **kw)

        steps.append(step)
        nbytes.append(decode_bytes(inp.kv_lens, Hkv, D))
        inps.append(inp)
        all_masks.append(masks)
    with torch.cuda.stream(stream):
        times = timed_steps(steps[0], K, warmup, flush, stream)
        steady = None
        if sets > 1:
            ms = steady_ms(steps, K, warmup, stream)
            steady = (ms, sum(nbytes[i % sets] for i in range(K)) / K)
    err = S.sinkattn_get_error(stream)
    if err:
        raise RuntimeError(f"device error {S.status_string(err)}")
    return inps[0], steps[0], times, nbytes[0], steady, all_masks[0]


YARN_GPT_OSS = dict(theta=150000.0, factor=32.0, original_max_position=4096, beta_fast=32.0, beta_slow=1.0)


def bench_prologue_chunked(S, W, rank, K, warmup, flush, stream):
    """The chunked prefill with the fused prologue in front: QKV bias + YaRN rotary of the new tokens
    (q out, k/v into the pages), then the paged prefill.  Returns (inputs, step, ms list, flops,
    prologue ms list, prologue bytes moved, (qkv, bias))."""
    inp = W.chunked_prefill(device="cuda", seed=rank)
    T, Hq, D = inp.q.shape
    Hkv = inp.k_pages.shape[1]
    g = torch.Generator(device="cuda")
    g.manual_seed(1000 + rank)
    qkv = torch.randn(T, (Hq + 2 * Hkv) * D, generator=g, device="cuda").to(torch.bfloat16)
    bias = torch.randn((Hq + 2 * Hkv) * D, generator=g, device="cuda").to(torch.bfloat16)
    q = torch.empty_like(inp.q)
    out = torch.empty_like(inp.q)
    lse = torch.empty(T, Hq, dtype=torch.float32, device="cuda")

    def prologue():
        S.sinkattn_qkv_prologue(qkv, bias, inp.cu_seqlens, inp.start_pos, inp.page_table, inp.k_pages, inp.v_pages,
                                Hq, q_out=q, stream=stream, **YARN_GPT_OSS)

    def step():
        prologue()
        S.sinkattn_prefill_paged(q, inp.k_pages, inp.v_pages, inp.page_table, inp.cu_seqlens, inp.start_pos,
                                 inp.sinks, inp.scale, max_seqlen=inp.max_seqlen, out=out, lse=lse, stream=stream)

    with torch.cuda.stream(stream):
        times = timed_steps(step, K, warmup, flush, stream)
        ptimes = timed_steps(prologue, K, warmup, flush, stream)
    err = S.sinkattn_get_error(stream)
    if err:
        raise RuntimeError(f"device error {S.status_string(err)}")
    moved = (qkv.numel() + q.numel() + 2 * T * Hkv * D) * 2 + bias.numel() * 2  # bytes read + written
    return inp, step, times, 4 * D * Hq * inp.visible_pairs(), ptimes, moved, (qkv, bias)


def bench_chunked(S, W, rank, K, warmup, flush, stream):
    """One step = the serving step of a chunked prefill: append the new tokens' K/V into the pages,
    then the paged prefill over prefix + new tokens.  Returns the attention flops per step."""
    inp = W.chunked_prefill(device="cuda", seed=rank)
    out = torch.empty_like(inp.q)
    lse = torch.empty(inp.q.shape[0], inp.q.shape[1], dtype=torch.float32, device="cuda")

    def step():
        S.sinkattn_kv_append(inp.k_new, inp.v_new, inp.cu_seqlens, inp.start_pos, inp.page_table, inp.k_pages,
                             inp.v_pages, stream=stream)
        S.sinkattn_prefill_paged(inp.q, inp.k_pages, inp.v_pages, inp.page_table, inp.cu_seqlens, inp.start_pos,
                                 inp.sinks, inp.scale, max_seqlen=inp.max_seqlen, out=out, lse=lse, stream=stream)

    with torch.cuda.stream(stream):
        times = timed_steps(step, K, warmup, flush, stream)
    err = S.sinkattn_get_error(stream)
    if err:
        raise RuntimeError(f"device error {S.status_string(err)}")
    return inp, step, times, 4 * 64 * inp.q.shape[1] * inp.visible_pairs()


def bench_prefill(S, W, name, rank, K, warmup, flush, stream):
    inp = (W.mixed_serving_prefill if name == "mixed_serving" else W.causal_prefill)(device="cuda", seed=rank)
    out = torch.empty_like(inp.q)
    lse = torch.empty(inp.q.shape[0], inp.q.shape[1], dtype=torch.float32, device="cuda")

    def step():
        S.sinkattn_prefill(inp.q, inp.k, inp.v, inp.cu_seqlens, inp.sinks, inp.scale, True,
                           max_seqlen=inp.max_seqlen, out=out, lse=lse, stream=stream)

    with torch.cuda.stream(stream):
        times = timed_steps(step, K, warmup, flush, stream)
    err = S.sinkattn_get_error(stream)
    if err:
        raise RuntimeError(f"device error {S.status_string(err)}")
    flops = 4 * 64 * inp.q.shape[1] * inp.visible_pairs()
    return inp, step, times, flops


def oracle_request(inp, b, masks=None):
    """Runs the fp64 oracle on every query row of request b of a decode / verification workload
    (inputs on the host); returns the cache bytes that request reads."""
    import oracle

    B, Hq = inp.q.shape[0], inp.q.shape[-2]
    Hkv = inp.k_pages.shape[1]
    args = (inp.q, inp.k_pages, inp.v_pages, inp.page_table, inp.kv_lens)
    if inp.q.dim() == 4:  # verification inputs carry q_len query tokens per request
        QL = inp.q.shape[1]
        rows = torch.tensor([[b, i, h] for i in range(QL) for h in range(Hq)], dtype=torch.int32).numpy()
        if masks is None:
            oracle.verify(*args, inp.sinks, inp.scale, rows=rows)
        else:
            oracle.verify_tree(*args, masks, inp.sinks, inp.scale, rows=rows)
    else:
        rows = torch.tensor([[b, h] for h in range(Hq)], dtype=torch.int32).numpy()
        oracle.decode(*args, inp.sinks, inp.scale, rows=rows)
    return int(inp.kv_lens[b]) * Hkv * 64 * 4


def one_thread(fn, fargs, budget_s=4.0):
    """The same oracle baseline on one host thread (a shorter sample), for the per-core figure."""
    import oracle

    n = oracle.num_threads()
    oracle.set_num_threads(1)
    try:
        r = fn(*fargs, budget_s=budget_s)
    finally:
        oracle.set_num_threads(n)
    return {"value": r["value"], "unit": r["unit"], "cores": 1, "sample": r["sample"]}


def cpu_baseline_decode(inp, masks=None, budget_s=12.0):
    """The fp64 oracle on the host cores, on whole requests of the same workload, ~budget_s of CPU work."""
    import oracle

    inp = inp.to("cpu")
    masks = masks.cpu() if masks is not None else None
    B, Hq = inp.q.shape[0], inp.q.shape[-2]
    QL = inp.q.shape[1] if inp.q.dim() == 4 else 1
    done_bytes, reqs = 0, 0
    t0 = time.perf_counter()
    while time.perf_counter() - t0 < budget_s:
        done_bytes += oracle_request(inp, reqs % B, masks)
        reqs += 1
    dt = time.perf_counter() - t0
    return {"value": done_bytes / dt / 1e9, "unit": "GB/s", "cores": oracle.num_threads(), "kind": "oracle",
            "sample": f"{reqs} whole requests (all {QL} x {Hq} query rows) of the same workload, fp64, {dt:.1f} s"}


def cpu_baseline_chunked(inp, budget_s=8.0):
    """The fp64 oracle (append, then paged prefill of random rows) on the host cores."""
    import numpy as np

    import oracle

    kb, vb = oracle.kv_append(inp.k_new, inp.v_new, inp.cu_seqlens, inp.start_pos, inp.page_table, inp.k_pages,
                              inp.v_pages)
    q, pt, cu, sp, sk = inp.q.cpu(), inp.page_table.cpu(), inp.cu_seqlens.cpu(), inp.start_pos.cpu(), inp.sinks.cpu()
    T, Hq, _ = q.shape
    rng = np.random.default_rng(0)
    cul, spl = cu.tolist(), sp.tolist()
    pairs, n = 0, 0
    t0 = time.perf_counter()
    while time.perf_counter() - t0 < budget_s:
        t = int(rng.integers(0, T))
        rows = np.stack([np.full(Hq, t), np.arange(Hq)], 1).astype(np.int32)
        oracle.prefill_paged(q, kb, vb, pt, cu, sp, sk, inp.scale, rows=rows)
        s = max(i for i in range(len(cul) - 1) if cul[i] <= t)
        pairs += (spl[s] + t - cul[s] + 1) * Hq
        n += 1
    dt = time.perf_counter() - t0
    return {"value": 4 * 64 * pairs / dt / 1e12, "unit": "TFLOP/s", "cores": oracle.num_threads(), "kind": "oracle",
            "sample": f"{n} random new-token rows (all {Hq} heads) of the workload after the append, fp64, {dt:.1f} s"}


def cpu_baseline_serving(inp, qkv, bias, budget_s=10.0):
    """The fp64 oracle for the serving step: the prologue of every new token (bias + YaRN rotary,
    k/v into the pages), then the paged prefill of random rows, the prefill part scaled to the whole
    step by its share of the step's pairs."""
    import numpy as np

    import oracle

    inp = inp.to("cpu")
    qkv, bias = qkv.cpu(), bias.cpu()
    T, Hq, _ = inp.q.shape
    Hkv = inp.k_pages.shape[1]
    to_bf16 = lambda a: torch.from_numpy(a).float().to(torch.bfloat16)
    t0 = time.perf_counter()
    q, k, v = oracle.qkv_prologue(qkv, bias, inp.cu_seqlens, inp.start_pos, Hq, Hkv, **YARN_GPT_OSS)
    kb, vb = oracle.kv_append(to_bf16(k), to_bf16(v), inp.cu_seqlens, inp.start_pos, inp.page_table, inp.k_pages,
                              inp.v_pages)
    q = to_bf16(q)
    t_pro = time.perf_counter() - t0
    rng = np.random.default_rng(0)
    cul, spl = inp.cu_seqlens.tolist(), inp.start_pos.tolist()
    pairs, n = 0, 0
    t1 = time.perf_counter()
    while time.perf_counter() - t1 < budget_s:
        t = int(rng.integers(0, T))
        rows = np.stack([np.full(Hq, t), np.arange(Hq)], 1).astype(np.int32)
        oracle.prefill_paged(q, kb, vb, inp.page_table, inp.cu_seqlens, inp.start_pos, inp.sinks, inp.scale,
                             rows=rows)
        s = max(i for i in range(len(cul) - 1) if cul[i] <= t)
        pairs += (spl[s] + t - cul[s] + 1) * Hq
        n += 1
    t_rows = time.perf_counter() - t1
    total_pairs = Hq * inp.visible_pairs()
    step_s = t_pro + t_rows * total_pairs / pairs
    return {"value": 4 * 64 * total_pairs / step_s / 1e12, "unit": "TFLOP/s", "cores": oracle.num_threads(),
            "kind": "oracle",
            "sample": f"the prologue + append of all {T} new tokens ({t_pro:.1f} s), then {n} random new-token rows "
                      f"(all {Hq} heads) of the paged prefill ({t_rows:.1f} s), scaled to the step's "
                      f"{total_pairs} (row, key) pairs; fp64"}


def cpu_baseline_prefill(inp, budget_s=8.0):
    import numpy as np

    import oracle

    q, k, v, cu, sk = inp.q.cpu(), inp.k.cpu(), inp.v.cpu(), inp.cu_seqlens.cpu(), inp.sinks.cpu()
    T, Hq, _ = q.shape
    rng = np.random.default_rng(0)
    cul = cu.tolist()
    pairs, n = 0, 0
    t0 = time.perf_counter()
    while time.perf_counter() - t0 < budget_s:
        t = int(rng.integers(0, T))
        rows = np.stack([np.full(Hq, t), np.arange(Hq)], 1).astype(np.int32)
        oracle.prefill(q, k, v, cu, sk, inp.scale, True, rows=rows)
        s = max(i for i in range(len(cul) - 1) if cul[i] <= t)
        pairs += (t - cul[s] + 1) * Hq
        n += 1
    dt = time.perf_counter() - t0
    return {"value": 4 * 64 * pairs / dt / 1e12, "unit": "TFLOP/s", "cores": oracle.num_threads(), "kind": "oracle",
            "sample": f"{n} random query rows (all {Hq} heads) of the workload, fp64, {dt:.1f} s"}


# ----------------------------------------------------------------------------- arms

def run_reference(args):
    """Reference arm: the fp64 oracle, as it stands, on the host cores (rank 0 only), on the same
    workload, metric and unit as the GPU arm.  Decode-type workloads: one step = whole requests
    (every query row); prefill-type workloads: one step = a fixed number of random new-token rows
    (all heads), counted by the (row, key) pairs they cover."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    import numpy as np

    from gqa_attention_learned_head_gb300 import workloads as W
    import oracle

    name = args.workload
    masks, pre = None, None
    if name in ("batched_paged_decode", "long_context_decode", "tiny_decode", "speculative_verify", "tree_verify"):
        if name == "tree_verify":
            inp, masks = W.tree_verify(device="cpu", seed=0)
        else:
            inp = getattr(W, name)(device="cpu", seed=0)
        B, Hq = inp.q.shape[0], inp.q.shape[-2]
        # about a quarter of a second of oracle work per step on 16 cores; a 131072-token request is a step of its own
        per_step = {"long_context_decode": 1, "speculative_verify": 8, "tree_verify": 4}.get(name, B)
        unit, scale_units = "GB/s", 1e9
        step_text = f"{per_step} whole request(s) x all query rows through the fp64 CPU oracle"

        def step(i):
            return sum(oracle_request(inp, (i * per_step + j) % B, masks) for j in range(per_step))
    else:
        to_bf16 = lambda a: torch.from_numpy(a).float().to(torch.bfloat16)
        if name in ("causal_prefill",):
            inp = W.causal_prefill(device="cpu", seed=0)
            starts = [0] * len(inp.seqlens)
            run_rows = lambda rows: oracle.prefill(inp.q, inp.k, inp.v, inp.cu_seqlens, inp.sinks, inp.scale, True,
                                                   rows=rows)
        else:
            inp = W.chunked_prefill(device="cpu", seed=0)
            starts = inp.start_pos.tolist()
            if name == "serving_step":  # the prologue's output is the prefill's q / k / v (setup, not timed)
                T, Hq = inp.q.shape[:2]
                Hkv = inp.k_pages.shape[1]
                g = torch.Generator().manual_seed(1000)
                qkv = torch.randn(T, (Hq + 2 * Hkv) * 64, generator=g).to(torch.bfloat16)
                bias = torch.randn((Hq + 2 * Hkv) * 64, generator=g).to(torch.bfloat16)
                q, k, v = oracle.qkv_prologue(qkv, bias, inp.cu_seqlens, inp.start_pos, Hq, Hkv, **YARN_GPT_OSS)
                inp.q, inp.k_new, inp.v_new = to_bf16(q), to_bf16(k), to_bf16(v)
            kb, vb = oracle.kv_append(inp.k_new, inp.v_new, inp.cu_seqlens, inp.start_pos, inp.page_table,
                                      inp.k_pages, inp.v_pages)
            run_rows = lambda rows: oracle.prefill_paged(inp.q, kb, vb, inp.page_table, inp.cu_seqlens,
                                                         inp.start_pos, inp.sinks, inp.scale, rows=rows)
        T, Hq = inp.q.shape[:2]
        cul = inp.cu_seqlens.tolist()
        rng = np.random.default_rng(0)
        per_step = 2
        unit, scale_units = "TFLOP/s", 1e12
        step_text = (f"{per_step} random new-token rows x {Hq} heads through the fp64 CPU oracle"
                     + (" (the append / prologue done once, untimed)" if name != "causal_prefill" else ""))

        def step(i):
            flops = 0
            for _ in range(per_step):
                t = int(rng.integers(0, T))
                run_rows(np.stack([np.full(Hq, t), np.arange(Hq)], 1).astype(np.int32))
                n = max(j for j in range(len(cul) - 1) if cul[j] <= t)
                flops += 4 * 64 * Hq * (starts[n] + t - cul[n] + 1)
            return flops

    for i in range(args.warmup):
        step(i)
    t0 = time.perf_counter()
    units = sum(step(args.warmup + i) for i in range(args.steps))
    dt = time.perf_counter() - t0
    value = units / dt / scale_units
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": unit, "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt / args.steps * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": WORKLOAD_TEXT[name], "step": step_text},
            "cpu_baseline": {"value": value, "unit": unit, "cores": oracle.num_threads(), "kind": "oracle",
                             "sample": f"{step_text}, per step; {args.steps} steps"},
            "e2e": {"value": value, "unit": unit, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def run_ours(args):
    rank, world, local = dist_setup(args)
    from gqa_attention_learned_head_gb300 import sinkattn as S
    from gqa_attention_learned_head_gb300 import workloads as W

    hbm_peak, tc_peak, tc_sustained, peak_src = peaks()
    stream = torch.cuda.Stream()
    flush_buf = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device="cuda")
    flush_src = torch.ones(2 * L2_FLUSH_BYTES // 4, dtype=torch.float32, device="cuda")
    flush_acc = torch.zeros(1, dtype=torch.float32, device="cuda")

    def flush():
        # Write a buffer twice the size of L2, then read another one: the L2 ends up full of clean
        # lines of unrelated data, so the timed step neither hits its own data nor pays for writing
        # back dirty flush lines.
        flush_buf.fill_(rank & 0x7f)
        flush_acc.copy_(flush_src.sum().view(1))

    sampler = ClockSampler(local) if rank == 0 else None
    if sampler:
        sampler.start()
        time.sleep(0.3)

    K, Wu = args.steps, args.warmup
    name = args.workload
    barrier(world)
    torch.cuda.synchronize()
    t_load0 = time.time()
    masks = None
    if name in ("batched_paged_decode", "long_context_decode", "tiny_decode", "speculative_verify", "tree_verify"):
        workers = 0
        # the tiny case (32 KB) is latency-bound: per call, flushed; the others steady-state over
        # independent input sets that together outgrow L2 (the long context: 1 GiB per set)
        sets = 1 if name == "tiny_decode" else 2 if name == "long_context_decode" else STEADY_SETS
        if name in ("speculative_verify", "tree_verify"):
            inp, step, times, nbytes, steady, masks = bench_verify(S, W, rank, K, Wu, flush, stream, sets=sets,
                                                                    tree=name == "tree_verify")
        else:
            inp, step, times, nbytes, steady = bench_decode(S, W, name, rank, K, Wu, flush, stream, workers,
                                                            sets=sets)
        flushed_ms = statistics.mean(times)
        ms, step_bytes = steady if steady else (flushed_ms, nbytes)
        torch.cuda.synchronize()
        barrier(world)
        ms_max = max_over_ranks(ms, world)
        total_bytes = sum_over_ranks(float(step_bytes), world)
        value = total_bytes / (ms_max * 1e-3) / 1e9
        unit = "GB/s"
        achieved = step_bytes / (ms * 1e-3) / 1e9
        verify = name in ("speculative_verify", "tree_verify")
        kname, call = ("verify_tc_kernel", "sinkattn_verify" + ("_tree" if name == "tree_verify" else "")) if verify \
            else ("decode_split_kernel", "sinkattn_decode")
        per_call = decode_launches_per_call(inp.q.shape[0], inp.k_pages.shape[1], inp.page_table.shape[1], workers)
        roof = {"bound": "hbm",
                "kernel": f"{kname} and, behind it, split_merge_kernel (the kernels of a {call} call); achieved over "
                          "the whole call" if per_call == 2 else f"{kname} (the only kernel of a {call} call)",
                "achieved": achieved, "peak": hbm_peak, "unit": "GB/s", "frac": achieved / hbm_peak,
                "peak_source": f"{peak_src} hbm_gbs",
                "traffic": profiled_traffic(kname, name, KERNEL_SOURCES[kname])}
        launches = per_call * K
        cfg_extra = {"kv_tokens": int(inp.kv_lens.sum()), "kv_bytes_per_step": step_bytes}
        if steady:
            flushed_gbs = nbytes / (flushed_ms * 1e-3) / 1e9
            cfg_extra["per_call_flushed"] = {
                "value": flushed_gbs, "unit": "GB/s", "ms_per_step": flushed_ms, "frac_of_hbm_peak": flushed_gbs / hbm_peak,
                "kv_bytes_per_step": nbytes,
                "method": "input set 0 alone, one call per step between its own event pair, L2 flushed before each "
                          "(256 MiB write, then 512 MiB read); the event pair and the stream launch after the flush "
                          "add a few microseconds of front-end time to every step"}
        if name == "long_context_decode":
            cfg_extra["split"] = ("automatic: one share per resident CTA (the configuration's 32 chunks per "
                                  "(request, KV head) are timed in the secondary lines)")
    elif name in ("chunked_prefill", "serving_step"):
        if name == "chunked_prefill":
            inp, step, times, flops = bench_chunked(S, W, rank, K, Wu, flush, stream)
        else:
            inp, step, times, flops, ptimes, moved, (qkv, bias) = bench_prologue_chunked(S, W, rank, K, Wu, flush,
                                                                                        stream)
        total_flops = sum_over_ranks(float(flops), world)
        ms = statistics.mean(times)
        torch.cuda.synchronize()
        barrier(world)
        ms_max = max_over_ranks(ms, world)
        value = total_flops / (ms_max * 1e-3) / 1e12
        unit = "TFLOP/s"
        achieved = flops / (ms * 1e-3) / 1e12
        first = "kv_append_kernel" if name == "chunked_prefill" else "qkv_prologue_kernel"
        roof = {"bound": "tensor", "kernel": f"prefill_pp_kernel<paged> + {first} (the two kernels of a step); "
                                             "achieved over the whole step",
                "achieved": achieved, "peak": tc_peak, "unit": "TFLOP/s", "frac": achieved / tc_peak,
                "peak_source": f"{peak_src} bf16_tflops",
                "traffic": profiled_traffic("prefill_pp_kernel_paged", "chunked_prefill",
                                            KERNEL_SOURCES["prefill_pp_kernel_paged"])}
        if name == "serving_step":
            p_ms = statistics.mean(ptimes)
            p_gbs = moved / (p_ms * 1e-3) / 1e9
            roof["prologue"] = {"bound": "hbm", "kernel": "qkv_prologue_kernel, timed alone", "ms": p_ms,
                                "achieved": p_gbs, "peak": hbm_peak, "unit": "GB/s", "frac": p_gbs / hbm_peak,
                                "bytes_per_launch": moved,
                                "traffic": profiled_traffic("qkv_prologue_kernel", name,
                                                            KERNEL_SOURCES["qkv_prologue_kernel"])}
        launches = 2 * K  # append (or prologue) + paged prefill per step
        cfg_extra = {"new_tokens": int(inp.q.shape[0]), "cached_tokens": int(inp.start_pos.sum()),
                     "flops_per_step": flops}
    else:
        inp, step, times, flops = bench_prefill(S, W, name, rank, K, Wu, flush, stream)
        total_flops = sum_over_ranks(float(flops), world)
        ms = statistics.mean(times)
        torch.cuda.synchronize()
        barrier(world)
        ms_max = max_over_ranks(ms, world)
        value = total_flops / (ms_max * 1e-3) / 1e12
        unit = "TFLOP/s"
        achieved = flops / (ms * 1e-3) / 1e12
        # an even query-head group runs the two-head kernel, an odd one the one-head kernel
        kname = "prefill_pp_kernel" if (inp.q.shape[1] // inp.k.shape[1]) % 2 == 0 else "prefill_tc_kernel"
        roof = {"bound": "tensor", "kernel": f"{kname} (the only kernel of a sinkattn_prefill call)",
                "achieved": achieved, "peak": tc_peak, "unit": "TFLOP/s", "frac": achieved / tc_peak,
                "peak_source": f"{peak_src} bf16_tflops",
                "traffic": profiled_traffic(kname, name, KERNEL_SOURCES[kname])}
        launches = K
        cfg_extra = {"tokens": int(inp.q.shape[0]), "flops_per_step": flops}
    if unit == "GB/s" and name != "tiny_decode":
        l2_text = (f"inputs larger than L2: the K timed steps run back to back over {sets} independent input sets "
                   f"({sets} x {step_bytes / 1e6:.0f} MB of K/V), so each step's cache was last read {sets - 1} steps "
                   "earlier; the K steps captured in one CUDA graph and timed as one replay between an event pair")
    else:
        l2_text = "flushed before every timed step (256 MiB write, then 512 MiB read)"
    # keep the GPU under the same load for >= 1.5 s of clock samples (not timed)
    while not args.kernels_only and time.time() - t_load0 < 1.5:
        with torch.cuda.stream(stream):
            for _ in range(50):
                flush()
                step()
        torch.cuda.synchronize()
    t_load1 = time.time()

    # ---- end to end through the public API: per-step inputs from pinned host memory, result read back.
    # A step's inputs travel in one host-to-device copy and its results in one device-to-host copy
    # (Staging), as a serving loop that stages each step's tensors in one buffer would do.
    e2e = None
    if not args.kernels_only:
        bf16, i32, f32 = torch.bfloat16, torch.int32, torch.float32
        if name == "chunked_prefill":
            srcs = (inp.q, inp.k_new, inp.v_new, inp.cu_seqlens, inp.start_pos, inp.page_table)
            res = [(inp.q.shape, bf16), (inp.q.shape[:2], f32)]
            metric_units, unit_scale, e_unit = total_flops, 1e12, "TFLOP/s"
            note = ("the page pools stay resident (they are the cache); new tokens' q/k/v and the metadata come from "
                    "pinned host memory every step and the output + lse are read back")

            def api(d, o):
                q, kn, vn, cu, sp, pt = d
                S.sinkattn_kv_append(kn, vn, cu, sp, pt, inp.k_pages, inp.v_pages, stream=stream)
                S.sinkattn_prefill_paged(q, inp.k_pages, inp.v_pages, pt, cu, sp, inp.sinks, inp.scale,
                                         max_seqlen=inp.max_seqlen, out=o[0], lse=o[1], stream=stream)
        elif name == "serving_step":
            srcs = (qkv, inp.cu_seqlens, inp.start_pos, inp.page_table)
            res = [(inp.q.shape, bf16), (inp.q.shape[:2], f32)]
            metric_units, unit_scale, e_unit = total_flops, 1e12, "TFLOP/s"
            note = ("the page pools and the QKV bias stay resident; the new tokens' fused QKV projection output and "
                    "the metadata come from pinned host memory every step and the output + lse are read back")
            d_q = torch.empty_like(inp.q)
            Hq = inp.q.shape[1]

            def api(d, o):
                x, cu, sp, pt = d
                S.sinkattn_qkv_prologue(x, bias, cu, sp, pt, inp.k_pages, inp.v_pages, Hq, q_out=d_q, stream=stream,
                                        **YARN_GPT_OSS)
                S.sinkattn_prefill_paged(d_q, inp.k_pages, inp.v_pages, pt, cu, sp, inp.sinks, inp.scale,
                                         max_seqlen=inp.max_seqlen, out=o[0], lse=o[1], stream=stream)
        elif name == "causal_prefill":
            srcs = (inp.q, inp.k, inp.v, inp.cu_seqlens)
            res = [(inp.q.shape, bf16), (inp.q.shape[:2], f32)]
            metric_units, unit_scale, e_unit = total_flops, 1e12, "TFLOP/s"
            note = "q, k, v and cu_seqlens come from pinned host memory every step and the output + lse are read back"

            def api(d, o):
                S.sinkattn_prefill(d[0], d[1], d[2], d[3], inp.sinks, inp.scale, True, max_seqlen=inp.max_seqlen,
                                   out=o[0], lse=o[1], stream=stream)
        else:
            srcs = (inp.q, inp.page_table, inp.kv_lens) + ((masks,) if masks is not None else ())
            res = [(inp.q.shape, bf16), (inp.q.shape[:-1], f32)]
            metric_units, unit_scale, e_unit = total_bytes, 1e9, "GB/s"
            note = ("KV pool stays resident in HBM (it is the cache); q, page table and lengths"
                    + (" and the tree masks" if masks is not None else "")
                    + " come from pinned host memory every step and the output + lse are read back")
            verify = name in ("speculative_verify", "tree_verify")
            ws_size = S.sinkattn_verify_workspace_size if verify else S.sinkattn_decode_workspace_size
            ws = torch.empty(ws_size(inp.q, inp.k_pages, inp.page_table), dtype=torch.uint8, device="cuda")

            def api(d, o):
                kw = dict(out=o[0], lse=o[1], workspace=ws, stream=stream)
                if masks is not None:
                    S.sinkattn_verify_tree(d[0], inp.k_pages, inp.v_pages, d[1], d[2], d[3], inp.sinks, inp.scale, **kw)
                elif verify:
                    S.sinkattn_verify(d[0], inp.k_pages, inp.v_pages, d[1], d[2], inp.sinks, inp.scale, **kw)
                else:
                    S.sinkattn_decode(d[0], inp.k_pages, inp.v_pages, d[1], d[2], inp.sinks, inp.scale, **kw)

        ins = [Staging([(t.shape, t.dtype) for t in srcs]) for _ in range(2)]
        for slot in ins:
            for h, t in zip(slot.h, srcs):
                h.copy_(t)
        outs = [Staging(res) for _ in range(2)]

        def e2e_step():
            ins[0].to_device()
            api(ins[0].d, outs[0].d)
            outs[0].to_host()

        with torch.cuda.stream(stream):
            et = timed_steps(e2e_step, K, Wu, flush, stream)
        e_ms = max_over_ranks(statistics.mean(et), world)
        try:
            p_ms, p_err = pipelined_ms(api, ins, outs, K, Wu, stream), None
        except Exception as exc:  # report, never hide (every rank still joins the reduction below)
            p_ms, p_err = float("nan"), f"{type(exc).__name__}: {exc}"
        p_ms = max_over_ranks(p_ms, world)
        e2e = {"value": metric_units / (e_ms * 1e-3) / unit_scale, "unit": e_unit, "ms_per_step": e_ms,
               "h2d_bytes_per_step": ins[0].nbytes, "d2h_bytes_per_step": outs[0].nbytes,
               "copies_per_step": {"h2d": 1, "d2h": 1}, "note": note,
               "pipelined": {"value": metric_units / (p_ms * 1e-3) / unit_scale, "unit": e_unit, "ms_per_step": p_ms,
                             "mode": "double-buffered serving loop captured in one CUDA graph, no L2 flush: step "
                                     "i+1's inputs copy in and step i-1's results copy out on their own streams "
                                     "while step i computes; K steps timed as one replay",
                             **({"error": p_err} if p_err else {})}}

    # ---- secondary workloads (rank 0 reports its own numbers)
    secondary = []
    if not args.no_secondary:
        Ks = max(3, min(K, 20))
        try:
            for split, workers in (("the configuration's 32 chunks per (request, KV head): 1024 shares, 1.7 waves "
                                    "of resident CTAs", 4 * 8 * W.LONG_CONTEXT_CHUNKS),
                                   ("automatic: one share per resident CTA, ~19 pieces per (request, KV head)", 0)):
                li, _, lt, lb, lsteady = bench_decode(S, W, "long_context_decode", rank, Ks, Wu, flush, stream,
                                                      num_workers=workers, sets=2)
                lms, lsb = lsteady
                secondary.append({"workload": WORKLOAD_TEXT["long_context_decode"], "split": split,
                                  "value": lsb / (lms * 1e-3) / 1e9, "unit": "GB/s", "ms_per_step": lms,
                                  "frac_of_hbm_peak": lsb / (lms * 1e-3) / 1e9 / hbm_peak,
                                  "method": "steady state over 2 input sets (1 GiB of K/V each)",
                                  "per_call_flushed_ms": statistics.mean(lt),
                                  "traffic": profiled_traffic("decode_split_kernel", "long_context_decode",
                                                              KERNEL_SOURCES["decode_split_kernel"])})
                del li
            # the two decode configurations also replayed from a CUDA graph (launch overhead stripped)
            gi, gstep, gt, gb, _ = bench_decode(S, W, "tiny_decode", rank, Ks, Wu, flush, stream)
            g_ms = graph_ms(gstep, 100, 5, stream)
            tms = statistics.mean(gt)
            secondary.append({"workload": WORKLOAD_TEXT["tiny_decode"], "value": gb / (tms * 1e-3) / 1e9,
                              "unit": "GB/s", "ms_per_step": tms, "us_per_call": tms * 1e3,
                              "graph": {"us_per_call": g_ms * 1e3, "value": gb / (g_ms * 1e-3) / 1e9, "unit": "GB/s",
                                        "method": "100 calls back to back in one CUDA graph, replayed 5 times "
                                                  "(32 KB of K/V: no flush)"}})
            del gi
            bi, bstep, _, bb, _ = bench_decode(S, W, "batched_paged_decode", rank, 3, Wu, flush, stream)
            b_ms = graph_ms(bstep, 20, 5, stream, flush=flush)
            secondary.append({"workload": WORKLOAD_TEXT["batched_paged_decode"], "value": bb / (b_ms * 1e-3) / 1e9,
                              "unit": "GB/s", "ms_per_step": b_ms, "frac_of_hbm_peak": bb / (b_ms * 1e-3) / 1e9 / hbm_peak,
                              "graph": {"method": "20 x (L2 flush, call) in one CUDA graph, replayed 5 times, minus a "
                                                  "graph of the 20 flushes alone"}})
            del bi
            vi, _, vt, vb0, (vms, vb), _ = bench_verify(S, W, rank, Ks, Wu, flush, stream, sets=STEADY_SETS)
            secondary.append({"workload": WORKLOAD_TEXT["speculative_verify"], "value": vb / (vms * 1e-3) / 1e9,
                              "unit": "GB/s", "ms_per_step": vms, "frac_of_hbm_peak": vb / (vms * 1e-3) / 1e9 / hbm_peak,
                              "method": f"steady state over {STEADY_SETS} input sets",
                              "per_call_flushed": {"ms_per_step": statistics.mean(vt),
                                                   "value": vb0 / (statistics.mean(vt) * 1e-3) / 1e9},
                              "traffic": profiled_traffic("verify_tc_kernel", "speculative_verify",
                                                          KERNEL_SOURCES["verify_tc_kernel"])})
            del vi
            ti, _, tt, tb0, (tms, tb), _ = bench_verify(S, W, rank, Ks, Wu, flush, stream, sets=STEADY_SETS,
                                                         tree=True)
            secondary.append({"workload": WORKLOAD_TEXT["tree_verify"], "value": tb / (tms * 1e-3) / 1e9,
                              "unit": "GB/s", "ms_per_step": tms, "frac_of_hbm_peak": tb / (tms * 1e-3) / 1e9 / hbm_peak,
                              "method": f"steady state over {STEADY_SETS} input sets",
                              "per_call_flushed": {"ms_per_step": statistics.mean(tt),
                                                   "value": tb0 / (statistics.mean(tt) * 1e-3) / 1e9},
                              "traffic": profiled_traffic("verify_tc_kernel", "tree_verify",
                                                          KERNEL_SOURCES["verify_tc_kernel"])})
            del ti
            pi, _, pt_, pf = bench_prefill(S, W, "causal_prefill", rank, Ks, Wu, flush, stream)
            pms = statistics.mean(pt_)
            secondary.append({"workload": WORKLOAD_TEXT["causal_prefill"], "value": pf / (pms * 1e-3) / 1e12,
                              "unit": "TFLOP/s", "ms_per_step": pms,
                              "frac_of_bf16_peak": pf / (pms * 1e-3) / 1e12 / tc_peak})
            del pi
            ci, _, ct, cf = bench_chunked(S, W, rank, Ks, Wu, flush, stream)
            cms = statistics.mean(ct)
            secondary.append({"workload": WORKLOAD_TEXT["chunked_prefill"], "value": cf / (cms * 1e-3) / 1e12,
                              "unit": "TFLOP/s", "ms_per_step": cms,
                              "frac_of_bf16_peak": cf / (cms * 1e-3) / 1e12 / tc_peak})
            del ci
            _, _, st_, sf, pt2, moved, _ = bench_prologue_chunked(S, W, rank, Ks, Wu, flush, stream)
            sms, pms2 = statistics.mean(st_), statistics.mean(pt2)
            secondary.append({"workload": "serving step of the chunked prefill: fused prologue (QKV bias + YaRN "
                                          "rotary, k/v into the pages) + paged prefill, same sequences",
                              "value": sf / (sms * 1e-3) / 1e12, "unit": "TFLOP/s", "ms_per_step": sms,
                              "frac_of_bf16_peak": sf / (sms * 1e-3) / 1e12 / tc_peak,
                              "prologue_ms": pms2, "prologue_GB/s": moved / (pms2 * 1e-3) / 1e9,
                              "prologue_frac_of_hbm_peak": moved / (pms2 * 1e-3) / 1e9 / hbm_peak})
            secondary.append(bench_mixed(S, W, rank, Ks, Wu, flush, hbm_peak, tc_peak))
        except Exception as e:  # report, never hide
            secondary.append({"error": f"{type(e).__name__}: {e}"})

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        fn, fargs = ((cpu_baseline_decode, (inp, masks)) if unit == "GB/s" else
                     (cpu_baseline_chunked, (inp,)) if name == "chunked_prefill" else
                     (cpu_baseline_serving, (inp, qkv, bias)) if name == "serving_step" else
                     (cpu_baseline_prefill, (inp,)))
        cpu = fn(*fargs)
        cpu["one_thread"] = one_thread(fn, fargs)

    clocks = None
    if sampler:
        sampler.stop()
        clocks = sampler.summary(t_load0, t_load1)

    if rank == 0:
        line = {"metric": METRIC, "value": value, "unit": unit, "n_gpus": world, "steps": K, "warmup": Wu,
                "ms_per_step": ms_max, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
                "dtype": "bf16", "data": "synthetic (seeded, drawn on the device; input set j of rank r: seed 16 r + j)",
                "config": {"workload": WORKLOAD_TEXT[name], "l2": l2_text, **cfg_extra},
                "roofline": roof, "cpu_baseline": cpu, "e2e": e2e, "gpu_launches": launches, "clocks": clocks,
                "secondary": secondary}
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist

        dist.destroy_process_group()


def bench_mixed(S, W, rank, K, Wu, flush, hbm_peak, tc_peak):
    """Prefill and decode halves of the mixed batch on two streams; time vs t* = bytes/BW + flops/peak.
    Schedule: the decode goes first with two shares per SM, then the prefill with share_sms (the
    one-head kernel), so every SM runs two decode CTAs beside one prefill CTA -- the HBM-bound half
    beside the tensor-bound one.  With the default kernels each half fills whole SMs and the two run
    one after the other (reported as serial_ms)."""
    pre = W.mixed_serving_prefill(device="cuda", seed=rank)
    dec = W.mixed_serving_decode(device="cuda", seed=rank)
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    workers = 2 * torch.cuda.get_device_properties(torch.cuda.current_device()).multi_processor_count
    ws = torch.empty(S.sinkattn_decode_workspace_size(dec.q, dec.k_pages, dec.page_table, workers), dtype=torch.uint8,
                     device="cuda")
    ws_auto = torch.empty(S.sinkattn_decode_workspace_size(dec.q, dec.k_pages, dec.page_table), dtype=torch.uint8,
                          device="cuda")
    po, dout = torch.empty_like(pre.q), torch.empty_like(dec.q)
    main = torch.cuda.current_stream()

    def step():
        s1.wait_stream(main)
        s2.wait_stream(main)
        S.sinkattn_decode(dec.q, dec.k_pages, dec.v_pages, dec.page_table, dec.kv_lens, dec.sinks, dec.scale,
                          out=dout, return_lse=False, workspace=ws, num_workers=workers, stream=s2)
        S.sinkattn_prefill(pre.q, pre.k, pre.v, pre.cu_seqlens, pre.sinks, pre.scale, True,
                           max_seqlen=pre.max_seqlen, out=po, return_lse=False, share_sms=True, stream=s1)
        main.wait_stream(s1)
        main.wait_stream(s2)

    def serial():  # the default kernels, one after the other
        S.sinkattn_decode(dec.q, dec.k_pages, dec.v_pages, dec.page_table, dec.kv_lens, dec.sinks, dec.scale,
                          out=dout, return_lse=False, workspace=ws_auto, stream=main)
        S.sinkattn_prefill(pre.q, pre.k, pre.v, pre.cu_seqlens, pre.sinks, pre.scale, True,
                           max_seqlen=pre.max_seqlen, out=po, return_lse=False, stream=main)

    times = timed_steps(step, K, Wu, flush, main)
    serial_times = timed_steps(serial, K, Wu, flush, main)
    if S.sinkattn_get_error(main):
        raise RuntimeError("device error in mixed batch")
    ms = statistics.mean(times)
    nbytes = decode_bytes(dec.kv_lens, 8)
    flops = 4 * 64 * 64 * pre.visible_pairs()
    t_star = nbytes / (hbm_peak * 1e9) + flops / (tc_peak * 1e12)
    t_overlap = max(nbytes / (hbm_peak * 1e9), flops / (tc_peak * 1e12))
    return {"workload": WORKLOAD_TEXT["mixed_serving"], "value": ms, "unit": "ms", "higher_is_better": False,
            "t_star_ms": t_star * 1e3, "frac_of_t_star": t_star * 1e3 / ms,
            "overlap_bound_ms": t_overlap * 1e3, "frac_of_overlap_bound": t_overlap * 1e3 / ms,
            "bounds": "t_star = bytes / BW + flops / peak (the halves one after the other); overlap bound = "
                      "max(bytes / BW, flops / peak) (the halves fully overlapped)",
            "decode_bytes": nbytes,
            "prefill_flops": flops, "serial_ms": statistics.mean(serial_times),
            "schedule": f"decode first with {workers} shares (two per SM), then the prefill with share_sms "
                        "(one-head kernel) on a second stream; serial_ms = the default kernels one after the other"}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="batched_paged_decode",
                    choices=["batched_paged_decode", "long_context_decode", "tiny_decode", "speculative_verify",
                             "tree_verify", "causal_prefill", "chunked_prefill", "serving_step"])
    ap.add_argument("--no-secondary", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--kernels-only", action="store_true",
                    help="only the warm-up and timed steps of the headline workload (for profiler runs)")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.kernels_only:
        args.no_secondary = args.no_cpu_baseline = True
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
