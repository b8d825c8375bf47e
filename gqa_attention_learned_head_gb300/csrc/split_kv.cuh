// split_kv.cuh -- the work split shared by the paged kernels (decode and draft
// verification): the flattened list of (request b, KV head g, page) units, cut
// into contiguous per-CTA shares; a share is cut at segment ends into pieces;
// the pieces of a segment held by several CTAs are merged after the kernel by
// the split-merge kernel (slot of CTA c's piece of segment seg: c + seg).
//
// Source of the split: "GPT-OSS on day 0" (Perplexity), section "Kernels for
// GPT-OSS / Sink Attention": attention runs in parallel along the KV length as
// well as over heads, and the blocks along the sequence are combined by their
// running max and scale, with the sink held by the first block only.
#pragma once
#include <cstdint>

namespace sinkattn {

__device__ __forceinline__ int clamp_len(int L, int cap) { return L < 0 ? 0 : (L > cap ? cap : L); }

// One piece of a CTA's share: units [ps, pe) of segment (b, g) whose first unit is seg_start.
struct SegPiece {
    long long ps, pe, seg_start;
    int b, g, n, idx;
    __device__ int len() const { return (int)(pe - ps); }
    __device__ int page0() const { return (int)(ps - seg_start); }
};

// prefix[b] = units (pages) of requests before b; a segment (b, g) spans Hkv-major blocks of n pages.
__device__ __forceinline__ void piece_first(SegPiece& p, const int* prefix, int B, int Hkv, long long x0,
                                            long long x1) {
    int lo = 0, hi = B - 1;  // smallest b with prefix[b+1]*Hkv > x0
    while (lo < hi) {
        const int mid = (lo + hi) >> 1;
        if ((long long)prefix[mid + 1] * Hkv > x0) hi = mid;
        else lo = mid + 1;
    }
    p.b = lo;
    p.n = prefix[lo + 1] - prefix[lo];
    const long long off = x0 - (long long)prefix[lo] * Hkv;
    p.g = (int)(off / p.n);
    p.seg_start = (long long)prefix[lo] * Hkv + (long long)p.g * p.n;
    p.ps = x0;
    p.pe = min(x1, p.seg_start + p.n);
    p.idx = 0;
}

// Moves to the next piece; p.ps >= x1 afterwards means the share is done.
__device__ __forceinline__ void piece_next(SegPiece& p, const int* prefix, int B, int Hkv, long long x1) {
    p.ps = p.pe;
    ++p.idx;
    if (p.ps >= x1) return;
    p.seg_start = p.pe;  // a piece that ends before x1 ends at its segment's end
    if (++p.g == Hkv) {
        p.g = 0;
        do { ++p.b; } while (p.b < B && prefix[p.b + 1] == prefix[p.b]);
        p.n = prefix[p.b + 1] - prefix[p.b];
    }
    p.pe = min(x1, p.seg_start + p.n);
}

// CTA count actually used for U units (identical in every CTA).  workers: the planned count;
// fixed: use it exactly (capped at U); otherwise never cut shares finer than min_pages units.
__device__ __forceinline__ long long effective_shares(long long workers, int fixed, int min_pages, long long U) {
    long long c = workers;
    if (!fixed) {
        const long long want = (U + min_pages - 1) / min_pages;
        if (want < c) c = want;
    }
    if (c > U) c = U;
    return c < 1 ? 1 : c;
}

// Shares (CTAs) that hold units of the segment starting at unit seg_start with n units: first share and count.
__device__ __forceinline__ void segment_pieces(long long seg_start, int n, long long C, long long U, long long& c_first,
                                               int& pieces) {
    c_first = ((seg_start + 1) * C - 1) / U;
    const long long c_last = ((seg_start + n) * C - 1) / U;
    pieces = (int)(c_last - c_first + 1);
}

}  // namespace sinkattn
