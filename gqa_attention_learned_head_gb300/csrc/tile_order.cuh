// tile_order.cuh -- maps a CTA's linear tile index to (sequence, query tile)
// for packed variable-length prefill, heaviest tiles first.
//
// With causal masking, query tile t of a sequence attends to t+1 key tiles, so
// the last tile of a sequence is its heaviest.  Tiles are enumerated by
// "distance from the sequence's last tile" r = 0, 1, 2, ...; within one r, by
// sequence index.  Every CTA derives the order itself from cu_seqlens (no host
// knowledge of the lengths, no workspace): a histogram of tiles per sequence,
// two block-wide scans, a binary search and a ballot search.
#pragma once
#include "ptx.cuh"

namespace sinkattn {

// In-place exclusive scan of arr[0, n) in shared memory; returns the total.
// Every thread of the block must call it.  s_warp holds kThreads/32 ints.
template <int kThreads>
__device__ int block_exclusive_scan(int* arr, int n, int* s_warp) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int running = 0;
    for (int base = 0; base < n; base += kThreads) {
        const int i = base + threadIdx.x;
        const int v = i < n ? arr[i] : 0;
        int incl = v;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += y;
        }
        if (lane == 31) s_warp[warp] = incl;
        __syncthreads();
        int woff = 0, tot = 0;
#pragma unroll
        for (int w = 0; w < kThreads / 32; ++w) {
            const int t = s_warp[w];
            woff += (w < warp) ? t : 0;
            tot += t;
        }
        if (i < n) arr[i] = running + woff + incl - v;
        running += tot;
        __syncthreads();
    }
    return running;
}

// Shared-memory ints needed by TileOrder for N sequences and kmax tiles per sequence.
__host__ __device__ inline size_t tile_order_smem_ints(int N, int kmax) { return size_t(N) + size_t(kmax) + 1 + 40; }

template <int kThreads>
struct TileOrder {
    int* s_nt;    // [N]       tiles of each sequence (capped at kmax)
    int* s_c;     // [kmax+1]  C(r) = number of tiles with distance < r
    int* s_misc;  // [40]      scan scratch + broadcast slots
    int N, kmax, total;

    // Phase A: every thread of the block calls this once.
    // Sequences whose rows fall outside [0, T) or whose length is negative or
    // above max_seqlen are flagged; a negative or out-of-range one gets no tile,
    // a too-long one is cut to max_seqlen rows.
    __device__ void build(int* smem, const int* cu, int N_, int T, int max_seqlen, int bm, unsigned* err) {
        N = N_;
        kmax = (max_seqlen + bm - 1) / bm;
        s_nt = smem;
        s_c = smem + N;
        s_misc = s_c + kmax + 1;
        for (int r = threadIdx.x; r <= kmax; r += kThreads) s_c[r] = 0;
        __syncthreads();
        for (int n = threadIdx.x; n < N; n += kThreads) {
            const int lo = cu[n], hi = cu[n + 1];
            int L = hi - lo;
            if (lo < 0 || hi > T || L < 0 || L > max_seqlen) {
                if (blockIdx.x == 0) atomicOr(err, kErrBadLength);
                L = (lo < 0 || hi > T || L < 0) ? 0 : max_seqlen;
            }
            const int nt = (L + bm - 1) / bm;
            s_nt[n] = nt;
            if (nt > 0) atomicAdd(&s_c[nt - 1], 1);  // histogram of (tiles - 1)
        }
        __syncthreads();
        // cnt(r) = #{n : nt(n) > r} = live - (#{n : nt(n) - 1 < r})
        const int live = block_exclusive_scan<kThreads>(s_c, kmax, s_misc);
        for (int r = threadIdx.x; r < kmax; r += kThreads) s_c[r] = live - s_c[r];
        __syncthreads();
        total = block_exclusive_scan<kThreads>(s_c, kmax, s_misc);
        if (threadIdx.x == 0) s_c[kmax] = total;
        __syncthreads();
    }

    // Phase A done by warp 0 alone with shuffle scans; the caller then needs one block barrier
    // before any thread reads the tables.  Same tables as build().
    __device__ void build_warp0(int* smem, const int* cu, int N_, int T, int max_seqlen, int bm, unsigned* err) {
        N = N_;
        kmax = (max_seqlen + bm - 1) / bm;
        s_nt = smem;
        s_c = smem + N;
        s_misc = s_c + kmax + 1;
        total = 0;
        if (threadIdx.x >= 32) return;
        const int lane = threadIdx.x;
        for (int r = lane; r <= kmax; r += 32) s_c[r] = 0;
        __syncwarp();
        int live = 0;
        for (int n = lane; n < N; n += 32) {
            const int lo = __ldg(&cu[n]), hi = __ldg(&cu[n + 1]);
            int L = hi - lo;
            if (lo < 0 || hi > T || L < 0 || L > max_seqlen) {
                if (blockIdx.x == 0) atomicOr(err, kErrBadLength);
                L = (lo < 0 || hi > T || L < 0) ? 0 : max_seqlen;
            }
            const int nt = (L + bm - 1) / bm;
            s_nt[n] = nt;
            if (nt > 0) {
                atomicAdd(&s_c[nt - 1], 1);  // histogram of (tiles - 1)
                ++live;
            }
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) live += __shfl_xor_sync(0xffffffffu, live, o);
        __syncwarp();
        // cnt(r) = live - #{n : nt(n) - 1 < r}; C(r) = sum_{r' < r} cnt(r')
        int run_h = 0, run_c = 0;
        for (int base = 0; base < kmax; base += 32) {
            const int r = base + lane;
            const int hv = r < kmax ? s_c[r] : 0;
            int ih = hv;  // inclusive scan of the histogram
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int y = __shfl_up_sync(0xffffffffu, ih, o);
                if (lane >= o) ih += y;
            }
            const int cnt = r < kmax ? live - (run_h + ih - hv) : 0;
            int ic = cnt;  // inclusive scan of cnt
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int y = __shfl_up_sync(0xffffffffu, ic, o);
                if (lane >= o) ic += y;
            }
            __syncwarp();
            if (r < kmax) s_c[r] = run_c + ic - cnt;
            run_h += __shfl_sync(0xffffffffu, ih, 31);
            run_c += __shfl_sync(0xffffffffu, ic, 31);
        }
        total = run_c;
        if (lane == 0) {
            s_c[kmax] = total;
            s_misc[0] = total;
        }
    }
    // After the block barrier that follows build_warp0: every thread learns the total.
    __device__ void finish_warp0_build() { total = s_misc[0]; }

    // Phase B: every thread calls it with the same idx < total.  Returns
    // the sequence and the query-tile index inside it.
    __device__ void lookup(int idx, int& seq, int& tile) {
        int lo = 0, hi = kmax - 1;  // largest r with C(r) <= idx
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (s_c[mid] <= idx) lo = mid;
            else hi = mid - 1;
        }
        const int r = lo, j = idx - s_c[r];
        // j-th sequence (in index order) with nt > r
        const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
        int base = 0, found = -1;
        for (int c = 0; c < N && found < 0; c += kThreads) {
            const int n = c + threadIdx.x;
            const bool f = n < N && s_nt[n] > r;
            const unsigned bal = __ballot_sync(0xffffffffu, f);
            if (lane == 0) s_misc[warp] = __popc(bal);
            __syncthreads();
            int woff = 0, tot = 0;
#pragma unroll
            for (int w = 0; w < kThreads / 32; ++w) {
                const int t = s_misc[w];
                woff += (w < warp) ? t : 0;
                tot += t;
            }
            if (f && base + woff + __popc(bal & ((1u << lane) - 1)) == j) s_misc[32] = n;
            __syncthreads();
            if (base + tot > j) found = s_misc[32];
            base += tot;
            __syncthreads();
        }
        seq = found;
        tile = s_nt[found] - 1 - r;
    }

    // Phase B for one warp on its own (no block barrier): all 32 lanes call it with the same
    // idx < total and get the same answer.
    __device__ void lookup_warp(int idx, int& seq, int& tile) const {
        int lo = 0, hi = kmax - 1;  // largest r with C(r) <= idx
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (s_c[mid] <= idx) lo = mid;
            else hi = mid - 1;
        }
        const int r = lo, lane = threadIdx.x & 31;
        int j = idx - s_c[r], found = 0;
        for (int c = 0; c < N; c += 32) {  // j-th sequence (in index order) with nt > r
            const int n = c + lane;
            unsigned bal = __ballot_sync(0xffffffffu, n < N && s_nt[n] > r);
            const int cnt = __popc(bal);
            if (j < cnt) {
                for (int t = 0; t < j; ++t) bal &= bal - 1;
                found = c + __ffs(bal) - 1;
                break;
            }
            j -= cnt;
        }
        seq = found;
        tile = s_nt[found] - 1 - r;
    }
};

// Sequence-major order, for the tcgen05 prefills: the query tiles of one sequence are consecutive,
// from its last (heaviest) tile to its first, so the CTAs running at any moment share one
// sequence's K and V and L2 keeps them between tiles.  (An order that visits every sequence for
// each tile distance re-reads their K/V from memory once the batch's K/V outgrows L2.)  Sequences
// come by descending weight, ties by index; the weight is the key count of the sequence's heaviest
// tile (cached prefix + new tokens), so the CTAs that start last are the lightest ones of the
// least-weighted sequence.  Up to kSortMax sequences are ranked by a warp bitonic sort; a larger
// batch keeps index order.
constexpr int kSortMax = 128;  // 32 lanes x 4 keys

__host__ __device__ inline size_t seq_order_smem_ints(int N) {
    return size_t(N) + 1 + (N <= kSortMax ? 2 * size_t(N) : 0);
}

// Bitonic sort, descending, of the 32 * E keys held by one warp: lane l holds positions l*E .. l*E+E-1.
template <int E>
__device__ __forceinline__ void warp_sort_desc(unsigned long long (&v)[E]) {
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int k = 2; k <= 32 * E; k <<= 1) {
#pragma unroll
        for (int j = k >> 1; j > 0; j >>= 1) {
            unsigned long long o[E];
#pragma unroll
            for (int e = 0; e < E; ++e) o[e] = j < E ? v[(e ^ j) & (E - 1)] : __shfl_xor_sync(0xffffffffu, v[e], j / E);
#pragma unroll
            for (int e = 0; e < E; ++e) {
                const int i = lane * E + e;
                // a block of size k runs descending when (i & k) == 0; the lower position of a
                // compared pair keeps the larger key in a descending block, the smaller otherwise
                const bool keep_max = ((i & j) == 0) == ((i & k) == 0);
                v[e] = keep_max ? (v[e] > o[e] ? v[e] : o[e]) : (v[e] < o[e] ? v[e] : o[e]);
            }
        }
    }
}

// Exclusive scan of arr[0, n) in place by one warp; returns the total.
__device__ __forceinline__ int warp_exclusive_scan(int* arr, int n) {
    const int lane = threadIdx.x & 31;
    int run = 0;
    for (int base = 0; base < n; base += 32) {
        const int i = base + lane;
        const int v = i < n ? arr[i] : 0;
        int inc = v;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, inc, o);
            if (lane >= o) inc += y;
        }
        if (i < n) arr[i] = run + inc - v;
        run += __shfl_sync(0xffffffffu, inc, 31);
    }
    return run;
}

struct SeqOrder {
    int* s_pre;   // [N+1] tiles before each rank; s_pre[N] = total
    int* s_perm;  // [N]   sequence of each rank (sorted batches only)
    int* s_nt;    // [N]   tiles of each sequence (sorted batches only)
    int N, total;
    bool sorted;

    // Warp 0 builds the tables; the caller then needs one block barrier before any thread reads them
    // (finish_build, lookup_warp).  start = cache position of each sequence's first new token, null
    // without a cached prefix.  Sequences whose rows fall outside [0, T) or whose length is negative
    // or above max_seqlen are flagged; a negative or out-of-range one gets no tile, a too-long one is
    // cut to max_seqlen rows.
    __device__ void build_warp0(int* smem, const int* cu, const int* start, int N_, int T, int max_seqlen, int bm,
                                unsigned* err) {
        N = N_;
        sorted = N <= kSortMax;
        s_pre = smem;
        s_perm = smem + N + 1;
        s_nt = s_perm + N;
        total = 0;
        if (threadIdx.x >= 32) return;
        const int lane = threadIdx.x;
        auto rows = [&](int n) {
            const int lo = __ldg(&cu[n]), hi = __ldg(&cu[n + 1]);
            int L = hi - lo;
            if (lo < 0 || hi > T || L < 0 || L > max_seqlen) {
                if (blockIdx.x == 0) atomicOr(err, kErrBadLength);
                L = (lo < 0 || hi > T || L < 0) ? 0 : max_seqlen;
            }
            return L;
        };
        if (!sorted) {
            for (int n = lane; n < N; n += 32) s_pre[n] = (rows(n) + bm - 1) / bm;
            __syncwarp();
        } else {
            // key = weight << 32 | ~index: descending order = heaviest first, then lowest index;
            // the padding keys (0) sort after every sequence
            auto key = [&](int n) -> unsigned long long {
                if (n >= N) return 0ull;
                const int L = rows(n), nt = (L + bm - 1) / bm;
                s_nt[n] = nt;
                const int s0 = start ? min(max(__ldg(&start[n]), 0), 1 << 30) : 0;
                const unsigned w = nt > 0 ? (unsigned)(s0 + min(L, 1 << 30)) : 0u;
                return ((unsigned long long)w << 32) | (0xffffffffu - (unsigned)n);
            };
            auto place = [&](unsigned long long k, int i) {
                if (i < N) s_perm[i] = (int)(0xffffffffu - (unsigned)(k & 0xffffffffull));
            };
            if (N <= 32) {
                unsigned long long v[1] = {key(lane)};
                warp_sort_desc<1>(v);
                place(v[0], lane);
            } else {
                constexpr int E = kSortMax / 32;
                unsigned long long v[E];
#pragma unroll
                for (int e = 0; e < E; ++e) v[e] = key(lane * E + e);
                warp_sort_desc<E>(v);
#pragma unroll
                for (int e = 0; e < E; ++e) place(v[e], lane * E + e);
            }
            __syncwarp();
            for (int i = lane; i < N; i += 32) s_pre[i] = s_nt[s_perm[i]];
            __syncwarp();
        }
        const int tot = warp_exclusive_scan(s_pre, N);
        if (lane == 0) s_pre[N] = tot;
    }
    // After the block barrier that follows build_warp0: every thread learns the total.
    __device__ void finish_build() { total = s_pre[N]; }

    // Every lane of a warp calls it with the same idx < total and gets the sequence and the query
    // tile inside it.
    __device__ void lookup_warp(int idx, int& seq, int& tile) const {
        int lo = 0, hi = N - 1;  // largest rank k with s_pre[k] <= idx (an empty rank is passed over)
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (s_pre[mid] <= idx) lo = mid;
            else hi = mid - 1;
        }
        seq = sorted ? s_perm[lo] : lo;
        tile = s_pre[lo + 1] - 1 - idx;  // heaviest (last) tile at the sequence's first rank
    }
};

}  // namespace sinkattn
