// tile_order.cuh -- maps a CTA's linear tile index to (sequence, query tile)
// for packed variable-length prefill, heaviest tiles first, sequence by
// sequence.
//
// With causal masking, query tile t of a sequence attends to t+1 key tiles, so
// the last tile of a sequence is its heaviest.  Every CTA derives the order
// itself from cu_seqlens (and start_pos over a paged cache): no host knowledge
// of the lengths, no workspace.
#pragma once
#include "ptx.cuh"

namespace sinkattn {

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
