// verify_tc.cu -- attention of drafted tokens over the paged cache (verification in
// speculative decoding) on the fifth-generation tensor cores.
//
// Source: "Accelerating Sonar through speculation" (Perplexity), sections
// "Speculative decoding" and "Inference with speculative decoding" (the target
// model scores every drafted token in one pass over the paged KV cache) and
// section "EAGLE" (a tree of drafts checked with a custom attention mask); the
// attention is the sink attention of "GPT-OSS on day 0", section "Kernels for
// GPT-OSS / Sink Attention".  Query token i of request b is the cache token at
// position kv_len - q_len + i and sees cache tokens 0 .. that position (or, for
// a tree, every token before the draft and the drafted tokens its mask names).
//
// GB300 design.  The R = q_len x G query rows of one (request b, KV head g) --
// row r = i * G + h is drafted token i of query head g * G + h -- form ONE
// tcgen05 tile (R <= 64, padded to the MMA's 128 rows), so the group's K/V pass
// costs the cache bytes once and every product runs on the tensor core:
//   warps 0, 3  TMA producers: warp 0 loads the rows of Q with one 3-D copy
//               (64 dims x G heads x q_len tokens, landing as rows i * G + h)
//               and the K tiles, warp 3 the V tiles; a 128-key tile is 8 page
//               copies of 2 KB (lanes 0-7), 128-byte swizzle.
//   warp 1      allocates 256 TMEM columns; one lane issues S_j = Q K_j^T.
//   warp 2      one lane issues O += P_j V_j (P read from TMEM).
//   warps 4-7   softmax, thread r = row r (only the warps that hold rows work):
//               each row masked at its own causal limit or by its tree mask.
// A (request, KV head) segment is cut into chunks of whole 128-key tiles, one CTA
// each; the chunk holding token 0 is seeded with the sink.  A segment of several
// chunks writes fp32 partials per row and the CTA that completes it (an epoch-
// tagged arrival counter) merges them by log-sum-exp.  Every wait is bounded.
#include "args_verify.h"
#include "ptx.cuh"
#include "split_kv.cuh"
#include "tc_tile.cuh"

namespace sinkattn {
namespace {

using namespace tc;

constexpr int kThreads = 256;
constexpr uint32_t kTmemCols = 256;
constexpr uint32_t kColS = 0, kColO = 128, kColP = 192;
constexpr int kKStages = 3, kVStages = 2;
constexpr int kPagesPerTile = kBN / kPageSize;  // 8

struct __align__(1024) Smem {
    uint8_t q[kTileBytes];
    uint8_t k[kKStages][kTileBytes];
    uint8_t v[kVStages][kTileBytes];
    uint64_t q_full, k_full[kKStages], k_empty[kKStages], v_full[kVStages], v_empty[kVStages];
    uint64_t s_full, s_free, p_full, o_done, mma_done, v_fixed;
    uint32_t tmem_base;
    int last;  // this CTA completes its segment and merges it
};

// TMA row of page pg of segment (b, g) in the 2-D map over the page pool; a page past the cache
// end and a page id outside the pool give a row past the pool's end, which the copy fills with zeros.
__device__ __forceinline__ int page_row(const VerifyArgs& a, int b, int g, int pg, int kv_len) {
    const int oob = a.num_pages * a.Hkv * kPageSize;
    if (pg >= a.max_pages || pg * kPageSize >= kv_len) return oob;
    const int pid = __ldg(&a.page_table[(long long)b * a.max_pages + pg]);
    if (pid < 0 || pid >= a.num_pages) {
        atomicOr(a.err, kErrBadPage);
        return oob;
    }
    return (pid * a.Hkv + g) * kPageSize;
}

__device__ __forceinline__ void softmax_bar() { asm volatile("bar.sync 1, 128;" ::: "memory"); }

// 128-key tiles of request i's cache (its length clamped to the page table's reach)
__device__ __forceinline__ int request_tiles(const VerifyArgs& a, int i) {
    return (clamp_len(__ldg(&a.kv_lens[i]), a.max_pages * kPageSize) + kBN - 1) / kBN;
}

// Chunks of request i (every KV head of the request has that many): chunks of at most
// ceil(U / target) tiles, so that the U tiles of all segments make at most target + segments chunks.
__device__ __forceinline__ int request_chunks(long long tiles, long long target, long long U) {
    if (U <= 0 || tiles <= 1) return 1;
    const long long size = (U + target - 1) / target;
    return (int)((tiles + size - 1) / size);
}

struct Located {
    int b, x0, n, tiles;  // request, index of its first chunk, chunks per KV head, tiles per segment
};

// Finds the request whose chunks hold CTA index x (chunk index = request-major, then KV head, then
// chunk): U over all requests, then a running block-wide scan of the chunk counts.  Every CTA
// computes the same plan; false if x is past the last chunk.  All threads take part.
__device__ bool locate(const VerifyArgs& a, long long x, int* scratch, Located& loc) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    constexpr int kWarpsPerCta = kThreads / 32;
    long long part = 0;
    for (int i = tid; i < a.B; i += kThreads) {
        const int raw = __ldg(&a.kv_lens[i]);
        if ((raw < 0 || raw > a.max_pages * kPageSize) && blockIdx.x == 0) atomicOr(a.err, kErrBadLength);
        part += request_tiles(a, i);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) part += __shfl_xor_sync(0xffffffffu, part, o);
    long long* red = reinterpret_cast<long long*>(scratch);  // [kWarpsPerCta] warp totals
    if (lane == 0) red[warp] = part;
    __syncthreads();
    long long U = 0;
#pragma unroll
    for (int w = 0; w < kWarpsPerCta; ++w) U += red[w];
    U *= a.Hkv;
    int* found = scratch + 2 * kWarpsPerCta;  // [0] flag, [1] b, [2] x0, [3] n, [4] tiles
    if (tid == 0) found[0] = 0;
    __syncthreads();
    long long base = 0;
    for (int p0 = 0; p0 < a.B; p0 += kThreads) {
        const int i = p0 + tid;
        int tb = 0, nb = 0;
        long long cnt = 0;
        if (i < a.B) {
            tb = request_tiles(a, i);
            nb = request_chunks(tb, a.tc_target, U);
            cnt = (long long)nb * a.Hkv;
        }
        long long incl = cnt;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const long long y = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += y;
        }
        __syncthreads();  // the previous pass has read red[]
        if (lane == 31) red[warp] = incl;
        __syncthreads();
        long long woff = 0, total = 0;
#pragma unroll
        for (int w = 0; w < kWarpsPerCta; ++w) {
            woff += w < warp ? red[w] : 0;
            total += red[w];
        }
        const long long lo = base + woff + incl - cnt;
        if (i < a.B && cnt > 0 && x >= lo && x < lo + cnt) {
            found[0] = 1;
            found[1] = i;
            found[2] = (int)lo;
            found[3] = nb;
            found[4] = tb;
        }
        base += total;
        __syncthreads();
        if (found[0]) break;
    }
    loc.b = found[1];
    loc.x0 = found[2];
    loc.n = found[3];
    loc.tiles = found[4];
    return found[0] != 0;
}

// ---- a segment of several chunks: the CTA whose arrival completes it merges the partials, by the
// four softmax warps (after their partials are written) with one thread per row
__device__ __forceinline__ void merge_segment(const VerifyArgs& a, Smem& sm, int seg, long long slot0, int b, int g,
                                              int nchunks) {
    const int R = a.R, QL = a.QL, G = a.G;
    softmax_bar();  // every partial of this CTA is written (CTA scope) ...
    if (threadIdx.x == 128) sm.last = arrive_last(&a.counters[seg], a.epoch, nchunks) ? 1 : 0;  // ... and published
    softmax_bar();
    const int r = threadIdx.x - 128;
    if (!sm.last || r >= R) return;
    const float* lp = a.part_lse + slot0 * R + r;
    const float* op = a.part_o + (slot0 * R + r) * kHeadDim;
    float M = kNegInf;
    for (int k = 0; k < nchunks; ++k) M = fmaxf(M, __ldcg(lp + (long long)k * R));
    const int i = r / G, h = r % G;
    const long long row = ((long long)b * QL + i) * a.Hq + g * G + h;
    uint4* dst = reinterpret_cast<uint4*>(a.out + row * kHeadDim);
    if (M == kNegInf) {  // no live key and no finite sink in any chunk
#pragma unroll
        for (int e = 0; e < 8; ++e) dst[e] = make_uint4(0u, 0u, 0u, 0u);
        if (a.lse) a.lse[row] = kNegInf;
        return;
    }
    float sum = 0.f;
    float acc[64];
#pragma unroll
    for (int e = 0; e < 64; ++e) acc[e] = 0.f;
    for (int k = 0; k < nchunks; ++k) {
        const float l = __ldcg(lp + (long long)k * R);
        if (l == kNegInf) continue;
        const float w = exp2f(l - M);
        sum += w;
        const float4* src = reinterpret_cast<const float4*>(op + (long long)k * R * kHeadDim);
#pragma unroll
        for (int e = 0; e < 16; ++e) {
            const float4 v = __ldcg(src + e);
            acc[4 * e + 0] += w * v.x;
            acc[4 * e + 1] += w * v.y;
            acc[4 * e + 2] += w * v.z;
            acc[4 * e + 3] += w * v.w;
        }
    }
    const float inv = 1.f / sum;
#pragma unroll
    for (int e = 0; e < 8; ++e)
        dst[e] = make_uint4(pack_bf16(acc[8 * e + 0] * inv, acc[8 * e + 1] * inv),
                            pack_bf16(acc[8 * e + 2] * inv, acc[8 * e + 3] * inv),
                            pack_bf16(acc[8 * e + 4] * inv, acc[8 * e + 5] * inv),
                            pack_bf16(acc[8 * e + 6] * inv, acc[8 * e + 7] * inv));
    if (a.lse) a.lse[row] = (M + log2f(sum)) * kLn2;
}

__global__ void __launch_bounds__(kThreads, 2)
    verify_tc_kernel(const __grid_constant__ CUtensorMap tmap_q, const __grid_constant__ CUtensorMap tmap_k,
                     const __grid_constant__ CUtensorMap tmap_v, const VerifyArgs a) {
    extern __shared__ uint8_t smem_raw[];
    Smem& sm = *reinterpret_cast<Smem*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    Located loc;
    if (!locate(a, blockIdx.x, reinterpret_cast<int*>(sm.k[0]), loc)) return;  // whole CTA: past the last chunk
    const int nchunks = loc.n, local = (int)(blockIdx.x - loc.x0);
    const int b = loc.b, g = local / nchunks, c = local % nchunks;
    const int seg = b * a.Hkv + g;
    const long long slot0 = (long long)loc.x0 + (long long)g * nchunks;  // partial slot of the segment's chunk 0
    const int kv_len = clamp_len(__ldg(&a.kv_lens[b]), a.max_pages * kPageSize);
    const int tiles = loc.tiles;
    // chunk c of the segment: tiles [c * tiles / n, (c + 1) * tiles / n)
    const int t0 = (int)((long long)c * tiles / nchunks), t1 = (int)((long long)(c + 1) * tiles / nchunks);
    const int ntile = t1 - t0;
    const bool whole = nchunks == 1;
    const int R = a.R, QL = a.QL, G = a.G;
    const int pos0 = kv_len - QL;  // cache position of drafted token 0 (negative for a short cache)
    const int active = (R + 31) / 32;  // softmax warps that hold rows
    // the last V tile may end inside a page whose later slots hold anything
    const bool fix_last_v = ntile > 0 && t1 == tiles && tiles * kBN > kv_len;

    if (threadIdx.x == 0) {
        mbar_init(&sm.q_full, 1);
        for (int i = 0; i < kKStages; ++i) {
            mbar_init(&sm.k_full[i], 1);
            mbar_init(&sm.k_empty[i], 1);
        }
        for (int i = 0; i < kVStages; ++i) {
            mbar_init(&sm.v_full[i], 1);
            mbar_init(&sm.v_empty[i], 1);
        }
        mbar_init(&sm.s_full, 1);
        mbar_init(&sm.s_free, 32 * active);
        mbar_init(&sm.p_full, 32 * active);
        mbar_init(&sm.o_done, 1);
        mbar_init(&sm.mma_done, 2);
        mbar_init(&sm.v_fixed, 1);
        sm.last = 0;
        fence_mbar_init();
        fence_proxy_async_smem();
    }
    if (warp == 1) {
        tmem_alloc(&sm.tmem_base, kTmemCols);
        tmem_relinquish();
    }
    // Q rows R..127 (no query) are zeros, so their scores stay finite; the TMA writes rows 0..R-1
    for (int e = R * 8 + (int)threadIdx.x; e < kBM * 8; e += kThreads)
        reinterpret_cast<uint4*>(sm.q)[e] = make_uint4(0u, 0u, 0u, 0u);
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tbase = sm.tmem_base;

    if (warp < 4) {
        asm volatile("setmaxnreg.dec.sync.aligned.u32 56;");
        if (ntile > 0 && (warp == 0 || warp == 3)) {
            // ------------------------------------------------------------ TMA producers
            const bool is_k = warp == 0;
            const int stages = is_k ? kKStages : kVStages;
            uint64_t* full = is_k ? sm.k_full : sm.v_full;
            uint64_t* empty = is_k ? sm.k_empty : sm.v_empty;
            const CUtensorMap* map = is_k ? &tmap_k : &tmap_v;
            if (lane == 0) {
                tma_prefetch_desc(map);
                if (is_k) {
                    tma_prefetch_desc(&tmap_q);
                    mbar_arrive_expect_tx(&sm.q_full, (uint32_t)R * 128u);
                    tma_load_3d(sm.q, &tmap_q, 0, g * G, b * QL, &sm.q_full);
                }
            }
            int issued = 0;
            bool ok = true;
            for (int j = 0; j < ntile; ++j) {
                const int st = j % stages;
                if (j >= stages) {
                    int got = 0;
                    if (lane == 0) got = mbar_wait(&empty[st], ((j / stages) - 1) & 1);
                    if (!(ok = __shfl_sync(0xffffffffu, got, 0) != 0)) break;
                }
                const int row = page_row(a, b, g, (t0 + j) * kPagesPerTile + (lane & 7), kv_len);
                if (lane == 0) mbar_arrive_expect_tx(&full[st], kTileBytes);
                __syncwarp();
                uint8_t* tile = is_k ? sm.k[st] : sm.v[st];
                if (lane < kPagesPerTile) tma_load_2d(tile + lane * (kPageSize * 128), map, 0, row, &full[st]);
                issued = j + 1;
            }
            if (!ok && lane == 0) atomicOr(a.err, kErrTimeout);
            if (!is_k && ok && fix_last_v) {
                // zero the rows of the last V tile at or past the cache end, then hand it over
                const int j = ntile - 1, st = j % kVStages;
                const bool landed = __all_sync(0xffffffffu, mbar_wait(&sm.v_full[st], (j / kVStages) & 1));
                if (landed) {
                    const int r0 = kv_len - (t1 - 1) * kBN;
                    for (int i = r0 * 8 + lane; i < kBN * 8; i += 32)
                        reinterpret_cast<uint4*>(sm.v[st])[i] = make_uint4(0u, 0u, 0u, 0u);
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&sm.v_fixed);
                } else if (lane == 0) {
                    atomicOr(a.err, kErrTimeout);
                }
            }
            // every copy this warp started has landed before the CTA can exit (bounded)
            if (lane == 0) {
                if (is_k) (void)mbar_wait(&sm.q_full, 0);
                for (int j = issued - stages < 0 ? 0 : issued - stages; j < issued; ++j)
                    (void)mbar_wait(&full[j % stages], (j / stages) & 1);
            }
        } else if (ntile > 0 && warp == 1 && lane == 0) {
            // ------------------------------------------------------------ S issuer: S_j = Q K_j^T
            const uint32_t tS = tbase + kColS;
            const uint32_t qaddr = smem_u32(sm.q);
            bool ok = mbar_wait(&sm.q_full, 0);
            for (int j = 0; ok && j < ntile; ++j) {
                const int st = j % kKStages;
                ok = mbar_wait(&sm.k_full[st], (j / kKStages) & 1) && (j == 0 || mbar_wait(&sm.s_free, (j - 1) & 1));
                if (!ok) break;
                tc_fence_after();
                const uint32_t kaddr = smem_u32(sm.k[st]);
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)
                    tc_mma_ss(tS, sw128_desc(qaddr + kk * 32), sw128_desc(kaddr + kk * 32), kIdescQK, kk > 0);
                tc_commit(&sm.s_full);
                tc_commit(&sm.k_empty[st]);
            }
            if (!ok) atomicOr(a.err, kErrTimeout);
            tc_commit(&sm.mma_done);  // every MMA of both issuers has finished before TMEM is released
            (void)mbar_wait(&sm.mma_done, 0);
        } else if (ntile > 0 && warp == 2 && lane == 0) {
            // ------------------------------------------------------------ PV issuer: O += P_j V_j
            const uint32_t tO = tbase + kColO, tP = tbase + kColP;
            bool ok = true;
            for (int j = 0; ok && j < ntile; ++j) {
                ok = ((fix_last_v && j == ntile - 1) ? mbar_wait(&sm.v_fixed, 0)
                                                     : mbar_wait(&sm.v_full[j % kVStages], (j / kVStages) & 1)) &&
                     mbar_wait(&sm.p_full, j & 1);
                if (!ok) break;
                tc_fence_after();
                const uint32_t vaddr = smem_u32(sm.v[j % kVStages]);
#pragma unroll
                for (int ks = 0; ks < 8; ++ks)
                    tc_mma_ts(tO, tP + ks * 8, sw128_desc(vaddr + ks * 2048), kIdescPV, (j > 0 || ks > 0) ? 1u : 0u);
                tc_commit(&sm.v_empty[j % kVStages]);
                tc_commit(&sm.o_done);
            }
            if (!ok) atomicOr(a.err, kErrTimeout);
            tc_commit(&sm.mma_done);
            (void)mbar_wait(&sm.mma_done, 0);
        }
    } else {
        // 128 x 56 + 128 x 200 = 256 x 128, the launch's registers
        asm volatile("setmaxnreg.inc.sync.aligned.u32 200;");
        const int r = threadIdx.x - 128;
        const bool live = r < R;
        const int i = live ? r / G : 0, h = live ? r % G : 0;
        if (warp - 4 < active) {
            // ---------------------------------------------------------------- softmax
            const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;
            const uint32_t tS = tbase + lane_off + kColS, tO = tbase + lane_off + kColO, tP = tbase + lane_off + kColP;
            const bool tree = a.tree_mask != nullptr;
            // the drafted keys this tree row sees (q_len <= 16 bits)
            const uint32_t dbits =
                (tree && live) ? (uint32_t)(__ldg(&a.tree_mask[(long long)b * QL + i]) & ((1ull << QL) - 1)) : 0u;
            // a linear row sees keys [0, lim)
            const int lim = live ? pos0 + i + 1 : 0;
            const float scale_log2 = a.scale_log2;
            float m = (c == 0 && live) ? __ldg(&a.sinks[g * G + h]) * kLog2e : kNegInf;  // seeded with the sink
            float d = (c == 0 && live) ? 1.f : 0.f;                                      // e^(sink - m) = 1
            bool ok = true;
            for (int j = 0; j < ntile; ++j) {
                if (!(ok = warp_wait(&sm.s_full, j & 1))) break;
                tc_fence_after();
                float s[128];
#pragma unroll
                for (int cc = 0; cc < 4; ++cc)
                    tmem_ld32(tS + cc * 32, *reinterpret_cast<uint32_t(*)[32]>(&s[cc * 32]));
                tc_wait_ld();
                tc_fence_before();
                mbar_arrive(&sm.s_free);

                const int kb = (t0 + j) * kBN;
                float mul = scale_log2;
                if (!(scale_log2 > 0.f)) {  // zero or negative scale: scale first, mask after
#pragma unroll
                    for (int cc = 0; cc < 128; ++cc) s[cc] *= scale_log2;
                    mul = 1.f;
                }
                if (kb + kBN > pos0) {
                    // the tile holds drafted keys or the cache end: this row's visible keys of the tile
                    // as four 32-bit words -- every key before the draft, then (tree) the drafted keys
                    // its mask names or (linear) the drafted keys up to its own
                    const int lo = pos0 - kb;  // keys of the tile before the draft
                    uint32_t vis[4];
#pragma unroll
                    for (int w = 0; w < 4; ++w) {
                        const int n = (tree ? lo : lim - kb) - 32 * w;
                        uint32_t bitsw = n <= 0 ? 0u : n >= 32 ? 0xFFFFFFFFu : ((1u << n) - 1u);
                        const int off = lo - 32 * w;
                        if (tree && off > -32 && off < 32) bitsw |= off >= 0 ? (dbits << off) : (dbits >> -off);
                        vis[w] = bitsw;
                    }
#pragma unroll
                    for (int cc = 0; cc < 128; ++cc) s[cc] = ((vis[cc >> 5] >> (cc & 31)) & 1u) ? s[cc] : kNegInf;
                }
                float acc[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) acc[e] = fmax3(s[e], s[8 + e], s[16 + e]);
#pragma unroll
                for (int cc = 24; cc < 120; cc += 16)
#pragma unroll
                    for (int e = 0; e < 8; ++e) acc[e] = fmax3(acc[e], s[cc + e], s[cc + 8 + e]);
#pragma unroll
                for (int e = 0; e < 8; ++e) acc[e] = fmaxf(acc[e], s[120 + e]);
                const float mx_raw =
                    fmaxf(fmax3(acc[0], acc[1], acc[2]), fmax3(acc[3], acc[4], fmax3(acc[5], acc[6], acc[7])));
                const float mx = mx_raw == kNegInf ? kNegInf : mx_raw * mul;
                const float m_new = fmaxf(m, mx);
                float factor = 1.f;
                bool rescale_o = false;
                if (j == 0 || m_new > m + kRescaleThreshold) {
                    factor = (m_new == kNegInf) ? 1.f : fast_exp2(m - m_new);
                    rescale_o = (j > 0);
                    m = m_new;
                    d *= factor;
                }
                const float neg_m = (m == kNegInf) ? 0.f : -m;
                const float2 mul2 = make_float2(mul, mul), negm2 = make_float2(neg_m, neg_m);
                float2 sums[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f),
                                  make_float2(0.f, 0.f)};
                uint32_t pk[64];
#pragma unroll
                for (int cc = 0; cc < 64; ++cc) {
                    const float2 xx = ffma2(make_float2(s[2 * cc], s[2 * cc + 1]), mul2, negm2);
                    const float2 pp = make_float2(fast_exp2(xx.x), fast_exp2(xx.y));
                    sums[cc & 3] = fadd2(sums[cc & 3], pp);
                    pk[cc] = pack_bf16(pp.x, pp.y);
                }
                const float2 s01 = fadd2(fadd2(sums[0], sums[1]), fadd2(sums[2], sums[3]));
                d += s01.x + s01.y;
                if (j > 0) {  // P_{j-1} consumed and O_{j-1} final before P and O are touched
                    if (!(ok = warp_wait(&sm.o_done, (j - 1) & 1))) break;
                    tc_fence_after();
                    if (__any_sync(0xffffffffu, rescale_o)) {
#pragma unroll
                        for (int cc = 0; cc < 2; ++cc) {
                            uint32_t o[32];
                            tmem_ld32(tO + cc * 32, o);
                            tc_wait_ld();
#pragma unroll
                            for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * factor);
                            tmem_st32(tO + cc * 32, o);
                        }
                    }
                }
                tmem_st32(tP, *reinterpret_cast<uint32_t(*)[32]>(&pk[0]));
                tmem_st32(tP + 32, *reinterpret_cast<uint32_t(*)[32]>(&pk[32]));
                tc_wait_st();
                tc_fence_before();
                mbar_arrive(&sm.p_full);
            }
            if (ok && ntile > 0) ok = warp_wait(&sm.o_done, (ntile - 1) & 1);
            if (!ok) {
                if (lane == 0) atomicOr(a.err, kErrTimeout);
            } else {
                // O / d of this row (zero when the chunk has no key: only an empty cache's single chunk)
                uint32_t o[64];
                if (ntile > 0) {
                    tc_fence_after();
                    tmem_ld32(tO, *reinterpret_cast<uint32_t(*)[32]>(&o[0]));
                    tmem_ld32(tO + 32, *reinterpret_cast<uint32_t(*)[32]>(&o[32]));
                    tc_wait_ld();
                } else {
#pragma unroll
                    for (int e = 0; e < 64; ++e) o[e] = 0u;
                }
                if (live) {
                    const float inv = d > 0.f ? 1.f / d : 0.f;
                    const float l2 = d > 0.f ? m + log2f(d) : kNegInf;
                    if (whole) {
                        const long long row = ((long long)b * QL + i) * a.Hq + g * G + h;
                        uint4* dst = reinterpret_cast<uint4*>(a.out + row * kHeadDim);
#pragma unroll
                        for (int e = 0; e < 8; ++e) {
                            uint4 w;
                            w.x = pack_bf16(__uint_as_float(o[8 * e + 0]) * inv, __uint_as_float(o[8 * e + 1]) * inv);
                            w.y = pack_bf16(__uint_as_float(o[8 * e + 2]) * inv, __uint_as_float(o[8 * e + 3]) * inv);
                            w.z = pack_bf16(__uint_as_float(o[8 * e + 4]) * inv, __uint_as_float(o[8 * e + 5]) * inv);
                            w.w = pack_bf16(__uint_as_float(o[8 * e + 6]) * inv, __uint_as_float(o[8 * e + 7]) * inv);
                            dst[e] = w;
                        }
                        if (a.lse) a.lse[row] = l2 * kLn2;
                    } else {
                        const long long slot = slot0 + c;
                        float4* dst = reinterpret_cast<float4*>(a.part_o + (slot * R + r) * kHeadDim);
#pragma unroll
                        for (int e = 0; e < 16; ++e)
                            dst[e] = make_float4(__uint_as_float(o[4 * e + 0]) * inv, __uint_as_float(o[4 * e + 1]) * inv,
                                                 __uint_as_float(o[4 * e + 2]) * inv, __uint_as_float(o[4 * e + 3]) * inv);
                        a.part_lse[slot * R + r] = l2;
                    }
                }
            }
        }
        if (!whole) merge_segment(a, sm, seg, slot0, b, g, nchunks);
    }
    tc_fence_before();
    __syncthreads();  // TMEM is no longer read
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tbase, kTmemCols);
    }
}

}  // namespace

size_t verify_tc_smem() { return 1024 + sizeof(Smem); }

cudaError_t verify_tc_occupancy(int* per_sm) {
    static thread_local bool set[64] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev >= 64 || !set[dev]) {
        e = cudaFuncSetAttribute(verify_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)verify_tc_smem());
        if (e != cudaSuccess) return e;
        if (dev < 64) set[dev] = true;
    }
    return cudaOccupancyMaxActiveBlocksPerMultiprocessor(per_sm, verify_tc_kernel, kThreads, verify_tc_smem());
}

cudaError_t verify_tc_launch(const VerifyArgs& a, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                             cudaStream_t stream) {
    if (a.B == 0) return cudaSuccess;
    const long long grid = a.tc_grid;
    if (grid > 0x7fffffffll) return cudaErrorInvalidConfiguration;
    int per_sm = 0;  // also sets the kernel's shared-memory limit
    cudaError_t e = verify_tc_occupancy(&per_sm);
    if (e != cudaSuccess) return e;
    verify_tc_kernel<<<(unsigned)grid, kThreads, verify_tc_smem(), stream>>>(tq, tk, tv, a);
    return cudaGetLastError();
}

}  // namespace sinkattn
