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
// costs the cache bytes once and every product runs on the tensor core.
// Work: the flattened list of (request, KV head, 128-key tile) units, one
// contiguous share per CTA (one CTA per resident slot), cut at segment ends
// into pieces (the split of split_kv.cuh with tiles as units).  The pipeline
// runs on across the pieces of a share:
//   warps 0, 3  TMA producers: warp 0 loads each piece's Q rows with one 3-D
//               copy (64 dims x G heads x q_len tokens, landing as rows
//               i * G + h) into a 2-slot Q ring and the K tiles, warp 3 the V
//               tiles; a tile is 8 page copies of 2 KB (lanes 0-7), 128-byte
//               swizzle.
//   warp 1      allocates 256 TMEM columns; issues S_j = Q K_j^T.
//   warp 2      issues O += P_j V_j (P read from TMEM; the first tile of a
//               piece starts O afresh).  Both issuers walk their loops
//               warp-wide and one elected lane issues the products.
//   warps 4-7   softmax, thread r = row r (only the warps that hold rows work),
//               each row masked at its own causal limit or by its tree mask; at
//               a piece's end they read O and write the rows (or fp32 partials).
// A piece holding token 0 is seeded with the sink.  The pieces of a segment
// split between CTAs write fp32 partials; the CTA holding the segment's first
// piece lists it, and the split-merge kernel, launched right behind this one as
// a programmatic dependent, combines them (no CTA waits for another).  The
// kernel itself is a programmatic dependent of what precedes it on the stream.
// Every wait is bounded.
#include "args_merge.h"
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
constexpr int kKStages = 2, kVStages = 2;
constexpr int kPagesPerTile = kBN / kPageSize;  // 8
constexpr int kMinTiles = kVerifyMinTiles;  // automatic mode: never cut shares finer than this


__device__ __forceinline__ int kv_len_of(const VerifyArgs& a, int i) {
    return clamp_len(__ldg(&a.kv_lens[i]), a.max_pages * kPageSize);
}
__device__ __forceinline__ int tiles_of(int kv_len) { return (kv_len + kBN - 1) / kBN; }

// One piece: tiles [ta, tb) of segment (b, g), whose first unit is seg_start and which has `tiles` tiles.
struct Piece {
    int b, g, ta, tb, tiles, kv_len;
    long long seg_start;
};

// Walks the pieces of units [x, x1); every role of the CTA runs its own walker over the same share.
struct Walk {
    int b, g, tiles, kv_len;
    long long seg_start, x, x1;
    int B, Hkv;

    // the next segment with at least one tile (a walk never passes the share's end)
    __device__ void advance(const VerifyArgs& a) {
        seg_start += tiles;
        if (++g == Hkv) {
            g = 0;
            do {
                ++b;
                kv_len = kv_len_of(a, b);
                tiles = tiles_of(kv_len);
            } while (tiles == 0 && b + 1 < B);
        }
    }
    __device__ bool next(const VerifyArgs& a, Piece& p) {
        if (x >= x1) return false;
        while (x >= seg_start + tiles) advance(a);
        p.b = b;
        p.g = g;
        p.tiles = tiles;
        p.kv_len = kv_len;
        p.seg_start = seg_start;
        p.ta = (int)(x - seg_start);
        const long long end = x1 < seg_start + tiles ? x1 : seg_start + tiles;
        p.tb = (int)(end - seg_start);
        x = end;
        return true;
    }
};

struct __align__(1024) Smem {
    uint8_t q[2][kTileBytes];
    uint8_t k[kKStages][kTileBytes];
    uint8_t v[kVStages][kTileBytes];
    uint64_t q_full[2], q_empty[2], k_full[kKStages], k_empty[kKStages], v_full[kVStages], v_empty[kVStages];
    uint64_t s_full, s_free, p_full, o_done, mma_done;
    uint32_t tmem_base;
    long long red[8];    // block reductions
    long long found[4];  // share start: request, its first unit, its tiles, flag
    Walk walk[4];        // the softmax warps' walkers (kept out of their registers)
    Piece piece[4];      // ... and their current pieces
};

__global__ void __launch_bounds__(kThreads, 2)
    verify_tc_kernel(const __grid_constant__ CUtensorMap tmap_q, const __grid_constant__ CUtensorMap tmap_k,
                     const __grid_constant__ CUtensorMap tmap_v, const VerifyArgs a) {
    extern __shared__ uint8_t smem_raw[];
    Smem& sm = *reinterpret_cast<Smem*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int B = a.B, Hkv = a.Hkv, R = a.R, QL = a.QL, G = a.G;
    const int active = (R + 31) / 32;  // softmax warps that hold rows

    // ---- 0. set-up that reads no input (barriers, tensor memory, the Q padding): done before the wait
    // below, so it overlaps the preceding kernel's tail
    if (tid == 0) {
        for (int i = 0; i < 2; ++i) {
            mbar_init(&sm.q_full[i], 1);
            mbar_init(&sm.q_empty[i], 1);
        }
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
        fence_mbar_init();
        fence_proxy_async_smem();
    }
    if (warp == 1) {
        tmem_alloc(&sm.tmem_base, kTmemCols);
        tmem_relinquish();
    }
    // Q rows R..127 (no query) are zeros, so their scores stay finite; the TMA writes rows 0..R-1
    for (int e = R * 8 + tid; e < kBM * 8; e += kThreads) {
        reinterpret_cast<uint4*>(sm.q[0])[e] = make_uint4(0u, 0u, 0u, 0u);
        reinterpret_cast<uint4*>(sm.q[1])[e] = make_uint4(0u, 0u, 0u, 0u);
    }
    fence_proxy_async_smem();

    // a programmatic dependent of what precedes it on the stream: no input is read before that has
    // completed; the split merge behind this kernel may be scheduled once every CTA runs
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

    // ---- 1. units (Hkv x tiles) per request: their total U and, by a running block-wide scan, the
    // request holding this share's first unit (one pass when the batch fits the CTA's threads)
    if (tid == 0) sm.found[3] = 0;
    long long U = 0, base = 0, lo = 0, cnt = 0;
    for (int p0 = 0; p0 < B; p0 += kThreads) {
        const int i = p0 + tid;
        int ti = 0;
        if (i < B) {
            const int raw = __ldg(&a.kv_lens[i]);
            if ((raw < 0 || raw > a.max_pages * kPageSize) && blockIdx.x == 0) atomicOr(a.err, kErrBadLength);
            ti = tiles_of(clamp_len(raw, a.max_pages * kPageSize));
        }
        const long long c = (long long)ti * Hkv;
        long long incl = c;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const long long y = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += y;
        }
        __syncthreads();  // red[] is free
        if (lane == 31) sm.red[warp] = incl;
        __syncthreads();
        long long woff = 0, total = 0;
#pragma unroll
        for (int w = 0; w < kThreads / 32; ++w) {
            woff += w < warp ? sm.red[w] : 0;
            total += sm.red[w];
        }
        if (B <= kThreads) {  // one pass: this thread's request and its units stay in registers
            lo = woff + incl - c;
            cnt = c;
        }
        U = base + total;
        base = U;
    }
    {  // rows of requests with an empty cache carry only the sink
        const long long rows = (long long)B * QL * a.Hq;
        for (long long r = (long long)blockIdx.x * kThreads + tid; r < rows; r += (long long)gridDim.x * kThreads) {
            const int b = (int)(r / ((long long)QL * a.Hq));
            if (kv_len_of(a, b) != 0) continue;
            uint4* dst = reinterpret_cast<uint4*>(a.out + r * kHeadDim);
#pragma unroll
            for (int e = 0; e < 8; ++e) dst[e] = make_uint4(0u, 0u, 0u, 0u);
            if (a.lse) a.lse[r] = __ldg(&a.sinks[r % a.Hq]);
        }
    }
    const long long C = U > 0 ? effective_shares(a.tc_grid, a.fixed_workers, kMinTiles, U) : 0;
    const long long cta = blockIdx.x;
    if (cta >= C) {  // no share: release the tensor memory taken above (the whole CTA is here)
        if (tid == 0 && a.merge_list) a.merge_list[cta] = make_int2(-1, 0);
        tc_fence_before();
        __syncthreads();
        if (warp == 1) {
            tc_fence_after();
            tmem_dealloc(sm.tmem_base, kTmemCols);
        }
        return;
    }
    const long long x0 = cta * U / C, x1 = (cta + 1) * U / C;
    if (B <= kThreads) {
        if (cnt > 0 && x0 >= lo && x0 < lo + cnt) {
            sm.found[0] = tid;
            sm.found[1] = lo;
            sm.found[2] = cnt / Hkv;
        }
        __syncthreads();
    } else {
        // ---- 2. a second scan, now that U (and so x0) is known
        base = 0;
        for (int p0 = 0; p0 < B; p0 += kThreads) {
            const int i = p0 + tid;
            const int ti = i < B ? tiles_of(kv_len_of(a, i)) : 0;
            const long long c = (long long)ti * Hkv;
            long long incl = c;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const long long y = __shfl_up_sync(0xffffffffu, incl, o);
                if (lane >= o) incl += y;
            }
            __syncthreads();  // red[] (and found[3]) are settled
            if (lane == 31) sm.red[warp] = incl;
            __syncthreads();
            long long woff = 0, total = 0;
#pragma unroll
            for (int w = 0; w < kThreads / 32; ++w) {
                woff += w < warp ? sm.red[w] : 0;
                total += sm.red[w];
            }
            const long long l0 = base + woff + incl - c;
            if (c > 0 && x0 >= l0 && x0 < l0 + c) {
                sm.found[0] = i;
                sm.found[1] = l0;
                sm.found[2] = ti;
                sm.found[3] = 1;
            }
            base += total;
            __syncthreads();
            if (sm.found[3]) break;
        }
    }
    Walk walk;
    walk.B = B;
    walk.Hkv = Hkv;
    walk.b = (int)sm.found[0];
    walk.tiles = (int)sm.found[2];
    walk.kv_len = kv_len_of(a, walk.b);
    walk.g = (int)((x0 - sm.found[1]) / walk.tiles);
    walk.seg_start = sm.found[1] + (long long)walk.g * walk.tiles;
    walk.x = x0;
    walk.x1 = x1;
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tbase = sm.tmem_base;

    if (warp < 4) {
        asm volatile("setmaxnreg.dec.sync.aligned.u32 56;");
        if (warp == 0 || warp == 3) {
            // ------------------------------------------------------------ TMA producers
            const bool is_k = warp == 0;
            const int stages = is_k ? kKStages : kVStages;
            uint64_t* full = is_k ? sm.k_full : sm.v_full;
            uint64_t* empty = is_k ? sm.k_empty : sm.v_empty;
            const CUtensorMap* map = is_k ? &tmap_k : &tmap_v;
            if (lane == 0) {
                tma_prefetch_desc(map);
                if (is_k) tma_prefetch_desc(&tmap_q);
            }
            int J = 0, p = 0, issued = 0;  // tiles, pieces (their Q issued) and tile copies issued so far
            bool ok = true;
            Piece pc;
            while (ok && walk.next(a, pc)) {
                if (is_k) {  // this piece's Q rows into Q slot p & 1, once the piece two back has used it
                    int got = 1;
                    if (lane == 0) {
                        if (p >= 2) got = mbar_wait(&sm.q_empty[p & 1], ((p >> 1) - 1) & 1);
                        if (got) {
                            mbar_arrive_expect_tx(&sm.q_full[p & 1], (uint32_t)R * 128u);
                            tma_load_3d(sm.q[p & 1], &tmap_q, 0, pc.g * G, pc.b * QL, &sm.q_full[p & 1]);
                        }
                    }
                    if (!(ok = __shfl_sync(0xffffffffu, got, 0) != 0)) break;
                }
                ++p;
                for (int t = pc.ta; ok && t < pc.tb; ++t, ++J) {
                    const int st = J % stages;
                    if (J >= stages) {
                        int got = 0;
                        if (lane == 0) got = mbar_wait(&empty[st], ((J / stages) - 1) & 1);
                        if (!(ok = __shfl_sync(0xffffffffu, got, 0) != 0)) break;
                    }
                    const int row = page_tile_row(a, pc.b, pc.g, t * kPagesPerTile + (lane & 7), pc.kv_len);
                    if (lane == 0) mbar_arrive_expect_tx(&full[st], kTileBytes);
                    __syncwarp();
                    uint8_t* tile = is_k ? sm.k[st] : sm.v[st];
                    if (lane < kPagesPerTile) tma_load_2d(tile + lane * (kPageSize * 128), map, 0, row, &full[st]);
                    issued = J + 1;
                }
            }
            if (!ok && lane == 0) atomicOr(a.err, kErrTimeout);
            // every copy this warp started has landed before the CTA can exit (bounded)
            if (lane == 0) {
                for (int j = issued - stages < 0 ? 0 : issued - stages; j < issued; ++j)
                    (void)mbar_wait(&full[j % stages], (j / stages) & 1);
                if (is_k)
                    for (int q = p - 2 < 0 ? 0 : p - 2; q < p; ++q) (void)mbar_wait(&sm.q_full[q & 1], (q >> 1) & 1);
            }
        } else if (warp == 1) {
            // ------------------------------------------------------------ S issuer: S_j = Q K_j^T
            // (the whole warp walks the loop, one elected lane issues)
            const uint32_t tS = tbase + kColS;
            int J = 0, p = 0;
            bool ok = true;
            Piece pc;
            while (ok && walk.next(a, pc)) {
                if (!(ok = warp_wait(&sm.q_full[p & 1], (p >> 1) & 1))) break;
                const uint32_t qaddr = smem_u32(sm.q[p & 1]);
                for (int t = pc.ta; t < pc.tb; ++t, ++J) {
                    const int st = J % kKStages;
                    ok = warp_wait(&sm.k_full[st], (J / kKStages) & 1) && (J == 0 || warp_wait(&sm.s_free, (J - 1) & 1));
                    if (!ok) break;
                    tc_fence_after();
                    const uint32_t kaddr = smem_u32(sm.k[st]);
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk)
                        tc_mma_ss_warp(tS, sw128_desc(qaddr + kk * 32), sw128_desc(kaddr + kk * 32), kIdescQK, kk > 0);
                    tc_commit_warp(&sm.s_full);
                    tc_commit_warp(&sm.k_empty[st]);
                }
                tc_commit_warp(&sm.q_empty[p & 1]);  // this piece's Q slot is free once its products end
                ++p;
            }
            if (!ok && lane == 0) atomicOr(a.err, kErrTimeout);
            tc_commit_warp(&sm.mma_done);  // every MMA of both issuers has finished before TMEM is released
            (void)warp_wait(&sm.mma_done, 0);
        } else if (warp == 2) {
            // ------------------------------------------------------------ PV issuer: O += P_j V_j
            // One elected lane issues; the whole warp zeroes the rows past the cache end of a segment's last V
            // tile (they may hold anything, and a 0 weight times NaN is NaN) before its product.
            const uint32_t tO = tbase + kColO, tP = tbase + kColP;
            int J = 0;
            bool ok = true;
            Piece pc;
            while (ok && walk.next(a, pc)) {
                for (int t = pc.ta; t < pc.tb; ++t, ++J) {
                    const int st = J % kVStages;
                    ok = warp_wait(&sm.v_full[st], (J / kVStages) & 1);
                    if (!ok) break;
                    if (t == pc.tiles - 1 && pc.tiles * kBN > pc.kv_len) {
                        for (int e = (pc.kv_len - t * kBN) * 8 + lane; e < kBN * 8; e += 32)
                            reinterpret_cast<uint4*>(sm.v[st])[e] = make_uint4(0u, 0u, 0u, 0u);
                        fence_proxy_async_smem();
                        __syncwarp();
                    }
                    if (!(ok = warp_wait(&sm.p_full, J & 1))) break;
                    tc_fence_after();
                    const uint32_t vaddr = smem_u32(sm.v[st]);
                    // P_j is written only after the softmax has read the previous piece's O, so the first tile of
                    // a piece may start O afresh
#pragma unroll
                    for (int ks = 0; ks < 8; ++ks)
                        tc_mma_ts_warp(tO, tP + ks * 8, sw128_desc(vaddr + ks * 2048), kIdescPV,
                                       (t > pc.ta || ks > 0) ? 1u : 0u);
                    tc_commit_warp(&sm.v_empty[st]);
                    tc_commit_warp(&sm.o_done);
                }
            }
            if (!ok && lane == 0) atomicOr(a.err, kErrTimeout);
            tc_commit_warp(&sm.mma_done);
            (void)warp_wait(&sm.mma_done, 0);
        }
    } else {
        // 128 x 56 + 128 x 200 = 256 x 128, the launch's registers
        asm volatile("setmaxnreg.inc.sync.aligned.u32 200;");
        const int r = tid - 128;
        const bool live = r < R;
        const int i = live ? r / G : 0, h = live ? r % G : 0;
        int2 head = make_int2(-1, 0);  // the share's last piece, if it starts a segment it does not end
        if (warp - 4 < active) {
            // ---------------------------------------------------------------- softmax
            const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;
            const uint32_t tS = tbase + lane_off + kColS, tO = tbase + lane_off + kColO, tP = tbase + lane_off + kColP;
            const bool tree = a.tree_mask != nullptr;
            const float scale_log2 = a.scale_log2;
            int J = 0;
            bool ok = true;
            const int sw = warp - 4;
            if (lane == 0) sm.walk[sw] = walk;
            __syncwarp();
            while (ok) {
                int has = 0;
                __syncwarp();  // every lane is done with the previous piece
                if (lane == 0) has = sm.walk[sw].next(a, sm.piece[sw]) ? 1 : 0;
                if (!__shfl_sync(0xffffffffu, has, 0)) break;
                __syncwarp();
                const Piece& pc = sm.piece[sw];
                const int pos0 = pc.kv_len - QL;  // cache position of drafted token 0 (negative: short cache)
                // the drafted keys this tree row sees (q_len <= 16 bits); a linear row sees keys [0, lim)
                const uint32_t dbits =
                    (tree && live) ? (uint32_t)(__ldg(&a.tree_mask[(long long)pc.b * QL + i]) & ((1ull << QL) - 1))
                                   : 0u;
                const int lim = live ? pos0 + i + 1 : 0;
                const int ta = pc.ta, tb = pc.tb;
                const bool seeded = ta == 0;
                float m = (seeded && live) ? __ldg(&a.sinks[pc.g * G + h]) * kLog2e : kNegInf;
                float d = (seeded && live) ? 1.f : 0.f;  // the sink's own e^(sink - m) = 1
                // page ids of a tile (lanes 0-7), loaded one tile ahead: a page outside the pool was
                // fetched as zeros, and its tokens count as absent
                const int kvl = pc.kv_len;
                const int* row_pt = a.page_table + (long long)pc.b * a.max_pages;
                auto page_id = [&](int t) {
                    const int pg = t * kPagesPerTile + (lane & 7);
                    return (lane < kPagesPerTile && pg < a.max_pages && pg * kPageSize < kvl) ? __ldg(&row_pt[pg]) : 0;
                };
                int pid = page_id(ta);
                for (int t = ta; t < tb; ++t, ++J) {
                    const uint32_t bad8 = __ballot_sync(0xffffffffu, pid < 0 || pid >= a.num_pages);
                    if (t + 1 < tb) pid = page_id(t + 1);
                    if (!(ok = warp_wait(&sm.s_full, J & 1))) break;
                    tc_fence_after();
                    float s[128];
#pragma unroll
                    for (int cc = 0; cc < 4; ++cc)
                        tmem_ld32(tS + cc * 32, *reinterpret_cast<uint32_t(*)[32]>(&s[cc * 32]));
                    tc_wait_ld();
                    tc_fence_before();
                    mbar_arrive(&sm.s_free);

                    const int kb = t * kBN;
                    float mul = scale_log2;
                    if (!(scale_log2 > 0.f)) {  // zero or negative scale: scale first, mask after
#pragma unroll
                        for (int cc = 0; cc < 128; ++cc) s[cc] *= scale_log2;
                        mul = 1.f;
                    }
                    const bool draft_tile = kb + kBN > pos0;
                    if (draft_tile || bad8 != 0u) {
                        // the tile holds drafted keys, the cache end or an absent page: this row's
                        // visible keys of the tile as four 32-bit words -- every key before the draft,
                        // then (tree) the drafted keys its mask names or (linear) the drafted keys up
                        // to its own, less the keys of absent pages
                        const int lo = pos0 - kb;  // keys of the tile before the draft
                        uint32_t vis[4];
#pragma unroll
                        for (int w = 0; w < 4; ++w) {
                            const int n = draft_tile ? (tree ? lo : lim - kb) - 32 * w : 32;
                            uint32_t bitsw = n <= 0 ? 0u : n >= 32 ? 0xFFFFFFFFu : ((1u << n) - 1u);
                            const int off = lo - 32 * w;
                            if (tree && off > -32 && off < 32) bitsw |= off >= 0 ? (dbits << off) : (dbits >> -off);
                            const uint32_t absent = ((bad8 >> (2 * w)) & 1u ? 0x0000FFFFu : 0u) |
                                                    ((bad8 >> (2 * w + 1)) & 1u ? 0xFFFF0000u : 0u);
                            vis[w] = bitsw & ~absent;
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
                    const bool first = t == ta;  // O starts afresh with this piece
                    float factor = 1.f;
                    bool rescale_o = false;
                    if (first || m_new > m + kRescaleThreshold) {
                        factor = (m_new == kNegInf) ? 1.f : fast_exp2(m - m_new);
                        rescale_o = !first;
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
                    if (!first) {  // P_{j-1} consumed and O_{j-1} final before P and O are touched
                        if (!(ok = warp_wait(&sm.o_done, (J - 1) & 1))) break;
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
                if (!ok) break;
                // ---- end of the piece (the PV of its last tile has finished): O / d of this row
                if (!(ok = warp_wait(&sm.o_done, (J - 1) & 1))) break;
                tc_fence_after();
                uint32_t o[64];
                tmem_ld32(tO, *reinterpret_cast<uint32_t(*)[32]>(&o[0]));
                tmem_ld32(tO + 32, *reinterpret_cast<uint32_t(*)[32]>(&o[32]));
                tc_wait_ld();
                tc_fence_before();
                const bool whole = seeded && tb == pc.tiles;
                const int seg = pc.b * Hkv + pc.g;
                if (seeded && !whole) {
                    long long c_first = 0;
                    int pieces = 0;
                    segment_pieces(pc.seg_start, pc.tiles, C, U, c_first, pieces);
                    head = make_int2(seg, pieces);
                }
                if (live) {
                    const float inv = d > 0.f ? 1.f / d : 0.f;
                    const float l2 = d > 0.f ? m + log2f(d) : kNegInf;
                    if (whole) {
                        const long long row = ((long long)pc.b * QL + i) * a.Hq + pc.g * G + h;
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
                        const long long slot = cta + seg;  // partial slot of this piece
                        float4* dst = reinterpret_cast<float4*>(a.part_o + (slot * R + r) * kHeadDim);
#pragma unroll
                        for (int e = 0; e < 16; ++e)
                            dst[e] = make_float4(__uint_as_float(o[4 * e + 0]) * inv, __uint_as_float(o[4 * e + 1]) * inv,
                                                 __uint_as_float(o[4 * e + 2]) * inv, __uint_as_float(o[4 * e + 3]) * inv);
                        a.part_lse[slot * R + r] = l2;
                    }
                }
            }
            if (!ok && lane == 0) atomicOr(a.err, kErrTimeout);
        }
        // ---- list the segment whose first piece this share holds without completing it (the
        // split merge combines its partials once every CTA has finished)
        if (tid == 128 && a.merge_list) a.merge_list[cta] = head;
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tbase, kTmemCols);
    }
}

// An empty pool: one thread per (request, drafted token, query head) row writes out = 0 and
// lse = sink (every cached token is absent); the first row of a request checks its length.
__global__ void __launch_bounds__(256) verify_empty_pool_kernel(const VerifyArgs a) {
    const long long rows = (long long)a.B * a.QL * a.Hq;
    const long long r = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    if (r >= rows) return;
    uint4* dst = reinterpret_cast<uint4*>(a.out + r * kHeadDim);
#pragma unroll
    for (int c = 0; c < kHeadDim / 8; ++c) dst[c] = make_uint4(0u, 0u, 0u, 0u);
    if (a.lse) a.lse[r] = __ldg(&a.sinks[r % a.Hq]);
    if (r % ((long long)a.QL * a.Hq) == 0) {
        const int L = __ldg(&a.kv_lens[r / ((long long)a.QL * a.Hq)]);
        if (L < 0 || L > a.max_pages * kPageSize) atomicOr(a.err, kErrBadLength);
        else if (L > 0) atomicOr(a.err, kErrBadPage);
    }
}

}  // namespace

cudaError_t verify_empty_pool_launch(const VerifyArgs& a, cudaStream_t stream) {
    const long long rows = (long long)a.B * a.QL * a.Hq;
    if (rows == 0) return cudaSuccess;
    verify_empty_pool_kernel<<<(unsigned)((rows + 255) / 256), 256, 0, stream>>>(a);
    return cudaGetLastError();
}

size_t verify_tc_smem() { return 1024 + sizeof(Smem); }

// CTAs of this kernel that fit on one SM, from its registers, its shared memory (with the per-block
// reservation) and its tensor memory (512 columns per SM, kTmemCols per CTA).  Computed here because
// the runtime's occupancy query reports one CTA per SM for this kernel whatever its size, while the
// hardware keeps two resident.
cudaError_t verify_tc_occupancy(int* per_sm) {
    static thread_local int cached[64] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 64 && cached[dev] > 0) {
        *per_sm = cached[dev];
        return cudaSuccess;
    }
    e = cudaFuncSetAttribute(verify_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)verify_tc_smem());
    if (e != cudaSuccess) return e;
    cudaFuncAttributes fa;
    if ((e = cudaFuncGetAttributes(&fa, verify_tc_kernel)) != cudaSuccess) return e;
    int smem_sm = 0, reserved = 0, regs_sm = 0;
    if ((e = cudaDeviceGetAttribute(&smem_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev)) != cudaSuccess ||
        (e = cudaDeviceGetAttribute(&reserved, cudaDevAttrReservedSharedMemoryPerBlock, dev)) != cudaSuccess ||
        (e = cudaDeviceGetAttribute(&regs_sm, cudaDevAttrMaxRegistersPerMultiprocessor, dev)) != cudaSuccess)
        return e;
    const size_t block_smem = verify_tc_smem() + fa.sharedSizeBytes + (size_t)reserved;
    const int regs_warp = ((fa.numRegs * 32 + 255) / 256) * 256;  // allocated per warp in units of 256
    int n = 512 / (int)kTmemCols;
    n = n < (int)(smem_sm / block_smem) ? n : (int)(smem_sm / block_smem);
    n = n < regs_sm / (regs_warp * (kThreads / 32)) ? n : regs_sm / (regs_warp * (kThreads / 32));
    if (n < 1) return cudaErrorInvalidConfiguration;
    if (dev < 64) cached[dev] = n;
    *per_sm = n;
    return cudaSuccess;
}

cudaError_t verify_plan(int B, int QL, int Hq, int Hkv, int num_workers, VerifyPlan* plan) {
    const int G = Hq / Hkv, R = QL * G;
    // one share of the (request, KV head, 128-key tile) units per resident slot (num_workers > 0:
    // that many shares)
    int per_sm = 0, sms = 0, dev = 0;
    cudaError_t e;
    if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
    if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
    if ((e = verify_tc_occupancy(&per_sm)) != cudaSuccess) return e;
    const long long segs = (long long)B * Hkv;
    plan->tc_grid = num_workers > 0 ? num_workers : (long long)sms * (per_sm > 0 ? per_sm : 1);
    plan->slots = (size_t)plan->tc_grid + (size_t)segs;  // partial slot = share + segment
    size_t bytes = plan->slots * R * kHeadDim * 4;       // partial o
    bytes += plan->slots * R * 4;                        // partial lse (base 2)
    plan->merge_list_offset = (bytes + 255) & ~size_t(255);
    plan->ws_bytes = plan->merge_list_offset + (size_t)plan->tc_grid * sizeof(int2);
    return cudaSuccess;
}

cudaError_t verify_tc_launch(const VerifyArgs& args, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                             bool may_split, cudaStream_t stream) {
    if (args.B == 0) return cudaSuccess;
    if (args.tc_grid > 0x7fffffffll || args.tc_grid < 1) return cudaErrorInvalidConfiguration;
    int per_sm = 0;  // also sets the kernel's shared-memory limit
    cudaError_t e = verify_tc_occupancy(&per_sm);
    if (e != cudaSuccess) return e;
    VerifyArgs a = args;
    if (!may_split) a.merge_list = nullptr;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)a.tc_grid);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = verify_tc_smem();
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, verify_tc_kernel, tq, tk, tv, a);
    if (e != cudaSuccess || !may_split) return e;
    SplitMergeArgs m;
    m.part_o = a.part_o;
    m.part_lse = a.part_lse;
    m.list = a.merge_list;
    m.out = a.out;
    m.lse = a.lse;
    m.listed = (int)a.tc_grid;
    m.R = a.R;
    m.G = a.G;
    m.QL = a.QL;
    m.Hq = a.Hq;
    m.Hkv = a.Hkv;
    return split_merge_launch(m, stream);
}

}  // namespace sinkattn
