// decode.cu -- paged split-KV decode with a per-head learned sink.
//
// Source of the method: "GPT-OSS on day 0" (Perplexity), section "Kernels for
// GPT-OSS / Sink Attention": attention is parallelised over independent heads
// and along the KV length; the softmax runs online with a running max m and
// scale d, and seeding m from the head's sink makes the sink count in the
// normaliser -- in the first block along the sequence only.  Pages come from a
// per-request page table ("Accelerating Sonar through speculation", section
// "Inference with speculative decoding": KV pages allocated per request, page
// metadata copied to the GPU).
//
// GB300 design (not the pages' FlashInfer template):
//  * Work = the flattened list of (request b, KV head g, page) units; a
//    (b, g) pair is a "segment".  Every CTA recomputes the per-request page
//    prefix sum from kv_lens in shared memory, so the split needs no host-side
//    knowledge of the lengths (no host sync; graph-capturable).  CTA c takes
//    the contiguous share [c*U/C, (c+1)*U/C) of the U units: balanced to one
//    page.  The share is cut at segment ends into "pieces".
//  * The warps of a CTA deal the pages of their share round robin, one page
//    each in turn, and the turn carries on across piece boundaries, so every
//    warp streams the same number of pages (+-1) however the share is cut.  A
//    piece shorter than the warp count goes whole to the warp whose turn it is.
//  * Piece ends need no CTA barrier: each warp drops its online-softmax state
//    for the piece into one of two shared-memory slots and counts itself in;
//    the last warp to arrive combines the states and writes the result while
//    the others carry on streaming.
//  * A piece that is a whole segment writes the final output.  Any other piece
//    writes an fp32 partial (o_c, lse_c) into its slot of the workspace; the
//    CTA holding a split segment's page 0 lists the segment, and a small merge
//    kernel, launched as a programmatic dependent of this one (its launch
//    overlaps this kernel; it waits for this grid to finish), combines the
//    partials by log-sum-exp.  No CTA ever waits for another, and nothing in
//    the workspace carries over between calls.  Only the piece holding page 0
//    is seeded with the sink, so the sink is counted exactly once.
//  * Each warp streams its pages through a private ring of kStages shared-
//    memory stages.  One stage = the K and V slices of one (page, KV head):
//    2 x 2 KiB, loaded by two TMA tensor copies with 128-byte swizzle (so the
//    ldmatrix reads below are bank-conflict free) and tracked by one mbarrier.
//  * All G <= 8 query heads of the group share one pass over K/V.  Scores are
//    computed transposed, S^T[16 tokens x 8 heads] = K * Q^T, with
//    mma.m16n8k16 (no padding: M = a page, N = the group); the row max per
//    head is a 3-step shuffle; P^T is re-laid out for the next MMA with
//    movmatrix; O^T[64 x 8] += V^T * P^T.  Everything stays in registers.
#include "args_decode.h"
#include "args_merge.h"
#include "ptx.cuh"
#include "split_kv.cuh"

#ifndef SINKATTN_DECODE_STAGES
#define SINKATTN_DECODE_STAGES 2
#endif
#ifndef SINKATTN_DECODE_MIN_PAGES
#define SINKATTN_DECODE_MIN_PAGES 32
#endif
#ifndef SINKATTN_DECODE_MIN_BLOCKS
#define SINKATTN_DECODE_MIN_BLOCKS 4
#endif
#ifndef SINKATTN_DECODE_WARPS
#define SINKATTN_DECODE_WARPS 4
#endif

namespace sinkattn {
namespace {

constexpr int kWarps = SINKATTN_DECODE_WARPS;    // warps per CTA
constexpr int kStages = SINKATTN_DECODE_STAGES;  // ring depth per warp
constexpr int kSliceBytes = kPageSize * kHeadDim * 2;  // 2048: one (page, KV head) of K or V
constexpr int kStageBytes = 2 * kSliceBytes;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kNegInf = -__builtin_huge_valf();

// Shared memory: ring | mbarriers | bad-page flags | combine slots | slot words | scan | prefix[B+1].
template <int NT>
struct SmemLayout {
    static constexpr int kHeads = 8 * NT;
    static constexpr size_t ring = size_t(kWarps) * kStages * kStageBytes;
    static constexpr size_t bars = ring;
    static constexpr size_t bad = bars + size_t(kWarps) * kStages * 8;
    static constexpr size_t cmb_o = bad + size_t(kWarps) * kStages * 4;                   // [2][warps][heads][64] f32
    static constexpr size_t cmb_md = cmb_o + 2 * size_t(kWarps) * kHeads * kHeadDim * 4;  // [2][warps][heads] m, d
    static constexpr size_t slot = cmb_md + 2 * size_t(kWarps) * kHeads * 8;  // [2] arrivals, [2] generation
    static constexpr size_t scan = slot + 4 * 4;                             // [kWarps] scan scratch
    static constexpr size_t prefix = scan + kWarps * 4;
    static constexpr size_t fixed = prefix + 1024 /* alignment slack */;
};

__device__ __forceinline__ uint32_t ld_u32(const __nv_bfloat16* p) {
    return __ldg(reinterpret_cast<const unsigned int*>(p));
}

__device__ __forceinline__ void allow_dependent_launch() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void wait_for_prerequisite_grids() {
    asm volatile("griddepcontrol.wait;" ::: "memory");
}

// A piece as the decode processes it.  `rot` is the warp whose turn it is at the piece's first
// page (the deal carries on from the previous piece of the share).  A piece of >= kWarps pages
// is dealt page by page from warp rot on; a shorter one goes whole to warp rot.
struct Piece : SegPiece {
    int rot;
    __device__ bool split() const { return len() >= kWarps; }
    __device__ int offset(int w) const { return (w - rot + kWarps) % kWarps; }
    // Units of this piece that warp w processes, and the page of its t-th one.
    __device__ int count(int w) const {
        if (split()) {
            const int o = offset(w);
            return len() > o ? (len() - o + kWarps - 1) / kWarps : 0;
        }
        return rot == w ? len() : 0;
    }
    __device__ int page(int w, int t) const { return page0() + (split() ? offset(w) + t * kWarps : t); }
    __device__ void first(const int* prefix, int B, int Hkv, long long x0, long long x1) {
        piece_first(*this, prefix, B, Hkv, x0, x1);
        rot = 0;
    }
    __device__ void next(const int* prefix, int B, int Hkv, long long x1) {
        rot = (rot + len()) % kWarps;
        piece_next(*this, prefix, B, Hkv, x1);
    }
};

// Bounded spin until a shared-memory word reaches `want`; false on give-up.
__device__ __forceinline__ bool wait_word(const int* w, int want) {
    for (uint32_t i = 0; i < kMaxPolls; ++i)
        if (*reinterpret_cast<const volatile int*>(w) == want) return true;
    return false;
}

template <int NT>  // NT = ceil(G / 8) groups of 8 query heads
__global__ void __launch_bounds__(kWarps * 32, SINKATTN_DECODE_MIN_BLOCKS)
    decode_split_kernel(const __grid_constant__ CUtensorMap tmap_k, const __grid_constant__ CUtensorMap tmap_v,
                        const DecodeArgs a) {
    using L = SmemLayout<NT>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t* bars = reinterpret_cast<uint64_t*>(sm + L::bars);
    int* bad = reinterpret_cast<int*>(sm + L::bad);
    float* cmb_o = reinterpret_cast<float*>(sm + L::cmb_o);
    float* cmb_md = reinterpret_cast<float*>(sm + L::cmb_md);
    int* slot_arr = reinterpret_cast<int*>(sm + L::slot);  // [2] warps counted in for the slot's piece
    int* slot_gen = slot_arr + 2;                          // [2] pieces the slot has combined
    int* scan = reinterpret_cast<int*>(sm + L::scan);
    int* prefix = reinterpret_cast<int*>(sm + L::prefix);  // [B + 1] exclusive prefix of pages per request

    // Launched as a programmatic dependent of whatever precedes it on the stream: the launch
    // overlaps that kernel's tail, and nothing is read before it has completed.  The merge kernel
    // may be scheduled as soon as every CTA of this grid is running.
    wait_for_prerequisite_grids();
    allow_dependent_launch();

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int B = a.B, Hkv = a.Hkv, G = a.G, cap = a.max_pages * kPageSize;
    const long long cta = blockIdx.x;

    // ---- 1. pages per request -> exclusive prefix sum (every CTA, in shared memory)
    int running = 0;
    for (int base = 0; base < B; base += kWarps * 32) {
        int b = base + tid, n = 0;
        if (b < B) {
            int Lb = a.kv_lens[b];
            if ((Lb < 0 || Lb > cap) && blockIdx.x == 0) atomicOr(a.err, kErrBadLength);
            n = (clamp_len(Lb, cap) + kPageSize - 1) / kPageSize;
        }
        int incl = n;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            int y = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += y;
        }
        if (lane == 31) scan[warp] = incl;
        __syncthreads();
        int woff = 0, tot = 0;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) {
            int v = scan[w];
            woff += (w < warp) ? v : 0;
            tot += v;
        }
        if (b < B) prefix[b] = running + woff + incl - n;
        running += tot;
        __syncthreads();
    }
    if (tid == 0) {
        prefix[B] = running;
        slot_arr[0] = slot_arr[1] = 0;
        slot_gen[0] = slot_gen[1] = 0;
    }
    __syncthreads();

    // ---- 2. requests with no cached token: all mass on the sink (out = 0, lse = sink)
    {
        const long long rows = (long long)B * a.Hq;
        for (long long r = (long long)blockIdx.x * blockDim.x + tid; r < rows; r += (long long)gridDim.x * blockDim.x) {
            const int b = (int)(r / a.Hq);
            if (prefix[b + 1] != prefix[b]) continue;
            uint4* dst = reinterpret_cast<uint4*>(a.out + r * kHeadDim);
#pragma unroll
            for (int c = 0; c < 8; ++c) dst[c] = make_uint4(0, 0, 0, 0);
            if (a.lse) a.lse[r] = __ldg(&a.sinks[r - (long long)b * a.Hq]);
        }
    }

    const long long U = (long long)running * Hkv;
    const long long C = U > 0 ? effective_shares(a.workers, a.fixed_workers, a.min_pages_per_worker, U) : 0;
    if (cta >= C) {
        if (tid == 0 && a.merge_list) a.merge_list[cta] = make_int2(-1, 0);
        return;
    }
    const long long x0 = cta * U / C, x1 = (cta + 1) * U / C;

    uint8_t* my_ring = sm + warp * kStages * kStageBytes;
    uint64_t* my_bars = bars + warp * kStages;
    int* my_bad = bad + warp * kStages;
    if (lane == 0) {
        for (int s = 0; s < kStages; ++s) mbar_init(&my_bars[s], 1);
        fence_mbar_init();
        fence_proxy_async_smem();
        tma_prefetch_desc(&tmap_k);
        tma_prefetch_desc(&tmap_v);
    }
    __syncwarp();

    // ---- 3. producer: walks this warp's units piece by piece; lanes resolve 32 page ids at a time
    Piece pp;
    pp.first(prefix, B, Hkv, x0, x1);
    int pt = 0, pcnt = pp.count(warp), win_base = -64, win_row = -1, issued = 0;
    auto issue = [&]() -> bool {  // warp-uniform
        while (pt >= pcnt) {
            pp.next(prefix, B, Hkv, x1);
            if (pp.ps >= x1) return false;
            pt = 0;
            pcnt = pp.count(warp);
            win_base = -64;
        }
        if (pt - win_base >= 32) {
            win_base = pt;
            int row = -1;
            if (pt + lane < pcnt) {
                const int pid = __ldg(&a.page_table[(long long)pp.b * a.max_pages + pp.page(warp, pt + lane)]);
                if (pid >= 0 && pid < a.num_pages) row = (pid * Hkv + pp.g) * kPageSize;
            }
            win_row = row;
        }
        const int row = __shfl_sync(0xffffffffu, win_row, pt - win_base);
        if (lane == 0) {
            const int s = issued % kStages;
            uint8_t* dst = my_ring + s * kStageBytes;
            if (row >= 0) {
                my_bad[s] = 0;
                mbar_arrive_expect_tx(&my_bars[s], kStageBytes);
                tma_load_2d(dst, &tmap_k, 0, row, &my_bars[s]);
                tma_load_2d(dst + kSliceBytes, &tmap_v, 0, row, &my_bars[s]);
            } else {
                my_bad[s] = 1;
                atomicOr(a.err, kErrBadPage);
                mbar_arrive(&my_bars[s]);
            }
        }
        ++pt;
        ++issued;
        return true;
    };
    bool more = true;
    for (int j = 0; j < kStages && more; ++j) more = issue();

    // ---- 4. consumer: piece by piece
    const int gq = lane >> 2, tq = lane & 3;  // mma fragment coordinates
    float O[4][NT][4];
    float m[NT][2], d[NT][2];
    int consumed = 0;
    bool failed = false;  // a wait gave up: skip all further work, keep the barriers
    int nsplit = 0;       // dealt pieces met so far (they take the combine slots in turn)
    int head_seg = -1;    // segment whose page 0 this share holds without completing it

    // Per-piece inputs (query fragments, sink logits, cache length), fetched one piece ahead.
    struct PieceIn {
        uint32_t qf[NT][4][2];
        float sink2[NT][2];
        int kv_len;
    };
    auto fetch = [&](const Piece& p, PieceIn& in) {
        in.kv_len = clamp_len(__ldg(&a.kv_lens[p.b]), cap);
        const __nv_bfloat16* qb = a.q + ((long long)p.b * a.Hq + (long long)p.g * G) * kHeadDim;
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
            const int hl = nt * 8 + gq;
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
                in.qf[nt][kk][0] = hl < G ? ld_u32(qb + hl * kHeadDim + kk * 16 + 2 * tq) : 0u;
                in.qf[nt][kk][1] = hl < G ? ld_u32(qb + hl * kHeadDim + kk * 16 + 8 + 2 * tq) : 0u;
            }
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                const int h = nt * 8 + 2 * tq + e;
                in.sink2[nt][e] = h < G ? __ldg(&a.sinks[p.g * G + h]) * kLog2e : kNegInf;
            }
        }
    };
    PieceIn cur, nxt;
    Piece cp;
    cp.first(prefix, B, Hkv, x0, x1);
    fetch(cp, cur);

    while (cp.ps < x1) {
        Piece np = cp;
        np.next(prefix, B, Hkv, x1);
        if (np.ps < x1) fetch(np, nxt);  // in flight while this piece is processed

        const int cnt = cp.count(warp);
        const bool first = cp.page0() == 0;  // this piece holds the segment's page 0
        // ... and this warp carries the sink (for a dealt piece, warp 0: it always has a page)
        const bool seeded = first && (cp.split() ? warp == 0 : cnt > 0);
        const int seg = cp.b * Hkv + cp.g;
        const bool whole = first && (cp.pe == cp.seg_start + cp.n);
        if (first && !whole) head_seg = seg;
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                m[nt][e] = seeded ? cur.sink2[nt][e] : kNegInf;
                d[nt][e] = (seeded && lane < 4) ? 1.f : 0.f;  // the sink's own e^(sink-m)=1, once per head
            }
#pragma unroll
            for (int mt = 0; mt < 4; ++mt)
#pragma unroll
                for (int e = 0; e < 4; ++e) O[mt][nt][e] = 0.f;
        }

        for (int t = 0; t < cnt && !failed; ++t) {
            const int s = consumed % kStages;
            if (!__all_sync(0xffffffffu, mbar_wait(&my_bars[s], (consumed / kStages) & 1))) {
                failed = true;
                if (lane == 0) atomicOr(a.err, kErrTimeout);
                break;
            }
            const int page = cp.page(warp, t);
            const int valid = my_bad[s] ? 0 : min(kPageSize, cur.kv_len - page * kPageSize);
            uint8_t* st = my_ring + s * kStageBytes;
            if (valid < kPageSize) {
                // Rows past the cache end (or a skipped page) may hold anything; zero the
                // value rows so that 0-weight * garbage cannot produce NaN.
                uint4* vz = reinterpret_cast<uint4*>(st + kSliceBytes);
                for (int c = valid * 8 + lane; c < kPageSize * 8; c += 32) vz[c] = make_uint4(0, 0, 0, 0);
                __syncwarp();
            }
            const uint32_t kb = smem_u32(st), vb = kb + kSliceBytes;

            // S^T = K Q^T : 16 tokens x 8 heads per n-tile
            float acc[NT][4];
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                for (int e = 0; e < 4; ++e) acc[nt][e] = 0.f;
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
                const int row = ((lane >> 3) & 1) * 8 + (lane & 7);
                const int chunk = 2 * kk + (lane >> 4);
                uint32_t af[4];
                ldmatrix_x4(af, kb + row * 128 + ((chunk ^ (row & 7)) << 4));
#pragma unroll
                for (int nt = 0; nt < NT; ++nt) mma_bf16_16816(acc[nt], af, cur.qf[nt][kk][0], cur.qf[nt][kk][1]);
            }

            // online softmax (base 2); this thread holds tokens gq, gq+8 and heads 2tq, 2tq+1
            uint32_t pb[NT][2];
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
                float sc[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int tok = gq + (e >= 2 ? 8 : 0);
                    sc[e] = tok < valid ? acc[nt][e] * a.scale_log2 : kNegInf;
                }
                float mx0 = fmaxf(sc[0], sc[2]), mx1 = fmaxf(sc[1], sc[3]);
#pragma unroll
                for (int o = 4; o < 32; o <<= 1) {
                    mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, o));
                    mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, o));
                }
                const float mn0 = fmaxf(m[nt][0], mx0), mn1 = fmaxf(m[nt][1], mx1);
                const bool dead0 = (mn0 == kNegInf), dead1 = (mn1 == kNegInf);
                const float al0 = dead0 ? 1.f : fast_exp2(m[nt][0] - mn0);
                const float al1 = dead1 ? 1.f : fast_exp2(m[nt][1] - mn1);
                const float p0 = dead0 ? 0.f : fast_exp2(sc[0] - mn0);
                const float p2 = dead0 ? 0.f : fast_exp2(sc[2] - mn0);
                const float p1 = dead1 ? 0.f : fast_exp2(sc[1] - mn1);
                const float p3 = dead1 ? 0.f : fast_exp2(sc[3] - mn1);
                d[nt][0] = d[nt][0] * al0 + (p0 + p2);
                d[nt][1] = d[nt][1] * al1 + (p1 + p3);
                m[nt][0] = mn0;
                m[nt][1] = mn1;
#pragma unroll
                for (int mt = 0; mt < 4; ++mt) {
                    O[mt][nt][0] *= al0;
                    O[mt][nt][1] *= al1;
                    O[mt][nt][2] *= al0;
                    O[mt][nt][3] *= al1;
                }
                pb[nt][0] = movmatrix_trans(pack_bf16(p0, p1));  // tokens 0..7  -> B rows k = 2tq, 2tq+1
                pb[nt][1] = movmatrix_trans(pack_bf16(p2, p3));  // tokens 8..15
            }

            // O^T += V^T P^T : 4 tiles of 16 head-dims
#pragma unroll
            for (int mt = 0; mt < 4; ++mt) {
                const int j = lane >> 3;
                const int row = (j >> 1) * 8 + (lane & 7);
                const int chunk = 2 * mt + (j & 1);
                uint32_t af[4];
                ldmatrix_x4_trans(af, vb + row * 128 + ((chunk ^ (row & 7)) << 4));
#pragma unroll
                for (int nt = 0; nt < NT; ++nt) mma_bf16_16816(O[mt][nt], af, pb[nt][0], pb[nt][1]);
            }

            // release the stage and refill it
            fence_proxy_async_smem();
            __syncwarp();
            ++consumed;
            if (more) more = issue();
        }

        // ---- end of the piece: this warp's normaliser over its lanes
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int e = 0; e < 2; ++e)
#pragma unroll
                for (int o = 4; o < 32; o <<= 1) d[nt][e] += __shfl_xor_sync(0xffffffffu, d[nt][e], o);

        const long long slot = cta + seg;  // partial slot of this piece
        if (!cp.split()) {
            if (cnt > 0) {
                // one warp holds the whole piece: normalise and write
#pragma unroll
                for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
                    for (int mt = 0; mt < 4; ++mt)
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const int h = nt * 8 + 2 * tq + (e & 1);
                            const int dim = mt * 16 + gq + (e >= 2 ? 8 : 0);
                            if (h >= G) continue;
                            const float dt = d[nt][e & 1];
                            const float v = dt > 0.f ? O[mt][nt][e] / dt : 0.f;
                            if (whole)
                                a.out[((long long)cp.b * a.Hq + cp.g * G + h) * kHeadDim + dim] =
                                    __float2bfloat16_rn(v);
                            else
                                a.part_o[(slot * G + h) * kHeadDim + dim] = v;
                        }
                    if (lane < 4) {
#pragma unroll
                        for (int e = 0; e < 2; ++e) {
                            const int h = nt * 8 + 2 * tq + e;
                            if (h >= G) continue;
                            const float l2 = d[nt][e] > 0.f ? m[nt][e] + log2f(d[nt][e]) : kNegInf;
                            if (whole) {
                                if (a.lse) a.lse[(long long)cp.b * a.Hq + cp.g * G + h] = l2 * kLn2;
                            } else {
                                a.part_lse[slot * G + h] = l2;
                            }
                        }
                    }
                }
            }
        } else {
            // ---- a dealt piece: drop this warp's state into the piece's combine slot; the last
            // warp to count itself in combines the states and writes the result
            const int sl = nsplit & 1, gen = nsplit >> 1;
            ++nsplit;
            if (!wait_word(&slot_gen[sl], gen)) {  // the slot's previous piece is combined
                failed = true;
                if (lane == 0) atomicOr(a.err, kErrTimeout);
            }
            __threadfence_block();
            float* co = cmb_o + sl * (kWarps * L::kHeads * kHeadDim);
            float* cmd = cmb_md + sl * (kWarps * L::kHeads * 2);
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
                for (int mt = 0; mt < 4; ++mt)
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const int h = nt * 8 + 2 * tq + (e & 1);
                        const int dim = mt * 16 + gq + (e >= 2 ? 8 : 0);
                        co[(warp * L::kHeads + h) * kHeadDim + dim] = O[mt][nt][e];
                    }
                if (lane < 4) {
#pragma unroll
                    for (int e = 0; e < 2; ++e) {
                        const int h = nt * 8 + 2 * tq + e;
                        cmd[(warp * L::kHeads + h) * 2 + 0] = m[nt][e];
                        cmd[(warp * L::kHeads + h) * 2 + 1] = d[nt][e];
                    }
                }
            }
            __syncwarp();
            int before = 0;
            if (lane == 0) {
                __threadfence_block();  // this warp's state is written before it counts itself in
                before = atomicAdd(&slot_arr[sl], 1);
                __threadfence_block();  // ... and the other warps' states are read after
            }
            before = __shfl_sync(0xffffffffu, before, 0);
            __syncwarp();
            if (before == kWarps - 1) {
                // the lanes split the G x 64 outputs: kLanesPerHead lanes per head, each with a run
                // of kDims consecutive head-dims, all loads of a run issued together
                constexpr int kLanesPerHead = 32 / L::kHeads;       // 4 (NT = 1) or 2 (NT = 2)
                constexpr int kDims = kHeadDim / kLanesPerHead;     // 16 or 32
                const int h = lane / kLanesPerHead, d0 = (lane % kLanesPerHead) * kDims;
                if (h < G) {
                    float sw[kWarps], M = kNegInf;
#pragma unroll
                    for (int w = 0; w < kWarps; ++w) {
                        sw[w] = cmd[(w * L::kHeads + h) * 2];
                        M = fmaxf(M, sw[w]);
                    }
                    float dt = 0.f;
#pragma unroll
                    for (int w = 0; w < kWarps; ++w) {
                        sw[w] = (M == kNegInf || sw[w] == kNegInf) ? 0.f : fast_exp2(sw[w] - M);
                        dt += sw[w] * cmd[(w * L::kHeads + h) * 2 + 1];
                    }
                    const float inv = dt > 0.f ? 1.f / dt : 0.f;
                    const float l2 = dt > 0.f ? M + log2f(dt) : kNegInf;
                    const long long row = (long long)cp.b * a.Hq + cp.g * G + h;
#pragma unroll
                    for (int part = 0; part < kDims / 8; ++part) {  // 8 head-dims at a time
                        float acc[8];
#pragma unroll
                        for (int i = 0; i < 8; ++i) acc[i] = 0.f;
#pragma unroll
                        for (int w = 0; w < kWarps; ++w) {
                            const float4* src =
                                reinterpret_cast<const float4*>(co + (w * L::kHeads + h) * kHeadDim + d0 + 8 * part);
                            const float4 v0 = src[0], v1 = src[1];
                            acc[0] += sw[w] * v0.x;
                            acc[1] += sw[w] * v0.y;
                            acc[2] += sw[w] * v0.z;
                            acc[3] += sw[w] * v0.w;
                            acc[4] += sw[w] * v1.x;
                            acc[5] += sw[w] * v1.y;
                            acc[6] += sw[w] * v1.z;
                            acc[7] += sw[w] * v1.w;
                        }
                        if (whole) {
                            reinterpret_cast<uint4*>(a.out + row * kHeadDim + d0)[part] =
                                make_uint4(pack_bf16(acc[0] * inv, acc[1] * inv), pack_bf16(acc[2] * inv, acc[3] * inv),
                                           pack_bf16(acc[4] * inv, acc[5] * inv), pack_bf16(acc[6] * inv, acc[7] * inv));
                        } else {
                            float4* dst = reinterpret_cast<float4*>(a.part_o + (slot * G + h) * kHeadDim + d0 + 8 * part);
                            dst[0] = make_float4(acc[0] * inv, acc[1] * inv, acc[2] * inv, acc[3] * inv);
                            dst[1] = make_float4(acc[4] * inv, acc[5] * inv, acc[6] * inv, acc[7] * inv);
                        }
                    }
                    if (d0 == 0) {
                        if (whole) {
                            if (a.lse) a.lse[row] = l2 * kLn2;
                        } else {
                            a.part_lse[slot * G + h] = l2;
                        }
                    }
                }
                __syncwarp();
                if (lane == 0) {  // free the slot for the piece after next
                    slot_arr[sl] = 0;
                    __threadfence_block();
                    *reinterpret_cast<volatile int*>(&slot_gen[sl]) = gen + 1;
                }
            }
        }
        cp = np;
        if (cp.ps < x1) cur = nxt;
    }

    if (failed) {
        // let copies already in flight land (bounded) before the CTA's shared memory is released
        for (int j = consumed; j < issued; ++j) (void)mbar_wait(&my_bars[j % kStages], (j / kStages) & 1);
    }

    // ---- 5. list the segment whose page 0 this share holds but does not complete: the merge
    // kernel combines its pieces (slots cta + seg .. cta + pieces - 1 + seg)
    if (tid == 0 && a.merge_list) {
        int2 e = make_int2(-1, 0);
        if (head_seg >= 0) {
            const int b = head_seg / Hkv, g = head_seg - b * Hkv;
            const int n = prefix[b + 1] - prefix[b];
            long long c_first;
            int pieces;
            segment_pieces((long long)prefix[b] * Hkv + (long long)g * n, n, C, U, c_first, pieces);
            e = make_int2(head_seg, pieces);
        }
        a.merge_list[cta] = e;
    }
}

template <int NT>
cudaError_t ensure_smem_attr(size_t smem) {
    static thread_local size_t set_to[64] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 64 && set_to[dev] >= smem) return cudaSuccess;
    e = cudaFuncSetAttribute(decode_split_kernel<NT>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e == cudaSuccess && dev < 64) set_to[dev] = smem;
    return e;
}

}  // namespace

// Resident CTAs per SM x SM count for one (device, group width, shared memory) triple,
// remembered so that repeated calls skip the occupancy query.
cudaError_t resident_ctas(int NT, size_t smem, long long* ctas) {
    struct Entry {
        int dev, NT;
        size_t smem;
        long long ctas;
    };
    static thread_local Entry cache[8] = {};
    static thread_local int next = 0;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    for (const Entry& c : cache)
        if (c.ctas > 0 && c.dev == dev && c.NT == NT && c.smem == smem) {
            *ctas = c.ctas;
            return cudaSuccess;
        }
    e = NT == 1 ? ensure_smem_attr<1>(smem) : ensure_smem_attr<2>(smem);
    if (e != cudaSuccess) return e;
    int sms = 0, per_sm = 0;
    if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
    e = NT == 1 ? cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, decode_split_kernel<1>, kWarps * 32, smem)
                : cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, decode_split_kernel<2>, kWarps * 32, smem);
    if (e != cudaSuccess) return e;
    if (per_sm < 1) return cudaErrorInvalidConfiguration;
    cache[next] = Entry{dev, NT, smem, (long long)sms * per_sm};
    next = (next + 1) % 8;
    *ctas = (long long)sms * per_sm;
    return cudaSuccess;
}

cudaError_t decode_plan(int B, int Hq, int Hkv, int num_workers, DecodePlan* plan) {
    const int G = Hq / Hkv;
    const int NT = G <= 8 ? 1 : 2;
    const size_t smem = (NT == 1 ? SmemLayout<1>::fixed : SmemLayout<2>::fixed) + size_t(B + 1) * 4;
    long long resident = 0;
    cudaError_t e = resident_ctas(NT, smem, &resident);
    if (e != cudaSuccess) return e;
    const long long shares = num_workers > 0 ? num_workers : resident;
    plan->workers = (int)shares;
    plan->min_pages = SINKATTN_DECODE_MIN_PAGES;
    plan->grid = (int)shares;
    plan->smem = smem;
    plan->slots = (size_t)shares + (size_t)B * Hkv;
    size_t bytes = plan->slots * G * kHeadDim * 4;   // partial o
    bytes += plan->slots * G * 4;                    // partial lse (base 2)
    plan->merge_list_offset = (bytes + 255) & ~size_t(255);
    plan->ws_bytes = plan->merge_list_offset + (size_t)shares * sizeof(int2);
    return cudaSuccess;
}

cudaError_t decode_launch(const DecodeArgs& args, const DecodePlan& plan, const CUtensorMap& tk,
                          const CUtensorMap& tv, bool may_split, cudaStream_t stream) {
    if (args.B == 0) return cudaSuccess;
    DecodeArgs a = args;
    if (!may_split) a.merge_list = nullptr;
    // Both kernels are programmatic dependents of what precedes them on the stream (each waits,
    // griddepcontrol.wait, for its predecessor to complete before reading anything), so a launch
    // overlaps the tail of the kernel before it instead of starting after it.
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)plan.grid);
    cfg.blockDim = dim3(kWarps * 32);
    cfg.dynamicSmemBytes = plan.smem;
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaError_t e = a.G <= 8 ? cudaLaunchKernelEx(&cfg, decode_split_kernel<1>, tk, tv, a)
                             : cudaLaunchKernelEx(&cfg, decode_split_kernel<2>, tk, tv, a);
    if (e != cudaSuccess || !may_split) return e;
    // the merge: its CTAs are scheduled while the decode runs and wait for the decode grid to
    // complete before they read its partials
    SplitMergeArgs m;
    m.part_o = a.part_o;
    m.part_lse = a.part_lse;
    m.list = a.merge_list;
    m.out = a.out;
    m.lse = a.lse;
    m.listed = plan.grid;
    m.R = a.G;
    m.G = a.G;
    m.QL = 1;
    m.Hq = a.Hq;
    m.Hkv = a.Hkv;
    return split_merge_launch(m, stream);
}

}  // namespace sinkattn
